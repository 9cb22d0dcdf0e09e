"""Multi-GPU use of the step is replicas only: each rank verifies its own
sequences and nothing crosses ranks but the timing.  These world-size-2 tests
run the bench's host logic over the gloo backend on CPU: disjoint sequence
shards, the max-over-ranks step time, the whole-job rate, and that different
ranks really get different synthetic inputs."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from speculative_decoding_eagle_gb300 import workloads as W

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        sets, batch = 3, 4
        offs = bench.shard_offsets(rank, sets, batch)
        gathered = [None] * WORLD
        dist.all_gather_object(gathered, offs)
        local_ms = 1.5 * (rank + 1)           # rank 1 is the slower one
        step_ms = bench.reduce_step_ms(local_ms, WORLD)
        wl = W.WORKLOADS["tiny"]
        roots = W.root_tokens(wl, (rank + 1) * 64)[rank * 64:(rank + 1) * 64]
        roots_all = [None] * WORLD
        dist.all_gather_object(roots_all, roots.tolist())
        out[rank] = dict(offs=gathered, step_ms=step_ms, rate=bench.whole_job_rate(step_ms, WORLD),
                         roots=roots_all)
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def results():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(WORLD)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0, p.exitcode
        return dict(out)


def test_shards_are_disjoint_and_cover_a_contiguous_range(results):
    offs = results[0]["offs"]
    assert offs == results[1]["offs"]
    flat = sorted(o + i for shard in offs for o in shard for i in range(4))
    assert flat == list(range(WORLD * 3 * 4))


def test_step_time_is_the_slowest_rank_and_rate_counts_every_rank(results):
    for r in range(WORLD):
        assert results[r]["step_ms"] == pytest.approx(3.0)
        assert results[r]["rate"] == pytest.approx(WORLD * 1000.0 / 3.0)


def test_ranks_draw_different_sequences(results):
    a, b = results[0]["roots"]
    assert len(a) == len(b) == 64
    assert not np.array_equal(np.asarray(a), np.asarray(b))


def test_single_rank_needs_no_collective():
    assert bench.reduce_step_ms(2.5, 1) == 2.5
    assert bench.whole_job_rate(2.0, 1) == pytest.approx(500.0)
    assert bench.shard_offsets(0, 2, 8) == [0, 8]
