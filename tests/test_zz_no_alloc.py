"""The allocation-free expansion entry point against the ordinary one.

et_tree_expand_noalloc exists for callers that cannot give the library device
scratch memory (their framework forbids allocation while it executes them,
all device memory is reserved up front, or a stream is being captured).  It
takes its scratch from an array the library keeps on the device, so its
results must equal et_tree_expand's, call after call, even though every call
reuses (and leaves behind) the same scratch.  This file is collected last so
that a failure here never hides the other tests.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_eagle_gb300 import binding as E

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_eagle_gb300 import build_lib
    build_lib.build()
    E.load()


def _state(tb):
    torch.cuda.synchronize()
    return [t.cpu().numpy().copy() for t in (tb.cand_tok, tb.cand_parent, tb.cand_lp, tb.cand_key, tb.frontier)]


def test_noalloc_expand_matches_workspace_expand_two_calls_in_a_row():
    cfg = E.TreeCfg(B=3, V=32000, depth=3, topk=10, m=10, n=60)
    C = E.et_num_candidates(cfg)
    rng = np.random.default_rng(2024)
    table = torch.from_numpy((rng.standard_normal((cfg.B * (C + 1), cfg.V)) * 2).astype(np.float32)).cuda()
    rmap = torch.from_numpy((np.arange(cfg.B)[:, None] * (C + 1) + np.arange(C + 1)[None, :]).astype(np.int32)).cuda()
    ref = E.TreeBuffers.allocate(cfg)
    got = E.TreeBuffers.allocate(cfg)
    ws = E.new_workspace(E.et_tree_workspace_size(cfg))
    # two calls in a row (layers 0 and 1), each compared with the workspace path
    for layer in range(2):
        E.et_tree_expand(cfg, layer, table, ref, ws, row_of_node=rmap)
        E.et_tree_expand_noalloc(cfg, layer, table, got, row_of_node=rmap)
        for a, b in zip(_state(ref), _state(got)):
            np.testing.assert_array_equal(a, b)
    # and the same layer again on fresh buffers: leftovers of the previous
    # calls in the shared scratch must not leak into the result
    again = E.TreeBuffers.allocate(cfg)
    for layer in range(2):
        E.et_tree_expand_noalloc(cfg, layer, table, again, row_of_node=rmap)
    for a, b in zip(_state(ref), _state(again)):
        np.testing.assert_array_equal(a, b)


def test_noalloc_expand_past_one_cluster_two_calls_in_a_row():
    """V = 65536 takes the chunked kernel (per-chunk partials and per-row
    counters in the library's array, laid out for B * m_l rows), not the
    cluster kernel; two layers in a row must equal the workspace path."""
    cfg = E.TreeCfg(B=1, V=65536, depth=2, topk=4, m=4, n=8)
    C = E.et_num_candidates(cfg)
    rng = np.random.default_rng(2025)
    table = torch.from_numpy((rng.standard_normal((cfg.B * (C + 1), cfg.V)) * 2).astype(np.float32)).cuda()
    ref = E.TreeBuffers.allocate(cfg)
    got = E.TreeBuffers.allocate(cfg)
    ws = E.new_workspace(E.et_tree_workspace_size(cfg))
    for layer in range(2):
        E.et_tree_expand(cfg, layer, table, ref, ws)
        E.et_tree_expand_noalloc(cfg, layer, table, got)
        for a, b in zip(_state(ref), _state(got)):
            np.testing.assert_array_equal(a, b)


def test_noalloc_expand_rejects_shapes_beyond_its_scratch():
    # 1000 root rows of a 262144-token vocabulary with k = 32 need ~34 MB of
    # partials: more than the 4 MiB the library keeps, so nothing is launched
    cfg = E.TreeCfg(B=1000, V=262144, depth=2, topk=32, m=32, n=32)
    tb = E.TreeBuffers.allocate(E.TreeCfg(B=1, V=16, depth=2, topk=2, m=2, n=2))
    logits = torch.zeros((1, 262144), dtype=torch.float32, device="cuda")
    with pytest.raises(E.EtError) as ex:
        E.et_tree_expand_noalloc(cfg, 0, logits, tb)
    assert ex.value.status == E.ET_ERR_WORKSPACE
