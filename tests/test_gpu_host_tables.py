"""Logit tables in page-locked host memory.

The tree build, the per-layer expansion and the acceptance take their logit
tables as plain pointers: device memory, or page-locked host memory that the
GPU addresses (the kernels then read only the rows they use over the host
link).  Results must be bit-for-bit those of the same tables in device
memory; pageable host memory is refused before anything launches.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from speculative_decoding_eagle_gb300 import binding as E
from speculative_decoding_eagle_gb300 import step as S
from speculative_decoding_eagle_gb300 import workloads as W
from tests.parity_util import gpu_tree_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_eagle_gb300 import build_lib
    build_lib.build()
    E.load()


CASES = [  # workload, batch, per-layer calls, acceptance mode
    ("tiny", 3, False, None),                          # one cluster launch for the tree
    ("llama2-7b", 1, False, None),
    ("llama2-7b", 1, True, E.ET_ACCEPT_STOCH_POINT),   # per-layer expansion calls
    ("llama2-7b", 9, False, E.ET_ACCEPT_STOCH_POINT),  # the work-queue tree; the walk acceptance
    ("tiny", 2, False, E.ET_ACCEPT_STOCH_DRAFTQ),      # the draft table read by the acceptance as well
]


@pytest.mark.parametrize("wl_name,B,per_layer,mode", CASES)
def test_host_tables_match_device_tables(wl_name, B, per_layer, mode):
    wl = W.WORKLOADS[wl_name].with_(B=B)
    if mode == E.ET_ACCEPT_STOCH_DRAFTQ:
        wl = wl.with_(temperature=0.7)
    on_dev = S.VerifyStep(wl, mode=mode, per_layer=per_layer)
    on_host = S.VerifyStep(wl, mode=mode, per_layer=per_layer)
    h = S.host_inputs(wl, on_dev.C)
    dev = S.to_device(wl, h)
    host = dataclasses.replace(dev, draft=dev.draft.cpu().pin_memory(), target=dev.target.cpu().pin_memory())
    assert not host.draft.is_cuda and host.draft.is_pinned()
    on_dev.run(dev)
    on_host.run(host)
    torch.cuda.synchronize()
    want, got = gpu_tree_np(on_dev.tree), gpu_tree_np(on_host.tree)
    for name in want:
        np.testing.assert_array_equal(got[name], want[name], err_msg=name)
    for a, b in ((on_dev.mask, on_host.mask), (on_dev.posids, on_host.posids), (on_dev.accept_len, on_host.accept_len),
                 (on_dev.path, on_host.path), (on_dev.tokens, on_host.tokens)):
        assert torch.equal(a, b)
    assert int(on_host.dev_status.item()) == 0


def test_pageable_host_table_is_refused_before_launch():
    wl = W.WORKLOADS["tiny"].with_(B=1)
    st = S.VerifyStep(wl)
    cfg = st.cfg
    pageable = torch.zeros((st.C + 1, wl.V), dtype=torch.float32)  # plain host memory, not page-locked
    with pytest.raises(ValueError):
        E.et_tree_expand(cfg, 0, pageable, st.tree, st.ws)
    # through the C ABI itself: refused with ET_ERR_INVALID_ARG, nothing written
    st.tree.cand_tok.fill_(-5)
    before = st.tree.cand_tok.clone()
    lib = E.load()
    rc = lib.et_tree_expand(ctypes.byref(cfg.c()), 0, pageable.data_ptr(), wl.V, None, ctypes.byref(st.tree.c()),
                            None, st.ws.data_ptr(), st.ws.numel() * st.ws.element_size(),
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == E.ET_ERR_INVALID_ARG
    assert torch.equal(st.tree.cand_tok, before)
    rc = lib.et_verify_accept(ctypes.byref(cfg.c()), E.ET_ACCEPT_GREEDY, ctypes.byref(st.tree.c()),
                              pageable.data_ptr(), wl.V, None, None, 0, None, None, st.accept_len.data_ptr(),
                              st.path.data_ptr(), st.tokens.data_ptr(), None, st.ws.data_ptr(),
                              st.ws.numel() * st.ws.element_size(), torch.cuda.current_stream().cuda_stream)
    assert rc == E.ET_ERR_INVALID_ARG
