"""Bounded device waits that run out, on purpose, on small cases.

Every wait on the GPU side of the library is bounded.  et_set_wait_limit
shortens the bound of the kernels launched after it; with a bound of one
cycle any wait that is not already satisfied runs out.  The kernel must then
report ET_DEV_TIMEOUT, let its copies and MMAs in flight finish, free its
tensor memory and return, so that the next call on the same stream (with the
default bound) is correct.  Nothing here faults or hangs the GPU: the waits
that run out are ordinary waits for copies that do land.
"""
import numpy as np
import pytest
import torch

import oracle as O
from speculative_decoding_eagle_gb300 import binding as E
from speculative_decoding_eagle_gb300 import step as S
from speculative_decoding_eagle_gb300 import workloads as W
from tests.parity_util import BF16_MAX_ABS, BF16_REL_L2, gpu_tree_np, rel_l2
from tests.test_gpu_parity import _attn_case, _lm_operands

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _default_bound_afterwards():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_eagle_gb300 import build_lib
    build_lib.build()
    E.load()
    yield
    E.et_set_wait_limit(0)


@pytest.mark.parametrize("splits", [1, 2])
def test_attention_wait_runs_out_then_next_call_is_exact(splits):
    case = dict(B=1, N=17, Hq=4, Hkv=4, d=128, prefixes=[300], dtype="bf16", seed=3, splits=splits,
                impl=E.ATTN_TCGEN05)
    E.et_set_wait_limit(1)
    *_, status = _attn_case(**case)
    E.et_set_wait_limit(0)
    assert status & E.ET_DEV_TIMEOUT
    got, _, ref, _, status = _attn_case(**case)
    assert status == 0
    assert np.abs(got - ref).max() <= BF16_MAX_ABS and rel_l2(got, ref) <= BF16_REL_L2


def test_lm_head_wait_runs_out_then_next_call_is_exact():
    M, H, V = 10, 256, 1000
    x, w = _lm_operands(M, H, V, seed=5)
    xf, wf = x.float().numpy(), w.float().numpy()
    x, w = x.cuda(), w.cuda()
    out = torch.zeros((M, V), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.et_set_wait_limit(1)
    E.et_lm_head(x, w, out, dev_status=status)
    torch.cuda.synchronize()
    E.et_set_wait_limit(0)
    assert int(status.item()) & E.ET_DEV_TIMEOUT
    status.zero_()
    E.et_lm_head(x, w, out, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.lm_head_logits(xf, wf)
    bound = O.lm_head_error_bound(xf, wf) + 1e-30
    assert np.all(np.abs(out.cpu().numpy() - ref) <= bound)


@pytest.fixture(params=["cluster", "block"])
def build_form(request):
    """et_tree_build in its cluster form (every cluster resident) and in its work-queue form."""
    prev = E.et_set_expand_kernel(E.ET_EXPAND_CLUSTER if request.param == "cluster" else E.ET_EXPAND_BLOCK)
    yield request.param
    E.et_set_expand_kernel(prev)


def test_tree_build_frontier_wait_runs_out_then_next_call_is_exact(build_form):
    wl = W.WORKLOADS["tiny"].with_(B=2)
    one = S.VerifyStep(wl, per_layer=False)
    if E.et_tree_build_launches(one.cfg) not in (1, 2):
        pytest.skip("the clusters of the one-launch layers do not fit here")
    ref = S.VerifyStep(wl, per_layer=True)
    h = S.host_inputs(wl, one.C)
    inp = S.to_device(wl, h)
    ref.prepare(inp)
    ref.build_tree(inp)
    one.prepare(inp)
    E.et_set_wait_limit(1)
    one.build_tree(inp)
    torch.cuda.synchronize()
    E.et_set_wait_limit(0)
    assert int(one.dev_status.item()) & E.ET_DEV_TIMEOUT
    # after a wait that ran out the layers may have finished out of order:
    # the workspace's counters must be zeroed again before the next call
    one.dev_status.zero_()
    one.ws.zero_()
    one.build_tree(inp)
    torch.cuda.synchronize()
    assert int(one.dev_status.item()) == 0
    got, want = gpu_tree_np(one.tree), gpu_tree_np(ref.tree)
    for name in want:
        np.testing.assert_array_equal(got[name], want[name], err_msg=name)
    np.testing.assert_array_equal(one.mask.cpu().numpy(), ref.mask.cpu().numpy())
