"""CUDA path vs the CPU oracle on the same seeded inputs, through the C ABI.

Bars: token ids, parents, frontiers, flat trees, masks, position ids and
accepted tokens bit-exact; log-probs within 1e-5; bf16 attention within
max-abs 2e-2 and rel-L2 5e-3 (fp32 path: 1e-4 / 1e-5).  Every case states
the near-tie margins the oracle reports, so a bit-exact comparison is only
demanded where fp32 rounding cannot decide it.
"""
import numpy as np
import pytest
import torch

import oracle as O
from speculative_decoding_eagle_gb300 import binding as E
from speculative_decoding_eagle_gb300 import step as S
from speculative_decoding_eagle_gb300 import workloads as W
from tests.parity_util import (BF16_MAX_ABS, BF16_REL_L2, F32_MAX_ABS, F32_REL_L2, KEY_TOL_PER_LEVEL, compare_layer,
                               gpu_tree_np, ocfg, oracle_attention_from_host, out_as_float, rel_l2,
                               upload_oracle_tree)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_eagle_gb300 import build_lib
    build_lib.build()
    E.load()


@pytest.fixture(params=["cluster", "block"])
def expand_kernel(request):
    """Runs the test once with each expansion kernel (a cluster per row, one block per row)."""
    which = E.ET_EXPAND_CLUSTER if request.param == "cluster" else E.ET_EXPAND_BLOCK
    prev = E.et_set_expand_kernel(which)
    yield request.param
    E.et_set_expand_kernel(prev)


def _random_table(rows, V, seed, scale=2.0, ties=False):
    rng = np.random.default_rng(seed)
    if ties:
        return rng.integers(-4, 4, (rows, V)).astype(np.float32)
    return (rng.standard_normal((rows, V)) * scale).astype(np.float32)


def _rmap(B, C):
    return (np.arange(B)[:, None] * (C + 1) + np.arange(C + 1)[None, :]).astype(np.int32)


# ---------------------------------------------------------------------------
# expand, layer by layer, given the oracle's state before each layer
# ---------------------------------------------------------------------------
EXPAND_CASES = [
    # (B, V, D, k, m, n, ties, stride_pad)
    (1, 1000, 4, 4, 4, 16, False, 0),          # tiny shape
    (2, 32000, 3, 10, 10, 60, False, 0),       # 7B vocabulary, ragged last chunk (32000 % 2048)
    (3, 4099, 3, 7, 5, 20, False, 3),          # V % 4 != 0, unaligned row stride (scalar loads)
    (2, 300, 3, 32, 32, 100, True, 0),         # k = m = 32, many tied logits
    (1, 5000, 4, 1, 1, 4, False, 0),           # chain tree (k = 1)
    (4, 2048, 3, 3, 8, 12, False, 0),          # m > layer width
    (9, 32000, 3, 10, 8, 40, False, 0),        # 72 rows a layer: the automatic choice is one block per row
]


@pytest.mark.parametrize("B,V,D,k,m,n,ties,pad", EXPAND_CASES)
def test_expand_each_layer_matches_oracle(B, V, D, k, m, n, ties, pad, expand_kernel):
    cfg = E.TreeCfg(B=B, V=V, depth=D, topk=k, m=m, n=n)
    C = E.et_num_candidates(cfg)
    assert C == O.num_candidates(ocfg(cfg))
    table = _random_table(B * (C + 1), V, seed=V + k, ties=ties)
    rmap = _rmap(B, C)
    # device table with optional row padding (row stride V + pad)
    dev = torch.zeros((B * (C + 1), V + pad), dtype=torch.float32, device="cuda")
    dev[:, :V] = torch.from_numpy(table)
    dev_t = dev[:, :V] if pad else dev
    tb = E.TreeBuffers.allocate(cfg)
    ws = E.new_workspace(E.et_tree_workspace_size(cfg))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ot = O.Tree.empty(ocfg(cfg))
    for layer in range(D):
        upload_oracle_tree(ot, tb)
        O.tree_expand(ot, layer, table, rmap)
        E.et_tree_expand(cfg, layer, dev_t, tb, ws, row_of_node=torch.from_numpy(rmap).cuda(), dev_status=status)
        ties_here = [x for x in O.near_tie_selections(ot) if x[1] == "frontier" and x[3] == layer + 1]
        compare_layer(cfg, layer, gpu_tree_np(tb), ot, check_frontier=not ties_here)
    assert int(status.item()) == 0


def test_expand_slot_ordered_rows_and_nonfinite(expand_kernel):
    """Rows given in expansion order (no row map), with NaN / +-inf logits."""
    B, V = 2, 3000
    cfg = E.TreeCfg(B=B, V=V, depth=2, topk=5, m=3, n=8)
    C = E.et_num_candidates(cfg)
    ot = O.Tree.empty(ocfg(cfg))
    tb = E.TreeBuffers.allocate(cfg)
    ws = E.new_workspace(E.et_tree_workspace_size(cfg))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = _random_table(B, V, 1)
    t0[0, 17] = np.nan
    t0[1, 5] = -np.inf
    t0[1, 6] = np.inf
    O.tree_expand(ot, 0, t0, None)
    E.et_tree_expand(cfg, 0, torch.from_numpy(t0).cuda(), tb, ws, dev_status=status)
    compare_layer(cfg, 0, gpu_tree_np(tb), ot)
    assert int(status.item()) & E.ET_DEV_NONFINITE
    t1 = _random_table(B * 3, V, 2)
    upload_oracle_tree(ot, tb)
    O.tree_expand(ot, 1, t1, None)
    E.et_tree_expand(cfg, 1, torch.from_numpy(t1).cuda(), tb, ws)
    compare_layer(cfg, 1, gpu_tree_np(tb), ot)
    assert C == 5 + 15


def test_expand_all_neg_inf_row(expand_kernel):
    cfg = E.TreeCfg(B=1, V=100, depth=1, topk=3, m=1, n=3)
    tb = E.TreeBuffers.allocate(cfg)
    ws = E.new_workspace(E.et_tree_workspace_size(cfg))
    z = np.full((1, 100), -np.inf, np.float32)
    E.et_tree_expand(cfg, 0, torch.from_numpy(z).cuda(), tb, ws)
    g = gpu_tree_np(tb)
    assert list(g["cand_tok"][0]) == [0, 1, 2]
    assert (g["cand_key"][0] == O.KEY_MIN).all()


@pytest.mark.parametrize("k", [10, 32])
def test_expand_constant_row_takes_lowest_ids(k, expand_kernel):
    # every logit equal: the top-k by (value desc, id asc) are ids 0..k-1, each
    # with log-prob -ln V (k = 32 makes every warp rank more tied keys than it
    # counts directly, so the exact argmin rounds decide)
    V = 32000
    cfg = E.TreeCfg(B=2, V=V, depth=2, topk=k, m=k, n=k + 1)
    tb = E.TreeBuffers.allocate(cfg)
    ws = E.new_workspace(E.et_tree_workspace_size(cfg))
    z = np.full((2, V), 1.25, np.float32)
    z[1] = -3.5
    E.et_tree_expand(cfg, 0, torch.from_numpy(z).cuda(), tb, ws)
    g = gpu_tree_np(tb)
    for b in range(2):
        assert list(g["cand_tok"][b][:k]) == list(range(k))
        np.testing.assert_allclose(g["cand_lp"][b][:k], -np.log(V), rtol=1e-5)
        assert list(g["frontier"][b][:k]) == list(range(k))


# ---------------------------------------------------------------------------
# rerank + mask/posids, given the oracle's keys
# ---------------------------------------------------------------------------
RERANK_CASES = [(1, 4, 4, 4, 16), (3, 6, 10, 10, 60), (2, 8, 8, 8, 80), (2, 6, 10, 10, 100), (1, 3, 2, 2, 10),
                (2, 16, 2, 1, 9), (1, 2, 32, 32, 127)]


@pytest.mark.parametrize("B,D,k,m,n", RERANK_CASES)
@pytest.mark.parametrize("ties", [False, True])
def test_rerank_mask_posids_match_oracle(B, D, k, m, n, ties):
    V = 64
    cfg = E.TreeCfg(B=B, V=V, depth=D, topk=k, m=m, n=n)
    C = E.et_num_candidates(cfg)
    table = _random_table(B * (C + 1), V, seed=D * 100 + k, ties=ties)
    if ties:  # many equal values across parents: shallow-first tie-break must hold
        table[:] = np.round(table)
    root = np.arange(B, dtype=np.int32) + 7
    ot = O.build_tree(ocfg(cfg), table, _rmap(B, C), root)
    tb = E.TreeBuffers.allocate(cfg, root_tok=torch.from_numpy(root).cuda())
    upload_oracle_tree(ot, tb)
    tb.flat_node.fill_(-5)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.et_tree_rerank(cfg, tb, dev_status=status)
    g = gpu_tree_np(tb)
    for name, want in (("flat_node", ot.flat_node), ("flat_tok", ot.flat_tok), ("flat_parent", ot.flat_parent),
                       ("flat_depth", ot.flat_depth)):
        np.testing.assert_array_equal(g[name], want, err_msg=name)
    assert int(status.item()) == 0
    prefix = (np.arange(B, dtype=np.int32) * 37 + 5)
    N = cfg.N
    mask = torch.zeros((B, N, (N + 63) // 64), dtype=torch.int64, device="cuda")
    pos = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    E.et_tree_mask_posids(cfg, tb, torch.from_numpy(prefix).cuda(), mask, pos)
    om, op = O.mask_posids(ot.flat_parent, ot.flat_depth, prefix)
    np.testing.assert_array_equal(mask.cpu().numpy().view(np.uint64), om)
    np.testing.assert_array_equal(pos.cpu().numpy(), op)
    # the fused call writes the same flat tree, mask and positions in one launch
    for buf in (tb.flat_node, tb.flat_tok, tb.flat_parent, tb.flat_depth):
        buf.fill_(-5)
    mask.fill_(-1)
    pos.fill_(-1)
    E.et_tree_rerank_mask(cfg, tb, torch.from_numpy(prefix).cuda(), mask, pos, dev_status=status)
    g = gpu_tree_np(tb)
    for name, want in (("flat_node", ot.flat_node), ("flat_tok", ot.flat_tok), ("flat_parent", ot.flat_parent),
                       ("flat_depth", ot.flat_depth)):
        np.testing.assert_array_equal(g[name], want, err_msg="fused " + name)
    np.testing.assert_array_equal(mask.cpu().numpy().view(np.uint64), om)
    np.testing.assert_array_equal(pos.cpu().numpy(), op)
    assert int(status.item()) == 0


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def _attn_case(B, N, Hq, Hkv, d, prefixes, dtype, seed, splits=0, head_stride=0, impl=E.ATTN_AUTO, nan_tail=False):
    rng = np.random.default_rng(seed)
    wl = W.Workload("t", 99, V=16, Hq=Hq, Hkv=Hkv, d=d, prefix=0, dtype=dtype, depth=3, topk=2, m=2, n=N - 1,
                    sigma=0.5, accept=("greedy",), B=B)
    # random tree topology: parent of row i uniform in [0, i)
    fp = np.full((B, N), -1, np.int32)
    depth = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(1, N):
            fp[b, i] = rng.integers(0, i)
            depth[b, i] = depth[b, fp[b, i]] + 1
    mask, _ = O.mask_posids(fp, depth, np.zeros(B, np.int32))
    L = np.asarray(prefixes, np.int32)
    hs = head_stride
    rows_per_seq = [Hkv * (hs if hs else int(L[b])) for b in range(B)]
    kv_row0 = np.concatenate([[0], np.cumsum(rows_per_seq)[:-1]]).astype(np.int64)
    total = max(int(sum(rows_per_seq)), 1)
    f32 = lambda *s: rng.standard_normal(s).astype(np.float32)
    enc = (lambda x: W.bf16_bits(x)) if dtype == "bf16" else (lambda x: x)
    h = dict(q=enc(f32(B, N, Hq, d)), k_tree=enc(f32(B, N, Hkv, d)), v_tree=enc(f32(B, N, Hkv, d)),
             k_prefix=enc(f32(total, d)), v_prefix=enc(f32(total, d)), prefix_len=L, kv_row0=kv_row0)
    if nan_tail and hs:  # cache rows past each prefix hold NaN: they must never reach the output
        nan = W.bf16_bits(np.array([np.nan], np.float32))[0] if dtype == "bf16" else np.float32(np.nan)
        for b in range(B):
            for g in range(Hkv):
                lo = kv_row0[b] + g * hs + int(L[b])
                h["k_prefix"][lo:kv_row0[b] + (g + 1) * hs] = nan
                h["v_prefix"][lo:kv_row0[b] + (g + 1) * hs] = nan
    # oracle view of the prefix (respecting the head stride)
    kpf, vpf = W.as_float(wl, h["k_prefix"]), W.as_float(wl, h["v_prefix"])
    kp, vp = [], []
    for b in range(B):
        stride = hs if hs else int(L[b])
        idx = kv_row0[b] + np.arange(Hkv)[:, None] * stride + np.arange(int(L[b]))[None, :]
        kp.append(kpf[idx].astype(np.float64))
        vp.append(vpf[idx].astype(np.float64))
    ref, lse = O.tree_attention(W.as_float(wl, h["q"]).astype(np.float64), kp, vp,
                                W.as_float(wl, h["k_tree"]).astype(np.float64),
                                W.as_float(wl, h["v_tree"]).astype(np.float64), mask, d ** -0.5)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32

    def up(x):
        if dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()

    shape = E.AttnShape(B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, dtype=E.ET_BF16 if dtype == "bf16" else E.ET_F32,
                        scale=d ** -0.5, max_prefix=int(L.max()) if B else 0, kv_rows=total,
                        kv_head_stride=hs, num_splits=splits, impl=impl)
    out = torch.full((B, N, Hq, d), float("nan"), dtype=dt, device="cuda")
    lse_g = torch.zeros((B, Hq, N), dtype=torch.float32, device="cuda")
    ws = E.new_workspace(E.et_tree_attention_workspace_size(shape))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.et_tree_attention(shape, up(h["q"]), up(h["k_prefix"]), up(h["v_prefix"]),
                        torch.from_numpy(kv_row0).cuda(), torch.from_numpy(L).cuda(), up(h["k_tree"]),
                        up(h["v_tree"]), torch.from_numpy(mask.view(np.int64)).cuda(), out, lse=lse_g, ws=ws,
                        dev_status=status)
    torch.cuda.synchronize()
    return out_as_float(out), lse_g.cpu().numpy(), ref, lse, int(status.item())


ATTN_CASES = [
    # B, N, Hq, Hkv, d, prefixes, dtype, splits, head_stride
    (1, 17, 4, 4, 64, [128], "f32", 0, 0),          # tiny shape
    (2, 9, 2, 1, 128, [70, 3], "f32", 0, 0),
    (1, 61, 32, 32, 128, [1024], "bf16", 0, 0),     # 7B shape at its bench prefix
    (1, 61, 4, 4, 128, [1000], "bf16", 1, 0),       # single split, ragged last tile
    (1, 61, 4, 4, 128, [1000], "bf16", 7, 0),       # uneven splits
    (2, 81, 16, 2, 128, [300, 129], "bf16", 0, 0),  # GQA group 8, N > 64
    (1, 81, 64, 8, 128, [700], "bf16", 0, 0),       # 70B heads: 648 rows per KV head, 6 row tiles
    (3, 101, 4, 4, 128, [64, 0, 513], "bf16", 0, 0),  # empty prefix, N = 101 (two mask words)
    (2, 33, 8, 2, 64, [200, 77], "bf16", 3, 0),     # d = 64
    (2, 20, 4, 2, 128, [100, 60], "bf16", 2, 128),  # static cache layout (head stride)
    (1, 128, 2, 2, 128, [257], "bf16", 0, 0),       # maximum N
    (2, 7, 4, 4, 128, [0, 0], "bf16", 0, 0),        # no prefix at all
    (1, 61, 8, 8, 128, [4096], "bf16", 32, 0),      # many splits (16 on the tcgen05 path: one cluster)
    (1, 61, 8, 8, 128, [1000], "bf16", 5, 0),       # odd cluster size
    (1, 61, 2, 2, 128, [8192], "bf16", 7, 0),       # 7 splits of 129 key tiles
    (1, 61, 4, 4, 128, [1024], "bf16", 9, 0),       # 9 splits (a non-portable cluster) of 17 key tiles
    (2, 81, 16, 2, 128, [3000, 700], "bf16", 12, 0),  # 12 splits, GQA rows merged through L2
    (5, 33, 4, 4, 128, [513, 64, 513, 1000, 64], "bf16", 0, 0),  # ragged batch out longest first, equal lengths
    (66, 9, 2, 2, 128, [(37 * i) % 301 for i in range(66)], "bf16", 0, 0),  # past 64 sequences: grid order
]


@pytest.mark.parametrize("impl", [E.ATTN_MMA_SYNC, E.ATTN_TCGEN05])
@pytest.mark.parametrize("B,N,Hq,Hkv,d,prefixes,dtype,splits,hs", ATTN_CASES)
def test_attention_matches_oracle(B, N, Hq, Hkv, d, prefixes, dtype, splits, hs, impl):
    if dtype == "f32":
        if impl != E.ATTN_MMA_SYNC:
            pytest.skip("fp32 has one path")
        impl = E.ATTN_AUTO
    if impl == E.ATTN_TCGEN05 and d != 128:
        pytest.skip("the tcgen05 path is built for d = 128")
    got, lse_g, ref, lse_o, status = _attn_case(B, N, Hq, Hkv, d, prefixes, dtype, seed=N * 7 + d, splits=splits,
                                                head_stride=hs, impl=impl)
    assert status == 0
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    rl = rel_l2(got, ref)
    if dtype == "bf16":
        assert err <= BF16_MAX_ABS and rl <= BF16_REL_L2, (err, rl)
    else:
        assert err <= F32_MAX_ABS and rl <= F32_REL_L2, (err, rl)
    assert np.abs(lse_g - lse_o).max() < 1e-3


@pytest.mark.parametrize("impl", [E.ATTN_MMA_SYNC, E.ATTN_TCGEN05])
def test_attention_ignores_cache_rows_past_the_prefix(impl):
    """A static cache whose rows past the prefix hold NaN: the output stays exact."""
    got, _, ref, _, status = _attn_case(2, 24, 4, 2, 128, [100, 37], "bf16", seed=5, splits=2, head_stride=192,
                                        impl=impl, nan_tail=True)
    assert status == 0 and np.isfinite(got).all()
    assert np.abs(got - ref).max() <= BF16_MAX_ABS and rel_l2(got, ref) <= BF16_REL_L2


def test_tcgen05_and_mma_paths_agree_at_the_7b_shape():
    a = _attn_case(1, 61, 32, 32, 128, [1024], "bf16", seed=1, impl=E.ATTN_TCGEN05)[0]
    b = _attn_case(1, 61, 32, 32, 128, [1024], "bf16", seed=1, impl=E.ATTN_MMA_SYNC)[0]
    assert np.abs(a - b).max() <= 2 * BF16_MAX_ABS


# ---------------------------------------------------------------------------
# the whole tree in one launch (et_tree_build)
# ---------------------------------------------------------------------------
BUILD_CASES = [  # workload, B, changed fields, expected launches (None: whatever fits)
    ("tiny", 4, {}, 1),
    ("llama2-7b", 1, {}, 1),
    ("llama2-70b", 1, {}, 1),
    ("llama2-7b", 3, {"n": 100}, None),
    ("llama2-7b", 1, {"topk": 16, "m": 16}, 2),  # n + the widest layer > 256: the rerank as a second launch
    ("tiny", 2, {"V": 50000}, 5),                # past one cluster: the per-layer launches
]


# forms of et_tree_build chosen by et_tree_expand's row code: (expansion kernel, cases)
FORM_CASES = [
    # the work-queue form (one block per row, layers of different sequences overlapping, rerank inside)
    (E.ET_EXPAND_BLOCK, "tiny", 4, {}, 1),
    (E.ET_EXPAND_BLOCK, "llama2-7b", 1, {}, 1),
    (E.ET_EXPAND_BLOCK, "llama2-7b", 3, {"n": 100}, 1),
    (E.ET_EXPAND_BLOCK, "llama2-7b", 1, {"topk": 16, "m": 16}, 1),  # n + the widest layer > 256: still inside
    (E.ET_EXPAND_BLOCK, "llama2-70b", 1, {}, 1),
    (E.ET_EXPAND_BLOCK, "llama2-7b", 9, {}, 1),
    (E.ET_EXPAND_BLOCK, "tiny", 2, {"V": 50000}, 5),  # past one cluster: the per-layer launches
    # the cluster row code where the one-launch clusters do not fit: the per-layer launches
    (E.ET_EXPAND_CLUSTER, "llama2-7b", 9, {}, None),
]


@pytest.mark.parametrize("kernel,wl_name,B,changes,launches", FORM_CASES)
def test_tree_build_forms_match_per_layer_path_and_oracle(kernel, wl_name, B, changes, launches):
    """et_tree_build with the expansion row code forced: the work-queue form
    (one block per row) against the per-layer launches of the same row code,
    bit for bit, twice in a row, and the oracle."""
    prev = E.et_set_expand_kernel(kernel)
    try:
        test_tree_build_matches_per_layer_path_and_oracle(wl_name, B, changes, launches)
    finally:
        E.et_set_expand_kernel(prev)


@pytest.mark.parametrize("kernel", [E.ET_EXPAND_CLUSTER, E.ET_EXPAND_BLOCK])
def test_tree_build_nonfinite_logits_both_forms(kernel):
    """NaN (counted as -inf), +inf (counted as FLT_MAX) and -inf logits in
    the draft rows, including a whole -inf row: both build forms write what
    the per-layer launches of the same row code write, bit for bit, and flag
    ET_DEV_NONFINITE."""
    prev = E.et_set_expand_kernel(kernel)
    try:
        wl = W.WORKLOADS["llama2-7b"].with_(B=3)
        one = S.VerifyStep(wl, per_layer=False)
        ref = S.VerifyStep(wl, per_layer=True)
        h = S.host_inputs(wl, one.C)
        C = one.C
        d = h["draft"].copy()
        rng = np.random.default_rng(7)
        for b in range(wl.B):
            for node in range(-1, C, 37):  # the root and every 37th candidate's row
                row = h["row_of_node"][b, node + 1]
                cols = rng.integers(0, wl.V, 6)
                d[row, cols[:2]] = np.nan
                d[row, cols[2]] = np.inf
                d[row, cols[3:]] = -np.inf
            d[h["row_of_node"][b, 5], :] = -np.inf  # a whole row of -inf (a child of the root)
        h = dict(h, draft=d)
        inp = S.to_device(wl, h)
        for st in (one, ref):
            st.prepare(inp)
            st.build_tree(inp)
        torch.cuda.synchronize()
        got, want = gpu_tree_np(one.tree), gpu_tree_np(ref.tree)
        for name in want:
            np.testing.assert_array_equal(got[name], want[name], err_msg=name)
        np.testing.assert_array_equal(one.mask.cpu().numpy(), ref.mask.cpu().numpy())
        assert int(one.dev_status.item()) & E.ET_DEV_NONFINITE
        assert int(ref.dev_status.item()) & E.ET_DEV_NONFINITE
    finally:
        E.et_set_expand_kernel(prev)


@pytest.mark.parametrize("wl_name,B,changes,launches", BUILD_CASES)
def test_tree_build_matches_per_layer_path_and_oracle(wl_name, B, changes, launches):
    """et_tree_build (all layers and the rerank in one launch, or the rerank
    as a second launch) writes exactly what D et_tree_expand calls and
    et_tree_rerank_mask write; twice in a row (its per-layer counters must be
    back at zero for the second call), and equal to the oracle's tree."""
    wl = W.WORKLOADS[wl_name].with_(B=B, **changes)
    one = S.VerifyStep(wl, per_layer=False)
    ref = S.VerifyStep(wl, per_layer=True)
    if launches is not None:
        assert E.et_tree_build_launches(one.cfg) == launches
    h = S.host_inputs(wl, one.C)
    inp = S.to_device(wl, h)
    for st in (one, ref):
        st.prepare(inp)
        st.build_tree(inp)
    torch.cuda.synchronize()
    first = gpu_tree_np(one.tree)
    want = gpu_tree_np(ref.tree)
    for name in want:
        np.testing.assert_array_equal(first[name], want[name], err_msg=name)
    np.testing.assert_array_equal(one.mask.cpu().numpy(), ref.mask.cpu().numpy())
    np.testing.assert_array_equal(one.posids.cpu().numpy(), ref.posids.cpu().numpy())
    one.tree.flat_node.fill_(-7)
    one.mask.zero_()
    one.build_tree(inp)
    torch.cuda.synchronize()
    again = gpu_tree_np(one.tree)
    for name in want:
        np.testing.assert_array_equal(again[name], want[name], err_msg=name)
    np.testing.assert_array_equal(one.mask.cpu().numpy(), ref.mask.cpu().numpy())
    assert int(one.dev_status.item()) == 0
    ot = O.build_tree(ocfg(one.cfg), h["draft"], h["row_of_node"], h["root_tok"])
    assert not O.near_tie_selections(ot)
    for name, o in (("flat_node", ot.flat_node), ("flat_tok", ot.flat_tok), ("flat_parent", ot.flat_parent),
                    ("flat_depth", ot.flat_depth), ("cand_tok", ot.tok), ("cand_parent", ot.parent)):
        np.testing.assert_array_equal(again[name], o, err_msg=name)


# ---------------------------------------------------------------------------
# acceptance, given the oracle's flat tree
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode", [E.ET_ACCEPT_GREEDY, E.ET_ACCEPT_STOCH_POINT, E.ET_ACCEPT_STOCH_DRAFTQ])
@pytest.mark.parametrize("wl_name,B,V", [("tiny", 4, None), ("llama2-7b", 2, None), ("tiny", 3, 50000),
                                          # 8 or more sequences: greedy and point-mass walk each path in one cluster
                                          ("tiny", 8, None), ("llama2-7b", 9, None)])
def test_verify_matches_oracle(mode, wl_name, B, V):
    """V = 50000 is past one cluster (32768 tokens): one block per 2048-token chunk, merged by the last."""
    wl = W.WORKLOADS[wl_name].with_(B=B, temperature=0.7 if mode == E.ET_ACCEPT_STOCH_DRAFTQ else 1.0)
    if V is not None:
        wl = wl.with_(V=V)
    cfg = S.tree_cfg(wl)
    C = E.et_num_candidates(cfg)
    h = S.host_inputs(wl, C)
    ot = O.build_tree(ocfg(cfg), h["draft"], h["row_of_node"], h["root_tok"])
    ref = O.verify_accept(ocfg(cfg), mode, ot.flat_tok, ot.flat_parent, ot.flat_node, h["target"], h["row_of_node"],
                          uniforms=h["uniforms"], draft_table=h["draft"], draft_row_of_node=h["row_of_node"])
    inp = S.to_device(wl, h)
    st = S.VerifyStep(wl, mode=mode)
    upload_oracle_tree(ot, st.tree)
    st.accept(inp)
    torch.cuda.synchronize()
    bad_b = {b for b, _, _ in ref.near_ties}
    for b in range(B):
        if b in bad_b:
            continue
        assert st.accept_len[b].item() == ref.accept_len[b]
        np.testing.assert_array_equal(st.path[b].cpu().numpy(), ref.path[b])
        np.testing.assert_array_equal(st.tokens[b].cpu().numpy(), ref.tokens[b])
    assert len(bad_b) < B
    assert int(st.dev_status.item()) == 0


@pytest.mark.parametrize("wl_name,B,V,T,squeeze", [("tiny", 8, None, 1.3, 0.1), ("llama2-7b", 4, None, 0.7, 0.02),
                                                    ("tiny", 4, 50000, 0.7, 0.02)])
def test_draftq_chained_rejections(wl_name, B, V, T, squeeze):
    """Uniforms pushed toward 1 reject several children in a row: the residual
    after each rejection (its sum from phase 1, replayed per token by the walk)
    and the bonus draw from the last residual, on both phase-1 layouts."""
    wl = W.WORKLOADS[wl_name].with_(B=B, temperature=T)
    if V is not None:
        wl = wl.with_(V=V)
    cfg = S.tree_cfg(wl)
    C = E.et_num_candidates(cfg)
    h = S.host_inputs(wl, C)
    h["uniforms"] = (1.0 - (1.0 - h["uniforms"].astype(np.float64)) * squeeze).astype(np.float32)
    ot = O.build_tree(ocfg(cfg), h["draft"], h["row_of_node"], h["root_tok"])
    ref = O.verify_accept(ocfg(cfg), O.STOCH_DRAFTQ, ot.flat_tok, ot.flat_parent, ot.flat_node, h["target"],
                          h["row_of_node"], uniforms=h["uniforms"], draft_table=h["draft"],
                          draft_row_of_node=h["row_of_node"])
    inp = S.to_device(wl, h)
    st = S.VerifyStep(wl, mode=E.ET_ACCEPT_STOCH_DRAFTQ)
    upload_oracle_tree(ot, st.tree)
    st.accept(inp)
    torch.cuda.synchronize()
    bad_b = {b for b, _, _ in ref.near_ties}
    multi = 0
    for b in range(B):
        if b in bad_b:
            continue
        a = int(ref.accept_len[b])
        multi += int((ot.flat_parent[b] == ref.path[b][a]).sum()) >= 2
        assert st.accept_len[b].item() == a
        np.testing.assert_array_equal(st.path[b].cpu().numpy(), ref.path[b])
        np.testing.assert_array_equal(st.tokens[b].cpu().numpy(), ref.tokens[b])
    assert len(bad_b) < B and multi >= 1  # at least one bonus drawn after two or more rejections
    assert int(st.dev_status.item()) == 0


def _rejections(ot, ref, b):
    """Children the oracle's walk rejected in sequence b: at each row of the
    accepted path the siblings tried before the accepted one, and every child
    of the row where it stopped."""
    ch = {}
    for j in range(1, ot.flat_parent.shape[1]):
        ch.setdefault(int(ot.flat_parent[b, j]), []).append(j)
    a = int(ref.accept_len[b])
    path = [int(x) for x in ref.path[b, :a + 1]]
    n = sum(ch.get(path[s], []).index(path[s + 1]) for s in range(a))
    return n + len(ch.get(path[-1], []))


@pytest.mark.parametrize("wl_name,B,V", [("llama2-7b", 4, None), ("tiny", 3, 50000), ("llama2-7b", 8, None)])
@pytest.mark.parametrize("slope,T,squeeze", [(7.0, 0.5, 3e-5), (4.0, 1.0, 1e-2), (7.0, 1.5, 1e-4), (2.5, 0.5, 1e-3)])
def test_point_mass_steep_targets(wl_name, B, V, slope, T, squeeze):
    """Steep targets, low temperatures and uniforms pushed toward 1 reject long
    runs of children that hold almost all of a row's mass (the regime where a
    1 - R form of the ratio cancels in fp32), on both phase-1 layouts: every
    decision the oracle does not flag as a near tie is bit-exact."""
    wl = W.WORKLOADS[wl_name].with_(B=B, temperature=T, slope=slope)
    if V is not None:
        wl = wl.with_(V=V)
    cfg = S.tree_cfg(wl)
    C = E.et_num_candidates(cfg)
    h = S.host_inputs(wl, C)
    h["uniforms"] = (1.0 - (1.0 - h["uniforms"].astype(np.float64)) * squeeze).astype(np.float32)
    ot = O.build_tree(ocfg(cfg), h["draft"], h["row_of_node"], h["root_tok"])
    ref = O.verify_accept(ocfg(cfg), O.STOCH_POINT, ot.flat_tok, ot.flat_parent, ot.flat_node, h["target"],
                          h["row_of_node"], uniforms=h["uniforms"])
    inp = S.to_device(wl, h)
    st = S.VerifyStep(wl, mode=E.ET_ACCEPT_STOCH_POINT)
    upload_oracle_tree(ot, st.tree)
    st.accept(inp)
    torch.cuda.synchronize()
    bad_b = {b for b, _, _ in ref.near_ties}
    longest = 0
    for b in range(B):
        if b in bad_b:
            continue
        longest = max(longest, _rejections(ot, ref, b))
        assert st.accept_len[b].item() == ref.accept_len[b]
        np.testing.assert_array_equal(st.path[b].cpu().numpy(), ref.path[b])
        np.testing.assert_array_equal(st.tokens[b].cpu().numpy(), ref.tokens[b])
    assert len(bad_b) < B and longest >= 3  # long rejection chains occurred
    assert int(st.dev_status.item()) == 0


def test_point_mass_repeated_sibling_tokens():
    """Siblings that repeat a token (a user-built tree): a repeat of a rejected
    token has no residual mass and is never accepted, and the rejected mass
    counts once; the oracle's rule, on both phase-1 layouts."""
    for V in (32000, 50000):
        wl = W.WORKLOADS["tiny"].with_(B=4, V=V, slope=3.0, temperature=0.7)
        cfg = S.tree_cfg(wl)
        C = E.et_num_candidates(cfg)
        h = S.host_inputs(wl, C)
        h["uniforms"] = (1.0 - (1.0 - h["uniforms"].astype(np.float64)) * 1e-2).astype(np.float32)
        ot = O.build_tree(ocfg(cfg), h["draft"], h["row_of_node"], h["root_tok"])
        tok = ot.flat_tok.copy()
        for b in range(cfg.B):  # every second child of each row takes its previous sibling's token
            seen = {}
            for j in range(1, tok.shape[1]):
                p = int(ot.flat_parent[b, j])
                seen[p] = seen.get(p, 0) + 1
                if seen[p] % 2 == 0:
                    tok[b, j] = tok[b, j - 1] if int(ot.flat_parent[b, j - 1]) == p else tok[b, j]
        ot.flat_tok = tok
        ref = O.verify_accept(ocfg(cfg), O.STOCH_POINT, ot.flat_tok, ot.flat_parent, ot.flat_node, h["target"],
                              h["row_of_node"], uniforms=h["uniforms"])
        inp = S.to_device(wl, h)
        st = S.VerifyStep(wl, mode=E.ET_ACCEPT_STOCH_POINT)
        upload_oracle_tree(ot, st.tree)
        st.accept(inp)
        torch.cuda.synchronize()
        bad_b = {b for b, _, _ in ref.near_ties}
        for b in range(cfg.B):
            if b in bad_b:
                continue
            np.testing.assert_array_equal(st.path[b].cpu().numpy(), ref.path[b])
            np.testing.assert_array_equal(st.tokens[b].cpu().numpy(), ref.tokens[b])
        assert len(bad_b) < cfg.B


# ---------------------------------------------------------------------------
# the whole step, every configuration
# ---------------------------------------------------------------------------
STEP_CASES = [("tiny", None, None, None), ("tiny", None, E.ET_ACCEPT_STOCH_POINT, None),
              ("llama2-7b", None, None, None), ("llama2-13b", None, None, None), ("llama2-70b", None, None, None),
              ("llama2-70b", None, E.ET_ACCEPT_STOCH_POINT, None), ("sweep-7b", 4, None, None),
              # the batched sweep: ragged prefixes of 512..16384 tokens, kept trees of 16, 32 and 100 nodes
              ("sweep-7b", 16, None, 16), ("sweep-7b", 32, None, 32), ("sweep-7b", 16, None, 100)]
ATTN_SAMPLE_FROM_B = 16  # from this batch on, attention is checked on sampled sequences


def _attention_sample(h, B):
    """Sequences whose attention the oracle recomputes at large batch: the
    first, the longest and shortest prefix, and one seeded pick."""
    L = h["prefix_len"]
    pick = int(np.random.default_rng(B).integers(0, B))
    return sorted({0, int(np.argmax(L)), int(np.argmin(L)), pick})


@pytest.mark.parametrize("wl_name,B,mode,n", STEP_CASES)
def test_full_step_matches_oracle(wl_name, B, mode, n):
    wl = W.WORKLOADS[wl_name]
    if B is not None:
        wl = wl.with_(B=B)
    if n is not None:
        wl = wl.with_(n=n)
    st = S.VerifyStep(wl, mode=mode)
    cfg = st.cfg
    h = S.host_inputs(wl, st.C)
    inp = S.to_device(wl, h)
    st.run(inp)
    torch.cuda.synchronize()
    oc = ocfg(cfg)
    ot = O.build_tree(oc, h["draft"], h["row_of_node"], h["root_tok"])
    assert not O.near_tie_selections(ot), O.near_tie_selections(ot)
    g = gpu_tree_np(st.tree)
    for name, want in (("flat_node", ot.flat_node), ("flat_tok", ot.flat_tok), ("flat_parent", ot.flat_parent),
                       ("flat_depth", ot.flat_depth), ("cand_tok", ot.tok), ("cand_parent", ot.parent)):
        np.testing.assert_array_equal(g[name], want, err_msg=name)
    assert np.abs(g["cand_lp"].astype(np.float64) - ot.lp).max() <= 1e-5
    assert np.abs(g["cand_key"] - ot.key).max() <= KEY_TOL_PER_LEVEL * cfg.depth
    om, op = O.mask_posids(ot.flat_parent, ot.flat_depth, h["prefix_len"])
    np.testing.assert_array_equal(st.mask.cpu().numpy().view(np.uint64), om)
    np.testing.assert_array_equal(st.posids.cpu().numpy(), op)
    got = out_as_float(st.out)
    tol = (BF16_MAX_ABS, BF16_REL_L2) if wl.dtype == "bf16" else (F32_MAX_ABS, F32_REL_L2)
    if cfg.B < ATTN_SAMPLE_FROM_B:
        ref, _ = oracle_attention_from_host(wl, h, om, cfg.B)
        assert np.abs(got - ref).max() <= tol[0] and rel_l2(got, ref) <= tol[1]
    else:
        for b in _attention_sample(h, cfg.B):
            hb = dict(h, q=h["q"][b:b + 1], k_tree=h["k_tree"][b:b + 1], v_tree=h["v_tree"][b:b + 1],
                      prefix_len=h["prefix_len"][b:b + 1], kv_row0=h["kv_row0"][b:b + 1])
            ref, _ = oracle_attention_from_host(wl, hb, om[b:b + 1], 1)
            assert np.abs(got[b] - ref[0]).max() <= tol[0] and rel_l2(got[b], ref[0]) <= tol[1], b
    acc = O.verify_accept(oc, st.mode, ot.flat_tok, ot.flat_parent, ot.flat_node, h["target"], h["row_of_node"],
                          uniforms=h["uniforms"])
    # a decision within fp32 rounding of its threshold may go either way:
    # such sequences are compared up to that decision
    tied = {b for b, _, _ in acc.near_ties}
    assert len(tied) < cfg.B
    for b in range(cfg.B):
        if b in tied:
            continue
        assert st.accept_len[b].item() == acc.accept_len[b]
        np.testing.assert_array_equal(st.path[b].cpu().numpy(), acc.path[b])
        np.testing.assert_array_equal(st.tokens[b].cpu().numpy(), acc.tokens[b])
    assert int(st.dev_status.item()) == 0


def test_step_is_deterministic_and_graph_capturable():
    wl = W.WORKLOADS["llama2-7b"]
    st = S.VerifyStep(wl)
    h = S.host_inputs(wl, st.C)
    inp = S.to_device(wl, h)
    st.run(inp)
    torch.cuda.synchronize()
    first = (st.out.clone(), st.tokens.clone(), st.tree.flat_node.clone())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        st.run(inp)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.run(inp)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(first[0], st.out) and torch.equal(first[1], st.tokens) and torch.equal(first[2], st.tree.flat_node)


# ---------------------------------------------------------------------------
# KV commit (the step after acceptance)
# ---------------------------------------------------------------------------
COMMIT_CASES = [  # (B, N, Hkv, d, depth, dtype, F)
    (3, 17, 4, 64, 4, "f32", 64),
    (2, 61, 32, 128, 6, "bf16", 4096),
    (4, 81, 8, 128, 8, "bf16", 0),
]


@pytest.mark.parametrize("B,N,Hkv,d,D,dtype,F", COMMIT_CASES)
def test_kv_commit_matches_oracle(B, N, Hkv, d, D, dtype, F):
    rng = np.random.default_rng(B * 1000 + N)
    np_dt = np.float32
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    cap = 300
    prefix = rng.integers(0, cap - D - 1, B).astype(np.int32)
    kv_row0 = (np.arange(B) * Hkv * cap).astype(np.int64)
    rows = B * Hkv * cap
    # accepted paths: a root-first chain of increasing flat rows, lengths 0..D
    alen = rng.integers(0, D + 1, B).astype(np.int32)
    alen[0] = D
    path = np.full((B, D + 1), -1, np.int32)
    for b in range(B):
        path[b, 0] = 0
        path[b, 1:alen[b] + 1] = np.sort(rng.choice(np.arange(1, N), alen[b], replace=False))

    def rnd(*shape):  # values exactly representable in the compute dtype
        x = rng.standard_normal(shape).astype(np_dt)
        return torch.from_numpy(x).to(tdt).float().numpy()
    kt, vt, kc, vc = rnd(B, N, Hkv, d), rnd(B, N, Hkv, d), rnd(rows, d), rnd(rows, d)
    feats = rnd(B, N, F) if F else None
    okc, ovc, olen, ofe = O.kv_commit(kt, vt, alen, path, kc, vc, kv_row0, prefix, cap, feats)
    dev = lambda x: torch.from_numpy(x).cuda()
    dkc, dvc = dev(kc).to(tdt), dev(vc).to(tdt)
    new_len = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    fout = torch.full((B, D + 1, F), 5.0, dtype=tdt, device="cuda") if F else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape = E.CommitShape(B=B, N=N, Hkv=Hkv, d=d, path_len=D + 1, dtype=E.ET_BF16 if dtype == "bf16" else E.ET_F32,
                          kv_head_stride=cap, kv_rows=rows, feat_dim=F)
    E.et_kv_commit(shape, dev(kt).to(tdt), dev(vt).to(tdt), dev(alen), dev(path), dkc, dvc, dev(kv_row0),
                   dev(prefix), new_len, features=None if feats is None else dev(feats).to(tdt), feat_out=fout,
                   dev_status=status)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dkc.float().cpu().numpy(), okc)
    np.testing.assert_array_equal(dvc.float().cpu().numpy(), ovc)
    np.testing.assert_array_equal(new_len.cpu().numpy(), olen)
    if F:
        np.testing.assert_array_equal(fout.float().cpu().numpy(), ofe)
    assert int(status.item()) == 0


def test_kv_commit_skips_and_flags_bad_rows():
    B, N, Hkv, d, D, cap = 2, 9, 2, 64, 3, 6
    tdt = torch.float32
    kt = torch.randn(B, N, Hkv, d, device="cuda")
    vt = torch.randn(B, N, Hkv, d, device="cuda")
    kc = torch.zeros(B * Hkv * cap, d, device="cuda")
    vc = torch.zeros_like(kc)
    kv_row0 = torch.tensor([0, Hkv * cap], dtype=torch.int64, device="cuda")
    prefix = torch.tensor([1, 4], dtype=torch.int32, device="cuda")   # sequence 1: only 2 free slots
    alen = torch.tensor([2, 3], dtype=torch.int32, device="cuda")
    path = torch.tensor([[0, 3, 99, -1], [0, 1, 2, 5]], dtype=torch.int32, device="cuda")  # 99 is no row
    new_len = torch.zeros(B, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape = E.CommitShape(B=B, N=N, Hkv=Hkv, d=d, path_len=D + 1, dtype=E.ET_F32, kv_head_stride=cap,
                          kv_rows=B * Hkv * cap)
    E.et_kv_commit(shape, kt, vt, alen, path, kc, vc, kv_row0, prefix, new_len, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & E.ET_DEV_BAD_INDEX
    # valid rows landed, the bad ones were skipped
    assert torch.equal(kc[0 * cap + 1], kt[0, 0, 0]) and torch.equal(kc[1 * cap + 2], kt[0, 3, 1])
    assert torch.count_nonzero(kc[0 * cap + 3]) == 0               # row 99 skipped
    assert torch.equal(kc[Hkv * cap + 0 * cap + 4], kt[1, 0, 0])   # positions 4 and 5 fit
    assert torch.equal(kc[Hkv * cap + 0 * cap + 5], kt[1, 1, 0])
    assert new_len.cpu().tolist() == [4, 8]


# ---------------------------------------------------------------------------
# static draft tree (fixed shape) -> flat tree -> verification
# ---------------------------------------------------------------------------
STATIC_CASES = [  # (B, V, widths, ties)
    (2, 1000, (3, 2, 1), False),
    (2, 32000, (4, 2, 2, 1, 1), False),
    (3, 300, (8, 4), True),
    (1, 5000, (1, 1, 1, 1), False),
]


def _static_case(B, V, widths, ties, seed=11):
    parent, rank = W.static_shape(widths)
    N = parent.size
    table = _random_table(B * N, V, seed=seed + V, ties=ties)
    rmap = (np.arange(B)[:, None] * N + np.arange(N)[None, :]).astype(np.int32)
    root = (np.arange(B) + 3).astype(np.int32)
    return parent, rank, table, rmap, root


@pytest.mark.parametrize("B,V,widths,ties", STATIC_CASES)
def test_static_tree_matches_oracle(B, V, widths, ties):
    parent, rank, table, rmap, root = _static_case(B, V, widths, ties)
    N, k = parent.size, max(widths)
    tb = E.TreeBuffers.allocate_flat(B, N, root_tok=torch.from_numpy(root).cuda())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.et_static_tree(B, V, k, torch.from_numpy(parent).cuda(), torch.from_numpy(rank).cuda(),
                     torch.from_numpy(table).cuda(), torch.from_numpy(rmap).cuda(), tb, dev_status=status)
    g = gpu_tree_np(tb)
    tok, fpar, fdep, node = O.static_tree(parent, rank, table, rmap, root)
    np.testing.assert_array_equal(g["flat_tok"], tok)
    np.testing.assert_array_equal(g["flat_parent"], fpar)
    np.testing.assert_array_equal(g["flat_depth"], fdep)
    np.testing.assert_array_equal(g["flat_node"], node)
    assert int(status.item()) == 0


def test_static_tree_then_mask_and_greedy_acceptance():
    B, V, widths = 3, 32000, (4, 2, 2, 1, 1)
    parent, rank, table, rmap, root = _static_case(B, V, widths, False, seed=3)
    N, D = parent.size, len(widths)
    tb = E.TreeBuffers.allocate_flat(B, N, root_tok=torch.from_numpy(root).cuda())
    E.et_static_tree(B, V, max(widths), torch.from_numpy(parent).cuda(), torch.from_numpy(rank).cuda(),
                     torch.from_numpy(table).cuda(), torch.from_numpy(rmap).cuda(), tb)
    # target rows in flat order: the target agrees with the draft's top token often enough to accept a few
    rng = np.random.default_rng(9)
    target = (table + 0.3 * rng.standard_normal(table.shape)).astype(np.float32)
    cfg = E.TreeCfg(B=B, V=V, depth=D, topk=4, m=4, n=N - 1)
    prefix = np.array([10, 20, 30], np.int32)
    mask = torch.zeros((B, N, (N + 63) // 64), dtype=torch.int64, device="cuda")
    pos = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    E.et_tree_mask_posids(cfg, tb, torch.from_numpy(prefix).cuda(), mask, pos)
    ws = E.new_workspace(E.et_tree_workspace_size(cfg))
    alen = torch.zeros(B, dtype=torch.int32, device="cuda")
    path = torch.zeros((B, D + 1), dtype=torch.int32, device="cuda")
    toks = torch.zeros((B, D + 1), dtype=torch.int32, device="cuda")
    E.et_verify_accept(cfg, E.ET_ACCEPT_GREEDY, tb, torch.from_numpy(target).cuda(), alen, path, toks, ws)
    tok, fpar, fdep, node = O.static_tree(parent, rank, table, rmap, root)
    om, op = O.mask_posids(fpar, fdep, prefix)
    np.testing.assert_array_equal(mask.cpu().numpy().view(np.uint64), om)
    np.testing.assert_array_equal(pos.cpu().numpy(), op)
    ref = O.verify_accept(ocfg(cfg), O.GREEDY, tok, fpar, node, target, None)
    np.testing.assert_array_equal(alen.cpu().numpy(), ref.accept_len)
    np.testing.assert_array_equal(path.cpu().numpy(), ref.path)
    np.testing.assert_array_equal(toks.cpu().numpy(), ref.tokens)


def test_static_tree_flags_a_bad_rank():
    parent = np.array([-1, 0, 0], np.int32)
    rank = np.array([-1, 0, 5], np.int32)  # rank 5 with topk 2
    table = _random_table(3, 100, seed=1)
    tb = E.TreeBuffers.allocate_flat(1, 3)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.et_static_tree(1, 100, 2, torch.from_numpy(parent).cuda(), torch.from_numpy(rank).cuda(),
                     torch.from_numpy(table).cuda(), torch.from_numpy(np.arange(3, dtype=np.int32)[None]).cuda(),
                     tb, dev_status=status)
    g = gpu_tree_np(tb)
    assert int(status.item()) & E.ET_DEV_BAD_INDEX
    assert g["flat_tok"][0, 2] == -1 and g["flat_tok"][0, 1] == int(np.argmax(table[0]))


# ---------------------------------------------------------------------------
# draft LM head on tcgen05, and its logits feeding the expansion
# ---------------------------------------------------------------------------
LMHEAD_CASES = [(1, 64, 1000), (10, 4096, 32000), (37, 512, 5000), (64, 128, 130), (16, 256, 128)]


def _lm_operands(M, H, V, seed):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((M, H)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy((0.05 * rng.standard_normal((V, H))).astype(np.float32)).to(torch.bfloat16)
    return x, w


@pytest.mark.parametrize("M,H,V", LMHEAD_CASES)
def test_lm_head_matches_oracle(M, H, V):
    x, w = _lm_operands(M, H, V, seed=M * 7 + V)
    ldo = V + 37
    out = torch.full((M, ldo), 12345.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.et_lm_head(x.cuda(), w.cuda(), out, dev_status=status)
    got = out.cpu().numpy()
    xf, wf = x.float().numpy(), w.float().numpy()
    ref = O.lm_head_logits(xf, wf)
    bound = O.lm_head_error_bound(xf, wf) + 1e-30
    err = np.abs(got[:, :V] - ref)
    assert np.all(err <= bound), float((err / bound).max())
    assert np.all(got[:, V:] == 12345.0)  # past the vocabulary: untouched
    assert int(status.item()) == 0


def test_lm_head_logits_feed_the_expansion():
    # one layer-0 expansion per sequence straight from the head's logits rows
    B, H, V, k = 3, 1024, 32000, 10
    x, w = _lm_operands(B, H, V, seed=2)
    logits = torch.zeros((B, V), device="cuda")
    E.et_lm_head(x.cuda(), w.cuda(), logits)
    cfg = E.TreeCfg(B=B, V=V, depth=2, topk=k, m=k, n=20)
    tb = E.TreeBuffers.allocate(cfg)
    ws = E.new_workspace(E.et_tree_workspace_size(cfg))
    E.et_tree_expand(cfg, 0, logits, tb, ws)
    g = gpu_tree_np(tb)
    table = logits.cpu().numpy()
    for b in range(B):
        want = O.topk_children(table[b], k)
        assert list(g["cand_tok"][b][:k]) == list(want)


SAMPLED_CASES = [(2, 1000, (3, 2, 1), 1.0), (2, 32000, (4, 2, 2, 1, 1), 1.0), (3, 5000, (6, 3), 0.7)]


@pytest.mark.parametrize("B,V,widths,T", SAMPLED_CASES)
def test_static_tree_sampled_matches_oracle(B, V, widths, T):
    parent, _, table, rmap, root = _static_case(B, V, widths, False, seed=21)
    N = parent.size
    u = np.random.default_rng(V + B).random((B, N)).astype(np.float32)
    tb = E.TreeBuffers.allocate_flat(B, N, root_tok=torch.from_numpy(root).cuda())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.et_static_tree_sampled(B, V, T, torch.from_numpy(parent).cuda(), torch.from_numpy(table).cuda(),
                             torch.from_numpy(rmap).cuda(), torch.from_numpy(u).cuda(), tb, dev_status=status)
    g = gpu_tree_np(tb)
    tok, fpar, fdep, node, gaps = O.static_tree_sampled(parent, table, rmap, u, T, root)
    np.testing.assert_array_equal(g["flat_parent"], fpar)
    np.testing.assert_array_equal(g["flat_depth"], fdep)
    np.testing.assert_array_equal(g["flat_node"], node)
    clear = gaps >= O.TIE_REL_CDF  # a uniform within 1e-5 of a CDF step may land on either side in fp32
    clear[:, 0] = True
    np.testing.assert_array_equal(g["flat_tok"][clear], tok[clear])
    assert clear.mean() > 0.5  # high-entropy rows at V = 32000 have CDF steps of about 1e-5: many near ties
    assert int(status.item()) == 0


def test_static_tree_sampled_then_draftq_acceptance():
    B, V, widths, T = 3, 32000, (4, 2, 2, 1, 1), 1.0
    parent, _, draft, rmap, root = _static_case(B, V, widths, False, seed=5)
    N, D = parent.size, len(widths)
    rng = np.random.default_rng(77)
    u_tree = rng.random((B, N)).astype(np.float32)
    u_acc = rng.random((B, N)).astype(np.float32)
    target = (draft + 0.5 * rng.standard_normal(draft.shape)).astype(np.float32)
    tb = E.TreeBuffers.allocate_flat(B, N, root_tok=torch.from_numpy(root).cuda())
    E.et_static_tree_sampled(B, V, T, torch.from_numpy(parent).cuda(), torch.from_numpy(draft).cuda(),
                             torch.from_numpy(rmap).cuda(), torch.from_numpy(u_tree).cuda(), tb)
    cfg = E.TreeCfg(B=B, V=V, depth=D, topk=4, m=4, n=N - 1, temperature=T)
    ws = E.new_workspace(E.et_tree_workspace_size(cfg))
    alen = torch.zeros(B, dtype=torch.int32, device="cuda")
    path = torch.zeros((B, D + 1), dtype=torch.int32, device="cuda")
    toks = torch.zeros((B, D + 1), dtype=torch.int32, device="cuda")
    E.et_verify_accept(cfg, E.ET_ACCEPT_STOCH_DRAFTQ, tb, torch.from_numpy(target).cuda(), alen, path, toks, ws,
                       draft_logits=torch.from_numpy(draft).cuda(), uniforms=torch.from_numpy(u_acc).cuda())
    g = gpu_tree_np(tb)
    ref = O.verify_accept(ocfg(cfg), O.STOCH_DRAFTQ, g["flat_tok"], g["flat_parent"], g["flat_node"], target, None,
                          uniforms=u_acc, draft_table=draft, draft_row_of_node=None)
    tied = {b for b, _, _ in ref.near_ties}
    for b in range(B):
        if b in tied:
            continue
        assert alen[b].item() == ref.accept_len[b]
        np.testing.assert_array_equal(path[b].cpu().numpy(), ref.path[b])
        np.testing.assert_array_equal(toks[b].cpu().numpy(), ref.tokens[b])
    assert len(tied) < B
