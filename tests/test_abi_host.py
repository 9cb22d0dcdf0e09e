"""The C ABI without a GPU: the library builds and loads, exports every symbol
the header declares, computes the tree geometry like the oracle, and rejects
bad arguments on the host before any launch (host-side fault injection)."""
import ctypes
import os
import re

import pytest

import oracle as O
from speculative_decoding_eagle_gb300 import binding as E
from speculative_decoding_eagle_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x100000  # a non-null, 256-byte aligned address that is never dereferenced


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return E.load()


def _declared():
    txt = open(os.path.join(ROOT, "include", "eagle_tree.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return set(re.findall(r"^\s*(?:et_status|int32_t|int64_t|size_t|const char \*)\s*(et_\w+)\s*\(", txt, flags=re.M))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 14
    assert names == set(E.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.et_abi_version() == 2


@pytest.mark.parametrize("D,k,m,n", [(4, 4, 4, 16), (6, 10, 10, 60), (8, 8, 8, 80), (1, 32, 1, 32), (16, 2, 2, 50),
                                     (3, 5, 25, 100)])
def test_geometry_matches_oracle(lib, D, k, m, n):
    cfg = E.TreeCfg(B=3, V=1000, depth=D, topk=k, m=m, n=n)
    oc = O.TreeCfg(B=3, V=1000, depth=D, topk=k, m=m, n=n)
    assert E.et_num_candidates(cfg) == O.num_candidates(oc)
    for layer in range(D):
        assert E.et_layer_expanded(cfg, layer) == O.expanded_count(oc, layer)
        if layer >= 1:
            assert E.et_layer_base(cfg, layer) == O.layer_base(oc, layer)
    assert E.et_layer_expanded(cfg, D) == -1
    assert E.et_tree_workspace_size(cfg) > 0


@pytest.mark.parametrize("bad", [dict(topk=0), dict(topk=33), dict(m=33), dict(depth=0), dict(depth=17),
                                 dict(n=0), dict(n=128), dict(V=3, topk=4), dict(temperature=0.0), dict(B=0),
                                 dict(depth=8, topk=32, m=32, n=10)])
def test_invalid_cfg_rejected(lib, bad):
    base = dict(B=1, V=1000, depth=4, topk=4, m=4, n=16, temperature=1.0)
    base.update(bad)
    cfg = E.TreeCfg(**base)
    assert E.et_num_candidates(cfg) == -1
    tree = E.TreeC(*([FAKE] * 10))
    st = lib.et_tree_expand(ctypes.byref(cfg.c()), 0, FAKE, 1000, None, ctypes.byref(tree), None, FAKE, 1 << 20, None)
    assert st == E.ET_ERR_INVALID_ARG


def test_expand_argument_checks(lib):
    cfg = E.TreeCfg(B=2, V=1000, depth=3, topk=4, m=4, n=10)
    need = E.et_tree_workspace_size(cfg)
    tree = E.TreeC(*([FAKE] * 10))
    call = lambda layer=0, logits=FAKE, stride=1000, ws=FAKE, wsb=need, tr=tree: lib.et_tree_expand(
        ctypes.byref(cfg.c()), layer, logits, stride, None, ctypes.byref(tr), None, ws, wsb, None)
    assert call(layer=3) == E.ET_ERR_INVALID_ARG
    assert call(layer=-1) == E.ET_ERR_INVALID_ARG
    assert call(logits=None) == E.ET_ERR_INVALID_ARG
    assert call(stride=999) == E.ET_ERR_INVALID_ARG
    assert call(logits=FAKE + 2) == E.ET_ERR_INVALID_ARG      # not 4-byte aligned
    assert call(ws=None) == E.ET_ERR_WORKSPACE
    assert call(wsb=need - 1) == E.ET_ERR_WORKSPACE
    assert call(ws=FAKE + 16) == E.ET_ERR_WORKSPACE          # not 256-byte aligned
    t2 = E.TreeC(*([FAKE] * 10))
    t2.cand_key = None
    assert call(tr=t2) == E.ET_ERR_INVALID_ARG


def test_attention_argument_checks(lib):
    def shape(**kw):
        s = dict(B=1, N=61, Hq=32, Hkv=32, d=128, dtype=E.ET_BF16, scale=0.088, max_prefix=1024,
                 kv_rows=32 * 1024, kv_head_stride=0, num_splits=0, impl=0)
        s.update(kw)
        return E.AttnShapeC(*s.values())

    def call(sh, q=FAKE, ws=FAKE, wsb=1 << 30):
        return lib.et_tree_attention(ctypes.byref(sh), q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
                                     ws, wsb, None)
    assert call(shape(d=96)) == E.ET_ERR_UNSUPPORTED
    assert call(shape(d=64, impl=2)) == E.ET_ERR_UNSUPPORTED     # tcgen05 path needs d = 128
    assert call(shape(dtype=E.ET_F32, impl=2)) == E.ET_ERR_UNSUPPORTED
    assert call(shape(impl=3)) == E.ET_ERR_INVALID_ARG
    assert call(shape(N=129)) == E.ET_ERR_INVALID_ARG
    assert call(shape(N=0)) == E.ET_ERR_INVALID_ARG
    assert call(shape(Hq=30, Hkv=4)) == E.ET_ERR_INVALID_ARG
    assert call(shape(scale=0.0)) == E.ET_ERR_INVALID_ARG
    assert call(shape(), q=FAKE + 8) == E.ET_ERR_INVALID_ARG   # bf16 tiles need 16-byte alignment
    assert call(shape(), q=None) == E.ET_ERR_INVALID_ARG
    assert call(shape(impl=1), ws=None) == E.ET_ERR_WORKSPACE    # the mma.sync path merges splits in ws
    sz = lib.et_tree_attention_workspace_size(ctypes.byref(shape(num_splits=4, impl=1)))
    assert sz > 0
    assert call(shape(num_splits=4, impl=1), wsb=sz - 1) == E.ET_ERR_WORKSPACE
    assert lib.et_tree_attention_splits(ctypes.byref(shape(num_splits=4))) == 4
    # the tcgen05 path: the splits of a tile form one cluster (at most 16) and merge through the
    # workspace: per split and 128-row tile, fp32 rows and a (max, sum) pair per row
    tc4 = lib.et_tree_attention_workspace_size(ctypes.byref(shape(num_splits=4, impl=2)))
    assert tc4 == 32 * 1 * 4 * 128 * (128 * 4 + 8)
    assert call(shape(num_splits=4, impl=2), ws=None) == E.ET_ERR_WORKSPACE
    assert call(shape(num_splits=4, impl=2), wsb=tc4 - 1) == E.ET_ERR_WORKSPACE
    assert lib.et_tree_attention_workspace_size(ctypes.byref(shape(num_splits=1, impl=2))) == 0
    assert lib.et_tree_attention_splits(ctypes.byref(shape(num_splits=20, impl=2))) == 16
    assert lib.et_tree_attention_workspace_size(ctypes.byref(shape(num_splits=1))) == 0
    assert lib.et_tree_attention_splits(ctypes.byref(shape(dtype=E.ET_F32))) == 1
    # workspace: tiles x splits x rows-per-tile x d floats (+ counters and (max, sum) pairs)
    mma = lib.et_tree_attention_workspace_size(ctypes.byref(shape(num_splits=4, impl=1)))
    assert mma >= 32 * 4 * 64 * 128 * 4


def test_attention_rejects_unknown_flags(lib):
    shape = E.AttnShapeC(1, 61, 32, 32, 128, E.ET_BF16, 0.088, 1024, 32 * 1024, 0, 0, 0, 4)
    assert lib.et_tree_attention_workspace_size(ctypes.byref(shape)) == 0  # not a valid shape
    assert lib.et_tree_attention_splits(ctypes.byref(shape)) == -1
    ok = E.AttnShapeC(1, 61, 32, 32, 128, E.ET_BF16, 0.088, 1024, 32 * 1024, 0, 0, 0, E.ET_ATTN_INPUTS_READY)
    assert lib.et_tree_attention_splits(ctypes.byref(ok)) >= 1


def test_verify_argument_checks(lib):
    cfg = E.TreeCfg(B=1, V=1000, depth=3, topk=4, m=4, n=10)
    need = E.et_tree_workspace_size(cfg)
    tree = E.TreeC(*([FAKE] * 10))

    def call(mode=E.ET_ACCEPT_GREEDY, uni=None, draft=None, wsb=need, target=FAKE, tstride=1000, dstride=1000,
             ws=FAKE, alen=FAKE, c=cfg):
        return lib.et_verify_accept(ctypes.byref(c.c()), mode, ctypes.byref(tree), target, tstride, None, draft,
                                    dstride, None, uni, alen, FAKE, FAKE, None, ws, wsb, None)
    assert call(mode=7) == E.ET_ERR_INVALID_ARG
    assert call(mode=E.ET_ACCEPT_STOCH_POINT) == E.ET_ERR_INVALID_ARG         # no uniforms
    assert call(mode=E.ET_ACCEPT_STOCH_DRAFTQ, uni=FAKE) == E.ET_ERR_INVALID_ARG  # no draft table
    assert call(mode=E.ET_ACCEPT_STOCH_DRAFTQ, uni=FAKE, draft=FAKE, dstride=999) == E.ET_ERR_INVALID_ARG
    assert call(tstride=999) == E.ET_ERR_INVALID_ARG                           # rows shorter than V
    assert call(target=FAKE + 2) == E.ET_ERR_INVALID_ARG                      # fp32 rows need 4-byte alignment
    assert call(target=None) == E.ET_ERR_INVALID_ARG
    assert call(alen=None) == E.ET_ERR_INVALID_ARG
    assert call(wsb=need - 1) == E.ET_ERR_WORKSPACE
    assert call(ws=FAKE + 128) == E.ET_ERR_WORKSPACE                          # 256-byte aligned workspace
    assert call(ws=None) == E.ET_ERR_WORKSPACE
    big = E.TreeCfg(B=600, V=1000, depth=3, topk=8, m=8, n=120)               # 600 x 121 flat rows > 65535
    assert call(c=big, wsb=E.et_tree_workspace_size(big)) == E.ET_ERR_UNSUPPORTED


def test_rerank_mask_argument_checks(lib):
    cfg = E.TreeCfg(B=1, V=1000, depth=3, topk=4, m=4, n=10)
    tree = E.TreeC(*([FAKE] * 10))
    call = lambda pl=FAKE, mask=FAKE, pos=FAKE, c=cfg: lib.et_tree_rerank_mask(
        ctypes.byref(c.c()), ctypes.byref(tree), pl, mask, pos, None, None)
    assert call(pl=None) == E.ET_ERR_INVALID_ARG
    assert call(mask=None) == E.ET_ERR_INVALID_ARG
    assert call(pos=None) == E.ET_ERR_INVALID_ARG
    assert call(mask=FAKE + 4) == E.ET_ERR_INVALID_ARG   # mask words need 8-byte alignment
    assert call(c=E.TreeCfg(B=1, V=1000, depth=3, topk=4, m=4, n=200)) == E.ET_ERR_INVALID_ARG


def test_kv_commit_argument_checks(lib):
    def shape(**kw):
        s = dict(B=2, N=61, Hkv=32, d=128, path_len=7, dtype=E.ET_BF16, kv_head_stride=4096, kv_rows=2 * 32 * 4096,
                 feat_dim=0)
        s.update(kw)
        return E.CommitShapeC(*s.values())

    def call(sh, kt=FAKE, npl=FAKE + 256, feat=None, fout=None):
        return lib.et_kv_commit(ctypes.byref(sh), kt, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, npl, feat, fout,
                                None, None)
    assert call(shape(d=100)) == E.ET_ERR_UNSUPPORTED            # rows must be whole 16-byte chunks
    assert call(shape(dtype=7)) == E.ET_ERR_INVALID_ARG
    assert call(shape(path_len=18)) == E.ET_ERR_INVALID_ARG      # depth <= 16
    assert call(shape(N=129)) == E.ET_ERR_INVALID_ARG
    assert call(shape(kv_head_stride=0)) == E.ET_ERR_INVALID_ARG  # appending needs a capacity per head
    assert call(shape(), kt=None) == E.ET_ERR_INVALID_ARG
    assert call(shape(), kt=FAKE + 8) == E.ET_ERR_INVALID_ARG     # 16-byte alignment
    assert call(shape(), npl=FAKE) == E.ET_ERR_INVALID_ARG        # new_prefix_len must not alias prefix_len
    assert call(shape(feat_dim=4096)) == E.ET_ERR_INVALID_ARG     # features asked for, no buffers


def test_lm_head_argument_checks(lib):
    def call(M=10, H=4096, V=32000, ldo=32000, x=FAKE, w=FAKE, out=FAKE):
        return lib.et_lm_head(ctypes.byref(E.LmHeadShapeC(M, H, V, ldo)), x, w, out, None, None)
    assert call(M=0) == E.ET_ERR_INVALID_ARG
    assert call(M=65) == E.ET_ERR_INVALID_ARG          # at most 64 feature rows per call
    assert call(H=100) == E.ET_ERR_UNSUPPORTED         # whole 64-element k slices
    assert call(ldo=31999) == E.ET_ERR_INVALID_ARG
    assert call(x=FAKE + 8) == E.ET_ERR_INVALID_ARG    # TMA needs 16-byte aligned operands
    assert call(w=None) == E.ET_ERR_INVALID_ARG


def test_static_tree_sampled_argument_checks(lib):
    cfg = E.StaticCfgC(2, 32000, 61, 1, 1.0)
    need = lib.et_static_tree_workspace_size(ctypes.byref(cfg))
    assert need == (2 * 61 * 8 * 2 * 4 + 255) // 256 * 256  # (max, sum) per 4096-token chunk of every row, 256-byte rounded
    tree = E.TreeC(*([FAKE] * 10))
    call = lambda c=cfg, u=FAKE, ws=FAKE, wsb=need: lib.et_static_tree_sampled(
        ctypes.byref(c), FAKE, FAKE, 32000, FAKE, u, ctypes.byref(tree), None, ws, wsb, None)
    assert call(c=E.StaticCfgC(2, 32000, 61, 1, 0.0)) == E.ET_ERR_INVALID_ARG   # temperature must be > 0
    assert call(c=E.StaticCfgC(2, 40000, 61, 1, 1.0)) == E.ET_ERR_UNSUPPORTED   # one cluster covers 32768 tokens
    assert call(u=None) == E.ET_ERR_INVALID_ARG
    assert call(wsb=need - 1) == E.ET_ERR_WORKSPACE
    assert call(ws=FAKE + 64) == E.ET_ERR_WORKSPACE


def test_status_strings(lib):
    for s in range(6):
        assert E.status_string(s)
    assert E.status_string(99) == "unknown status"


def test_tree_build_argument_checks(lib):
    """et_tree_build: host-side rejections; without a GPU nothing launches."""
    cfg = E.TreeCfgC(1, 32000, 6, 10, 10, 60, 1.0)
    bad_cfg = E.TreeCfgC(1, 32000, 6, 10, 10, 5000, 1.0)  # n > C
    tree = E.TreeC(*([FAKE] * 10))
    ws_sz = lib.et_tree_workspace_size(ctypes.byref(cfg))

    def call(c=cfg, logits=FAKE, stride=32000, t=tree, mask=None, posids=None, prefix=None, ws=FAKE, wsb=ws_sz):
        return lib.et_tree_build(ctypes.byref(c), logits, stride, None, ctypes.byref(t), prefix, mask, posids, None,
                                 ws, wsb, None)
    assert call(c=bad_cfg) == E.ET_ERR_INVALID_ARG
    assert call(logits=None) == E.ET_ERR_INVALID_ARG
    assert call(stride=31999) == E.ET_ERR_INVALID_ARG
    assert call(logits=FAKE + 2) == E.ET_ERR_INVALID_ARG                 # rows must be 4-byte aligned
    assert call(mask=FAKE) == E.ET_ERR_INVALID_ARG                       # mask without posids / prefix_len
    assert call(mask=FAKE + 4, posids=FAKE, prefix=FAKE) == E.ET_ERR_INVALID_ARG  # mask not 8-byte aligned
    assert call(ws=None) == E.ET_ERR_WORKSPACE
    assert call(wsb=ws_sz - 1) == E.ET_ERR_WORKSPACE
    assert call(ws=FAKE + 16) == E.ET_ERR_WORKSPACE
    broken = E.TreeC(*([FAKE] * 6 + [None] + [FAKE] * 3))               # no flat_node array
    assert call(t=broken) == E.ET_ERR_INVALID_ARG
    # past one cluster (V > 32768) the call issues the per-layer launches: D + 1 (else 1 or 2)
    assert lib.et_tree_build_launches(ctypes.byref(E.TreeCfgC(1, 50000, 4, 4, 4, 16, 1.0))) == 5
    assert lib.et_tree_build_launches(ctypes.byref(bad_cfg)) == -1


def test_expand_kernel_switch_round_trips_and_refuses_unknown_values(lib):
    """et_set_expand_kernel is host state only: it returns the previous choice, and -1 (changing nothing)
    for a value that names no kernel.  et_tree_build_launches follows it for V > 32768 (always the
    per-layer launches) without touching a device."""
    prev = lib.et_set_expand_kernel(E.ET_EXPAND_CLUSTER)
    try:
        assert prev in (E.ET_EXPAND_AUTO, E.ET_EXPAND_CLUSTER, E.ET_EXPAND_BLOCK)
        assert lib.et_set_expand_kernel(E.ET_EXPAND_BLOCK) == E.ET_EXPAND_CLUSTER
        assert lib.et_set_expand_kernel(7) == -1
        assert lib.et_set_expand_kernel(-1) == -1
        assert lib.et_set_expand_kernel(E.ET_EXPAND_AUTO) == E.ET_EXPAND_BLOCK  # unchanged by the refusals
        wide = E.TreeCfgC(1, 50000, 4, 4, 4, 16, 1.0)
        for which in (E.ET_EXPAND_AUTO, E.ET_EXPAND_CLUSTER, E.ET_EXPAND_BLOCK):
            lib.et_set_expand_kernel(which)
            assert lib.et_tree_build_launches(ctypes.byref(wide)) == 5
        lib.et_set_expand_kernel(E.ET_EXPAND_BLOCK)  # one block per row: always the one work-queue launch
        assert lib.et_tree_build_launches(ctypes.byref(E.TreeCfgC(3, 1000, 4, 4, 4, 16, 1.0))) == 1
    finally:
        lib.et_set_expand_kernel(prev)
    with pytest.raises(ValueError):
        E.et_set_expand_kernel(9)


def test_attention_split_plan_short_prefixes(lib):
    """The tcgen05 plan gives each split about three K/V tiles at short
    prefixes (fewer and the split merge outweighs the shorter loop), and at
    long prefixes the SM count and the portable cluster size bound it."""
    def splits(**kw):
        s = dict(B=1, N=61, Hq=32, Hkv=32, d=128, dtype=E.ET_BF16, scale=0.088, max_prefix=1024,
                 kv_rows=32 * 1024, kv_head_stride=0, num_splits=0, impl=2)
        s.update(kw)
        return lib.et_tree_attention_splits(ctypes.byref(E.AttnShapeC(*s.values())))
    assert splits() == 6                                         # 16 prefix tiles + 1 tree tile: ceil(17 / 3)
    assert splits(max_prefix=512, kv_rows=32 * 512) == 3         # 9 tiles
    assert splits(max_prefix=128, kv_rows=32 * 128) == 1         # 3 tiles: at least two a split
    assert 6 <= splits(max_prefix=4096, kv_rows=32 * 4096) <= 8  # 65 tiles: the SM count and cluster size bound it
    assert splits(num_splits=5) == 5                             # an explicit count is kept
