"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

No GPU.  Each test checks the oracle against something other than itself:
closed forms, invariants the EAGLE-2 article states (connected kept tree,
shallower-first ties, ancestors-only attention), brute-force enumeration on
tiny vocabularies, library routines on special cases (torch's
scaled_dot_product_attention for a chain tree), and chi-square tests of the
losslessness the EAGLE blog (section 1.2) and abstract claim.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle as O
from oracle.eagle_tree_oracle import (_children, layer_widths, mask_bit, num_candidates)


# ---------------------------------------------------------------------------
# log-softmax / top-k / keys
# ---------------------------------------------------------------------------
def test_log_softmax_uniform_row_is_minus_log_v():
    for V in (1, 7, 1000, 32000):
        lp = O.log_softmax(np.full(V, 3.25, np.float32))
        assert np.allclose(lp, -math.log(V), rtol=0, atol=1e-13)


def test_log_softmax_two_tokens_closed_form():
    # p0 = 1 / (1 + e^{z1 - z0})
    for z0, z1 in [(0.0, 0.0), (1.5, -2.0), (-3.0, 7.0), (20.0, -20.0)]:
        lp = O.log_softmax(np.array([z0, z1], np.float32))
        assert abs(lp[0] - (-math.log1p(math.exp(z1 - z0)))) < 1e-13
        assert abs(lp[1] - (-math.log1p(math.exp(z0 - z1)))) < 1e-13


def test_log_softmax_normalised_and_matches_scipy():
    rng = np.random.default_rng(1)
    for V in (5, 1000, 32000):
        z = (rng.standard_normal(V) * 4).astype(np.float32)
        lp = O.log_softmax(z)
        assert abs(np.exp(lp).sum() - 1.0) < 1e-12
        assert np.max(np.abs(lp - scipy.special.log_softmax(z.astype(np.float64)))) < 1e-12
        assert np.all(lp <= 0)


def test_log_softmax_nonfinite_policy():
    lp = O.log_softmax(np.array([0.0, -np.inf, np.nan, 0.0], np.float32))
    assert lp[1] == -np.inf and lp[2] == -np.inf
    assert abs(lp[0] - math.log(0.5)) < 1e-15
    assert np.all(O.log_softmax(np.full(4, -np.inf, np.float32)) == -np.inf)


def _check_topk(z, k, ids):
    ids = list(ids)
    assert len(set(ids)) == len(ids) == k
    rest = [v for v in range(z.size) if v not in ids]
    zs = z.astype(np.float64)
    for a, b in zip(ids, ids[1:]):  # descending, ids ascending on ties
        assert zs[a] > zs[b] or (zs[a] == zs[b] and a < b)
    if rest:
        lo = zs[ids[-1]]
        for v in rest:
            assert zs[v] < lo or (zs[v] == lo and v > ids[-1])


def test_topk_properties_and_ties():
    rng = np.random.default_rng(2)
    for V, k in [(10, 3), (50, 10), (1000, 32), (7, 7)]:
        z = rng.integers(-3, 3, V).astype(np.float32)  # many ties
        _check_topk(z, k, O.topk_children(z, k))
        z = rng.standard_normal(V).astype(np.float32)
        _check_topk(z, k, O.topk_children(z, k))
    assert list(O.topk_children(np.zeros(100, np.float32), 5)) == [0, 1, 2, 3, 4]


def test_fixed_key_exact_and_monotone():
    assert O.fixed_key(0.0) == 0
    assert O.fixed_key(-1.0) == -(1 << 32)
    assert O.fixed_key(-0.5) == -(1 << 31)
    assert O.fixed_key(-np.inf) == O.KEY_MIN
    xs = np.sort(-np.abs(np.random.default_rng(3).standard_normal(2000)).astype(np.float32))
    ks = [O.fixed_key(x) for x in xs]
    assert all(a <= b for a, b in zip(ks, ks[1:]))
    # one unit is 2**-32 nats
    assert abs(O.fixed_key(np.float32(-3.1415927)) / 2.0 ** 32 - float(np.float32(-3.1415927))) < 2 ** -32


# ---------------------------------------------------------------------------
# tree geometry
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("D,k,m,C", [(4, 4, 4, 52), (6, 10, 10, 510), (8, 8, 8, 456), (3, 5, 25, 155)])
def test_candidate_counts(D, k, m, C):
    cfg = O.TreeCfg(B=1, V=100, depth=D, topk=k, m=m, n=1)
    assert num_candidates(cfg) == C


# ---------------------------------------------------------------------------
# expand / rerank against brute-force enumeration of every path
# ---------------------------------------------------------------------------
def _prefix_rows(V, D, seed):
    rng = np.random.default_rng(seed)
    rows = {}
    for L in range(D):
        for pre in itertools.product(range(V), repeat=L):
            rows[pre] = (rng.standard_normal(V) * 2).astype(np.float32)
    return rows


def _grow(cfg, rows):
    """Run the oracle layer by layer, feeding each frontier node its row."""
    tree = O.Tree.empty(cfg)

    def prefix(b, c):
        out = []
        while c >= 0:
            out.append(int(tree.tok[b, c]))
            c = int(tree.parent[b, c])
        return tuple(reversed(out))

    for layer in range(cfg.depth):
        nodes = [-1] if layer == 0 else [int(x) for x in tree.frontier[0, :O.expanded_count(cfg, layer)]]
        table = np.stack([rows[() if c < 0 else prefix(0, c)] for c in nodes])
        O.tree_expand(tree, layer, table, None)
    return tree, prefix


@pytest.mark.parametrize("V,D,n,seed", [(3, 3, 7, 0), (4, 3, 20, 1), (5, 2, 11, 2), (2, 3, 13, 3), (5, 3, 60, 4)])
def test_rerank_equals_bruteforce_topn(V, D, n, seed):
    rows = _prefix_rows(V, D, seed)
    cfg = O.TreeCfg(B=1, V=V, depth=D, topk=V, m=V ** (D - 1), n=n)
    tree, prefix = _grow(cfg, rows)
    O.tree_rerank(tree)
    # brute force: value of a path = product of softmax probabilities along it
    val = {}
    for L in range(1, D + 1):
        for path in itertools.product(range(V), repeat=L):
            v = 0.0
            for i in range(L):
                v += scipy.special.log_softmax(rows[path[:i]].astype(np.float64))[path[i]]
            val[path] = v
    best = sorted(val, key=lambda p: (-val[p], len(p)))[:n]
    kept = {prefix(0, int(c)) for c in tree.flat_node[0, 1:]}
    assert kept == set(best)
    # every kept node's value is the product of its ancestors' confidences
    for c in tree.flat_node[0, 1:]:
        assert abs(tree.key[0, c] / 2.0 ** 32 - val[prefix(0, int(c))]) < 1e-6 * D


def test_frontier_is_topm_of_newest_layer_bruteforce():
    V, D, m = 6, 3, 4
    rows = _prefix_rows(V, D, 9)
    cfg = O.TreeCfg(B=1, V=V, depth=D, topk=3, m=m, n=5)
    tree, prefix = _grow(cfg, rows)
    # layer-1 nodes: top-3 tokens of the root row; all expanded (3 <= m)
    l1 = sorted(range(V), key=lambda t: -rows[()][t])[:3]
    assert [prefix(0, c) for c in range(3)] == [(t,) for t in l1]
    # layer-2 frontier: the m best of the 9 layer-2 nodes by path value
    lsm = lambda pre: scipy.special.log_softmax(rows[pre].astype(np.float64))
    l2 = []
    for t1 in l1:
        for t2 in sorted(range(V), key=lambda t: -rows[(t1,)][t])[:3]:
            l2.append(((t1, t2), lsm(())[t1] + lsm((t1,))[t2]))
    want = {p for p, _ in sorted(l2, key=lambda x: -x[1])[:m]}
    # the frontier chosen after layer 2 (its expansion created layer 3)
    got = {prefix(0, int(tree.parent[0, c])) for c in range(O.layer_base(cfg, 3), num_candidates(cfg))}
    assert got == want


def _random_tree(V=64, D=6, k=10, m=10, n=60, B=2, seed=5, equal=False):
    cfg = O.TreeCfg(B=B, V=V, depth=D, topk=k, m=m, n=n)
    C = num_candidates(cfg)
    rng = np.random.default_rng(seed)
    if equal:
        table = np.zeros((B * (C + 1), V), np.float32)
    else:
        table = (rng.standard_normal((B * (C + 1), V)) * 2).astype(np.float32)
    rmap = (np.arange(B)[:, None] * (C + 1) + np.arange(C + 1)[None, :]).astype(np.int32)
    return cfg, O.build_tree(cfg, table, rmap)


def test_kept_tree_connected_and_ancestor_closed():
    for seed in range(4):
        cfg, tree = _random_tree(seed=seed)
        for b in range(cfg.B):
            kept = set(int(c) for c in tree.flat_node[b, 1:])
            assert len(kept) == cfg.n
            for c in kept:
                p = int(tree.parent[b, c])
                while p >= 0:
                    assert p in kept
                    p = int(tree.parent[b, p])
            fp = tree.flat_parent[b]
            assert fp[0] == -1 and all(0 <= fp[i] < i for i in range(1, cfg.N))
            assert all(tree.flat_depth[b, i] == tree.flat_depth[b, fp[i]] + 1 for i in range(1, cfg.N))


def test_keep_all_when_n_equals_c():
    cfg, tree = _random_tree(V=16, D=3, k=3, m=2, n=3 + 6 + 6)
    assert list(tree.flat_node[0, 1:]) == list(range(15))


def test_equal_values_keep_shallower_first():
    # every row uniform: a node's value is (1/V)^depth, so rerank keeps whole
    # shallow layers first and lower ids within a layer
    cfg, tree = _random_tree(V=32, D=4, k=4, m=4, n=11, equal=True)
    assert list(tree.flat_node[0, 1:]) == list(range(11))
    assert list(tree.flat_depth[0, 1:]) == [1] * 4 + [2] * 7
    # and the frontier of each layer is its lowest-id nodes
    assert list(tree.frontier[0]) == [O.layer_base(cfg, 3) + i for i in range(4)]


def test_child_value_never_exceeds_parent():
    cfg, tree = _random_tree(seed=11)
    for b in range(cfg.B):
        for c in range(num_candidates(cfg)):
            p = tree.parent[b, c]
            if p >= 0:
                assert tree.key[b, c] <= tree.key[b, p]


# ---------------------------------------------------------------------------
# mask / position ids
# ---------------------------------------------------------------------------
def _closure(fp):
    N = fp.size
    A = np.eye(N, dtype=bool)
    for i in range(1, N):
        A[i, fp[i]] = True
    for kk in range(N):  # Floyd-Warshall transitive closure
        A = A | (A[:, [kk]] & A[[kk], :])
    return A


def test_mask_is_closure_of_parent_edges():
    cfg, tree = _random_tree(seed=21, n=100, B=1)
    mask, pos = O.mask_posids(tree.flat_parent, tree.flat_depth, np.array([777]))
    A = _closure(tree.flat_parent[0])
    got = np.array([[mask_bit(mask, 0, i, j) for j in range(cfg.N)] for i in range(cfg.N)])
    assert (got == A).all()
    assert mask.shape == (1, 101, 2)
    # no bit beyond column N-1
    assert int(mask[0, :, 1].max()) >> (cfg.N - 64) == 0
    assert (pos[0] == 777 + tree.flat_depth[0]).all()


def test_mask_chain_and_star():
    N = 70
    chain = np.arange(-1, N - 1, dtype=np.int32)[None]
    m, pos = O.mask_posids(chain, np.arange(N, dtype=np.int32)[None], np.array([100]))
    got = np.array([[mask_bit(m, 0, i, j) for j in range(N)] for i in range(N)])
    assert (got == np.tril(np.ones((N, N), bool))).all()
    assert list(pos[0]) == list(range(100, 100 + N))  # ordinary decoding positions
    star = np.zeros((1, N), np.int32)
    star[0, 0] = -1
    m, _ = O.mask_posids(star, np.minimum(np.arange(N), 1)[None].astype(np.int32), np.array([0]))
    got = np.array([[mask_bit(m, 0, i, j) for j in range(N)] for i in range(N)])
    want = np.eye(N, dtype=bool)
    want[:, 0] = True
    assert (got == want).all()


def test_mask_golden_it_is_a_has(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "mask_it_is_a_has.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                r, tok, par, vis = line.split()
                rows.append((int(r), tok, int(par), [int(x) for x in vis.split(",")]))
    fp = np.array([[r[2] for r in rows]], np.int32)
    depth = np.zeros_like(fp)
    for i in range(1, fp.shape[1]):
        depth[0, i] = depth[0, fp[0, i]] + 1
    mask, _ = O.mask_posids(fp, depth, np.array([0]))
    for r, tok, _, vis in rows:
        assert [j for j in range(len(rows)) if mask_bit(mask, 0, r, j)] == vis, tok


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def _attn_inputs(B, N, Hq, Hkv, d, L, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, N, Hq, d))
    kp = [rng.standard_normal((Hkv, L, d)) for _ in range(B)]
    vp = [rng.standard_normal((Hkv, L, d)) for _ in range(B)]
    kt = rng.standard_normal((B, N, Hkv, d))
    vt = rng.standard_normal((B, N, Hkv, d))
    return q, kp, vp, kt, vt


def _sdpa_chain(q, kp, vp, kt, vt, scale):
    """Chain tree == ordinary causal attention over [prefix; tree]."""
    B, N, Hq, d = q.shape
    Hkv = kt.shape[2]
    G = Hq // Hkv
    outs = []
    for b in range(B):
        L = kp[b].shape[1]
        K = np.concatenate([kp[b], kt[b].transpose(1, 0, 2)], axis=1)  # [Hkv, L+N, d]
        Vv = np.concatenate([vp[b], vt[b].transpose(1, 0, 2)], axis=1)
        K = np.repeat(K, G, axis=0)
        Vv = np.repeat(Vv, G, axis=0)
        qq = np.zeros((Hq, L + N, d))
        qq[:, L:] = q[b].transpose(1, 0, 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qq)[None], torch.from_numpy(K)[None], torch.from_numpy(Vv)[None],
            is_causal=True, scale=scale)[0].numpy()
        outs.append(o[:, L:].transpose(1, 0, 2))
    return np.stack(outs)


@pytest.mark.parametrize("Hq,Hkv,N,L", [(4, 4, 9, 33), (8, 2, 17, 64), (2, 1, 1, 5)])
def test_chain_tree_attention_is_causal_attention(Hq, Hkv, N, L):
    d = 16
    q, kp, vp, kt, vt = _attn_inputs(2, N, Hq, Hkv, d, L, 7)
    chain = np.tile(np.arange(-1, N - 1, dtype=np.int32), (2, 1))
    mask, _ = O.mask_posids(chain, np.tile(np.arange(N, dtype=np.int32), (2, 1)), np.array([L, L]))
    scale = 1 / math.sqrt(d)
    out, lse = O.tree_attention(q, kp, vp, kt, vt, mask, scale)
    ref = _sdpa_chain(q, kp, vp, kt, vt, scale)
    assert np.max(np.abs(out - ref)) < 1e-12
    # log-sum-exp of the scaled scores: check against scipy on one row
    b, h, i = 1, Hq - 1, N - 1
    s = scale * np.concatenate([kp[b][h // (Hq // Hkv)], kt[b, :i + 1, h // (Hq // Hkv)]]) @ q[b, i, h]
    assert abs(lse[b, h, i] - scipy.special.logsumexp(s)) < 1e-12


def test_attention_ignores_non_ancestors():
    cfg, tree = _random_tree(V=16, D=3, k=3, m=2, n=10, B=1, seed=4)
    mask, _ = O.mask_posids(tree.flat_parent, tree.flat_depth, np.array([20]))
    q, kp, vp, kt, vt = _attn_inputs(1, cfg.N, 2, 2, 8, 20, 8)
    out, _ = O.tree_attention(q, kp, vp, kt, vt, mask, 0.3)
    for j in range(cfg.N):
        kt2, vt2 = kt.copy(), vt.copy()
        kt2[0, j] += 5.0
        vt2[0, j] -= 3.0
        out2, _ = O.tree_attention(q, kp, vp, kt2, vt2, mask, 0.3)
        for i in range(cfg.N):
            same = np.allclose(out[0, i], out2[0, i], atol=0, rtol=0)
            assert same == (not mask_bit(mask, 0, i, j))


def test_attention_root_only_is_decode_attention():
    q, kp, vp, kt, vt = _attn_inputs(1, 1, 3, 3, 32, 50, 9)
    mask = np.ones((1, 1, 1), np.uint64)
    out, _ = O.tree_attention(q, kp, vp, kt, vt, mask, 0.2)
    K = torch.from_numpy(np.concatenate([kp[0], kt[0].transpose(1, 0, 2)], axis=1))
    Vv = torch.from_numpy(np.concatenate([vp[0], vt[0].transpose(1, 0, 2)], axis=1))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[0].transpose(1, 0, 2))[:, :, :], K, Vv, scale=0.2).numpy()
    assert np.max(np.abs(out[0, 0] - ref[:, 0])) < 1e-12


def test_attention_prefix_permutation_invariant():
    q, kp, vp, kt, vt = _attn_inputs(1, 5, 2, 2, 8, 40, 10)
    chain = np.arange(-1, 4, dtype=np.int32)[None]
    mask, _ = O.mask_posids(chain, np.arange(5, dtype=np.int32)[None], np.array([40]))
    perm = np.random.default_rng(0).permutation(40)
    a, _ = O.tree_attention(q, kp, vp, kt, vt, mask, 0.35)
    b, _ = O.tree_attention(q, [kp[0][:, perm]], [vp[0][:, perm]], kt, vt, mask, 0.35)
    assert np.max(np.abs(a - b)) < 1e-12


# ---------------------------------------------------------------------------
# greedy acceptance on hand-built trees
# ---------------------------------------------------------------------------
def _hand_tree():
    # flat rows: 0 root; 1,2,3 children of root (tokens 5,6,7); 4,5 children of
    # row 1 (tokens 1,2); 6 child of row 2 (token 3); 7 child of row 4 (token 0)
    tok = np.array([[9, 5, 6, 7, 1, 2, 3, 0]], np.int32)
    par = np.array([[-1, 0, 0, 0, 1, 1, 2, 4]], np.int32)
    node = np.arange(-1, 7, dtype=np.int32)[None]
    return tok, par, node


def _onehot_rows(argmaxes, V=10):
    t = np.full((len(argmaxes), V), -1.0, np.float32)
    for i, a in enumerate(argmaxes):
        t[i, a] = 4.0
    return t


@pytest.mark.parametrize("argmaxes,acc,path,toks", [
    # root prefers 5 (row 1), row 1 prefers 1 (row 4), row 4 prefers 0 (row 7), row 7 prefers 8 -> bonus
    ([5, 1, 3, 4, 0, 4, 4, 8], 3, [0, 1, 4, 7], [5, 1, 0, 8]),
    # root prefers 6 (row 2), row 2 prefers 9: not a child -> bonus 9
    ([6, 1, 9, 4, 0, 4, 4, 8], 1, [0, 2], [6, 9]),
    # root prefers 4: no child has it -> nothing accepted, bonus 4
    ([4, 1, 3, 4, 0, 4, 4, 8], 0, [0], [4]),
    # root prefers 7 (row 3, a leaf) -> accepted, bonus = argmax of row 3
    ([7, 1, 3, 2, 0, 4, 4, 8], 1, [0, 3], [7, 2]),
])
def test_greedy_walk_hand_tree(argmaxes, acc, path, toks):
    tok, par, node = _hand_tree()
    cfg = O.TreeCfg(B=1, V=10, depth=3, topk=3, m=3, n=7)
    r = O.verify_accept(cfg, O.GREEDY, tok, par, node, _onehot_rows(argmaxes), None)
    assert r.accept_len[0] == acc
    assert list(r.path[0, :acc + 1]) == path and (r.path[0, acc + 1:] == -1).all()
    assert list(r.tokens[0, :acc + 1]) == toks


def test_greedy_argmax_tie_goes_to_lower_id():
    tok, par, node = _hand_tree()
    cfg = O.TreeCfg(B=1, V=10, depth=3, topk=3, m=3, n=7)
    rows = _onehot_rows([5, 1, 3, 4, 0, 4, 4, 8])
    rows[0, 6] = 4.0  # root: tie between 5 and 6 -> 5
    r = O.verify_accept(cfg, O.GREEDY, tok, par, node, rows, None)
    assert r.tokens[0, 0] == 5


# ---------------------------------------------------------------------------
# stochastic acceptance: losslessness (chi-square) and special cases
# ---------------------------------------------------------------------------
def _chi2_ok(counts, probs, alpha=1e-3):
    counts = np.asarray(counts, float)
    exp = np.asarray(probs) * counts.sum()
    keep = exp > 0
    assert counts[~keep].sum() == 0
    return scipy.stats.chisquare(counts[keep], exp[keep]).pvalue > alpha


def _stoch_tree(V, rng):
    # root with 3 children (distinct tokens), each child with 2 children
    kids = rng.choice(V, 3, replace=False)
    tok = [int(rng.integers(V))] + [int(x) for x in kids]
    par = [-1, 0, 0, 0]
    for c in (1, 2, 3):
        for t in rng.choice(V, 2, replace=False):
            tok.append(int(t))
            par.append(c)
    return np.array([tok], np.int32), np.array([par], np.int32)


def _star(toks):
    k = len(toks)
    return (np.array([[0] + list(toks)], np.int32), np.array([[-1] + [0] * k], np.int32),
            np.arange(-1, k, dtype=np.int32)[None])


def test_stoch_point_hand_example():
    """p = (0.5, 0.3, 0.2), children tokens 0 then 1.  u = 0.6 rejects token 0
    (ratio 0.5); token 1 then has ratio 0.3 / (1 - 0.5) = 0.6, so u = 0.55
    accepts it and u = 0.65 rejects it, after which only token 2 is left for
    the bonus draw, whatever its uniform."""
    z = np.log(np.array([5.0, 3.0, 2.0])).astype(np.float32)
    tok, par, node = _star([0, 1])
    cfg = O.TreeCfg(B=1, V=3, depth=1, topk=2, m=1, n=2)
    rows = np.stack([z] * 3)
    r = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, rows, None,
                        uniforms=np.array([[0.3, 0.6, 0.55]], np.float32))
    assert r.accept_len[0] == 1 and list(r.path[0]) == [0, 2] and r.tokens[0, 0] == 1
    for u0 in (0.01, 0.5, 0.99):
        r = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, rows, None,
                            uniforms=np.array([[u0, 0.6, 0.65]], np.float32))
        assert r.accept_len[0] == 0 and list(r.tokens[0]) == [2, -1]
    # u = 0.45 accepts token 0 at once
    r = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, rows, None,
                        uniforms=np.array([[0.3, 0.45, 0.0]], np.float32))
    assert list(r.path[0]) == [0, 1] and r.tokens[0, 0] == 0


def test_stoch_point_repeated_token_has_no_residual_mass():
    """Once a sibling with token x is rejected, the residual holds no mass at
    x, so a later sibling with the same token is rejected even with u = 0, and
    the rejected mass is counted once: the third child (token 1) has ratio
    0.3 / 0.5."""
    z = np.log(np.array([5.0, 3.0, 2.0])).astype(np.float32)
    tok, par, node = _star([0, 0, 1])
    cfg = O.TreeCfg(B=1, V=3, depth=1, topk=3, m=1, n=3)
    rows = np.stack([z] * 4)
    r = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, rows, None,
                        uniforms=np.array([[0.5, 0.6, 0.0, 0.59]], np.float32))
    assert list(r.path[0]) == [0, 3] and r.tokens[0, 0] == 1
    r = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, rows, None,
                        uniforms=np.array([[0.5, 0.6, 0.0, 0.61]], np.float32))
    assert r.accept_len[0] == 0 and r.tokens[0, 0] == 2


def test_draftq_residual_closed_form():
    """The acceptance kernel evaluates the draft-q residual as max(p - c q, 0) / F
    with (c, F) = (0, 1), then c <- c + F and F <- sum max(p - c q, 0) per
    rejection (kept when that sum is 0); the rule iterates r <- norm(max(r - q, 0)).
    The two agree elementwise, and the oracle's bonus token after every child
    is rejected is the closed form's inverse CDF."""
    rng = np.random.default_rng(17)
    for trial in range(20):
        V = int(rng.integers(2, 40))
        p = scipy.special.softmax(rng.standard_normal(V) * rng.uniform(0.3, 3.0))
        q = scipy.special.softmax(rng.standard_normal(V) * rng.uniform(0.3, 3.0))
        if trial == 0:
            q = p.copy()  # every excess is 0: r stays p
        r, c, F = p.copy(), 0.0, 1.0
        for _ in range(12):
            d = np.maximum(r - q, 0.0)
            if d.sum() > 0.0:
                r = d / d.sum()
            c1 = c + F
            F1 = np.maximum(p - c1 * q, 0.0).sum()
            if F1 > 0.0:
                c, F = c1, F1
            assert np.abs(np.maximum(p - c * q, 0.0) / F - r).max() <= 1e-12
    V, k = 12, 5
    pz = (rng.standard_normal(V) * 1.5).astype(np.float32)
    qz = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p = O.softmax_t(pz, 1.0)
    q = O.softmax_t(qz, 1.0)
    c, F = 0.0, 1.0
    for _ in range(k):
        F1 = np.maximum(p - (c + F) * q, 0.0).sum()
        if F1 > 0.0:
            c, F = c + F, F1
    w = np.maximum(p - c * q, 0.0)
    cfg = O.TreeCfg(B=1, V=V, depth=1, topk=k, m=1, n=k)
    par = np.array([[-1] + [0] * k], np.int32)
    node = np.arange(-1, k, dtype=np.int32)[None]
    tok = np.array([[0] + list(rng.choice(V, k, p=q))], np.int32)
    seen = 0
    for u0 in np.linspace(0.01, 0.99, 25):
        us = np.array([[u0] + [1.0] * k], np.float32)  # u = 1 rejects every child
        res = O.verify_accept(cfg, O.STOCH_DRAFTQ, tok, par, node, np.stack([pz] * (k + 1)), None, uniforms=us,
                              draft_table=np.stack([qz] * (k + 1)))
        if res.near_ties:
            continue
        want = int(np.nonzero(np.cumsum(w) > float(us[0, 0]) * w.sum())[0][0])
        assert res.accept_len[0] == 0 and res.tokens[0, 0] == want
        seen += 1
    assert seen >= 20


def test_stoch_draftq_hand_example():
    """p = (0.5, 0.3, 0.2), q = (0.7, 0.2, 0.1), children tokens 0 then 1.
    Token 0 has ratio 0.5 / 0.7, so u = 0.8 rejects it; the residual
    norm(max(p - q, 0)) is (0, 0.5, 0.5), so token 1 has ratio
    min(1, 0.5 / 0.2) = 1 and is accepted even with u = 0.95."""
    z = np.log(np.array([0.5, 0.3, 0.2])).astype(np.float32)
    zq = np.log(np.array([0.7, 0.2, 0.1])).astype(np.float32)
    tok = np.array([[0, 0, 1]], np.int32)
    par = np.array([[-1, 0, 0]], np.int32)
    node = np.arange(-1, 2, dtype=np.int32)[None]
    cfg = O.TreeCfg(B=1, V=3, depth=1, topk=2, m=1, n=2)
    r = O.verify_accept(cfg, O.STOCH_DRAFTQ, tok, par, node, np.stack([z] * 3), None,
                        uniforms=np.array([[0.5, 0.8, 0.95]], np.float32), draft_table=np.stack([zq] * 3))
    assert list(r.path[0]) == [0, 2] and r.tokens[0, 0] == 1
    r = O.verify_accept(cfg, O.STOCH_DRAFTQ, tok, par, node, np.stack([z] * 3), None,
                        uniforms=np.array([[0.5, 0.7, 0.95]], np.float32), draft_table=np.stack([zq] * 3))
    assert list(r.path[0]) == [0, 1] and r.tokens[0, 0] == 0


def test_stoch_special_cases():
    tok, par, node = _hand_tree()
    cfg = O.TreeCfg(B=1, V=10, depth=3, topk=3, m=3, n=7)
    # one-hot target: stochastic acceptance is deterministic and equals greedy
    rows = np.full((8, 10), -np.inf, np.float32)
    for i, a in enumerate([5, 1, 3, 4, 0, 4, 4, 8]):
        rows[i, a] = 0.0
    g = O.verify_accept(cfg, O.GREEDY, tok, par, node, rows, None)
    for u in (0.0, 0.3, 0.999):
        s = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, rows, None, uniforms=np.full((1, 8), u, np.float32))
        assert (s.tokens == g.tokens).all() and (s.path == g.path).all()
    # draft == target in the q-variant: the first child is always accepted
    rng = np.random.default_rng(4)
    z = rng.standard_normal((8, 10)).astype(np.float32)
    s = O.verify_accept(cfg, O.STOCH_DRAFTQ, tok, par, node, z, None,
                        uniforms=np.full((1, 8), 0.999, np.float32), draft_table=z)
    assert list(s.path[0]) == [0, 1, 4, 7]


def test_uniform_slot_usage():
    # slot c decides node c, slot 0 draws the bonus: changing any other slot
    # (those of untested nodes) must not change the outcome
    tok, par, node = _hand_tree()
    cfg = O.TreeCfg(B=1, V=10, depth=3, topk=3, m=3, n=7)
    rng = np.random.default_rng(5)
    z = rng.standard_normal((8, 10)).astype(np.float32)
    u = rng.random((1, 8)).astype(np.float32)
    base = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, z, None, uniforms=u)
    tested = set()
    cur_path = list(base.path[0, :base.accept_len[0] + 1])
    ch = _children(par[0])
    for p in cur_path:
        for c in ch[p]:
            tested.add(c)
            if c in cur_path:
                break
    for s in range(1, 8):
        if s in tested:
            continue
        u2 = u.copy()
        u2[0, s] = 1.0 - u2[0, s]
        r = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, z, None, uniforms=u2)
        assert (r.tokens == base.tokens).all()


# ---------------------------------------------------------------------------
# KV commit after acceptance: the root row and the accepted rows, in path
# order, land at prefix_len.. of every head; values typed out by hand
# ---------------------------------------------------------------------------
def test_kv_commit_hand_example():
    B, N, Hkv = 2, 4, 2
    k_tree = np.zeros((B, N, Hkv, 1), np.float32)
    for b in range(B):
        for r in range(N):
            for g in range(Hkv):
                k_tree[b, r, g, 0] = 100 * b + 10 * r + g
    v_tree = -k_tree
    path = np.array([[0, 2, 3], [0, -1, -1]], np.int32)
    alen = np.array([2, 0], np.int32)
    feats = np.array([[[0.], [1.], [2.], [3.]], [[1000.], [1001.], [1002.], [1003.]]], np.float32)
    cache = np.full((32, 1), 7.0, np.float32)
    kc, vc, new_len, fo = O.kv_commit(k_tree, v_tree, alen, path, cache, cache, np.array([0, 16]),
                                      np.array([3, 5], np.int32), 8, feats)
    want = np.full(32, 7.0, np.float32)
    want[[3, 4, 5]] = [0, 20, 30]      # sequence 0, head 0: rows 0, 2, 3 at positions 3, 4, 5
    want[[11, 12, 13]] = [1, 21, 31]   # sequence 0, head 1 (8 rows further)
    want[21] = 100                     # sequence 1 (base row 16), head 0: the root at position 5
    want[29] = 101                     # sequence 1, head 1
    np.testing.assert_array_equal(kc[:, 0], want)
    np.testing.assert_array_equal(vc[:, 0], np.where(want == 7.0, 7.0, -want))
    assert list(new_len) == [6, 6]
    np.testing.assert_array_equal(fo[:, :, 0], [[0, 2, 3], [1000, 0, 0]])
    assert cache[3, 0] == 7.0  # inputs untouched


# ---------------------------------------------------------------------------
# static draft tree: each row's token is the rank-th best token at its parent
# ---------------------------------------------------------------------------
def test_static_tree_hand_example():
    # root row 0 -> rows 1, 2 (ranks 0, 1); row 1 -> row 3 (rank 0); row 2 -> row 4 (rank 2)
    parent = np.array([-1, 0, 0, 1, 2], np.int32)
    rank = np.array([-1, 0, 1, 0, 2], np.int32)
    table = np.array([[0.5, 3.0, -1.0, 3.0, 2.0, 0.0],     # root: order 1, 3 (tie -> lower id), 4, 0, 5, 2
                      [9.0, 0.0, 0.0, 0.0, 0.0, 0.0],      # row 1: best 0
                      [1.0, 2.0, 3.0, 4.0, 5.0, 6.0],      # row 2: order 5, 4, 3, ...
                      [0.0] * 6, [0.0] * 6], np.float32)
    tok, fpar, fdep, node = O.static_tree(parent, rank, table, np.array([[0, 1, 2, 3, 4]], np.int32),
                                          np.array([42], np.int32))
    assert tok.tolist() == [[42, 1, 3, 0, 3]]
    assert fpar.tolist() == [[-1, 0, 0, 1, 2]]
    assert fdep.tolist() == [[0, 1, 1, 2, 2]]
    assert node.tolist() == [[-1, 0, 1, 2, 3]]


def test_static_tree_chain_is_greedy_argmax():
    rng = np.random.default_rng(5)
    table = rng.standard_normal((6, 50)).astype(np.float32)
    parent = np.arange(-1, 5, dtype=np.int32)
    rank = np.zeros(6, np.int32)
    tok, _, fdep, _ = O.static_tree(parent, rank, table, np.arange(6, dtype=np.int32)[None], np.array([0]))
    assert tok[0, 1:].tolist() == [int(np.argmax(table[i])) for i in range(5)]
    assert fdep[0].tolist() == [0, 1, 2, 3, 4, 5]


# ---------------------------------------------------------------------------
# draft LM head: logits = W x, pinned on integers (exact in any precision)
# ---------------------------------------------------------------------------
def test_lm_head_integer_example():
    x = np.array([[1, 2, 3], [0, -1, 4]], np.float32)
    w = np.array([[1, 0, 0], [0, 1, 0], [1, 1, 1], [2, -1, 0.5]], np.float32)
    np.testing.assert_array_equal(O.lm_head_logits(x, w), [[1, 2, 6, 1.5], [0, -1, 3, 3]])
    b = O.lm_head_error_bound(x, w)
    # H * 2^-24 * sum |x w|: row 0 . w row 0 has sum |x w| = 1; row 1 . w row 0 has none
    np.testing.assert_allclose(b[0, 0], 3 * 2.0 ** -24)
    assert b[1, 0] == 0.0
    np.testing.assert_allclose(b[0, 2], 3 * 2.0 ** -24 * 6)


# ---------------------------------------------------------------------------
# temperature: p(z / T), closed forms on two tokens
# ---------------------------------------------------------------------------
def test_softmax_temperature_closed_form():
    z = np.array([0.0, np.log(3.0)], np.float32)
    l3 = float(np.float32(np.log(3.0)))  # the logit as stored
    np.testing.assert_allclose(O.softmax_t(z, 2.0)[1], np.exp(l3 / 2) / (1 + np.exp(l3 / 2)), rtol=1e-12)
    np.testing.assert_allclose(O.softmax_t(z, 0.5)[1], np.exp(2 * l3) / (1 + np.exp(2 * l3)), rtol=1e-12)
    np.testing.assert_allclose(O.softmax_t(z, 0.5)[1], 0.9, atol=1e-6)


def test_stoch_acceptance_depends_on_temperature():
    # root row p = softmax([0, ln 3] / T): token 1 has p = 0.9 at T = 1/2 and 0.75 at T = 1;
    # its one child (token 1) meets the uniform 0.85
    tok = np.array([[7, 1]], np.int32)
    par = np.array([[-1, 0]], np.int32)
    node = np.array([[-1, 0]], np.int32)
    table = np.array([[0.0, np.log(3.0)], [0.0, 0.0]], np.float32)
    u = np.array([[0.5, 0.85]], np.float32)
    hot = O.verify_accept(O.TreeCfg(B=1, V=2, depth=1, topk=1, m=1, n=1, temperature=0.5), O.STOCH_POINT,
                          tok, par, node, table, None, uniforms=u)
    cold = O.verify_accept(O.TreeCfg(B=1, V=2, depth=1, topk=1, m=1, n=1, temperature=1.0), O.STOCH_POINT,
                           tok, par, node, table, None, uniforms=u)
    assert hot.accept_len[0] == 1 and hot.tokens[0, 0] == 1
    assert cold.accept_len[0] == 0 and cold.tokens[0, 0] == 0  # rejected: the residual keeps token 0 only


def test_static_tree_sampled_inverse_cdf_by_hand():
    # q = softmax([0, ln 3, 0]) = (0.2, 0.6, 0.2): uniforms 0.1 / 0.5 / 0.9 pick tokens 0 / 1 / 2
    parent = np.array([-1, 0, 0, 0], np.int32)
    table = np.array([[0.0, np.log(3.0), 0.0]] + [[0.0, 0.0, 0.0]] * 3, np.float32)
    u = np.array([[0.0, 0.1, 0.5, 0.9]], np.float32)
    tok, fpar, fdep, node, gaps = O.static_tree_sampled(parent, table, np.array([[0, 1, 2, 3]], np.int32), u, 1.0,
                                                        np.array([9], np.int32))
    assert tok.tolist() == [[9, 0, 1, 2]]
    assert fdep.tolist() == [[0, 1, 1, 1]]
    np.testing.assert_allclose(gaps[0, 1:], [0.1, 0.3, 0.1], atol=1e-6)  # CDF steps at 0.2, 0.8, 1.0
    # temperature 1/2 sharpens q to (0.1/1.1... ): (1, 9, 1) / 11 -> u = 0.5 still picks token 1, u = 0.95 token 2
    tok2, *_ = O.static_tree_sampled(parent, table, np.array([[0, 1, 2, 3]], np.int32),
                                     np.array([[0, 0.05, 0.5, 0.95]], np.float32), 0.5, np.array([9], np.int32))
    assert tok2.tolist() == [[9, 0, 1, 2]]


# ---------------------------------------------------------------------------
# losslessness of the stochastic walks (chi-square, 2e5 trials each; last in
# the file so that a cheaper pin stops a mutated run first)
# ---------------------------------------------------------------------------
def test_stoch_point_is_lossless_chi_square():
    V, trials = 8, 200000
    rng = np.random.default_rng(123)
    tok, par = _stoch_tree(V, rng)
    N = tok.shape[1]
    logits = (rng.standard_normal((N, V)) * 1.2).astype(np.float32)
    P = np.stack([scipy.special.softmax(logits[i].astype(np.float64)) for i in range(N)])
    cfg = O.TreeCfg(B=1, V=V, depth=2, topk=3, m=3, n=N - 1)
    node = np.arange(-1, N - 1, dtype=np.int32)[None]
    first = np.zeros(V)
    second = {c: np.zeros(V) for c in (1, 2, 3)}
    u_all = rng.random((trials, N)).astype(np.float32)
    for t in range(trials):
        r = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, logits, None, uniforms=u_all[t][None])
        first[r.tokens[0, 0]] += 1
        if r.accept_len[0] >= 1:
            second[int(r.path[0, 1])][r.tokens[0, 1]] += 1
    assert _chi2_ok(first, P[0])
    for c in (1, 2, 3):
        assert second[c].sum() > 1000
        assert _chi2_ok(second[c], P[c])


def test_stoch_point_lossless_with_repeated_tokens_chi_square():
    """Children with repeated tokens (as i.i.d. draws give) keep the first
    emitted token distributed as p."""
    V, trials = 6, 200000
    rng = np.random.default_rng(31)
    z = (rng.standard_normal(V) * 1.4).astype(np.float32)
    p = scipy.special.softmax(z.astype(np.float64))
    top = int(np.argmax(p))
    toks = [top, (top + 1) % V, top, (top + 1) % V, top]
    tok, par, node = _star(toks)
    cfg = O.TreeCfg(B=1, V=V, depth=1, topk=len(toks), m=1, n=len(toks))
    rows = np.stack([z] * (len(toks) + 1))
    first = np.zeros(V)
    us = rng.random((trials, len(toks) + 1)).astype(np.float32)
    for t in range(trials):
        r = O.verify_accept(cfg, O.STOCH_POINT, tok, par, node, rows, None, uniforms=us[t][None])
        first[r.tokens[0, 0]] += 1
    assert _chi2_ok(first, p)


def test_stoch_draftq_single_child_is_speculative_sampling():
    V, trials = 8, 200000
    rng = np.random.default_rng(7)
    pz = (rng.standard_normal(V) * 1.5).astype(np.float32)
    qz = (rng.standard_normal(V) * 1.5).astype(np.float32)
    p = scipy.special.softmax(pz.astype(np.float64))
    q = scipy.special.softmax(qz.astype(np.float64))
    cfg = O.TreeCfg(B=1, V=V, depth=1, topk=1, m=1, n=1)
    first = np.zeros(V)
    accepted = 0
    par = np.array([[-1, 0]], np.int32)
    node = np.array([[-1, 0]], np.int32)
    xs = rng.choice(V, trials, p=q)
    us = rng.random((trials, 2)).astype(np.float32)
    for t in range(trials):
        tok = np.array([[0, xs[t]]], np.int32)
        r = O.verify_accept(cfg, O.STOCH_DRAFTQ, tok, par, node, np.stack([pz, pz]), None,
                            uniforms=us[t][None], draft_table=np.stack([qz, qz]))
        first[r.tokens[0, 0]] += 1
        accepted += int(r.accept_len[0])
    assert _chi2_ok(first, p)
    # acceptance rate of speculative sampling = sum_x min(p(x), q(x))
    rate = np.minimum(p, q).sum()
    assert abs(accepted / trials - rate) < 4 * math.sqrt(rate * (1 - rate) / trials)


def test_stoch_draftq_iid_children_lossless():
    V, k, trials = 6, 3, 200000
    rng = np.random.default_rng(99)
    pz = (rng.standard_normal(V) * 1.3).astype(np.float32)
    qz = (rng.standard_normal(V) * 1.3).astype(np.float32)
    p = scipy.special.softmax(pz.astype(np.float64))
    q = scipy.special.softmax(qz.astype(np.float64))
    cfg = O.TreeCfg(B=1, V=V, depth=1, topk=k, m=1, n=k)
    par = np.array([[-1] + [0] * k], np.int32)
    node = np.arange(-1, k, dtype=np.int32)[None]
    rows = np.stack([pz] * (k + 1))
    drows = np.stack([qz] * (k + 1))
    first = np.zeros(V)
    xs = rng.choice(V, (trials, k), p=q)
    us = rng.random((trials, k + 1)).astype(np.float32)
    for t in range(trials):
        tok = np.array([[0] + list(xs[t])], np.int32)
        r = O.verify_accept(cfg, O.STOCH_DRAFTQ, tok, par, node, rows, None, uniforms=us[t][None],
                            draft_table=drows)
        first[r.tokens[0, 0]] += 1
    assert _chi2_ok(first, p)
