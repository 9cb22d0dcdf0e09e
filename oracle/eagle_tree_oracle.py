"""CPU oracle for one EAGLE-2 draft-tree verification step.

TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously-correct
restatement of what the step computes, in float64 and Python integers, used to
check the CUDA path.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its CPU-baseline leg and ``--impl reference`` arm) may import it.
The CUDA library never calls it and it never calls the CUDA library; the two
share no code (the seeded input generators live in their own module).

Sources (web pages on EAGLE / EAGLE-2):

* [EAGLE-2 article] "Up to 5x lossless acceleration: EAGLE-2 lets an RTX 3060
  generate faster than an A100" (sbmmt.com, Japanese body):
  - expansion phase: the m highest-value nodes of the newest layer are fed to
    the draft model and its outputs become their children;
  - node value: the product of the draft confidences of the node and all its
    ancestors (a token is only accepted if all its ancestors are);
  - reranking phase: sort the whole tree by value, keep the first n nodes;
    on equal value the shallower node is kept first, so the kept tree stays
    connected; the kept nodes are flattened to one dimension;
  - attention mask: each token sees only its ancestors (the "a" sees "It" and
    "is" but not "has" example); position encoding adjusted to agree with
    ordinary autoregressive decoding.
* [EAGLE blog] "大模型系列——论文解读：eagle/eagle2" (CSDN), section 1.1
  (one target forward verifies a whole draft and keeps the output
  distribution identical) and section 1.2 (lossless under greedy and
  non-greedy decoding).
* [EAGLE abstract] "EAGLE: Speculative Sampling Requires Rethinking Feature
  Uncertainty" (chatpaper.ai), abstract: the acceleration is lossless.

Readings where the pages are silent (each one is listed in the design notes):

* confidence = draft softmax probability at temperature 1, as a log-prob;
* top-k children ranked by the fp32 draft logit, ties -> lower token id;
* value kept in the log domain as an integer fixed-point key
  ``key(child) = key(parent) + rint(lp32 * 2**32)`` where ``lp32`` is the
  child's log-prob rounded to fp32 (the kernel's precision, so both sides rank
  the same numbers); saturates at ``KEY_MIN``;
* node ids: layer-major; layer 1 ids are 0..k-1 in rank order, a layer's
  children are numbered by (frontier slot, rank) after the previous layer;
  frontier slots are in ascending id; so id order is depth order;
* frontier and rerank order: (key descending, id ascending);
* flat order: root at row 0, kept ids ascending after it;
* position of flat row i: prefix length + depth(i), root at depth 0;
* attention scale 1/sqrt(d), caller-rotated Q/K (no RoPE here), every flat
  row attends to the whole prefix plus its in-tree ancestors and itself;
* greedy acceptance: argmax (lowest id on ties), children in ascending flat
  index;
* stochastic acceptance: point-mass proposals for deterministic top-k
  children (accept child x with probability r(x)/sum(r), r = p with the
  tokens of the siblings already rejected removed, i.e. p(x)/(1-R) for
  distinct tokens; the bonus token is drawn from that residual), or the
  draft-q variant (accept with
  min(1, r(x)/q(x)), r <- norm(max(r - q, 0)) after a rejection);
  uniforms: slot c is node c's test, slot 0 the bonus draw.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

FRAC_BITS = 32
KEY_MIN = -((1 << 52) - 1)
FLT_MAX = float(np.finfo(np.float32).max)

GREEDY = 0
STOCH_POINT = 1
STOCH_DRAFTQ = 2

# near-tie tolerances (relative); a decision closer than this to its threshold
# is reported, because fp32 rounding on the GPU may take it either way
TIE_REL_ACCEPT = 1e-5
TIE_REL_CDF = 1e-5
TIE_LP = 4e-6  # per-level log-prob error budget of the fp32 kernel


@dataclasses.dataclass(frozen=True)
class TreeCfg:
    B: int
    V: int
    depth: int
    topk: int
    m: int
    n: int
    temperature: float = 1.0

    @property
    def N(self) -> int:
        return self.n + 1


# ---------------------------------------------------------------------------
# tree geometry (node-id convention)
# ---------------------------------------------------------------------------
def layer_widths(cfg: TreeCfg) -> List[int]:
    """Number of nodes in layers 0..D (layer 0 is the root alone)."""
    w = [1, cfg.topk]
    for _ in range(2, cfg.depth + 1):
        w.append(min(cfg.m, w[-1]) * cfg.topk)
    return w


def expanded_count(cfg: TreeCfg, layer: int) -> int:
    """How many nodes of ``layer`` are expanded (the root, or the top-m)."""
    return 1 if layer == 0 else min(cfg.m, layer_widths(cfg)[layer])


def layer_base(cfg: TreeCfg, layer: int) -> int:
    """First candidate id of ``layer`` (layer >= 1)."""
    return sum(layer_widths(cfg)[1:layer])


def num_candidates(cfg: TreeCfg) -> int:
    return sum(layer_widths(cfg)[1:])


# ---------------------------------------------------------------------------
# step a1/a2: log-softmax, top-k children, fixed-point path value
# ---------------------------------------------------------------------------
def sanitize(z32: np.ndarray) -> np.ndarray:
    """fp32 logits -> float64; NaN counts as -inf, +inf as the largest float."""
    z = np.asarray(z32, dtype=np.float32).astype(np.float64)
    z = np.where(np.isnan(z), -np.inf, z)
    return np.where(z == np.inf, FLT_MAX, z)


def log_softmax(z32: np.ndarray) -> np.ndarray:
    """Draft confidence as a log-probability, in float64."""
    z = sanitize(z32)
    M = z.max()
    if M == -np.inf:
        return np.full(z.shape, -np.inf)
    return (z - M) - math.log(float(np.sum(np.exp(z - M))))


def topk_children(z32: np.ndarray, k: int) -> np.ndarray:
    """The k tokens with the largest logits, largest first, lower id on ties."""
    z = sanitize(z32)
    order = np.lexsort((np.arange(z.size), -z))
    return order[:k].astype(np.int64)


def fixed_key(lp32: float) -> int:
    """Integer fixed-point image of an fp32 log-prob (2**-32 nats per unit)."""
    x = float(np.float32(lp32))
    if x == -math.inf or math.isnan(x):
        return KEY_MIN
    return max(int(np.rint(math.ldexp(x, FRAC_BITS))), KEY_MIN)


def add_keys(parent_key: int, k: int) -> int:
    return max(parent_key + k, KEY_MIN)


# ---------------------------------------------------------------------------
# tree state
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Tree:
    cfg: TreeCfg
    tok: np.ndarray        # int32 [B, C]
    parent: np.ndarray     # int32 [B, C]  candidate id of the parent, -1 = root
    depth: np.ndarray      # int32 [B, C]
    lp: np.ndarray         # float64 [B, C] log-prob of the token in its parent's row
    lp32: np.ndarray       # float32 [B, C] the same rounded to fp32
    key: np.ndarray        # int64 [B, C]
    frontier: np.ndarray   # int32 [B, m]   next layer's expanded ids (ascending), -1 pad
    flat_node: Optional[np.ndarray] = None    # int32 [B, N] (-1 = root)
    flat_tok: Optional[np.ndarray] = None
    flat_parent: Optional[np.ndarray] = None
    flat_depth: Optional[np.ndarray] = None
    # (sequence, selection, cut between siblings?, levels summed in the keys, gap in nats)
    margins: List[Tuple[int, str, int, int, float]] = dataclasses.field(default_factory=list)

    @staticmethod
    def empty(cfg: TreeCfg) -> "Tree":
        C = num_candidates(cfg)
        B = cfg.B
        return Tree(cfg,
                    tok=np.full((B, C), -1, np.int32), parent=np.full((B, C), -1, np.int32),
                    depth=np.zeros((B, C), np.int32), lp=np.zeros((B, C)),
                    lp32=np.zeros((B, C), np.float32), key=np.zeros((B, C), np.int64),
                    frontier=np.full((B, cfg.m), -1, np.int32))


def _rank_order(keys: Sequence[int], ids: Sequence[int]) -> List[int]:
    """ids ordered by (key descending, id ascending)."""
    return sorted(ids, key=lambda c: (-int(keys[c]), c))


def _record_margin(tree: Tree, b: int, what: str, levels: int, ranked: List[int], keep: int) -> None:
    """Gap between the last kept and the first dropped key, in nats."""
    if keep < len(ranked):
        gap = (int(tree.key[b, ranked[keep - 1]]) - int(tree.key[b, ranked[keep]])) / 2.0 ** FRAC_BITS
        a, c = ranked[keep - 1], ranked[keep]
        siblings = tree.parent[b, a] == tree.parent[b, c]
        tree.margins.append((b, what, int(siblings), levels, gap))


def tree_expand(tree: Tree, layer: int, table: np.ndarray, row_of_node: Optional[np.ndarray]) -> None:
    """One expansion layer (EAGLE-2 article, expansion phase).

    The expanded nodes are the root (layer 0) or the frontier picked by the
    previous layer.  Each gets the top-k tokens of its draft row as children;
    a child's value is its parent's value times its confidence (sum of keys).
    Then the next frontier is the top-m of the new layer by value.

    ``row_of_node[b, 1 + id]`` (``[b, 0]`` for the root) is the table row of a
    node's draft logits; without it, rows are in frontier-slot order.
    """
    cfg = tree.cfg
    k = cfg.topk
    m_l = expanded_count(cfg, layer)
    base = layer_base(cfg, layer + 1)
    for b in range(cfg.B):
        nodes = [-1] if layer == 0 else [int(x) for x in tree.frontier[b, :m_l]]
        for s, node in enumerate(nodes):
            row = int(row_of_node[b, node + 1]) if row_of_node is not None else b * m_l + s
            z = table[row]
            lp = log_softmax(z)
            kids = topk_children(z, k)
            pkey = 0 if node < 0 else int(tree.key[b, node])
            for r, t in enumerate(kids):
                c = base + s * k + r
                tree.tok[b, c] = t
                tree.parent[b, c] = node
                tree.depth[b, c] = layer + 1
                tree.lp[b, c] = lp[t]
                tree.lp32[b, c] = np.float32(lp[t])
                tree.key[b, c] = add_keys(pkey, fixed_key(tree.lp32[b, c]))
        if layer + 1 < cfg.depth:
            width = layer_widths(cfg)[layer + 1]
            m_next = min(cfg.m, width)
            ranked = _rank_order(tree.key[b], range(base, base + width))
            tree.frontier[b, :] = -1
            tree.frontier[b, :m_next] = sorted(ranked[:m_next])
            _record_margin(tree, b, "frontier", layer + 1, ranked, m_next)


# ---------------------------------------------------------------------------
# step a4: rerank + flatten
# ---------------------------------------------------------------------------
def tree_rerank(tree: Tree, root_tok: Optional[np.ndarray] = None) -> None:
    """Keep the n best nodes of the whole tree (EAGLE-2 article, reranking).

    Ties in value go to the smaller id, i.e. the shallower node.  The kept
    nodes are flattened: row 0 is the root, then kept ids ascending.
    """
    cfg = tree.cfg
    C = num_candidates(cfg)
    if not 1 <= cfg.n <= C:
        raise ValueError("n must be in [1, C]")
    N = cfg.N
    tree.flat_node = np.full((cfg.B, N), -1, np.int32)
    tree.flat_tok = np.full((cfg.B, N), -1, np.int32)
    tree.flat_parent = np.full((cfg.B, N), -1, np.int32)
    tree.flat_depth = np.zeros((cfg.B, N), np.int32)
    for b in range(cfg.B):
        ranked = _rank_order(tree.key[b], range(C))
        kept = sorted(ranked[:cfg.n])
        _record_margin(tree, b, "rerank", cfg.depth, ranked, cfg.n)
        row_of = {c: i + 1 for i, c in enumerate(kept)}
        tree.flat_tok[b, 0] = -1 if root_tok is None else int(root_tok[b])
        for i, c in enumerate(kept, start=1):
            p = int(tree.parent[b, c])
            if p >= 0 and p not in row_of:
                raise AssertionError("rerank kept a node without its parent")
            tree.flat_node[b, i] = c
            tree.flat_tok[b, i] = tree.tok[b, c]
            tree.flat_parent[b, i] = 0 if p < 0 else row_of[p]
            tree.flat_depth[b, i] = tree.depth[b, c]


# ---------------------------------------------------------------------------
# step a5: ancestor mask + position ids
# ---------------------------------------------------------------------------
def mask_posids(flat_parent: np.ndarray, flat_depth: np.ndarray, prefix_len: np.ndarray
                ) -> Tuple[np.ndarray, np.ndarray]:
    """Ancestor bitmask (uint64 words, bit j of word w = flat row 64w+j) and
    positions prefix_len + depth (EAGLE-2 article, attention-mask example and
    position-encoding sentence)."""
    B, N = flat_parent.shape
    W = (N + 63) // 64
    mask = np.zeros((B, N, W), np.uint64)
    for b in range(B):
        for i in range(N):
            j = i
            while j >= 0:
                mask[b, i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
                j = int(flat_parent[b, j])
    posids = (np.asarray(prefix_len, np.int64)[:, None] + flat_depth).astype(np.int32)
    return mask, posids


def mask_bit(mask: np.ndarray, b: int, i: int, j: int) -> bool:
    return bool((int(mask[b, i, j // 64]) >> (j % 64)) & 1)


# ---------------------------------------------------------------------------
# step a6: tree attention
# ---------------------------------------------------------------------------
def tree_attention(q: np.ndarray, k_prefix: Sequence[np.ndarray], v_prefix: Sequence[np.ndarray],
                   k_tree: np.ndarray, v_tree: np.ndarray, mask: np.ndarray, scale: float
                   ) -> Tuple[np.ndarray, np.ndarray]:
    """softmax(scale * q k^T) v over the prefix plus the row's in-tree ancestors.

    q ``[B, N, Hq, d]``; ``k_prefix[b]``/``v_prefix[b]`` ``[Hkv, L_b, d]``;
    k_tree/v_tree ``[B, N, Hkv, d]``; mask ``[B, N, W]`` uint64.
    Returns O ``[B, N, Hq, d]`` and the log-sum-exp ``[B, Hq, N]`` (natural
    log, of the scaled scores), both float64.
    """
    q = np.asarray(q, np.float64)
    B, N, Hq, d = q.shape
    Hkv = k_tree.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, N, Hq, d))
    lse = np.zeros((B, Hq, N))
    for b in range(B):
        Lb = k_prefix[b].shape[1]
        allowed = np.ones((N, Lb + N), dtype=bool)
        for i in range(N):
            for j in range(N):
                allowed[i, Lb + j] = mask_bit(mask, b, i, j)
        for h in range(Hq):
            g = h // G
            K = np.concatenate([np.asarray(k_prefix[b][g], np.float64), np.asarray(k_tree[b, :, g], np.float64)])
            Vv = np.concatenate([np.asarray(v_prefix[b][g], np.float64), np.asarray(v_tree[b, :, g], np.float64)])
            S = scale * (q[b, :, h] @ K.T)
            S = np.where(allowed, S, -np.inf)
            M = S.max(axis=1, keepdims=True)
            P = np.exp(S - M)
            l = P.sum(axis=1, keepdims=True)
            out[b, :, h] = (P @ Vv) / l
            lse[b, h] = (M + np.log(l))[:, 0]
    return out, lse


# ---------------------------------------------------------------------------
# step a7: acceptance walk
# ---------------------------------------------------------------------------
def _children(flat_parent_b: np.ndarray) -> List[List[int]]:
    N = flat_parent_b.size
    ch: List[List[int]] = [[] for _ in range(N)]
    for i in range(1, N):
        ch[int(flat_parent_b[i])].append(i)
    return ch


def softmax_t(z32: np.ndarray, T: float) -> np.ndarray:
    """Target (or draft) distribution at temperature T, float64."""
    z = sanitize(z32) / T
    M = z.max()
    e = np.exp(z - M)
    return e / e.sum()


def _inverse_cdf(weights: np.ndarray, u: float, total: float) -> Tuple[int, float]:
    """Smallest t with sum_{v<=t} weights[v] > u * total, and the distance of
    that threshold to the nearest CDF step (relative to total); -1 when no
    weight is positive."""
    pos = np.nonzero(weights > 0)[0]
    if pos.size == 0:
        return -1, math.inf  # nothing left to draw from
    cdf = np.cumsum(weights)
    thr = u * total
    idx = np.nonzero(cdf > thr)[0]
    t = int(idx[0]) if idx.size else int(pos[-1])
    hi = cdf[t]
    lo = cdf[t] - weights[t]
    gap = min(abs(hi - thr), abs(thr - lo)) / max(total, 1e-300)
    return t, gap


def point_mass_ratio(r: np.ndarray, x: int) -> float:
    """min(1, r(x)/q(x)) for the point-mass proposal q at token x, with r the
    residual kept unnormalised: r(x) / sum(r).  A token outside the row has
    no mass."""
    mass = float(r.sum())
    return float(r[x]) / mass if (0 <= x < r.size and mass > 0.0) else 0.0


def point_mass_reject(r: np.ndarray, x: int) -> None:
    """A rejection of the point-mass proposal at x: max(r - q, 0) removes
    x's mass (r(x) <= 1); the renormalisation is left to the next ratio."""
    if 0 <= x < r.size:
        r[x] = 0.0


def draftq_residual(r: np.ndarray, q: np.ndarray) -> np.ndarray:
    """One rejection under the draft-q rule: norm(max(r - q, 0)); when that
    excess has no mass, r is kept."""
    res = np.maximum(r - q, 0.0)
    s = res.sum()
    return res / s if s > 0.0 else r


@dataclasses.dataclass
class AcceptResult:
    accept_len: np.ndarray   # int32 [B]
    path: np.ndarray         # int32 [B, D+1]  flat rows, root first, -1 pad
    tokens: np.ndarray       # int32 [B, D+1]  accepted draft tokens then the bonus, -1 pad
    near_ties: List[Tuple[int, str, float]]


def verify_accept(cfg: TreeCfg, mode: int, flat_tok: np.ndarray, flat_parent: np.ndarray,
                  flat_node: np.ndarray, target_table: np.ndarray, target_row_of_node: Optional[np.ndarray],
                  uniforms: Optional[np.ndarray] = None, draft_table: Optional[np.ndarray] = None,
                  draft_row_of_node: Optional[np.ndarray] = None) -> AcceptResult:
    """Walk the kept tree from the root and emit the accepted tokens plus one
    bonus token (EAGLE blog sections 1.1 and 1.2: lossless in greedy and
    non-greedy decoding).

    Target rows: ``target_row_of_node[b, 1 + node]`` (node -1 = root), or
    flat order ``b * N + i`` without a map; draft rows likewise.
    """
    B, N = flat_tok.shape
    D = cfg.depth
    acc = np.zeros(B, np.int32)
    path = np.full((B, D + 1), -1, np.int32)
    toks = np.full((B, D + 1), -1, np.int32)
    ties: List[Tuple[int, str, float]] = []

    def trow(b: int, i: int) -> np.ndarray:
        if target_row_of_node is None:
            return target_table[b * N + i]
        return target_table[int(target_row_of_node[b, int(flat_node[b, i]) + 1])]

    def drow(b: int, i: int) -> np.ndarray:
        if draft_row_of_node is None:
            return draft_table[b * N + i]
        return draft_table[int(draft_row_of_node[b, int(flat_node[b, i]) + 1])]

    for b in range(B):
        ch = _children(flat_parent[b])
        cur = 0
        p_out: List[int] = [0]
        t_out: List[int] = []
        while True:
            z = trow(b, cur)
            nxt = -1
            if mode == GREEDY:
                a = int(topk_children(z, 1)[0])
                for c in ch[cur]:
                    if int(flat_tok[b, c]) == a:
                        nxt = c
                        break
                bonus = a
            elif mode == STOCH_POINT:
                # r: the residual, kept unnormalised.  A point-mass proposal
                # at x gives min(1, r(x)/q(x)) = r(x) / sum(r), and after a
                # rejection norm(max(r - q, 0)) is r with x zeroed (then
                # renormalised, which the next division by sum(r) does).
                # For distinct sibling tokens this is p(x) / (1 - R), R the
                # mass of the siblings already rejected; a token an earlier
                # sibling already took has no residual mass left.
                r = softmax_t(z, cfg.temperature)
                for c in ch[cur]:
                    x = int(flat_tok[b, c])
                    ratio = point_mass_ratio(r, x)
                    u = float(uniforms[b, c])
                    if abs(u - ratio) < TIE_REL_ACCEPT * max(1.0, ratio):
                        ties.append((b, "accept", abs(u - ratio)))
                    if u < ratio:
                        nxt = c
                        break
                    point_mass_reject(r, x)
                if nxt < 0:
                    bonus, gap = _inverse_cdf(r, float(uniforms[b, 0]), float(r.sum()))
                    if gap < TIE_REL_CDF:
                        ties.append((b, "cdf", gap))
            elif mode == STOCH_DRAFTQ:
                p = softmax_t(z, cfg.temperature)
                r = p
                if ch[cur]:
                    qd = softmax_t(drow(b, cur), cfg.temperature)
                for c in ch[cur]:
                    x = int(flat_tok[b, c])
                    ratio = 1.0 if qd[x] <= 0.0 else min(1.0, r[x] / qd[x])
                    u = float(uniforms[b, c])
                    if abs(u - ratio) < TIE_REL_ACCEPT * max(1.0, ratio):
                        ties.append((b, "accept", abs(u - ratio)))
                    if u < ratio:
                        nxt = c
                        break
                    r = draftq_residual(r, qd)
                if nxt < 0:
                    bonus, gap = _inverse_cdf(r, float(uniforms[b, 0]), float(r.sum()))
                    if gap < TIE_REL_CDF:
                        ties.append((b, "cdf", gap))
            else:
                raise ValueError("unknown acceptance mode")
            if nxt < 0:
                t_out.append(int(bonus))
                break
            t_out.append(int(flat_tok[b, nxt]))
            p_out.append(nxt)
            cur = nxt
        acc[b] = len(p_out) - 1
        path[b, :len(p_out)] = p_out
        toks[b, :len(t_out)] = t_out
    return AcceptResult(acc, path, toks, ties)


# ---------------------------------------------------------------------------
# whole step
# ---------------------------------------------------------------------------
def build_tree(cfg: TreeCfg, draft_table: np.ndarray, row_of_node: np.ndarray,
               root_tok: Optional[np.ndarray] = None) -> Tree:
    """Expand D layers, then rerank and flatten."""
    tree = Tree.empty(cfg)
    for layer in range(cfg.depth):
        tree_expand(tree, layer, draft_table, row_of_node)
    tree_rerank(tree, root_tok)
    return tree


def near_tie_selections(tree: Tree) -> List[Tuple[int, str, int, int, float]]:
    """Frontier/rerank cut points between non-siblings closer than the fp32
    log-prob error can resolve."""
    out = []
    for b, what, sib, levels, gap in tree.margins:
        if sib:
            continue  # siblings share the normaliser: their order is exact
        if gap <= 2 * TIE_LP * levels:
            out.append((b, what, sib, levels, gap))
    return out
