"""CPU oracle of the static draft tree (EAGLE-1 / Medusa style).

TEST INFRASTRUCTURE ONLY (same rules as the rest of ``oracle/``).

The [EAGLE-2 article] (sbmmt.com) contrasts its dynamic tree with the static
draft tree of earlier methods: the tree's shape is fixed in advance,
independent of the context, and every node takes a fixed set of children
from its draft distribution.  Here the fixed shape is a list of flat rows:
row 0 is the root, row i > 0 has a parent row ``parent[i] < i`` and a rank
``rank[i]``; its token is the rank[i]-th best token (largest draft logit
first, lower id on ties -- the same order as the dynamic tree's top-k) of the
draft logits at its parent.  Verification then runs unchanged on the
flattened tree (mask, attention, acceptance).
"""
from typing import Tuple

import numpy as np

from .eagle_tree_oracle import topk_children


def static_depths(parent: np.ndarray) -> np.ndarray:
    """Depth of every flat row (root 0), following parents (which precede children)."""
    depth = np.zeros(parent.size, np.int32)
    for i in range(1, parent.size):
        depth[i] = depth[int(parent[i])] + 1
    return depth


def static_tree(parent: np.ndarray, rank: np.ndarray, draft_table: np.ndarray, row_of_flat: np.ndarray,
                root_tok: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """parent, rank: [N] (parent[0] = -1); draft_table: [rows, V] fp32;
    row_of_flat: [B, N] table row of each flat row's draft logits (used for
    rows that have children).  Returns flat (tok, parent, depth, node) [B, N],
    node = flat row - 1 (root -1)."""
    B, N = row_of_flat.shape
    depth = static_depths(parent)
    k = int(rank[1:].max()) + 1 if N > 1 else 1
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        tok[b, 0] = root_tok[b]
        for i in range(1, N):
            p = int(parent[i])
            order = topk_children(draft_table[int(row_of_flat[b, p])], k)
            tok[b, i] = order[int(rank[i])]
    fparent = np.tile(parent.astype(np.int32), (B, 1))
    fdepth = np.tile(depth, (B, 1))
    node = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    return tok, fparent, fdepth, node


def static_tree_sampled(parent: np.ndarray, draft_table: np.ndarray, row_of_flat: np.ndarray,
                        uniforms: np.ndarray, temperature: float, root_tok: np.ndarray):
    """A static tree whose children are independent draws from the draft
    distribution at their parent, q = softmax(draft / T) (the proposal the
    draft-q acceptance rule needs to stay lossless): row i > 0 takes the
    smallest token t with sum_{v <= t} q(v) > uniforms[b, i].

    Returns (tok, parent, depth, node) like ``static_tree`` and the near-tie
    margin of every draw (distance of the uniform to the nearest CDF step)."""
    from .eagle_tree_oracle import _inverse_cdf, softmax_t
    B, N = row_of_flat.shape
    depth = static_depths(parent)
    tok = np.zeros((B, N), np.int32)
    gaps = np.full((B, N), np.inf)
    for b in range(B):
        tok[b, 0] = root_tok[b]
        for i in range(1, N):
            p = int(parent[i])
            q = softmax_t(draft_table[int(row_of_flat[b, p])], temperature)
            t, gap = _inverse_cdf(q, float(uniforms[b, i]), float(q.sum()))
            tok[b, i] = t
            gaps[b, i] = gap
    fparent = np.tile(parent.astype(np.int32), (B, 1))
    fdepth = np.tile(depth, (B, 1))
    node = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    return tok, fparent, fdepth, node, gaps
