"""CPU oracle of the KV commit that follows acceptance.

TEST INFRASTRUCTURE ONLY (same rules as the rest of ``oracle/``: only the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs use it).

After the acceptance walk of one verification step ([EAGLE-2 article]
sbmmt.com, reranking phase and attention mask: the kept tree is flattened, row
0 is the root, every row attends the prefix and its ancestors; [EAGLE blog]
section 1.1: one target forward verifies the draft and the accepted tokens are
kept), the flattened rows on the accepted path become part of the sequence:

* the root row (the last accepted token of the previous step, whose K/V were
  computed in this forward but are not in the cache yet) and the accepted
  draft rows ``path[1..accept_len]`` are appended to the KV cache, in path
  order, at positions ``prefix_len .. prefix_len + accept_len``;
* the features of the same rows (the target's hidden states, which the draft
  model reads in the next step) are gathered in the same order;
* the new prefix length is ``prefix_len + accept_len + 1`` (the bonus token
  becomes the next root).

Plain loops over (sequence, path position, head) with numpy row copies.
"""
from typing import Optional, Tuple

import numpy as np


def kv_commit(k_tree: np.ndarray, v_tree: np.ndarray, accept_len: np.ndarray, path: np.ndarray,
              k_cache: np.ndarray, v_cache: np.ndarray, kv_row0: np.ndarray, prefix_len: np.ndarray,
              head_stride: int, features: Optional[np.ndarray] = None
              ) -> Tuple[np.ndarray, np.ndarray, np.ndarray, Optional[np.ndarray]]:
    """k_tree, v_tree: [B, N, Hkv, d]; accept_len: [B]; path: [B, D+1] flat
    rows (path[b, 0] = 0, the root); k_cache, v_cache: [rows, d], head g of
    sequence b at row kv_row0[b] + g * head_stride + position; features:
    [B, N, F] or None.

    Returns (k_cache', v_cache', new_prefix_len, gathered features [B, D+1, F]
    with zero rows past each sequence's accepted length, or None).  Inputs are
    not modified."""
    B, N, Hkv, d = k_tree.shape
    Dp1 = path.shape[1]
    kc = k_cache.copy()
    vc = v_cache.copy()
    new_len = np.zeros(B, np.int32)
    feat = None
    if features is not None:
        feat = np.zeros((B, Dp1, features.shape[2]), features.dtype)
    for b in range(B):
        alen = int(accept_len[b])
        for i in range(alen + 1):
            row = int(path[b, i])
            pos = int(prefix_len[b]) + i
            for g in range(Hkv):
                dst = int(kv_row0[b]) + g * head_stride + pos
                kc[dst] = k_tree[b, row, g]
                vc[dst] = v_tree[b, row, g]
            if feat is not None:
                feat[b, i] = features[b, row]
        new_len[b] = int(prefix_len[b]) + alen + 1
    return kc, vc, new_len, feat
