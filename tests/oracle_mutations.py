"""pytest plugin: plant one plausible mistake in the oracle (on the CPU).

Loaded by ``tests/test_oracle_mutations.py`` in a child pytest run with
``ET_ORACLE_MUTATION=<name>``; the child runs the oracle's pins, which must
fail.  Each mutation stands for a mistake that could slip into a restatement
of the pages (a dropped term, a wrong sign, a reversed tie-break, an
off-by-one), so a surviving mutation marks a pin that is missing.
"""
import os

import numpy as np

import oracle
from oracle import eagle_tree_oracle as T
from oracle import kv_commit_oracle as K
from oracle import static_tree_oracle as ST


def _set(mod, name, fn):
    setattr(mod, name, fn)
    if hasattr(oracle, name):
        setattr(oracle, name, fn)


def _lsm_no_normaliser():
    def log_softmax(z32):
        z = T.sanitize(z32)
        return z - z.max()
    _set(T, "log_softmax", log_softmax)


def _topk_ties_high_id():
    def topk_children(z32, k):
        z = T.sanitize(z32)
        return np.lexsort((-np.arange(z.size), -z))[:k].astype(np.int64)
    _set(T, "topk_children", topk_children)
    ST.topk_children = topk_children


def _fixed_key_half_scale():
    orig = T.fixed_key
    _set(T, "fixed_key", lambda lp32: orig(lp32) // 2 if orig(lp32) != T.KEY_MIN else T.KEY_MIN)


def _add_keys_subtracts():
    _set(T, "add_keys", lambda parent_key, k: max(parent_key - k, T.KEY_MIN))


def _rerank_deeper_first():
    _set(T, "_rank_order", lambda keys, ids: sorted(ids, key=lambda c: (-int(keys[c]), -c)))


def _mask_without_self():
    orig = T.mask_posids

    def mask_posids(flat_parent, flat_depth, prefix_len):
        mask, pos = orig(flat_parent, flat_depth, prefix_len)
        B, N, _ = mask.shape
        for b in range(B):
            for i in range(N):
                mask[b, i, i // 64] &= ~(np.uint64(1) << np.uint64(i % 64))
        return mask, pos
    _set(T, "mask_posids", mask_posids)


def _attention_ignores_scale():
    orig = T.tree_attention
    _set(T, "tree_attention", lambda q, kp, vp, kt, vt, mask, scale: orig(q, kp, vp, kt, vt, mask, 1.0))


def _children_reversed():
    orig = T._children
    _set(T, "_children", lambda fp: [list(reversed(c)) for c in orig(fp)])


def _softmax_ignores_temperature():
    orig = T.softmax_t
    _set(T, "softmax_t", lambda z32, t: orig(z32, 1.0))


def _commit_skips_root():
    orig = K.kv_commit

    def kv_commit(k_tree, v_tree, accept_len, path, k_cache, v_cache, kv_row0, prefix_len, head_stride,
                  features=None):
        p2 = path.copy()
        p2[:, 0] = p2[:, 1].clip(min=0)  # the first accepted row where the root belongs
        return orig(k_tree, v_tree, accept_len, p2, k_cache, v_cache, kv_row0, prefix_len, head_stride, features)
    _set(K, "kv_commit", kv_commit)


def _static_rank_off_by_one():
    orig = ST.static_tree

    def static_tree(parent, rank, draft_table, row_of_flat, root_tok):
        r2 = rank.copy()
        r2[1:] += 1
        return orig(parent, r2, draft_table, row_of_flat, root_tok)
    _set(ST, "static_tree", static_tree)


def _residual_without_clamp():
    def draftq_residual(r, q):
        res = r - q
        s = np.abs(res).sum()
        return res / s if s > 0.0 else r
    _set(T, "draftq_residual", draftq_residual)


def _residual_not_renormalised():
    _set(T, "draftq_residual", lambda r, q: np.maximum(r - q, 0.0))


def _inverse_cdf_ignores_mass():
    orig = T._inverse_cdf
    _set(T, "_inverse_cdf", lambda weights, u, total: orig(weights, u, 1.0))  # threshold u, not u * mass


def _point_mass_keeps_rejected_mass():
    _set(T, "point_mass_reject", lambda r, x: None)


def _point_mass_not_renormalised():
    _set(T, "point_mass_ratio", lambda r, x: float(r[x]) if 0 <= x < r.size else 0.0)


MUTATIONS = {
    "log_softmax drops the log-sum-exp": _lsm_no_normaliser,
    "top-k ties go to the higher id": _topk_ties_high_id,
    "fixed-point key at half scale": _fixed_key_half_scale,
    "path keys subtract": _add_keys_subtracts,
    "rerank ties go to the deeper node": _rerank_deeper_first,
    "mask drops the row itself": _mask_without_self,
    "attention ignores the scale": _attention_ignores_scale,
    "children tried in descending row order": _children_reversed,
    "temperature ignored": _softmax_ignores_temperature,
    "KV commit skips the root row": _commit_skips_root,
    "static tree ranks off by one": _static_rank_off_by_one,
    "draft-q residual drops the clamp": _residual_without_clamp,
    "draft-q residual not renormalised": _residual_not_renormalised,
    "inverse CDF ignores the remaining mass": _inverse_cdf_ignores_mass,
    "point-mass rejection keeps the token's mass": _point_mass_keeps_rejected_mass,
    "point-mass ratio not renormalised": _point_mass_not_renormalised,
}


def pytest_configure(config):
    name = os.environ.get("ET_ORACLE_MUTATION")
    if name:
        MUTATIONS[name]()
