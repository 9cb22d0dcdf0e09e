"""Helpers shared by the GPU parity tests: run the oracle on the same seeded
inputs as the CUDA path, move tree state between the two, compare."""
import numpy as np
import torch

import oracle as O
from speculative_decoding_eagle_gb300 import binding as E
from speculative_decoding_eagle_gb300 import step as S
from speculative_decoding_eagle_gb300 import workloads as W

LP_TOL = 1e-5                                   # log-probs (spec tolerance)
KEY_TOL_PER_LEVEL = int(LP_TOL * 2 ** 32)       # fixed-point keys, per summed level
BF16_MAX_ABS, BF16_REL_L2 = 2e-2, 5e-3          # bf16 attention, fp32 accumulation
F32_MAX_ABS, F32_REL_L2 = 1e-4, 1e-5            # fp32 attention


def ocfg(cfg: E.TreeCfg) -> O.TreeCfg:
    return O.TreeCfg(B=cfg.B, V=cfg.V, depth=cfg.depth, topk=cfg.topk, m=cfg.m, n=cfg.n,
                     temperature=cfg.temperature)


def gpu_tree_np(tb: E.TreeBuffers):
    torch.cuda.synchronize()
    return {k: getattr(tb, k).cpu().numpy() for k in
            ("cand_tok", "cand_parent", "cand_lp", "cand_key", "frontier", "flat_node", "flat_tok", "flat_parent",
             "flat_depth")}


def upload_oracle_tree(tree: O.Tree, tb: E.TreeBuffers) -> None:
    """Copy the oracle's tree state into the device buffers (oracle -> GPU)."""
    tb.cand_tok.copy_(torch.from_numpy(tree.tok))
    tb.cand_parent.copy_(torch.from_numpy(tree.parent))
    tb.cand_lp.copy_(torch.from_numpy(tree.lp32))
    tb.cand_key.copy_(torch.from_numpy(tree.key))
    tb.frontier.copy_(torch.from_numpy(tree.frontier))
    if tree.flat_node is not None:
        for k, v in (("flat_node", tree.flat_node), ("flat_tok", tree.flat_tok), ("flat_parent", tree.flat_parent),
                     ("flat_depth", tree.flat_depth)):
            getattr(tb, k).copy_(torch.from_numpy(v))


def copy_oracle_tree(t: O.Tree) -> O.Tree:
    import copy
    return copy.deepcopy(t)


def compare_layer(cfg, layer, g, o: O.Tree, check_frontier=True):
    """GPU vs oracle for the nodes one expansion layer created."""
    base = O.layer_base(ocfg(cfg), layer + 1)
    width = O.layer_widths(ocfg(cfg))[layer + 1]
    sl = slice(base, base + width)
    np.testing.assert_array_equal(g["cand_tok"][:, sl], o.tok[:, sl])
    np.testing.assert_array_equal(g["cand_parent"][:, sl], o.parent[:, sl])
    lp_o = o.lp[:, sl]
    lp_g = g["cand_lp"][:, sl].astype(np.float64)
    fin = np.isfinite(lp_o)
    assert (np.isfinite(lp_g) == fin).all()
    assert np.max(np.abs(lp_g[fin] - lp_o[fin]), initial=0.0) <= LP_TOL
    dk = np.abs(g["cand_key"][:, sl].astype(np.int64) - o.key[:, sl])
    assert dk.max() <= KEY_TOL_PER_LEVEL * (layer + 1), dk.max()
    if check_frontier and layer + 1 < cfg.depth:
        np.testing.assert_array_equal(g["frontier"], o.frontier)


def rel_l2(a, b):
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-30))


def oracle_attention_from_host(wl: W.Workload, h, mask_np, B):
    q = W.as_float(wl, h["q"]).astype(np.float64)
    kt = W.as_float(wl, h["k_tree"]).astype(np.float64)
    vt = W.as_float(wl, h["v_tree"]).astype(np.float64)
    kp, vp = [], []
    kpf = W.as_float(wl, h["k_prefix"])
    vpf = W.as_float(wl, h["v_prefix"])
    for b in range(B):
        L = int(h["prefix_len"][b])
        r0 = int(h["kv_row0"][b])
        kp.append(kpf[r0:r0 + wl.Hkv * L].reshape(wl.Hkv, L, wl.d))
        vp.append(vpf[r0:r0 + wl.Hkv * L].reshape(wl.Hkv, L, wl.d))
    return O.tree_attention(q, kp, vp, kt, vt, mask_np, wl.d ** -0.5)


def out_as_float(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
