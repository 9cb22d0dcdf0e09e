"""Thin Python binding of ``libeagle_tree.so`` (the C ABI in ``include/eagle_tree.h``).

Argument marshalling only: each function checks that its torch tensors are
CUDA tensors of the right dtype and shape, passes their device pointers and
the current CUDA stream, and turns a non-OK status into an exception.  Every
step of the verification step runs in the library's kernels; there is no
fallback.  PyTorch is used for device memory and streams.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

from .build_lib import LIB

c_i32, c_i64, c_f32, c_vp, c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

ET_OK, ET_ERR_INVALID_ARG, ET_ERR_UNSUPPORTED, ET_ERR_WORKSPACE, ET_ERR_CUDA, ET_ERR_TIMEOUT = range(6)
ET_DEV_NONFINITE, ET_DEV_BAD_INDEX, ET_DEV_DISCONNECTED, ET_DEV_TIMEOUT = 1, 2, 4, 8
ET_BF16, ET_F32 = 0, 1
ET_ACCEPT_GREEDY, ET_ACCEPT_STOCH_POINT, ET_ACCEPT_STOCH_DRAFTQ = 0, 1, 2
ATTN_AUTO, ATTN_MMA_SYNC, ATTN_TCGEN05 = 0, 1, 2
ET_ATTN_INPUTS_READY = 1
ET_EXPAND_AUTO, ET_EXPAND_CLUSTER, ET_EXPAND_BLOCK = 0, 1, 2

EXPORTED = ("et_num_candidates", "et_layer_expanded", "et_layer_base", "et_tree_workspace_size",
            "et_tree_attention_workspace_size", "et_tree_attention_splits", "et_workspace_init",
            "et_status_string", "et_abi_version", "et_tree_expand", "et_tree_expand_noalloc", "et_tree_rerank", "et_tree_rerank_mask",
            "et_tree_build", "et_tree_build_launches", "et_set_wait_limit", "et_set_expand_kernel",
            "et_tree_mask_posids", "et_tree_attention", "et_verify_accept", "et_kv_commit", "et_static_tree", "et_lm_head", "et_static_tree_sampled",
            "et_static_tree_workspace_size")


class TreeCfgC(ctypes.Structure):
    _fields_ = [("B", c_i32), ("V", c_i32), ("depth", c_i32), ("topk", c_i32), ("m", c_i32), ("n", c_i32),
                ("temperature", c_f32)]


class TreeC(ctypes.Structure):
    _fields_ = [(f, c_vp) for f in ("cand_tok", "cand_parent", "cand_lp", "cand_key", "frontier", "root_tok",
                                    "flat_node", "flat_tok", "flat_parent", "flat_depth")]


class AttnShapeC(ctypes.Structure):
    _fields_ = [("B", c_i32), ("N", c_i32), ("Hq", c_i32), ("Hkv", c_i32), ("d", c_i32), ("dtype", c_i32),
                ("scale", c_f32), ("max_prefix", c_i32), ("kv_rows", c_i64), ("kv_head_stride", c_i64),
                ("num_splits", c_i32), ("impl", c_i32), ("flags", c_i32)]


class LmHeadShapeC(ctypes.Structure):
    _fields_ = [("M", c_i32), ("H", c_i32), ("V", c_i32), ("ldo", c_i64)]


class StaticCfgC(ctypes.Structure):
    _fields_ = [("B", c_i32), ("V", c_i32), ("N", c_i32), ("topk", c_i32), ("temperature", c_f32)]


class CommitShapeC(ctypes.Structure):
    _fields_ = [("B", c_i32), ("N", c_i32), ("Hkv", c_i32), ("d", c_i32), ("path_len", c_i32), ("dtype", c_i32),
                ("kv_head_stride", c_i64), ("kv_rows", c_i64), ("feat_dim", c_i32)]


class EtError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (built in-tree by ``build_lib.build``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with speculative_decoding_eagle_gb300.build_lib.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    sig = {
        "et_num_candidates": (c_i32, [P(TreeCfgC)]),
        "et_layer_expanded": (c_i32, [P(TreeCfgC), c_i32]),
        "et_layer_base": (c_i32, [P(TreeCfgC), c_i32]),
        "et_tree_workspace_size": (c_sz, [P(TreeCfgC)]),
        "et_tree_attention_workspace_size": (c_sz, [P(AttnShapeC)]),
        "et_tree_attention_splits": (c_i32, [P(AttnShapeC)]),
        "et_workspace_init": (c_i32, [c_vp, c_sz, c_vp]),
        "et_status_string": (ctypes.c_char_p, [c_i32]),
        "et_abi_version": (c_i32, []),
        "et_tree_expand": (c_i32, [P(TreeCfgC), c_i32, c_vp, c_i64, c_vp, P(TreeC), c_vp, c_vp, c_sz, c_vp]),
        "et_tree_expand_noalloc": (c_i32, [P(TreeCfgC), c_i32, c_vp, c_i64, c_vp, P(TreeC), c_vp, c_vp]),
        "et_tree_rerank": (c_i32, [P(TreeCfgC), P(TreeC), c_vp, c_vp]),
        "et_tree_rerank_mask": (c_i32, [P(TreeCfgC), P(TreeC), c_vp, c_vp, c_vp, c_vp, c_vp]),
        "et_tree_mask_posids": (c_i32, [P(TreeCfgC), P(TreeC), c_vp, c_vp, c_vp, c_vp]),
        "et_tree_build": (c_i32, [P(TreeCfgC), c_vp, c_i64, c_vp, P(TreeC), c_vp, c_vp, c_vp, c_vp, c_vp, c_sz,
                                  c_vp]),
        "et_tree_build_launches": (c_i32, [P(TreeCfgC)]),
        "et_set_wait_limit": (c_i64, [c_i64]),
        "et_set_expand_kernel": (c_i32, [c_i32]),
        "et_tree_attention": (c_i32, [P(AttnShapeC), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                      c_vp, c_vp, c_sz, c_vp]),
        "et_static_tree_workspace_size": (c_sz, [P(StaticCfgC)]),
        "et_static_tree_sampled": (c_i32, [P(StaticCfgC), c_vp, c_vp, c_i64, c_vp, c_vp, P(TreeC), c_vp, c_vp, c_sz,
                                           c_vp]),
        "et_lm_head": (c_i32, [P(LmHeadShapeC), c_vp, c_vp, c_vp, c_vp, c_vp]),
        "et_static_tree": (c_i32, [P(StaticCfgC), c_vp, c_vp, c_vp, c_i64, c_vp, P(TreeC), c_vp, c_vp]),
        "et_kv_commit": (c_i32, [P(CommitShapeC), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                 c_vp, c_vp]),
        "et_verify_accept": (c_i32, [P(TreeCfgC), c_i32, P(TreeC), c_vp, c_i64, c_vp, c_vp, c_i64, c_vp, c_vp,
                                     c_vp, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().et_status_string(status).decode()
    except Exception:  # library not loadable: still describe the code
        return {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "workspace", 4: "CUDA error",
                5: "timeout"}.get(status, "unknown")


def _check(fn: str, status: int) -> None:
    if status != ET_OK:
        raise EtError(fn, status)


def _ptr(t: Optional[torch.Tensor], dtype=None, what: str = "tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


def _table(t: torch.Tensor, what: str) -> int:
    """A logit table: fp32 [rows, >=V] with unit inner stride, in device memory or in page-locked host memory
    (the library reads the rows it needs over the host link)."""
    if t.dim() != 2 or t.stride(1) != 1 or t.dtype != torch.float32:
        raise ValueError(f"{what} must be an fp32 [rows, >=V] table with unit inner stride")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{what} must be a CUDA tensor or a pinned host tensor")
    return t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# ---------------------------------------------------------------------------
# shapes and buffers
# ---------------------------------------------------------------------------
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

    def c(self) -> TreeCfgC:
        return TreeCfgC(self.B, self.V, self.depth, self.topk, self.m, self.n, self.temperature)


def et_num_candidates(cfg: TreeCfg) -> int:
    return load().et_num_candidates(ctypes.byref(cfg.c()))


def et_layer_expanded(cfg: TreeCfg, layer: int) -> int:
    return load().et_layer_expanded(ctypes.byref(cfg.c()), layer)


def et_layer_base(cfg: TreeCfg, layer: int) -> int:
    return load().et_layer_base(ctypes.byref(cfg.c()), layer)


def et_tree_workspace_size(cfg: TreeCfg) -> int:
    return load().et_tree_workspace_size(ctypes.byref(cfg.c()))


@dataclasses.dataclass
class TreeBuffers:
    """Device tensors behind one ``et_tree`` (allocated with torch)."""

    cfg: TreeCfg
    cand_tok: torch.Tensor
    cand_parent: torch.Tensor
    cand_lp: torch.Tensor
    cand_key: torch.Tensor
    frontier: torch.Tensor
    flat_node: torch.Tensor
    flat_tok: torch.Tensor
    flat_parent: torch.Tensor
    flat_depth: torch.Tensor
    root_tok: Optional[torch.Tensor] = None

    @staticmethod
    def allocate(cfg: TreeCfg, device="cuda", root_tok: Optional[torch.Tensor] = None) -> "TreeBuffers":
        C = et_num_candidates(cfg)
        if C < 0:
            raise ValueError(f"tree configuration outside the library's limits: {cfg}")
        i32 = dict(dtype=torch.int32, device=device)
        B, N = cfg.B, cfg.N
        return TreeBuffers(cfg, torch.full((B, C), -1, **i32), torch.full((B, C), -1, **i32),
                           torch.zeros((B, C), dtype=torch.float32, device=device),
                           torch.zeros((B, C), dtype=torch.int64, device=device),
                           torch.full((B, cfg.m), -1, **i32), torch.full((B, N), -1, **i32),
                           torch.full((B, N), -1, **i32), torch.full((B, N), -1, **i32),
                           torch.zeros((B, N), **i32), root_tok)

    @staticmethod
    def allocate_flat(B: int, N: int, device="cuda", root_tok: Optional[torch.Tensor] = None) -> "TreeBuffers":
        """Only the flattened [B, N] arrays (a static tree has no candidate arrays)."""
        i32 = dict(dtype=torch.int32, device=device)
        one = lambda dt: torch.zeros(1, dtype=dt, device=device)
        return TreeBuffers(None, one(torch.int32), one(torch.int32), one(torch.float32), one(torch.int64),
                           one(torch.int32), torch.full((B, N), -1, **i32), torch.full((B, N), -1, **i32),
                           torch.full((B, N), -1, **i32), torch.zeros((B, N), **i32), root_tok)

    def c(self) -> TreeC:
        return TreeC(_ptr(self.cand_tok, torch.int32), _ptr(self.cand_parent, torch.int32),
                     _ptr(self.cand_lp, torch.float32), _ptr(self.cand_key, torch.int64),
                     _ptr(self.frontier, torch.int32), _ptr(self.root_tok, torch.int32),
                     _ptr(self.flat_node, torch.int32), _ptr(self.flat_tok, torch.int32),
                     _ptr(self.flat_parent, torch.int32), _ptr(self.flat_depth, torch.int32))


def new_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-filled, 256-byte aligned workspace (torch's allocator aligns to 512 B)."""
    ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


# ---------------------------------------------------------------------------
# the five calls of the step
# ---------------------------------------------------------------------------
def et_tree_expand(cfg: TreeCfg, layer: int, logits: torch.Tensor, tree: TreeBuffers, ws: torch.Tensor,
                   row_of_node: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    lp = _table(logits, "logits")
    st = load().et_tree_expand(ctypes.byref(cfg.c()), layer, lp, logits.stride(0),
                               _ptr(row_of_node, torch.int32, "row_of_node"), ctypes.byref(tree.c()),
                               _ptr(dev_status, torch.int32, "dev_status"), _ptr(ws, None, "ws"),
                               ws.numel() * ws.element_size(), _stream(stream))
    _check("et_tree_expand", st)


def et_tree_expand_noalloc(cfg: TreeCfg, layer: int, logits: torch.Tensor, tree: TreeBuffers,
                           row_of_node: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    """Same result as :func:`et_tree_expand` without a workspace argument.

    For callers that cannot hand the library device scratch memory (their
    framework forbids allocation inside its execute callback, all device
    memory is pre-reserved, or a stream is being captured): the scratch is a
    4 MiB array the library keeps on each device.  Calls on one device share
    it, so they must not overlap on the GPU.
    """
    lp = _table(logits, "logits")
    st = load().et_tree_expand_noalloc(ctypes.byref(cfg.c()), layer, lp, logits.stride(0),
                                       _ptr(row_of_node, torch.int32, "row_of_node"), ctypes.byref(tree.c()),
                                       _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("et_tree_expand_noalloc", st)


def et_tree_rerank(cfg: TreeCfg, tree: TreeBuffers, dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    st = load().et_tree_rerank(ctypes.byref(cfg.c()), ctypes.byref(tree.c()),
                               _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("et_tree_rerank", st)


def et_tree_rerank_mask(cfg: TreeCfg, tree: TreeBuffers, prefix_len: torch.Tensor, mask: torch.Tensor,
                        posids: torch.Tensor, dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    st = load().et_tree_rerank_mask(ctypes.byref(cfg.c()), ctypes.byref(tree.c()),
                                    _ptr(prefix_len, torch.int32, "prefix_len"), _ptr(mask, torch.int64, "mask"),
                                    _ptr(posids, torch.int32, "posids"), _ptr(dev_status, torch.int32, "dev_status"),
                                    _stream(stream))
    _check("et_tree_rerank_mask", st)


def et_tree_build(cfg: TreeCfg, logits: torch.Tensor, tree: TreeBuffers, ws: torch.Tensor,
                  row_of_node: Optional[torch.Tensor] = None, prefix_len: Optional[torch.Tensor] = None,
                  mask: Optional[torch.Tensor] = None, posids: Optional[torch.Tensor] = None,
                  dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    lp = _table(logits, "logits")
    st = load().et_tree_build(ctypes.byref(cfg.c()), lp, logits.stride(0),
                              _ptr(row_of_node, torch.int32, "row_of_node"), ctypes.byref(tree.c()),
                              _ptr(prefix_len, torch.int32, "prefix_len"), _ptr(mask, torch.int64, "mask"),
                              _ptr(posids, torch.int32, "posids"), _ptr(dev_status, torch.int32, "dev_status"),
                              _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    _check("et_tree_build", st)


def et_tree_build_launches(cfg: TreeCfg) -> int:
    return int(load().et_tree_build_launches(ctypes.byref(cfg.c())))


def et_set_wait_limit(cycles: int) -> int:
    """Bound (SM cycles) of device waits of later launches; 0 restores the default. Returns the previous bound."""
    return int(load().et_set_wait_limit(int(cycles)))


def et_set_expand_kernel(which: int) -> int:
    """Kernel of later expansion launches with V <= 32768 (ET_EXPAND_*); returns the previous choice."""
    prev = int(load().et_set_expand_kernel(int(which)))
    if prev < 0:
        raise ValueError(f"unknown expansion kernel {which}")
    return prev


def et_tree_mask_posids(cfg: TreeCfg, tree: TreeBuffers, prefix_len: torch.Tensor, mask: torch.Tensor,
                        posids: torch.Tensor, stream=None) -> None:
    st = load().et_tree_mask_posids(ctypes.byref(cfg.c()), ctypes.byref(tree.c()),
                                    _ptr(prefix_len, torch.int32, "prefix_len"), _ptr(mask, torch.int64, "mask"),
                                    _ptr(posids, torch.int32, "posids"), _stream(stream))
    _check("et_tree_mask_posids", st)


@dataclasses.dataclass(frozen=True)
class AttnShape:
    B: int
    N: int
    Hq: int
    Hkv: int
    d: int
    dtype: int = ET_BF16
    scale: float = 0.0
    max_prefix: int = 0
    kv_rows: int = 0
    kv_head_stride: int = 0
    num_splits: int = 0
    impl: int = ATTN_AUTO
    flags: int = 0

    def c(self) -> AttnShapeC:
        sc = self.scale if self.scale > 0 else self.d ** -0.5
        return AttnShapeC(self.B, self.N, self.Hq, self.Hkv, self.d, self.dtype, sc, self.max_prefix,
                          self.kv_rows, self.kv_head_stride, self.num_splits, self.impl, self.flags)


def et_tree_attention_workspace_size(shape: AttnShape) -> int:
    return load().et_tree_attention_workspace_size(ctypes.byref(shape.c()))


def et_tree_attention_splits(shape: AttnShape) -> int:
    return load().et_tree_attention_splits(ctypes.byref(shape.c()))


def et_tree_attention(shape: AttnShape, q, k_prefix, v_prefix, kv_row0, prefix_len, k_tree, v_tree, mask, out,
                      lse=None, ws=None, dev_status=None, stream=None) -> None:
    dt = torch.bfloat16 if shape.dtype == ET_BF16 else torch.float32
    st = load().et_tree_attention(
        ctypes.byref(shape.c()), _ptr(q, dt, "q"), _ptr(k_prefix, dt, "k_prefix"), _ptr(v_prefix, dt, "v_prefix"),
        _ptr(kv_row0, torch.int64, "kv_row0"), _ptr(prefix_len, torch.int32, "prefix_len"),
        _ptr(k_tree, dt, "k_tree"), _ptr(v_tree, dt, "v_tree"), _ptr(mask, torch.int64, "mask"),
        _ptr(out, dt, "out"), _ptr(lse, torch.float32, "lse"), _ptr(dev_status, torch.int32, "dev_status"),
        _ptr(ws, None, "ws"), 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check("et_tree_attention", st)


def et_verify_accept(cfg: TreeCfg, mode: int, tree: TreeBuffers, target_logits: torch.Tensor,
                     accept_len: torch.Tensor, path: torch.Tensor, tokens: torch.Tensor, ws: torch.Tensor,
                     target_row_of_node=None, draft_logits=None, draft_row_of_node=None, uniforms=None,
                     dev_status=None, stream=None) -> None:
    tp = _table(target_logits, "target_logits")
    dp = None if draft_logits is None else _table(draft_logits, "draft_logits")
    st = load().et_verify_accept(
        ctypes.byref(cfg.c()), mode, ctypes.byref(tree.c()), tp, target_logits.stride(0),
        _ptr(target_row_of_node, torch.int32, "target_row_of_node"),
        dp,
        0 if draft_logits is None else draft_logits.stride(0),
        _ptr(draft_row_of_node, torch.int32, "draft_row_of_node"), _ptr(uniforms, torch.float32, "uniforms"),
        _ptr(accept_len, torch.int32, "accept_len"), _ptr(path, torch.int32, "path"),
        _ptr(tokens, torch.int32, "tokens"), _ptr(dev_status, torch.int32, "dev_status"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream))
    _check("et_verify_accept", st)


@dataclasses.dataclass(frozen=True)
class CommitShape:
    B: int
    N: int
    Hkv: int
    d: int
    path_len: int
    dtype: int = ET_BF16
    kv_head_stride: int = 0
    kv_rows: int = 0
    feat_dim: int = 0

    def c(self) -> CommitShapeC:
        return CommitShapeC(self.B, self.N, self.Hkv, self.d, self.path_len, self.dtype, self.kv_head_stride,
                            self.kv_rows, self.feat_dim)


def et_kv_commit(shape: CommitShape, k_tree: torch.Tensor, v_tree: torch.Tensor, accept_len: torch.Tensor,
                 path: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, kv_row0: torch.Tensor,
                 prefix_len: torch.Tensor, new_prefix_len: torch.Tensor, features: Optional[torch.Tensor] = None,
                 feat_out: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                 stream=None) -> None:
    """Append each sequence's accepted path (root first) to the KV cache and gather its features."""
    dt = torch.bfloat16 if shape.dtype == ET_BF16 else torch.float32
    st = load().et_kv_commit(
        ctypes.byref(shape.c()), _ptr(k_tree, dt, "k_tree"), _ptr(v_tree, dt, "v_tree"),
        _ptr(accept_len, torch.int32, "accept_len"), _ptr(path, torch.int32, "path"),
        _ptr(k_cache, dt, "k_cache"), _ptr(v_cache, dt, "v_cache"), _ptr(kv_row0, torch.int64, "kv_row0"),
        _ptr(prefix_len, torch.int32, "prefix_len"), _ptr(new_prefix_len, torch.int32, "new_prefix_len"),
        _ptr(features, dt, "features"), _ptr(feat_out, dt, "feat_out"), _ptr(dev_status, torch.int32, "dev_status"),
        _stream(stream))
    _check("et_kv_commit", st)


def et_static_tree(B: int, V: int, topk: int, parent: torch.Tensor, rank: torch.Tensor, logits: torch.Tensor,
                   row_of_flat: torch.Tensor, tree: "TreeBuffers", dev_status: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """Flatten a static draft tree (fixed parent / rank per flat row) from the draft logits at each parent."""
    if logits.dim() != 2 or logits.stride(1) != 1 or logits.dtype != torch.float32 or not logits.is_cuda:
        raise ValueError("logits must be a CUDA fp32 [rows, >=V] table with unit inner stride")
    N = parent.numel()
    st = load().et_static_tree(ctypes.byref(StaticCfgC(B, V, N, topk, 1.0)), _ptr(parent, torch.int32, "parent"),
                               _ptr(rank, torch.int32, "rank"), logits.data_ptr(), logits.stride(0),
                               _ptr(row_of_flat, torch.int32, "row_of_flat"), ctypes.byref(tree.c()),
                               _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("et_static_tree", st)


def et_lm_head(features: torch.Tensor, weight: torch.Tensor, logits: torch.Tensor,
               dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """logits[m, :V] = features[m] @ weight.T (bf16 in, fp32 out) on the tcgen05 tensor cores."""
    M, H = features.shape
    V = weight.shape[0]
    if weight.shape[1] != H or logits.dim() != 2 or logits.shape[0] < M or logits.stride(1) != 1:
        raise ValueError("features [M, H], weight [V, H], logits [>=M, >=V] with unit inner stride")
    st = load().et_lm_head(ctypes.byref(LmHeadShapeC(M, H, V, logits.stride(0))),
                           _ptr(features, torch.bfloat16, "features"), _ptr(weight, torch.bfloat16, "weight"),
                           logits.data_ptr() if logits.dtype == torch.float32 and logits.is_cuda else None,
                           _ptr(dev_status, torch.int32, "dev_status"), _stream(stream))
    _check("et_lm_head", st)


def et_static_tree_sampled(B: int, V: int, temperature: float, parent: torch.Tensor, logits: torch.Tensor,
                           row_of_flat: torch.Tensor, uniforms: torch.Tensor, tree: "TreeBuffers",
                           ws: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    """Flatten a static tree whose children are draws from softmax(draft / T) at their parent."""
    if logits.dim() != 2 or logits.stride(1) != 1 or logits.dtype != torch.float32 or not logits.is_cuda:
        raise ValueError("logits must be a CUDA fp32 [rows, >=V] table with unit inner stride")
    N = parent.numel()
    cfg = StaticCfgC(B, V, N, 1, temperature)
    if ws is None:
        ws = new_workspace(load().et_static_tree_workspace_size(ctypes.byref(cfg)), logits.device)
    st = load().et_static_tree_sampled(ctypes.byref(cfg), _ptr(parent, torch.int32, "parent"), logits.data_ptr(),
                                       logits.stride(0), _ptr(row_of_flat, torch.int32, "row_of_flat"),
                                       _ptr(uniforms, torch.float32, "uniforms"), ctypes.byref(tree.c()),
                                       _ptr(dev_status, torch.int32, "dev_status"), _ptr(ws, None, "ws"),
                                       ws.numel() * ws.element_size(), _stream(stream))
    _check("et_static_tree_sampled", st)
