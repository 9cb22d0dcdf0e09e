"""One EAGLE-2 draft-tree verification step on the GPU, as a chain of the five
C-ABI calls (EAGLE-2 article on sbmmt.com: expansion, reranking, attention
mask / positions, ancestor-masked attention; EAGLE blog 1.2: lossless
acceptance).

``StepInputs`` holds the device copies of one batch of synthetic inputs;
``VerifyStep`` owns the output and workspace buffers and runs the calls in
stream order.  No arithmetic of the method happens here.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch

from . import binding as E
from . import workloads as W


@dataclasses.dataclass
class StepInputs:
    """Device tensors of one batch (all synthetic, seeded)."""

    draft: torch.Tensor          # fp32 [B*(C+1), V] node-indexed draft rows
    target: torch.Tensor         # fp32 [B*(C+1), V] node-indexed target rows
    row_of_node: torch.Tensor    # int32 [B, C+1]
    root_tok: torch.Tensor       # int32 [B]
    prefix_len: torch.Tensor     # int32 [B]
    kv_row0: torch.Tensor        # int64 [B]
    q: torch.Tensor              # [B, N, Hq, d]
    k_prefix: torch.Tensor       # [rows, d]
    v_prefix: torch.Tensor       # [rows, d]
    k_tree: torch.Tensor         # [B, N, Hkv, d]
    v_tree: torch.Tensor         # [B, N, Hkv, d]
    uniforms: torch.Tensor       # fp32 [B, N]
    host: Dict[str, np.ndarray]  # the numpy originals (for the oracle)


def tree_cfg(wl: W.Workload, B: Optional[int] = None) -> E.TreeCfg:
    return E.TreeCfg(B=wl.B if B is None else B, V=wl.V, depth=wl.depth, topk=wl.topk, m=wl.m, n=wl.n,
                     temperature=wl.temperature)


def host_inputs(wl: W.Workload, C: int, B: Optional[int] = None, b0: int = 0) -> Dict[str, np.ndarray]:
    """numpy inputs of sequences ``b0 .. b0+B-1``; ``C`` is the tree's candidate count."""
    B = wl.B if B is None else B
    # only nodes that can be expanded need draft rows: every layer but the last
    cfg = tree_cfg(wl, B)
    num_draft = E.et_layer_base(cfg, wl.depth) if wl.depth > 1 else 0
    target, draft, rmap = W.logit_tables(wl, C, num_draft, batch=range(b0, b0 + B))
    prefix = W.prefix_lengths(wl, b0 + B)[b0:b0 + B]
    qs, kps, vps, kts, vts = [], [], [], [], []
    for i in range(B):
        x = W.qkv(wl, b0 + i, int(prefix[i]))
        qs.append(x["q"]); kps.append(x["k_prefix"]); vps.append(x["v_prefix"])
        kts.append(x["k_tree"]); vts.append(x["v_tree"])
    kv_row0 = np.zeros(B, np.int64)
    acc = 0
    for i in range(B):
        kv_row0[i] = acc
        acc += wl.Hkv * int(prefix[i])
    dt = qs[0].dtype
    return dict(draft=draft, target=target, row_of_node=rmap, root_tok=W.root_tokens(wl, b0 + B)[b0:b0 + B],
                prefix_len=prefix, kv_row0=kv_row0, q=np.stack(qs),
                k_prefix=np.concatenate([k.reshape(-1, wl.d) for k in kps]) if acc else np.zeros((0, wl.d), dt),
                v_prefix=np.concatenate([v.reshape(-1, wl.d) for v in vps]) if acc else np.zeros((0, wl.d), dt),
                k_tree=np.stack(kts), v_tree=np.stack(vts),
                uniforms=np.stack([W.uniforms(wl, b0 + i) for i in range(B)]))


def to_device(wl: W.Workload, h: Dict[str, np.ndarray], device="cuda") -> StepInputs:
    def up(x, kind=None):
        x = np.ascontiguousarray(x)
        if kind == "bf16":  # uint16 bit patterns -> bf16 tensor
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(x).to(device)
    kind = "bf16" if wl.dtype == "bf16" else None
    kp = h["k_prefix"] if h["k_prefix"].size else np.zeros((1, wl.d), h["q"].dtype)
    vp = h["v_prefix"] if h["v_prefix"].size else np.zeros((1, wl.d), h["q"].dtype)
    return StepInputs(draft=up(h["draft"]), target=up(h["target"]), row_of_node=up(h["row_of_node"]),
                      root_tok=up(h["root_tok"]), prefix_len=up(h["prefix_len"]), kv_row0=up(h["kv_row0"]),
                      q=up(h["q"], kind), k_prefix=up(kp, kind), v_prefix=up(vp, kind),
                      k_tree=up(h["k_tree"], kind), v_tree=up(h["v_tree"], kind), uniforms=up(h["uniforms"]),
                      host=h)


# Measured on GB300 (7B heads, batch 1): a tcgen05 attention block spends
# about 1.4 us per 64-key K/V tile; one layer of the one-launch tree build
# takes about 7 us.
TILE_US = 1.4
LAYER_US = 7.0


def overlap_splits(tiles: int, depth: int, auto_splits: int, blocks_per_split: int, free_slots: int) -> int:
    """KV splits for the attention of a step whose tree is built in one launch.

    With ET_ATTN_INPUTS_READY the attention blocks stream their prefix while
    the latency-bound tree build runs, so a block may take long as long as it
    ends before the tree does: the fewest splits (at most the standalone
    plan's) whose blocks each stream within 80% of the tree's expected time
    and all find room beside the tree's blocks.  Fewer splits leave less to
    merge after the tree.  Falls back to the standalone plan."""
    budget = 0.8 * depth * LAYER_US
    for s in range(1, max(1, auto_splits) + 1):
        if -(-tiles // s) * TILE_US <= budget and s * blocks_per_split <= free_slots:
            return s
    return auto_splits


class VerifyStep:
    """Buffers and call chain of one verification step for a fixed shape."""

    def __init__(self, wl: W.Workload, B: Optional[int] = None, mode: Optional[int] = None, device="cuda",
                 num_splits: int = 0, max_prefix: Optional[int] = None, attn_impl: int = E.ATTN_AUTO,
                 per_layer: bool = False, overlap: bool = True):
        self.wl = wl
        self.per_layer = per_layer  # the tree by one et_tree_expand launch per layer, then et_tree_rerank_mask
        # with num_splits = 0: pick the attention's splits for streaming beside the
        # tree build (overlap_splits), else the standalone plan
        self.overlap = overlap
        self.cfg = tree_cfg(wl, B)
        self.B = self.cfg.B
        self.C = E.et_num_candidates(self.cfg)
        if self.C < 0:
            raise ValueError(f"workload {wl.name} is outside the library limits")
        if mode is None:
            mode = E.ET_ACCEPT_GREEDY if "greedy" in wl.accept else E.ET_ACCEPT_STOCH_POINT
        self.mode = mode
        self.device = device
        N = self.cfg.N
        self.tree = E.TreeBuffers.allocate(self.cfg, device)
        self.ws = E.new_workspace(E.et_tree_workspace_size(self.cfg), device)
        self.mask = torch.zeros((self.B, N, (N + 63) // 64), dtype=torch.int64, device=device)
        self.posids = torch.zeros((self.B, N), dtype=torch.int32, device=device)
        dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        self.out = torch.zeros((self.B, N, wl.Hq, wl.d), dtype=dt, device=device)
        self.lse = torch.zeros((self.B, wl.Hq, N), dtype=torch.float32, device=device)
        self.accept_len = torch.zeros(self.B, dtype=torch.int32, device=device)
        self.path = torch.zeros((self.B, wl.depth + 1), dtype=torch.int32, device=device)
        self.tokens = torch.zeros((self.B, wl.depth + 1), dtype=torch.int32, device=device)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=device)
        self.max_prefix = max_prefix
        self.num_splits = num_splits
        self.attn_impl = attn_impl
        self.attn_ws = None
        self.shape = None

    def attn_shape(self, inp: StepInputs) -> E.AttnShape:
        mp = self.max_prefix if self.max_prefix is not None else int(inp.host["prefix_len"].max())
        shape = E.AttnShape(B=self.B, N=self.cfg.N, Hq=self.wl.Hq, Hkv=self.wl.Hkv, d=self.wl.d,
                            dtype=E.ET_BF16 if self.wl.dtype == "bf16" else E.ET_F32, scale=self.wl.d ** -0.5,
                            max_prefix=mp, kv_rows=inp.k_prefix.shape[0], num_splits=self.num_splits,
                            impl=self.attn_impl,
                            # Q, K/V and the prefix lengths are step inputs; only the mask comes
                            # from the kernel before attention
                            flags=E.ET_ATTN_INPUTS_READY)
        if self.num_splits == 0 and self.overlap and not self.per_layer:
            shape = dataclasses.replace(shape, num_splits=self.step_splits(shape))
        return shape

    def step_splits(self, shape: E.AttnShape) -> int:
        """The attention's split count inside the step (see overlap_splits)."""
        auto = E.et_tree_attention_splits(shape)
        tc = shape.dtype == E.ET_BF16 and shape.d == 128 and self.attn_impl in (E.ATTN_AUTO, E.ATTN_TCGEN05)
        if auto <= 0 or not tc or E.et_tree_build_launches(self.cfg) != 1:
            return max(auto, 0)
        G = shape.Hq // shape.Hkv
        MT = -(-(shape.N * G) // 128)
        tiles = -(-shape.max_prefix // 64) + -(-shape.N // 64)
        slots = max(E.et_layer_expanded(self.cfg, l) for l in range(self.cfg.depth)) + 1
        # the cluster build's blocks; when they do not all fit, the work-queue build holds every SM
        tree_blocks = self.B * slots * -(-self.cfg.V // 4096)
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        return overlap_splits(tiles, self.cfg.depth, auto, self.B * shape.Hkv * MT, 2 * max(0, sms - tree_blocks))

    def prepare(self, inp: StepInputs) -> None:
        shape = self.attn_shape(inp)
        if self.shape != shape:
            self.shape = shape
            self.attn_ws = E.new_workspace(E.et_tree_attention_workspace_size(shape), self.device)
        self.tree.root_tok = inp.root_tok

    # the five calls -------------------------------------------------------
    def build_tree(self, inp: StepInputs, stream=None) -> None:
        """D expansion layers, rerank, mask and positions: one launch of et_tree_build (V <= 32768), or the
        per-layer calls when ``per_layer``."""
        self.tree.root_tok = inp.root_tok
        if self.per_layer:
            for layer in range(self.cfg.depth):
                E.et_tree_expand(self.cfg, layer, inp.draft, self.tree, self.ws, row_of_node=inp.row_of_node,
                                 dev_status=self.dev_status, stream=stream)
            E.et_tree_rerank_mask(self.cfg, self.tree, inp.prefix_len, self.mask, self.posids,
                                  dev_status=self.dev_status, stream=stream)
        else:
            E.et_tree_build(self.cfg, inp.draft, self.tree, self.ws, row_of_node=inp.row_of_node,
                            prefix_len=inp.prefix_len, mask=self.mask, posids=self.posids,
                            dev_status=self.dev_status, stream=stream)

    def attention(self, inp: StepInputs, stream=None) -> None:
        E.et_tree_attention(self.shape, inp.q, inp.k_prefix, inp.v_prefix, inp.kv_row0, inp.prefix_len,
                            inp.k_tree, inp.v_tree, self.mask, self.out, lse=self.lse, ws=self.attn_ws,
                            dev_status=self.dev_status, stream=stream)

    def accept(self, inp: StepInputs, stream=None) -> None:
        E.et_verify_accept(self.cfg, self.mode, self.tree, inp.target, self.accept_len, self.path, self.tokens,
                           self.ws, target_row_of_node=inp.row_of_node,
                           draft_logits=inp.draft if self.mode == E.ET_ACCEPT_STOCH_DRAFTQ else None,
                           draft_row_of_node=inp.row_of_node if self.mode == E.ET_ACCEPT_STOCH_DRAFTQ else None,
                           uniforms=inp.uniforms if self.mode != E.ET_ACCEPT_GREEDY else None,
                           dev_status=self.dev_status, stream=stream)

    def run(self, inp: StepInputs, stream=None) -> None:
        """The whole step: D expands, rerank with mask/posids (one launch), attention, acceptance."""
        self.prepare(inp)
        self.build_tree(inp, stream)
        self.attention(inp, stream)
        self.accept(inp, stream)

    def launches(self) -> int:
        """Kernel launches of one step: the tree (one launch, or D expands and the rerank with mask),
        attention, acceptance."""
        tree = self.cfg.depth + 1 if self.per_layer else E.et_tree_build_launches(self.cfg)
        return tree + 2
