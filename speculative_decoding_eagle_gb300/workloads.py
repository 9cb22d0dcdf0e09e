"""Seeded synthetic inputs for one draft-tree verification step.

This module only draws random numbers and lays them out; it computes nothing
the method defines (no softmax, no ranking, no attention).  Both the CUDA path
(through the tests and ``bench.py``) and the CPU oracle consume what it
returns, so it imports neither of them.

The shapes follow LLaMA2-like heads and vocabulary and EAGLE-2-sized trees
(EAGLE-2 article on sbmmt.com, expansion and reranking paragraphs, and the
EAGLE abstract's LLaMA2-Chat 7B/13B/70B setting); the published evaluation
suites (MT-bench, HumanEval, GSM8K, Alpaca, CNN/DM, Natural Questions) are
replaced by the recipe below, which mimics a confident draft model:

* target logits of node x: a seeded random permutation ``perm`` of the vocab,
  ``target[perm[r]] = -s * ln(r + 1) + N(0, 1)`` (Zipf-skewed ranks, slope
  s = 1.2 unless a test asks for a steeper one);
* draft logits of node x: ``target + sigma * N(0, 1)``;
* Q/K/V ~ N(0, 1), rounded to bf16 (round-to-nearest-even) or kept fp32;
* acceptance uniforms ~ U[0, 1) in fp32;
* ragged KV-prefix lengths ~ U{512 .. 16384} for the batched sweep.

Every draw comes from ``numpy.random.Generator(PCG64(SeedSequence([...])))``
keyed by (workload seed, sequence, node id / stream id), so any sub-part can be
regenerated alone.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

SEED_BASE = 0xEA61E000
ROOT_NODE_SEED_ID = 1 << 20  # seed id of the root node's logit rows
STREAM_QKV = 1
STREAM_UNIFORMS = 2
STREAM_PREFIXES = 3


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes of one synthetic verification step (batch B of sequences)."""

    name: str
    index: int           # selects the seed: SEED_BASE + index
    V: int               # vocabulary
    Hq: int              # query heads
    Hkv: int             # KV heads (Hq % Hkv == 0)
    d: int               # head dim
    prefix: int          # KV-prefix length (ignored when ragged)
    dtype: str           # "bf16" or "f32" for Q/K/V and the attention output
    depth: int           # D
    topk: int            # k
    m: int               # frontier width
    n: int               # kept draft nodes
    sigma: float         # draft noise
    accept: Tuple[str, ...]
    B: int = 1
    temperature: float = 1.0
    ragged: bool = False  # prefixes drawn from U{512..16384}
    slope: float = 1.2    # Zipf slope of the target logits (steeper: more mass on the top ranks)

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def N(self) -> int:
        return self.n + 1

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 0, V=1000, Hq=4, Hkv=4, d=64, prefix=128, dtype="f32",
                     depth=4, topk=4, m=4, n=16, sigma=0.5, accept=("greedy", "stoch")),
    "llama2-7b": Workload("llama2-7b", 1, V=32000, Hq=32, Hkv=32, d=128, prefix=1024,
                          dtype="bf16", depth=6, topk=10, m=10, n=60, sigma=0.5,
                          accept=("greedy",)),
    "llama2-13b": Workload("llama2-13b", 2, V=32000, Hq=40, Hkv=40, d=128, prefix=4096,
                           dtype="bf16", depth=6, topk=10, m=10, n=60, sigma=1.0,
                           accept=("stoch",)),
    "llama2-70b": Workload("llama2-70b", 3, V=32000, Hq=64, Hkv=8, d=128, prefix=8192,
                           dtype="bf16", depth=8, topk=8, m=8, n=80, sigma=0.5,
                           accept=("greedy", "stoch")),
    # batched sweep at the 7B shape; B and n are swept over {1,4,16,32} x {16,32,60,100}
    "sweep-7b": Workload("sweep-7b", 4, V=32000, Hq=32, Hkv=32, d=128, prefix=0,
                         dtype="bf16", depth=6, topk=10, m=10, n=60, sigma=0.5,
                         accept=("stoch",), B=32, ragged=True),
}
SWEEP_B = (1, 4, 16, 32)
SWEEP_N = (16, 32, 60, 100)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


# ---------------------------------------------------------------------------
# bf16 encoding of the inputs (round to nearest, ties to even)
# ---------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> uint16 bf16 bit patterns, round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> the fp32 values they encode (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# logits
# ---------------------------------------------------------------------------
def node_logits(wl: Workload, b: int, seed_id: int) -> Tuple[np.ndarray, np.ndarray]:
    """(target, draft) fp32 rows of one node, both of length V."""
    rng = _rng(wl.seed, b, seed_id)
    perm = rng.permutation(wl.V)
    target64 = np.empty(wl.V, dtype=np.float64)
    target64[perm] = -wl.slope * np.log(np.arange(1, wl.V + 1, dtype=np.float64)) + rng.standard_normal(wl.V)
    draft64 = target64 + wl.sigma * rng.standard_normal(wl.V)
    return target64.astype(np.float32), draft64.astype(np.float32)


def logit_tables(wl: Workload, num_nodes: int, num_draft_nodes: Optional[int] = None,
                 batch: Optional[range] = None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Node-indexed logit tables for a batch.

    Returns ``(target, draft, row_of_node)``:
    * ``target``/``draft``: fp32 ``[B * (num_nodes + 1), V]``; sequence b owns
      rows ``b*(num_nodes+1) ..``, its row 0 is the root, row ``1 + c`` is
      candidate node ``c``;
    * ``row_of_node``: int32 ``[B, num_nodes + 1]``, the table row of each node.

    Draft rows are only drawn for nodes ``c < num_draft_nodes`` (the ones that
    can ever be expanded); the others are left at zero and never read.
    """
    bs = list(batch) if batch is not None else list(range(wl.B))
    nd = num_nodes if num_draft_nodes is None else num_draft_nodes
    R = num_nodes + 1
    target = np.zeros((len(bs) * R, wl.V), dtype=np.float32)
    draft = np.zeros((len(bs) * R, wl.V), dtype=np.float32)
    for i, b in enumerate(bs):
        t, d = node_logits(wl, b, ROOT_NODE_SEED_ID)
        target[i * R], draft[i * R] = t, d
        for c in range(num_nodes):
            t, d = node_logits(wl, b, c)
            target[i * R + 1 + c] = t
            if c < nd:
                draft[i * R + 1 + c] = d
    row_of_node = (np.arange(len(bs), dtype=np.int32)[:, None] * R
                   + np.arange(R, dtype=np.int32)[None, :]).astype(np.int32)
    return target, draft, row_of_node


# ---------------------------------------------------------------------------
# attention operands, uniforms, prefixes
# ---------------------------------------------------------------------------
def prefix_lengths(wl: Workload, B: Optional[int] = None) -> np.ndarray:
    B = wl.B if B is None else B
    if not wl.ragged:
        return np.full(B, wl.prefix, dtype=np.int32)
    return _rng(wl.seed, STREAM_PREFIXES).integers(512, 16385, B).astype(np.int32)


def qkv(wl: Workload, b: int, L: int) -> Dict[str, np.ndarray]:
    """Q/K/V of one sequence.

    Layouts: ``q [N, Hq, d]``, ``k_prefix``/``v_prefix`` ``[Hkv, L, d]``,
    ``k_tree``/``v_tree`` ``[N, Hkv, d]``.  For bf16 workloads the arrays are
    uint16 bit patterns, else fp32.
    """
    rng = _rng(wl.seed, b, STREAM_QKV)
    N = wl.N
    shapes = {"q": (N, wl.Hq, wl.d), "k_prefix": (wl.Hkv, L, wl.d), "v_prefix": (wl.Hkv, L, wl.d),
              "k_tree": (N, wl.Hkv, wl.d), "v_tree": (N, wl.Hkv, wl.d)}
    out = {}
    for name, shp in shapes.items():
        x = rng.standard_normal(shp, dtype=np.float32)
        out[name] = bf16_bits(x) if wl.dtype == "bf16" else x
    return out


def as_float(wl: Workload, arr: np.ndarray) -> np.ndarray:
    """The exact fp32 values of an operand produced by :func:`qkv`."""
    return bf16_value(arr) if wl.dtype == "bf16" else np.asarray(arr, dtype=np.float32)


def uniforms(wl: Workload, b: int, N: Optional[int] = None) -> np.ndarray:
    N = wl.N if N is None else N
    return _rng(wl.seed, b, STREAM_UNIFORMS).random(N, dtype=np.float32)


def root_tokens(wl: Workload, B: Optional[int] = None) -> np.ndarray:
    """Token id of each sequence's root (the last accepted token)."""
    B = wl.B if B is None else B
    return _rng(wl.seed, 0x7007).integers(0, wl.V, B).astype(np.int32)


def static_shape(widths: Sequence[int]):
    """A static draft tree's shape as flat rows: every node at depth d gets
    widths[d] children with ranks 0..widths[d]-1, rows numbered depth by
    depth (parents first).  Returns (parent, rank) int32 [N], parent[0] = -1."""
    parent, rank = [-1], [-1]
    level = [0]
    for w in widths:
        nxt = []
        for p in level:
            for r in range(w):
                parent.append(p)
                rank.append(r)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.asarray(parent, np.int32), np.asarray(rank, np.int32)
