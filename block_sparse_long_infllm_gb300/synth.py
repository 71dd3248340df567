"""Seeded synthetic inputs for InfLLM v2 block-sparse attention.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no pooling, scoring, selection or attention).  Both the
CUDA path and the fp64 oracle are fed from it.

The pages measure MiniCPM4 on real long prompts (a 128K/140K prompt file, the
needle-in-a-haystack test); neither weights nor prompts exist here, so these
seeded tensors stand in for them, with the shapes the workloads name.

Recipe (one numpy PCG64 stream per workload, seed = 1000 + workload index,
+100 for the "decisive" variant), drawn in this order:
  1. Q  [B, Tq, Hq, d]        ~ N(0, 1) float32
  2. K  [B, Hkv, L_max, d]    ~ N(0, 1) float32, drawn one (b, g) slice at a time
  3. V  [B, Hkv, L_max, d]    ~ N(0, 1) float32, same order
  4. u  [B, Hkv, d]           ~ N(0, I), each row normalised to unit length
  5. planted block indices    per b: n_plant distinct blocks from the planting
                              range, shared by every KV head of that sequence
  6. (tree workloads) parents of the draft tree, then draft K, draft V
                              [B, Hkv, n_draft, d] ~ N(0, 1)
Then Q[b, :, h, :] += sqrt(d) * u[b, h // G] and, for every token of a planted
block, K[b, g, token, :] += beta * u[b, g]; finally every tensor is rounded to
bf16 (round to nearest even) once.  "As written" uses the workload's own
n_plant and beta = 0.5; "decisive" uses n_plant = topk and beta = 4.0.  A
planted block's neighbours share its boundary kernels (16 of their 32 tokens
are planted) and so score about beta/2 above noise; at beta = 4 the weakest
planted block still clears the strongest neighbour by a wide margin.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["Workload", "WORKLOADS", "WORKLOAD_ORDER", "make_inputs", "f32_to_bf16_bits",
           "bf16_bits_to_f32", "plant_range"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "prefill" (causal chunk), "decode" (one token) or "tree"
    B: int
    L: int               # KV tokens per sequence after the call (kv_len)
    Tq: int              # queries per sequence (chunk length, 1, or n_draft)
    Hq: int
    Hkv: int
    d: int
    block_size: int
    kernel_size: int
    kernel_stride: int
    topk: int
    n_init: int
    n_local: int
    dense_len: int
    n_plant: int
    seed: int
    tree_depth: int = 0
    tree_branch: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def L_max(self) -> int:
        return self.L

    @property
    def n_kernels(self) -> int:
        if self.L < self.kernel_size:
            return 0
        return (self.L - self.kernel_size) // self.kernel_stride + 1

    @property
    def q_pos0(self) -> int:
        """Position of the first query of the call (chunk queries are the last Tq tokens)."""
        return self.L - self.Tq if self.kind == "prefill" else self.L - 1

    def params(self) -> dict:
        return dict(block_size=self.block_size, kernel_size=self.kernel_size,
                    kernel_stride=self.kernel_stride, topk=self.topk,
                    n_init_blocks=self.n_init, n_local_blocks=self.n_local,
                    dense_len=self.dense_len, softmax_scale=0.0)

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: tiny causal prefill, 32K decode, 128K decode (batch 4),
# 32K-context chunked prefill, and 64K tree-speculative verification.
WORKLOADS = {
    "tiny_prefill_2k": Workload("tiny_prefill_2k", "prefill", B=1, L=2048, Tq=2048, Hq=2, Hkv=1, d=64,
                                block_size=64, kernel_size=32, kernel_stride=16, topk=4, n_init=1,
                                n_local=2, dense_len=0, n_plant=2, seed=1000),
    "decode_32k": Workload("decode_32k", "decode", B=1, L=32768, Tq=1, Hq=32, Hkv=2, d=128,
                           block_size=64, kernel_size=32, kernel_stride=16, topk=64, n_init=1,
                           n_local=2, dense_len=8192, n_plant=2, seed=1001),
    "decode_128k_b4": Workload("decode_128k_b4", "decode", B=4, L=131072, Tq=1, Hq=32, Hkv=2, d=128,
                               block_size=64, kernel_size=32, kernel_stride=16, topk=64, n_init=1,
                               n_local=2, dense_len=8192, n_plant=8, seed=1002),
    "chunked_prefill_32k": Workload("chunked_prefill_32k", "prefill", B=1, L=32768, Tq=4096, Hq=32,
                                    Hkv=2, d=128, block_size=128, kernel_size=32, kernel_stride=16,
                                    topk=16, n_init=1, n_local=4, dense_len=8192, n_plant=2,
                                    seed=1003),
    "tree_verify_64k": Workload("tree_verify_64k", "tree", B=1, L=65536, Tq=16, Hq=32, Hkv=2, d=128,
                                block_size=64, kernel_size=32, kernel_stride=16, topk=64, n_init=1,
                                n_local=2, dense_len=8192, n_plant=2, seed=1004, tree_depth=5,
                                tree_branch=3),
}
WORKLOAD_ORDER = list(WORKLOADS)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the raw 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def plant_range(w: Workload) -> tuple[int, int]:
    """Blocks that are top-k candidates for every query of the call (never forced).

    For a causal chunk the earliest query sees the fewest blocks; planted blocks
    are drawn below its local window.  A chunk that starts at position 0 has no
    such range, so its planted blocks go right after the initial blocks.
    """
    bt_min = w.q_pos0 // w.block_size
    if w.kind == "tree":
        bt_min = (w.L - 1) // w.block_size
    lo = w.n_init
    hi = bt_min - w.n_local + 1
    if w.kind == "prefill" and hi - lo < w.topk + 1:
        hi = lo + max(w.topk, w.n_plant) + 1
    return lo, hi


def _tree(rng: np.random.Generator, n: int, depth: int, branch: int):
    """Random draft tree: node 0 is the root (depth 1); node i picks its parent
    uniformly among earlier nodes with depth < `depth` and fewer than `branch` children."""
    parent = np.full(n, -1, dtype=np.int32)
    dep = np.zeros(n, dtype=np.int32)
    nchild = np.zeros(n, dtype=np.int32)
    dep[0] = 1
    for i in range(1, n):
        ok = [j for j in range(i) if dep[j] < depth and nchild[j] < branch]
        p = ok[int(rng.integers(len(ok)))]
        parent[i] = p
        dep[i] = dep[p] + 1
        nchild[p] += 1
    mask = np.zeros(n, dtype=np.uint64)
    for i in range(n):
        m = np.uint64(0)
        j = i
        while j >= 0:
            m |= np.uint64(1) << np.uint64(j)
            j = int(parent[j])
        mask[i] = m
    return parent, dep, mask


def make_inputs(w: Workload | str, decisive: bool = False) -> dict:
    """Draw the seeded inputs of workload `w`; bf16 tensors come back as uint16 bit patterns."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    n_plant = w.topk if decisive else w.n_plant
    beta = 4.0 if decisive else 0.5
    rng = np.random.Generator(np.random.PCG64(w.seed + (100 if decisive else 0)))
    B, Tq, Hq, Hkv, d, L = w.B, w.Tq, w.Hq, w.Hkv, w.d, w.L_max
    G = Hq // Hkv

    q = rng.standard_normal((B, Tq, Hq, d), dtype=np.float32)
    k = np.empty((B, Hkv, L, d), dtype=np.float32)
    v = np.empty((B, Hkv, L, d), dtype=np.float32)
    for b in range(B):
        for g in range(Hkv):
            k[b, g] = rng.standard_normal((L, d), dtype=np.float32)
    for b in range(B):
        for g in range(Hkv):
            v[b, g] = rng.standard_normal((L, d), dtype=np.float32)
    u = rng.standard_normal((B, Hkv, d))
    u /= np.linalg.norm(u, axis=-1, keepdims=True)
    lo, hi = plant_range(w)
    n_plant = min(n_plant, hi - lo)
    plant = np.stack([np.sort(rng.choice(np.arange(lo, hi), size=n_plant, replace=False))
                      for _ in range(B)]).astype(np.int32)

    out = {}
    if w.kind == "tree":
        parent, dep, mask = _tree(rng, Tq, w.tree_depth, w.tree_branch)
        dk = rng.standard_normal((B, Hkv, Tq, d), dtype=np.float32)
        dv = rng.standard_normal((B, Hkv, Tq, d), dtype=np.float32)
        out.update(parent=parent, depth=dep, tree_mask=np.tile(mask, (B, 1)),
                   draft_k=f32_to_bf16_bits(dk), draft_v=f32_to_bf16_bits(dv))

    for h in range(Hq):
        q[:, :, h, :] += (math.sqrt(d) * u[:, h // G, :])[:, None, :].astype(np.float32)
    bs = w.block_size
    for b in range(B):
        for g in range(Hkv):
            for blk in plant[b]:
                k[b, g, blk * bs:(blk + 1) * bs, :] += (beta * u[b, g]).astype(np.float32)

    out.update(q=f32_to_bf16_bits(q), k_cache=f32_to_bf16_bits(k), v_cache=f32_to_bf16_bits(v),
               kv_len=np.full(B, w.L, dtype=np.int32), plant=plant, u=u.astype(np.float32),
               beta=beta, n_plant=n_plant)
    return out
