"""Seeded synthetic inputs for the attention forward pass.

This module is the only code that both the CUDA path's tests/bench and the
oracle's tests use.  It draws random numbers and nothing else: it holds none
of the attention arithmetic.

Workloads (shapes and value distributions):

=====  ==========================  ======  ======================================
name   B, H, N, d                  causal  values
=====  ==========================  ======  ======================================
tiny   1, 1, 256, 64               no      Q, K, V i.i.d. N(0,1)
late   2, 8, 1024, 64              both    Q, V ~ N(0,1); K row j scaled by
                                           (1 + 4j/N) so the row max moves late
llama  1, 32, 8192, 128            yes     i.i.d. N(0,1) (Llama-3-8B layer shape)
batch  16, 16, 2048, 128           no      i.i.d. N(0,1)
long   1, 8, 32771, 128            yes     i.i.d. N(0,1); N = 256*128 + 3 leaves a
                                           ragged tail; checked on sampled rows
llama_ 1, 32 (8 K/V), 8192, 128    yes     i.i.d. N(0,1); grouped-query heads
gqa
decode 16, 32 (8 K/V), 8192, 128   n/a     one query row per head against an
                                           8192-position K/V cache (seed 7)
=====  ==========================  ======  ======================================

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; draw Q, then K, then V
with ``torch.randn(B, H, N, d, dtype=float32)`` (K and V with H_kv heads for
grouped-query workloads); apply the K row scaling (the
``late`` workload only, j the 0-based key position inside each head) in
fp32; round to bf16 (round-to-nearest-even).  Default seeds: tiny 1, late 2,
llama 3, batch 4, long 5, llama_gqa 6.  No public dataset is involved: the workloads are
shapes, and random N(0,1) values stand in for activations.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: tuple  # the mask settings this workload is run with
    seed: int
    k_row_ramp: bool = False  # K row j scaled by (1 + 4j/N)
    sampled_rows: int = 0  # >0: parity on this many seeded rows per head
    H_kv: int = 0  # K/V heads (grouped-query attention); 0 means H

    @property
    def scale(self) -> float:
        # 1/sqrt(d) rounded to fp32: the value both sides receive.
        return float(np.float32(1.0 / np.sqrt(self.d)))

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    def flops(self, causal: bool) -> float:
        """Nominal forward FLOPs 4*B*H*N^2*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if causal else f


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 256, 64, (False,), 1),
    "late": Workload("late", 2, 8, 1024, 64, (False, True), 2, k_row_ramp=True),
    "llama": Workload("llama", 1, 32, 8192, 128, (True,), 3),
    "batch": Workload("batch", 16, 16, 2048, 128, (False,), 4),
    "long": Workload("long", 1, 8, 32771, 128, (True,), 5, sampled_rows=512),
    # Llama-3-8B's own head layout: 32 query heads share 8 K/V heads
    "llama_gqa": Workload("llama_gqa", 1, 32, 8192, 128, (True,), 6, H_kv=8),
    # head dimension 256 at the llama workload's FLOP count (16 heads x 256)
    "d256": Workload("d256", 1, 16, 8192, 256, (True,), 8),
}

# Decoding: one new query row per (sequence, head) against a K/V cache of N
# positions; a batch of 16 Llama-3-8B sequences (32 query / 8 K/V heads).
DECODE_WORKLOADS = {
    "decode": Workload("decode", 16, 32, 8192, 128, (False,), 7, H_kv=8),
}


def make_decode(B: int, H: int, H_kv: int, N: int, d: int, seed: int):
    """q [B, H, d] (the newest token), then K, V [B, H_kv, N, d], drawn in
    that order as fp32 N(0,1) and rounded to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, H, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H_kv, N, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H_kv, N, d), generator=g, dtype=torch.float32)
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def make_qkv(B: int, H: int, N: int, d: int, seed: int,
             k_row_ramp: bool = False, H_kv: int = 0):
    """Q [B, H, N, d] and K, V [B, H_kv or H, N, d] as contiguous CPU bf16
    tensors (see the recipe)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    kv_shape = (B, H_kv or H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    v = torch.randn(kv_shape, generator=g, dtype=torch.float32)
    if k_row_ramp:
        j = torch.arange(N, dtype=torch.float32)
        k = k * (1.0 + 4.0 * j / N).view(1, 1, N, 1)
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def make_workload(w: Workload):
    return make_qkv(w.B, w.H, w.N, w.d, w.seed, w.k_row_ramp, w.H_kv)


def make_grad(B: int, H: int, N: int, d: int, seed: int):
    """Output gradient dO [B, H, N, d] for the backward pass: N(0,1) in fp32
    from ``seed + 1000``, rounded to bf16 (its own stream, so Q, K, V of the
    same seed are unchanged)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 1000)
    return torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(
        torch.bfloat16).contiguous()


def fixed_edge_rows(N: int, tile: int = 128) -> list:
    """Rows at tile edges and the ragged tail that are always checked."""
    cand = {0, 1, tile - 1, tile, N - 1}
    last_full = (N // tile) * tile
    cand.update({last_full - 1, last_full, last_full + 1, last_full + 2})
    return sorted(r for r in cand if 0 <= r < N)


def sample_rows(N: int, H: int, count: int, seed: int) -> np.ndarray:
    """Per-head query-row sample: ``default_rng(seed + h).choice(N, count)``
    without replacement, plus the fixed edge rows; int64 [H, R], each row
    sorted."""
    fixed = fixed_edge_rows(N)
    out = []
    for h in range(H):
        rng = np.random.default_rng(seed + h)
        pick = set(int(x) for x in rng.choice(N, size=min(count, N), replace=False))
        pick.update(fixed)
        out.append(sorted(pick))
    width = max(len(r) for r in out)
    # heads can differ in size only if a fixed row was also drawn; pad by
    # repeating the last row so the table is rectangular
    table = np.array([r + [r[-1]] * (width - len(r)) for r in out], dtype=np.int64)
    return table
