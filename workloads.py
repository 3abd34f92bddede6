"""Seeded synthetic inputs for the Purlin collective workloads.

This module only draws random inputs and per-rank counts.  It holds none of the
collectives' arithmetic (no sums, no layouts, no roundings of results), and both
sides of every parity check -- the CPU oracle and the CUDA library -- receive the
same bytes from it.

Workloads (all synthetic; the pages name no dataset):
  allreduce_r2_f32      AllReduce, R=2, fp32, 4096 elements per rank, integer
                        values uniform in [-8, 8] (sums are exact in any order).
  rs_ag_r8_bf16         ReduceScatter then AllGather, R=8, bf16, 64 MiB per rank
                        (8 partitions of 8 MiB), N(0,1).
  allreduce_sweep_r8    AllReduce, R=8, bf16, 4 KiB .. 256 MiB per rank in powers
                        of 4, N(0,1).
  moe_a2av_r8           AllToAllV MoE dispatch, R=8, 4096 tokens per source,
                        hidden 7168, bf16 N(0,1); destination of every token drawn
                        from Zipf(s=1.2) over the 8 ranks; then the inverse.
  dp_attn_agv_rsv_r8    AllGatherV + ReduceScatterV, R=8, per-rank token counts
                        uniform in [1, 2048], hidden 7168, bf16 N(0,1); plus a
                        1 GiB-total AllGather (128 MiB in per rank) and a 1 GiB per
                        rank AllReduce.

Random streams: values come from ``torch.Generator`` seeded per (workload, role,
rank) on the device the buffer is created on; counts come from numpy's PCG64.
"""
from __future__ import annotations

import numpy as np
import torch

SEED_BASE = 20260929

KiB = 1024
MiB = 1024 * KiB
GiB = 1024 * MiB

HIDDEN = 7168
ZIPF_S = 1.2

# Per-rank AllReduce message sizes of the sweep: 4 KiB * 4**i, i = 0..8.
SWEEP_BYTES = [4 * KiB * 4 ** i for i in range(9)]
# SNAC chunk sizes of the sweep (bytes per rank per step): 64 KiB .. 2 MiB.
SWEEP_CHUNKS = [64 * KiB * 2 ** i for i in range(6)]

WORKLOADS = {
    "allreduce_r2_f32": dict(R=2, dtype="f32", count=4096, values="int[-8,8]"),
    "rs_ag_r8_bf16": dict(R=8, dtype="bf16", count=64 * MiB // 2, values="N(0,1)"),
    "allreduce_sweep_r8": dict(R=8, dtype="bf16", bytes=SWEEP_BYTES, chunks=SWEEP_CHUNKS,
                               values="N(0,1)"),
    "moe_a2av_r8": dict(R=8, dtype="bf16", tokens=4096, hidden=HIDDEN, zipf_s=ZIPF_S,
                        values="N(0,1)"),
    "dp_attn_agv_rsv_r8": dict(R=8, dtype="bf16", tokens=(1, 2048), hidden=HIDDEN,
                               ag_bytes_per_rank=128 * MiB, ar_bytes_per_rank=1 * GiB,
                               values="N(0,1)"),
}

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def seed_for(workload: str, role: int = 0, rank: int = 0) -> int:
    """Deterministic seed for one buffer of one workload."""
    index = list(WORKLOADS).index(workload) + 1
    return SEED_BASE + 100_000 * index + 1_000 * role + rank


def torch_dtype(dtype: str) -> torch.dtype:
    return _TORCH_DTYPES[dtype]


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def normal_buffer(n: int, dtype: str, seed: int, device="cpu") -> torch.Tensor:
    """n draws of N(0,1) in fp32, narrowed to ``dtype`` by torch (ties to even)."""
    g = _generator(seed, device)
    x = torch.randn(n, generator=g, dtype=torch.float32, device=device)
    return x.to(_TORCH_DTYPES[dtype])


def int_buffer(n: int, lo: int, hi: int, dtype: str, seed: int, device="cpu") -> torch.Tensor:
    """n integers uniform in [lo, hi] (inclusive), stored as ``dtype``."""
    g = _generator(seed, device)
    x = torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int32, device=device)
    return x.to(_TORCH_DTYPES[dtype])


def rank_buffers(workload: str, R: int, n: int, dtype: str, role: int = 0,
                 device="cpu", values: str = "normal") -> list[torch.Tensor]:
    """One input buffer per virtual rank, each from its own seeded stream."""
    out = []
    for r in range(R):
        s = seed_for(workload, role, r)
        if values == "normal":
            out.append(normal_buffer(n, dtype, s, device))
        else:
            out.append(int_buffer(n, -8, 8, dtype, s, device))
    return out


def zipf_pair_counts(R: int, tokens_per_src: int, s: float, seed: int) -> np.ndarray:
    """Tokens sent from source rank a to destination rank b, as an R x R matrix.

    Every token of every source picks its destination independently with
    P(b) proportional to (b + 1) ** -s.  Grouping a source's tokens by destination
    (a stable sort, done as input preparation) makes each (a, b) block contiguous,
    so only the counts are needed to lay the send buffer out.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    p = np.arange(1, R + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    counts = np.zeros((R, R), dtype=np.int64)
    for a in range(R):
        dest = rng.choice(R, size=tokens_per_src, p=p)
        counts[a] = np.bincount(dest, minlength=R)
    return counts


def uniform_token_counts(R: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Per-rank token counts uniform on the integers lo..hi (inclusive)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(lo, hi + 1, size=R, dtype=np.int64)


def random_counts(R: int, max_count: int, seed: int, zero_prob: float = 0.2) -> np.ndarray:
    """Small random per-rank counts for edge-case tests (zeros included)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    c = rng.integers(0, max_count + 1, size=R, dtype=np.int64)
    c[rng.random(R) < zero_prob] = 0
    return c


def random_pair_counts(R: int, max_count: int, seed: int, zero_prob: float = 0.2) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    c = rng.integers(0, max_count + 1, size=(R, R), dtype=np.int64)
    c[rng.random((R, R)) < zero_prob] = 0
    return c
