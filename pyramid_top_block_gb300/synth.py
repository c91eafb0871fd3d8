"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only draws random numbers; it holds none of the selection method's
arithmetic.  Every tensor is drawn on the CPU from ``torch.Generator`` with a
fixed seed, in float32, then rounded to bfloat16, so the GPU path and the fp64
oracle see exactly the same values.

Workload shapes follow the selection-latency benchmark of "Block Sparse
Attention with Log-Linear Complexity" (§7.3 Selection latency): random bf16
queries and keys with a fixed seed, batch 1, 32 query heads, 2 KV heads,
d = 64, C = 64, K = 8, g = 2.
"""
from __future__ import annotations

import math

import numpy as np

import torch


def iid(B: int, N: int, Hq: int, Hkv: int, d: int = 64, seed: int = 0):
    """Q [B,N,Hq,d], K [B,N,Hkv,d]: i.i.d. N(0,1), drawn Q first then K, as bf16."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, N, Hq, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(B, N, Hkv, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return q, k


def structured(B: int, N: int, Hq: int, Hkv: int, d: int = 64, seed: int = 1, C: int = 64,
               offset_std: float = 0.5, q_mix: float = 0.5):
    """Keys with a per-block offset and queries that lean toward an earlier block.

    Draw order: offsets o[b, kv, j] ~ N(0, offset_std^2) for every block j of C
    tokens; key noise; query noise; the earlier block j'[b, t, kv], uniform over
    the blocks before t's own block (t's own block when t < C).
      K[b, t, kv, :] = noise + o[b, kv, t // C]               (all-ones direction)
      Q[b, t, h, :]  = noise + q_mix * o[b, kv(h), j'[b, t, kv(h)]]
    with kv(h) = h // (Hq // Hkv).
    """
    g = torch.Generator().manual_seed(seed)
    nblk = math.ceil(N / C)
    o = torch.randn(B, Hkv, nblk, generator=g, dtype=torch.float32) * offset_std
    kn = torch.randn(B, N, Hkv, d, generator=g, dtype=torch.float32)
    qn = torch.randn(B, N, Hq, d, generator=g, dtype=torch.float32)
    u = torch.rand(B, N, Hkv, generator=g, dtype=torch.float64)
    t = torch.arange(N)
    own = t // C
    jp = torch.floor(u * own.view(1, N, 1).to(torch.float64)).to(torch.int64)
    jp = torch.where(own.view(1, N, 1) == 0, torch.zeros_like(jp), jp)
    bidx = torch.arange(B).view(B, 1, 1)
    kvidx = torch.arange(Hkv).view(1, 1, Hkv)
    k_off = o[bidx, kvidx, own.view(1, N, 1)]            # [B, N, Hkv]
    q_off = o[bidx, kvidx, jp]                           # [B, N, Hkv]
    G = Hq // Hkv
    k = (kn + k_off.unsqueeze(-1)).to(torch.bfloat16)
    q_off_h = q_off.repeat_interleave(G, dim=2)          # [B, N, Hq]
    q = (qn + q_mix * q_off_h.unsqueeze(-1)).to(torch.bfloat16)
    return q, k


def decode_context(B: int, n_ctx: int, n_cap: int, Hkv: int, d: int = 64, seed: int = 2):
    """Key cache [B, n_cap, Hkv, d] whose first n_ctx tokens are N(0,1) bf16
    (the rest zero), plus the generator that continues the stream for the steps."""
    g = torch.Generator().manual_seed(seed)
    cache = torch.zeros(B, n_cap, Hkv, d, dtype=torch.bfloat16)
    cache[:, :n_ctx] = torch.randn(B, n_ctx, Hkv, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return cache, g


def decode_step(g: torch.Generator, B: int, Hq: int, Hkv: int, d: int = 64):
    """One decode step's new query [B, Hq, d] and new key [B, Hkv, d], N(0,1) bf16."""
    q = torch.randn(B, Hq, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(B, Hkv, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return q, k


# Named workloads (sizes of the selection-latency benchmark and its variants).
WORKLOADS = {
    "tiny-2k": dict(B=1, N=2048, Hq=4, Hkv=1, K=8, kind="iid", seed=0),
    "latency-4k": dict(B=1, N=4096, Hq=32, Hkv=2, K=8, kind="iid", seed=0),
    "latency-8k": dict(B=1, N=8192, Hq=32, Hkv=2, K=8, kind="iid", seed=0),
    "latency-16k": dict(B=1, N=16384, Hq=32, Hkv=2, K=8, kind="iid", seed=0),
    "latency-32k": dict(B=1, N=32768, Hq=32, Hkv=2, K=8, kind="iid", seed=0),
    "latency-64k": dict(B=1, N=65536, Hq=32, Hkv=2, K=8, kind="iid", seed=0),
    "latency-128k": dict(B=1, N=131072, Hq=32, Hkv=2, K=8, kind="iid", seed=0),
    "latency-256k": dict(B=1, N=262144, Hq=32, Hkv=2, K=8, kind="iid", seed=0),
    "ragged-16421": dict(B=2, N=16421, Hq=32, Hkv=2, K=32, kind="structured", seed=1),
}


def make(name: str):
    """Q, K for a named prefill workload, plus its parameters."""
    w = dict(WORKLOADS[name])
    fn = iid if w["kind"] == "iid" else structured
    q, k = fn(w["B"], w["N"], w["Hq"], w["Hkv"], 64, seed=w["seed"])
    return q, k, w


def random_blocks(B: int, Hkv: int, N: int, K: int, seed: int, C: int = 64, causal: bool = True):
    """Seeded block sets for stage-two tests: for every (b, kv, t), min(K, eligible)
    distinct leaves drawn uniformly from the eligible ones (start <= t when causal),
    ascending, -1 padded.  int32 [B, Hkv, N, K]."""
    rng = np.random.default_rng(seed)
    out = np.full((B, Hkv, N, K), -1, dtype=np.int32)
    M1 = -(-N // C)
    for b in range(B):
        for kv in range(Hkv):
            for t in range(N):
                n_el = min(M1, t // C + 1) if causal else M1
                k = min(K, n_el)
                out[b, kv, t, :k] = np.sort(rng.choice(n_el, size=k, replace=False))
    return torch.from_numpy(out)
