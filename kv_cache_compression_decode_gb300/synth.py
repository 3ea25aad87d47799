"""Seeded synthetic KV caches shaped like the CacheGen workloads.

This module only draws random numbers. It holds none of the codec's
arithmetic (no anchors, steps, quantization or coding), so that both the CPU
oracle and the CUDA path can take their inputs from it without sharing any
part of the method.

Recipe (one cache, ``[L][2][T][C]`` fp16, C = heads x head_dim):

* per layer ``l``: ``n_outlier`` outlier channels drawn without replacement,
  shared by K and V;
* per (layer, K/V): a per-channel scale ``sigma_c = exp(N(0, 0.5^2))``, times
  20 on the outlier channels; a zero-mean AR(1) process over tokens,
  ``x_0 ~ N(0,1)``, ``x_t = rho * x_{t-1} + sqrt(1 - rho^2) * eps_t``;
  value ``= sigma_c * x_t`` rounded to fp16.

The AR(1) recursion is evaluated in blocks of 64 tokens with a triangular
matrix of powers of rho plus a carried state, which is the same linear filter
evaluated in a different order (fp32 accumulation).  The numbers come from a
``torch.Generator`` seeded with ``seed``; CPU and CUDA generators give
different (equally valid) draws, so a parity check must hand the very same
tensor to both sides.

Token locality of this kind is what the CacheGen paper's "token-wise locality"
section and its Figure 3 (delta vs. original value distribution) describe;
per-channel scales with a few large outlier channels follow its "distribution
along layers, channels, and tokens" section.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

_BLOCK = 64


def _ar1_(eps: torch.Tensor, rho: float) -> torch.Tensor:
    """AR(1) filter over dim -2 of ``eps`` [..., T, C] (fp32)."""
    T, C = eps.shape[-2:]
    lead = eps.shape[:-2]
    a = math.sqrt(max(0.0, 1.0 - rho * rho))
    y = eps.clone()
    if T > 1:
        y[..., 1:, :] *= a
    nb = (T + _BLOCK - 1) // _BLOCK
    pad = nb * _BLOCK - T
    if pad:
        y = torch.cat([y, y.new_zeros(*lead, pad, C)], -2)
    i = torch.arange(_BLOCK, device=eps.device, dtype=torch.float64)
    diff = i[:, None] - i[None, :]
    tri = torch.where(diff >= 0, torch.pow(torch.tensor(rho, dtype=torch.float64), diff.clamp(min=0)),
                      torch.zeros((), dtype=torch.float64))
    tri = tri.to(device=eps.device, dtype=torch.float32)
    pw = torch.pow(torch.tensor(rho, dtype=torch.float64), i + 1).to(device=eps.device, dtype=torch.float32)
    xb = torch.matmul(tri, y.view(*lead, nb, _BLOCK, C))  # [..., nb, B, C]
    for b in range(1, nb):
        xb[..., b, :, :] += pw[:, None] * xb[..., b - 1, -1:, :]
    return xb.reshape(*lead, nb * _BLOCK, C)[..., :T, :]


def ar1_kv(L: int, T: int, C: int, rho: float, n_outlier: int, seed: int,
           device: str | torch.device = "cpu", sigma_log: float = 0.5,
           outlier_scale: float = 20.0, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Return a seeded synthetic KV cache ``[L][2][T][C]`` fp16 on ``device``.

    Draw order per layer: outlier permutation, then for K and V the channel
    scales and the [T][C] normal draws.  Layers are filtered in batches so the
    recursion runs over many layers at once."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    if out is None:
        out = torch.empty((L, 2, T, C), dtype=torch.float16, device=dev)
    assert out.shape == (L, 2, T, C) and out.dtype == torch.float16
    batch = max(1, min(L, (1 << 28) // max(1, 2 * T * C)))  # ~1 GiB of fp32 draws per batch
    for l0 in range(0, L, batch):
        l1 = min(L, l0 + batch)
        eps = torch.empty((l1 - l0, 2, T, C), dtype=torch.float32, device=dev)
        sig = torch.empty((l1 - l0, 2, C), dtype=torch.float32, device=dev)
        for l in range(l0, l1):
            outl = torch.randperm(C, generator=g, device=dev)[:n_outlier]
            for kv in range(2):
                sigma = torch.exp(torch.randn(C, generator=g, device=dev) * sigma_log)
                if n_outlier:
                    sigma[outl] *= outlier_scale
                sig[l - l0, kv] = sigma
                eps[l - l0, kv] = torch.randn((T, C), generator=g, device=dev)
        x = _ar1_(eps, rho)
        out[l0:l1].copy_((x * sig[:, :, None, :]).to(torch.float16))
        del eps, x
    return out


def seeded_ints(seed: int, low: int, high_inclusive: int, n: int) -> List[int]:
    """``n`` integers uniform in [low, high_inclusive] from a CPU generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return [int(v) for v in torch.randint(low, high_inclusive + 1, (n,), generator=g)]


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and generator parameters of one synthetic KV-cache workload."""
    name: str
    L: int
    T: int
    C: int
    rho: float
    n_outlier: int
    seed: int = 0
    chunk_tokens: int = 0        # 0: one chunk covering the whole cache
    tokens_per_stream: int = 1536
    group_size: int = 10

    @property
    def chunk(self) -> int:
        return self.chunk_tokens if self.chunk_tokens else self.T

    @property
    def values(self) -> int:
        return self.L * 2 * self.T * self.C

    @property
    def fp16_bytes(self) -> int:
        return 2 * self.values

    def generate(self, device="cpu") -> torch.Tensor:
        return ar1_kv(self.L, self.T, self.C, self.rho, self.n_outlier, self.seed, device=device)


# The five workload shapes (heads x head_dim = C).
TINY = Workload("tiny-4L-256T-8x128", 4, 256, 1024, 0.95, 2, 0, 0, 1536)
# Tokens per stream: a decode block serves one (layer, K/V, 32-channel group)
# with one warp per stream, so the stream length sets the warps per block --
# 12 for the 16384-token Llama-70B slices, 10 for the 4096-token Llama-7B
# slices, 3 per 1536-token chunk for the chunked Mistral-7B cache.
LLAMA7B = Workload("llama7b-mha-32L-4096T-32x128", 32, 4096, 4096, 0.95, 2, 0, 0, 410)
MISTRAL7B = Workload("mistral7b-gqa-32L-16384T-8x128-chunk1536", 32, 16384, 1024, 0.95, 2, 0, 1536, 512)
LLAMA70B = Workload("llama70b-gqa-80L-16384T-8x128", 80, 16384, 1024, 0.9, 4, 0, 0, 1366)

# Mixed-level chunk decode: three step multipliers, one level per chunk.
LEVEL_MULTIPLIERS = (1.0, 2.0, 4.0)


def mixed_levels(n_chunks: int, seed: int = 0) -> List[int]:
    """Per-chunk quality level (index into LEVEL_MULTIPLIERS), seeded."""
    return seeded_ints(seed, 0, len(LEVEL_MULTIPLIERS) - 1, n_chunks)


# Streamed batched decode: 64 contexts of a Llama-34B-shaped cache.
STREAM_L, STREAM_C, STREAM_CHUNK = 48, 1024, 1536
STREAM_CONTEXTS = 64


def stream_context_lengths(n: int = STREAM_CONTEXTS, seed: int = 0,
                           lo: int = 1400, hi: int = 16384) -> List[int]:
    """Context lengths uniform in [1.4K, 16K] tokens (seeded)."""
    return seeded_ints(seed, lo, hi, n)


def stream_context(j: int, T: int, L: int = STREAM_L, C: int = STREAM_C, device="cpu") -> torch.Tensor:
    """Context ``j`` of the streamed workload (seed 1 + j, rho 0.95, 2 outliers)."""
    return ar1_kv(L, T, C, 0.95, 2, 1 + j, device=device)


def small(name: str, L: int, T: int, C: int, seed: int = 0, rho: float = 0.95, n_outlier: int = 2,
          chunk_tokens: int = 0, tokens_per_stream: int = 1536, group_size: int = 10) -> Workload:
    """A reduced workload for tests (same recipe, chosen sizes)."""
    return Workload(name, L, T, C, rho, n_outlier, seed, chunk_tokens, tokens_per_stream, group_size)
