"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle's tests.

This module only draws random numbers and casts them to the storage dtype.  It holds none of the
attention arithmetic, so both the CPU oracle and the GPU path may consume what it produces
without sharing any of the method.

All tensors are drawn on the CPU from ``torch.Generator().manual_seed(seed)`` as standard normals
(the pages' workloads are "inputs ~N(0,1)") and then rounded to the storage dtype:

* ``"bf16"``  -> ``torch.bfloat16``
* ``"fp8"``   -> ``torch.float8_e5m2`` (per-tensor scale 1: the normal value is rounded directly)

The oracle consumes the *stored* values, dequantised exactly to float64.
"""
from __future__ import annotations

import torch

DTYPES = {"bf16": torch.bfloat16, "fp8": torch.float8_e5m2}

# Fixed per-role seed offsets, so that q, k, v, caches never share a stream.
SEED_Q, SEED_K, SEED_V, SEED_CACHE, SEED_LATENT = 0, 1, 2, 3, 4


def normal(shape, seed: int, dtype: str = "bf16", std: float = 1.0) -> torch.Tensor:
    """Return a CPU tensor of the given storage dtype filled with seeded N(0, std^2) draws."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(DTYPES[dtype])


def prefill_inputs(B, Hq, Hkv, S, D, dtype="bf16", seed=0):
    """q [B,Hq,S,D], k/v [B,Hkv,S,D], contiguous, storage dtype."""
    q = normal((B, Hq, S, D), 1000 * seed + SEED_Q, dtype)
    k = normal((B, Hkv, S, D), 1000 * seed + SEED_K, dtype)
    v = normal((B, Hkv, S, D), 1000 * seed + SEED_V, dtype)
    return q, k, v


def decode_inputs(B, Hq, Hkv, Lmax, D, cache_len, seed=0, dtype="bf16", cache_dtype=None):
    """q [B,Hq,D], k/v caches [B,Hkv,Lmax,D], cache_len int32 [B].

    ``cache_len`` may be an int (same for every sequence) or a sequence of B ints.  The caches
    use ``cache_dtype`` (default: ``dtype``).
    """
    cd = dtype if cache_dtype is None else cache_dtype
    q = normal((B, Hq, D), 1000 * seed + SEED_Q, dtype)
    k = normal((B, Hkv, Lmax, D), 1000 * seed + SEED_CACHE, cd)
    v = normal((B, Hkv, Lmax, D), 1000 * seed + SEED_CACHE + 10, cd)
    if isinstance(cache_len, int):
        lens = torch.full((B,), cache_len, dtype=torch.int32)
    else:
        lens = torch.tensor(list(cache_len), dtype=torch.int32)
    return q, k, v, lens


def latent_inputs(B, H, Lmax, cache_len, d_qk=512, seed=0, dtype="bf16", cache_dtype=None):
    """q [B,H,d_qk], latent cache [B,Lmax,d_qk] (``cache_dtype``, default ``dtype``),
    cache_len int32 [B]."""
    q = normal((B, H, d_qk), 1000 * seed + SEED_Q, dtype)
    c = normal((B, Lmax, d_qk), 1000 * seed + SEED_LATENT, dtype if cache_dtype is None else cache_dtype)
    if isinstance(cache_len, int):
        lens = torch.full((B,), cache_len, dtype=torch.int32)
    else:
        lens = torch.tensor(list(cache_len), dtype=torch.int32)
    return q, c, lens


def rope_input(B, H, S, D, dtype="bf16", seed=0):
    return normal((B, H, S, D), 1000 * seed + 7, dtype)
