"""Algorithmic work per launch (useful FLOPs and compulsory HBM bytes) for each entry point.

These counts are what the bench divides by measured time.  They are logical volumes, not
measured DRAM bytes, and useful FLOPs, not issued (padded) tensor-core work — the distinction the
Fixed-budget decode audit — 2026-09-11 draws in "What theory can and cannot establish".
"""
from __future__ import annotations

DTYPE_BYTES = {"bf16": 2, "fp8": 1}


def prefill_flops(B, Hq, S, D, causal, Dv=None):
    """Useful FLOPs of QK^T and PV.

    Non-causal: 2*S*S*D (QK^T) + 2*S*S*Dv (PV) per head.  Causal counts exactly the S(S+1)/2
    scored (query, key) pairs.
    """
    Dv = D if Dv is None else Dv
    pairs = S * (S + 1) // 2 if causal else S * S
    return 2 * B * Hq * pairs * (D + Dv)


def prefill_bytes(B, Hq, Hkv, S, D, dtype="bf16", out_bytes=2):
    """Compulsory HBM bytes: read Q, K, V once, write O once."""
    e = DTYPE_BYTES[dtype]
    return B * Hq * S * D * e + 2 * B * Hkv * S * D * e + B * Hq * S * D * out_bytes


def decode_bytes(B, Hq, Hkv, L, D, dtype="bf16"):
    """Compulsory HBM bytes of one decode step: the K and V history once, q in, o out.

    The history part is 2 * Hkv * D elements per token per sequence — for Hkv=8, D=128 that is
    the audit's 2048 BF16 elements per token per group, 1 GiB at batch 128 / context 2048.
    """
    e = DTYPE_BYTES[dtype]  # cache storage type; q and o are bf16
    return 2 * B * Hkv * L * D * e + B * Hq * D * 2 + B * Hq * D * 2


def decode_flops(B, Hq, L, D):
    """Useful FLOPs: q.k and p.v for every (query head, cached token): 4 * B * Hq * L * D."""
    return 4 * B * Hq * L * D


def latent_bytes(B, H, L, d_qk=512, d_v=448, dtype="bf16"):
    """Compulsory HBM bytes: the latent cache rows once (cache storage type), q in and o out
    (bf16)."""
    e = DTYPE_BYTES[dtype]
    return B * L * d_qk * e + B * H * d_qk * 2 + B * H * d_v * 2


def latent_flops(B, H, L, d_qk=512, d_v=448):
    return 2 * B * H * L * (d_qk + d_v)


def rope_bytes(n_rows, D, dtype="bf16"):
    """Read and write every element once (the cos/sin table is L2-resident and not charged)."""
    return 2 * n_rows * D * DTYPE_BYTES[dtype]
