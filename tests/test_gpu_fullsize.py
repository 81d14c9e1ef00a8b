"""Parity at the benchmark sizes, in the configuration bench.py times, on sampled outputs.

The full outputs are too large for the float64 oracle (one S=16384 head is an 2 GiB score
matrix), so the oracle recomputes selected rows one by one (each row's definition needs only
that query row and its head's keys and values).  The samples always include the first and last
rows, the rows on both sides of the 128-row tile and 256-row item boundaries, and seeded random
rows, spread over batches and heads.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_prefill_02_gb300 import binding, synthetic

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, FP8_MAX = 2e-2, 2e-3, 8e-2


def sample_rows(B, Hq, S, n_random=24, seed=0):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, 255, 256, S // 2, S // 2 + 127, S - 129, S - 128, S - 2, S - 1]
    rows = []
    for k, i in enumerate(fixed):
        rows.append((k % B, (7 * k) % Hq, min(max(i, 0), S - 1)))
    for _ in range(n_random):
        rows.append((int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(S))))
    return rows


def oracle_rows(q, k, v, rows, causal, rope, theta=10000.0):
    """Oracle rows, converting only the heads the samples touch to float64."""
    B, Hq, S, D = q.shape
    G = Hq // k.shape[1]
    out_o, out_l = [], []
    kv_cache = {}
    for (b, hq, i) in rows:
        h = hq // G
        if (b, h) not in kv_cache:
            kv_cache[(b, h)] = (oracle.as_f64(k[b:b + 1, h:h + 1]), oracle.as_f64(v[b:b + 1, h:h + 1]))
        kk, vv = kv_cache[(b, h)]
        qq = oracle.as_f64(q[b:b + 1, hq:hq + 1])
        # the row of the full problem equals the row of this one-head problem
        o, l = oracle.prefill_rows(qq, kk, vv, [(0, 0, i)], causal=causal, rope=rope, theta=theta)
        out_o.append(o[0])
        out_l.append(l[0])
    return np.array(out_o), np.array(out_l)


def check_rows(o, lse, rows, ro, rl, max_abs, mean_abs):
    got = np.array([oracle.as_f64(o[b, hq, i].cpu()) for (b, hq, i) in rows])
    d = np.abs(got - ro)
    assert np.all(np.isfinite(got))
    assert d.max() <= max_abs, f"max-abs {d.max():.3e}"
    if mean_abs is not None:
        assert d.mean() <= mean_abs, f"mean-abs {d.mean():.3e}"
    gl = np.array([float(lse[b, hq, i]) for (b, hq, i) in rows])
    assert np.abs(gl - rl).max() <= 2e-2


@pytest.mark.parametrize("rope", [1, 2])
def test_causal_prefill_s16384_rope_bf16(rope):
    """Causal GQA prefill, Z=4 Hq=32 Hkv=8 D=128 S=16384, bf16, RoPE 1e4 (the bench step):
    rope=1 rotates K once per call and Q in the kernel, rope=2 both in the kernel."""
    B, Hq, Hkv, S, D = 4, 32, 8, 16384, 128
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=17)
    binding.attn_rope_table_reserve(D, 10000.0, S)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, rope=rope,
                                  rope_theta=10000.0, want_lse=True)
    assert binding.attn_get_device_status() == 0
    rows = sample_rows(B, Hq, S)
    ro, rl = oracle_rows(q, k, v, rows, causal=True, rope=True)
    check_rows(o, lse, rows, ro, rl, BF16_MAX, BF16_MEAN)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_noncausal_prefill_d64_s16384(dtype):
    """Non-causal Z=4 H=32 D=64 S=16384 (the persistent-kernel shape), bf16 and fp8 e5m2."""
    B, H, S, D = 4, 32, 16384, 64
    q, k, v = synthetic.prefill_inputs(B, H, H, S, D, dtype, seed=18)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=False, want_lse=True)
    assert binding.attn_get_device_status() == 0
    rows = sample_rows(B, H, S, n_random=16, seed=1)
    ro, rl = oracle_rows(q, k, v, rows, causal=False, rope=False)
    check_rows(o, lse, rows, ro, rl, FP8_MAX if dtype == "fp8" else BF16_MAX,
               None if dtype == "fp8" else BF16_MEAN)


@pytest.mark.parametrize("rope", [False, True])
def test_causal_prefill_s16384_fp8(rope):
    """Causal GQA D=128 S=16384 in fp8 e5m2, with and without fused RoPE."""
    B, Hq, Hkv, S, D = 4, 32, 8, 16384, 128
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "fp8", seed=19)
    if rope:
        binding.attn_rope_table_reserve(D, 10000.0, S)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, rope=rope,
                                  rope_theta=10000.0, want_lse=True)
    assert binding.attn_get_device_status() == 0
    rows = sample_rows(B, Hq, S, n_random=16, seed=2)
    ro, rl = oracle_rows(q, k, v, rows, causal=True, rope=rope)
    check_rows(o, lse, rows, ro, rl, FP8_MAX, None)


def test_decode_b128_full_config():
    """GQA decode B=128 Hq=32 Hkv=8 D=128, cache 2048, q at 2048: 16 sampled sequences in full."""
    B, Hq, Hkv, L, D = 128, 32, 8, 2048, 128
    q, kc, vc, cl = synthetic.decode_inputs(B, Hq, Hkv, L, D, L, seed=21)
    o, lse = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda(), want_lse=True)
    assert binding.attn_get_device_status() == 0
    pick = sorted(set([0, 1, B - 1] + list(np.random.default_rng(3).integers(B, size=13))))
    ro, rl = oracle.decode(oracle.as_f64(q[pick]), oracle.as_f64(kc[pick]),
                           oracle.as_f64(vc[pick]), cl[pick].numpy())
    d = np.abs(oracle.as_f64(o[pick].cpu()) - ro)
    assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN, (d.max(), d.mean())
    assert np.abs(oracle.as_f64(lse[pick].cpu()) - rl).max() <= 5e-3


def test_latent_decode_b128_full_config():
    """Latent decode B=128, 16 heads, 448 + 64 dims, cache 2048: 16 sampled sequences."""
    B, H, L = 128, 16, 2048
    q, c, cl = synthetic.latent_inputs(B, H, L, L, seed=22)
    o, lse = binding.attn_decode_latent(q.cuda(), c.cuda(), cl.cuda(), want_lse=True)
    assert binding.attn_get_device_status() == 0
    pick = sorted(set([0, 1, B - 1] + list(np.random.default_rng(4).integers(B, size=13))))
    ro, rl = oracle.latent_decode(oracle.as_f64(q[pick]), oracle.as_f64(c[pick]), cl[pick].numpy())
    d = np.abs(oracle.as_f64(o[pick].cpu()) - ro)
    assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN, (d.max(), d.mean())
    assert np.abs(oracle.as_f64(lse[pick].cpu()) - rl).max() <= 5e-3


def test_causal_prefill_d256_s4096_sampled():
    """Causal GQA at head dim 256, Z=4 Hq=32 Hkv=8 S=4096 bf16 with RoPE (the D=256 shape the
    bench times): sampled rows against the oracle."""
    B, Hq, Hkv, S, D = 4, 32, 8, 4096, 256
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=23)
    binding.attn_rope_table_reserve(D, 10000.0, S)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, rope=1,
                                  rope_theta=10000.0, want_lse=True)
    assert binding.attn_get_device_status() == 0
    rows = sample_rows(B, Hq, S, n_random=16, seed=5)
    ro, rl = oracle_rows(q, k, v, rows, causal=True, rope=True)
    check_rows(o, lse, rows, ro, rl, BF16_MAX, BF16_MEAN)


def test_causal_prefill_fp8_d256_s4096_sampled():
    """fp8 e5m2 causal GQA at head dim 256, Z=4 Hq=32 Hkv=8 S=4096 (the shape the bench times in
    fp8; no RoPE at D = 256): sampled rows against the oracle on the dequantised inputs."""
    B, Hq, Hkv, S, D = 4, 32, 8, 4096, 256
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "fp8", seed=26)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, want_lse=True)
    assert binding.attn_get_device_status() == 0
    rows = sample_rows(B, Hq, S, n_random=16, seed=6)
    ro, rl = oracle_rows(q, k, v, rows, causal=True, rope=False)
    check_rows(o, lse, rows, ro, rl, FP8_MAX, 1e-2)


@pytest.mark.parametrize("path", [2, 1], ids=["tcgen05", "mma_sync"])
def test_backward_causal_d128_s4096_group_slice(path):
    """The backward at the size the bench times (causal GQA Z=4 Hq=32 Hkv=8 D=128 S=4096): the
    device computes the whole problem; dQ of the four query heads of one KV head of one batch,
    and that KV head's dK and dV (sums over those four heads), are compared with the oracle's
    gradients of that group in full (every row, every key)."""
    B, Hq, Hkv, S, D = 4, 32, 8, 4096, 128
    G = Hq // Hkv
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=24)
    do = synthetic.normal((B, Hq, S, D), 25, "bf16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = binding.attn_prefill(qd, kd, vd, causal=True, want_lse=True)
    binding.attn_set_backward_path(path)
    try:
        dq, dk, dv = binding.attn_prefill_backward(qd, kd, vd, o, lse, do.cuda(), causal=True)
    finally:
        binding.attn_set_backward_path(0)
    assert binding.attn_get_device_status() == 0
    b, h = 1, 3
    hs = slice(h * G, (h + 1) * G)
    rq, rk, rv = oracle.attention_backward(oracle.as_f64(q[b:b + 1, hs]), oracle.as_f64(k[b:b + 1, h:h + 1]),
                                           oracle.as_f64(v[b:b + 1, h:h + 1]), oracle.as_f64(do[b:b + 1, hs]), True)
    for what, got, ref in (("dQ", dq[b:b + 1, hs], rq), ("dK", dk[b:b + 1, h:h + 1], rk),
                           ("dV", dv[b:b + 1, h:h + 1], rv)):
        g = oracle.as_f64(got.cpu())
        d = np.abs(g - ref)
        assert np.all(np.isfinite(g)), what
        big, mean = np.abs(ref).max(), np.abs(ref).mean()
        # the bounds of the small-shape backward tests (relative to the largest entry and to the
        # mean magnitude; bf16 P and dS before every product, fp32 accumulation)
        assert d.max() <= 2e-2 * big, f"{what}: max-abs {d.max():.3e} > 2e-2 * {big:.3e}"
        assert d.mean() <= 5e-3 * mean, f"{what}: mean-abs {d.mean():.3e} > 5e-3 * {mean:.3e}"
