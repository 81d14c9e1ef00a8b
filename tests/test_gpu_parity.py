"""GPU parity: every entry point, called through the C ABI, against the float64 oracle on the
same seeded inputs.

Tolerances (the required parity bounds): bf16 outputs max-abs <= 2e-2 and mean-abs <= 2e-3; fp8 e5m2 max-abs
<= 8e-2 (oracle on the dequantised inputs).  LSE is compared to 5e-3 absolute (its error is the
relative error of the row sum, which bf16 rounding of P keeps near 1e-3).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_attn_prefill_02_gb300 import binding, synthetic

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, FP8_MAX, LSE_TOL = 2e-2, 2e-3, 8e-2, 5e-3
# LSE of a prefill whose Q and K are rotated by the library: the rotated values are rounded to
# bf16 before Q K^T, which moves each score by up to 2 * 2^-9 * scale * sum_i |q_i k_i| (about
# 0.03 worst case at D = 128 with N(0,1) inputs, ~1e-3 typical); 1e-2 bounds thousands of rows.
ROPE_LSE_TOL = 1e-2


def f64(t):
    return oracle.as_f64(t)


def check(gpu, ref, max_abs=BF16_MAX, mean_abs=BF16_MEAN, what=""):
    g = f64(gpu)
    d = np.abs(g - ref)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    assert d.max() <= max_abs, f"{what}: max-abs {d.max():.3e} > {max_abs}"
    if mean_abs is not None:
        assert d.mean() <= mean_abs, f"{what}: mean-abs {d.mean():.3e} > {mean_abs}"


def status_ok():
    assert binding.attn_get_device_status() == 0


# --------------------------------------------------------------------------------------------
# rope_apply
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("shape,pos0", [((2, 3, 37, 64), 5), ((1, 2, 130, 128), 0),
                                        ((1, 1, 3, 6), 11), ((2, 4, 256, 128), 16000),
                                        ((3, 9, 41, 128), 7),      # heads not a multiple of 4
                                        ((1, 32, 300, 64), 0)])
def test_rope_apply_bf16(shape, pos0):
    x = synthetic.rope_input(*shape, dtype="bf16", seed=1)
    y = binding.rope_apply(x.cuda(), pos0=pos0, theta=10000.0)
    torch.cuda.synchronize()
    ref = oracle.rope_rotate_half(f64(x), pos0 + np.arange(shape[2]), 10000.0)
    check(y.cpu(), ref, what="rope bf16")
    # the kernel rounds once to bf16: it must agree with the rounded oracle almost everywhere
    rounded = torch.from_numpy(ref).to(torch.bfloat16)
    assert (y.cpu() == rounded).float().mean() > 0.99


@pytest.mark.parametrize("H", [2, 7])
def test_rope_apply_fp8_heads(H):
    """fp8 e5m2 out of place, few heads and several (the per-position kernel walks the heads)."""
    x = synthetic.rope_input(2, H, 70, 128, dtype="fp8", seed=H)
    y = binding.rope_apply(x.cuda(), pos0=9, theta=10000.0)
    torch.cuda.synchronize()
    ref = oracle.rope_rotate_half(f64(x), 9 + np.arange(70), 10000.0)
    rounded = torch.from_numpy(ref).to(torch.float8_e5m2)
    g, r = f64(y.cpu()), f64(rounded)
    step = np.maximum(np.abs(r), 2.0 ** -14) * 0.25
    assert np.all(np.abs(g - r) <= step * 1.0001)
    assert (g == r).mean() > 0.99


def test_rope_apply_in_place_and_fp8():
    x = synthetic.rope_input(2, 2, 50, 64, dtype="fp8", seed=2)
    xd = x.cuda()
    binding.rope_apply(xd, xd, pos0=3, theta=500.0)
    torch.cuda.synchronize()
    ref = oracle.rope_rotate_half(f64(x), 3 + np.arange(50), 500.0)
    rounded = torch.from_numpy(ref).to(torch.float8_e5m2)
    agree = (xd.cpu().float() == rounded.float()).float().mean().item()
    assert agree > 0.99, agree
    # disagreements are at most one e5m2 step (rounding of a float32 vs float64 value)
    g, r = f64(xd.cpu()), f64(rounded)
    step = np.maximum(np.abs(r), 2.0 ** -14) * 0.25
    assert np.all(np.abs(g - r) <= step * 1.0001)


# --------------------------------------------------------------------------------------------
# prefill
# --------------------------------------------------------------------------------------------

PREFILL_CASES = [
    # B, Hq, Hkv, S, D, causal
    (1, 4, 1, 128, 64, True),      # the tiny config's shape
    (1, 4, 1, 128, 64, False),
    (2, 4, 2, 640, 128, True),     # several tiles, two items per head, GQA
    (1, 2, 2, 300, 128, True),     # ragged tail
    (1, 2, 1, 77, 64, False),      # shorter than one tile
    (1, 1, 1, 1, 128, True),       # S = 1
    (1, 8, 8, 513, 64, True),      # ragged, MHA
    (1, 2, 1, 1000, 128, False),   # ragged non-causal, many KV tiles
]


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", PREFILL_CASES)
def test_prefill_bf16(B, Hq, Hkv, S, D, causal):
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=S)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, want_lse=True)
    status_ok()
    ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=causal)
    check(o.cpu(), ro, what="O")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE")


@pytest.mark.parametrize("dtype,B,Hq,Hkv,S,D,causal,rope", [
    ("bf16", 2, 4, 2, 640, 128, True, 0),     # several items per head, GQA
    ("bf16", 1, 8, 8, 513, 64, True, 0),      # ragged, MHA, D = 64
    ("bf16", 1, 4, 1, 1100, 128, True, 1),    # RoPE through the rotation passes
    ("bf16", 1, 2, 2, 1030, 64, True, 2),     # RoPE inside the kernel
    ("bf16", 1, 2, 1, 1000, 128, False, 0),   # non-causal, ragged
    ("fp8", 1, 4, 1, 640, 128, True, 0),
    ("fp8", 2, 2, 2, 300, 128, True, 1),      # fp8 with the staged in-kernel RoPE
    ("fp8", 1, 4, 4, 256, 64, False, 0),
])
def test_prefill_one_tile_per_item(dtype, B, Hq, Hkv, S, D, causal, rope):
    """The second tile configuration (one 128-row Q tile per work item) gives the same
    attention as the oracle."""
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, dtype, seed=S + 71)
    try:
        binding.attn_set_prefill_tiles(1)
        o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, rope=rope,
                                      rope_theta=10000.0, want_lse=True)
        status_ok()
    finally:
        binding.attn_set_prefill_tiles(0)
    ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=causal, rope=bool(rope),
                            theta=10000.0)
    if dtype == "fp8":
        check(o.cpu(), ro, FP8_MAX, 1e-2, what="O fp8, one tile per item")
        check(lse.cpu(), rl, 2e-2, None, what="LSE fp8, one tile per item")
    else:
        check(o.cpu(), ro, what="O, one tile per item")
        check(lse.cpu(), rl, ROPE_LSE_TOL if rope else LSE_TOL, None,
              what="LSE, one tile per item")


def test_prefill_unfused_rope_tiny_config():
    """Tiny config: B=1, Hq=4, Hkv=1, S=128, D=64, RoPE 1e4 via rope_apply then attention."""
    q, k, v = synthetic.prefill_inputs(1, 4, 1, 128, 64, "bf16", seed=0)
    qd, kd = binding.rope_apply(q.cuda()), binding.rope_apply(k.cuda())
    o = binding.attn_prefill(qd, kd, v.cuda(), causal=True)
    status_ok()
    ro, _ = oracle.prefill(f64(q), f64(k), f64(v), causal=True, rope=True, theta=10000.0)
    check(o.cpu(), ro, what="O")


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,pos0,rope", [
    (1, 4, 1, 128, 64, True, 0, 1),       # the tiny config: RoPE fused into the Q/K loads
    (2, 8, 2, 700, 128, True, 0, 1),      # GQA, ragged tail, several items per head
    (1, 2, 2, 300, 64, False, 5000, 1),   # non-causal, positions offset
    (1, 4, 1, 257, 128, True, 3, 1),      # one row past a whole item
    (1, 4, 1, 1100, 128, True, 0, 1),     # long enough that K is rotated once per call
    (1, 4, 4, 1500, 64, False, 77, 1),    # the same path at D = 64, non-causal, offset
    (1, 4, 1, 1100, 128, True, 0, 2),     # forced: K rotated in every query block
    (1, 2, 2, 1030, 64, True, 9, 2),
])
def test_prefill_fused_rope(B, Hq, Hkv, S, D, causal, pos0, rope):
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=S + 1)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, rope=rope,
                                  rope_theta=10000.0, pos0=pos0, want_lse=True)
    status_ok()
    ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=causal, rope=True, theta=10000.0,
                            pos0=pos0)
    check(o.cpu(), ro, what="O")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE")


def test_prefill_fused_equals_unfused_closely():
    """Fused RoPE and rope_apply + attention round the rotated Q/K identically (both bf16)."""
    q, k, v = synthetic.prefill_inputs(1, 8, 2, 512, 128, "bf16", seed=4)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    of = binding.attn_prefill(qd, kd, vd, causal=True, rope=True)
    ou = binding.attn_prefill(binding.rope_apply(qd), binding.rope_apply(kd), vd, causal=True)
    status_ok()
    assert (of.float() - ou.float()).abs().max().item() <= 1e-2


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", [
    (1, 4, 4, 256, 64, False),     # non-causal D=64 (the persistent-kernel shape, fp8)
    (1, 4, 1, 640, 128, True),     # causal GQA D=128, several items
    (2, 2, 2, 333, 64, True),      # ragged, causal
    (1, 2, 1, 1000, 128, False),   # ragged non-causal
])
def test_prefill_fp8_e5m2(B, Hq, Hkv, S, D, causal):
    """fp8 e5m2 Q/K/V (per-tensor scale 1); the oracle runs on the dequantised values."""
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "fp8", seed=S + 3)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, want_lse=True)
    status_ok()
    ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=causal)
    check(o.cpu(), ro, FP8_MAX, 1e-2, what="O fp8")
    check(lse.cpu(), rl, 2e-2, None, what="LSE fp8")


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,pos0", [
    (1, 4, 1, 640, 128, True, 0),      # causal GQA fp8, RoPE fused (config shape, small S)
    (2, 2, 2, 300, 128, True, 7),      # ragged, offset positions
    (1, 2, 1, 520, 128, False, 0),     # non-causal
])
def test_prefill_fp8_fused_rope(B, Hq, Hkv, S, D, causal, pos0):
    """fp8 e5m2 Q/K/V with RoPE fused: rotated Q/K are kept in bf16 inside the kernel."""
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "fp8", seed=S + 11)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, rope=True,
                                  rope_theta=10000.0, pos0=pos0, want_lse=True)
    status_ok()
    ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=causal, rope=True, theta=10000.0,
                            pos0=pos0)
    check(o.cpu(), ro, FP8_MAX, 1e-2, what="O fp8 rope")
    check(lse.cpu(), rl, 2e-2, None, what="LSE fp8 rope")


def test_prefill_fp8_scales():
    """Dequantisation scales: q,k,v stored as x/scale give the same attention as x itself."""
    B, H, S, D = 1, 2, 200, 128
    q, k, v = synthetic.prefill_inputs(B, H, H, S, D, "fp8", seed=5)
    o1 = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=True)
    # halve the stored q (exact in e5m2 for normal values) and pass q_scale = 2
    qh = (q.float() / 2).to(torch.float8_e5m2)
    o2 = binding.attn_prefill(qh.cuda(), k.cuda(), v.cuda(), causal=True, q_scale=2.0)
    vh = (v.float() / 4).to(torch.float8_e5m2)
    o3 = binding.attn_prefill(q.cuda(), k.cuda(), vh.cuda(), causal=True, v_scale=4.0)
    status_ok()
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (o1.float() - o3.float()).abs().max().item() <= 1e-2


def test_prefill_large_logits_rescale_path():
    """Rows whose maximum grows late force the lazy O rescale; scale 1 makes logits large."""
    B, Hq, Hkv, S, D = 1, 2, 1, 700, 64
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=9)
    k = (f64(k) * np.linspace(0.2, 3.0, S)[None, None, :, None])
    k = torch.from_numpy(k).to(torch.bfloat16)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, softmax_scale=1.0,
                                  want_lse=True)
    status_ok()
    ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=True, scale=1.0)
    check(o.cpu(), ro, 3e-2, BF16_MEAN, what="O")
    np.testing.assert_allclose(f64(lse.cpu()), rl, rtol=2e-3, atol=2e-2)


# --------------------------------------------------------------------------------------------
# decode
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("B,Hq,Hkv,D,Lmax,lens", [
    (1, 32, 8, 128, 2048, [2048]),            # the decode config at batch 1 (split KV)
    (3, 32, 8, 128, 2048, [2048, 1, 777]),    # ragged lengths, one single-key sequence
    (8, 32, 8, 128, 2048, 2048),              # batch 8 (split KV)
    (2, 8, 1, 64, 300, [300, 129]),           # D = 64, group 8, Lmax not a tile multiple
    (2, 16, 1, 128, 100, [64, 100]),          # group of 16 fills the MMA tile
])
def test_decode_bf16(B, Hq, Hkv, D, Lmax, lens):
    q, kc, vc, cl = synthetic.decode_inputs(B, Hq, Hkv, Lmax, D, lens, seed=B)
    o, lse = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda(), want_lse=True)
    status_ok()
    ro, rl = oracle.decode(f64(q), f64(kc), f64(vc), cl.numpy(), rope=True, theta=10000.0)
    check(o.cpu(), ro, what="O")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE")


@pytest.mark.parametrize("B,Hq,Hkv,lens", [
    (1, 32, 8, [2048]), (3, 32, 8, [2048, 1, 777]), (8, 32, 8, 2048), (40, 32, 8, 1500),
    (2, 8, 8, [5, 2048]),            # group of 1
    (3, 64, 8, [300, 2048, 64]),     # group of 8: one full column tile
    (3, 24, 2, [1999, 65, 2048]),    # group of 12: two column tiles, the second ragged
    (2, 32, 2, [2048, 129]),         # group of 16
])
def test_decode_fp8_cache(B, Hq, Hkv, lens):
    """fp8 e5m2 K/V cache (q bf16): the kernel widens the cache exactly, so bf16 bounds hold."""
    q, kc, vc, cl = synthetic.decode_inputs(B, Hq, Hkv, 2048, 128, lens, seed=B + Hq + 50,
                                            cache_dtype="fp8")
    o, lse = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda(), want_lse=True)
    status_ok()
    ro, rl = oracle.decode(f64(q), f64(kc), f64(vc), cl.numpy(), rope=True, theta=10000.0)
    check(o.cpu(), ro, what="O fp8 cache")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE fp8 cache")


@pytest.mark.parametrize("nsplit", [1, 3, 32])
def test_decode_forced_splits(nsplit):
    """The global-split hook gives the same attention whatever the split count."""
    q, kc, vc, cl = synthetic.decode_inputs(3, 32, 8, 2048, 128, [2048, 77, 1500], seed=60 + nsplit)
    try:
        binding.attn_set_decode_splits(nsplit)
        o, lse = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda(), want_lse=True)
        status_ok()
    finally:
        binding.attn_set_decode_splits(0)
    ro, rl = oracle.decode(f64(q), f64(kc), f64(vc), cl.numpy(), rope=True, theta=10000.0)
    check(o.cpu(), ro, what=f"O split {nsplit}")
    check(lse.cpu(), rl, LSE_TOL, None, what=f"LSE split {nsplit}")


def test_decode_bad_cache_len_sets_status():
    q, kc, vc, cl = synthetic.decode_inputs(2, 8, 2, 64, 64, [64, 64], seed=1)
    cl[1] = 65  # > Lmax
    o = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda())
    assert binding.attn_get_device_status() == 7  # ATTN_ERR_DEVICE_ARG
    assert binding.attn_get_device_status() == 0  # cleared
    ro, _ = oracle.decode(f64(q[:1]), f64(kc[:1]), f64(vc[:1]), cl[:1].numpy())
    check(o[:1].cpu(), ro, what="valid row")
    assert torch.all(o[1].cpu() == 0)


# --------------------------------------------------------------------------------------------
# chunked prefill against a static cache
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,D,Hq,Hkv,Sq,Skv,pitch,rope", [
    ("bf16", 128, 8, 2, 32, 300, 320, True),     # a 32-row chunk, offset not a tile multiple
    ("bf16", 128, 8, 2, 1, 257, 257, True),      # one row after a ragged cache
    ("bf16", 128, 4, 1, 200, 700, 704, True),    # two query tiles, a partial item
    ("bf16", 128, 8, 2, 384, 384, 512, True),    # the whole prompt as one chunk
    ("bf16", 128, 8, 2, 96, 1000, 1000, False),
    ("bf16", 64, 8, 8, 64, 1000, 1024, True),
    ("fp8", 128, 8, 2, 128, 513, 640, True),     # fp8: rotated q in bf16, keys widened as stored
    ("fp8", 64, 4, 4, 50, 333, 333, False),
])
def test_prefill_chunk(dtype, D, Hq, Hkv, Sq, Skv, pitch, rope):
    B = 2
    q = synthetic.normal((B, Hq, Sq, D), 900 + Sq, dtype)
    kc = synthetic.normal((B, Hkv, pitch, D), 901 + Skv, dtype)
    vc = synthetic.normal((B, Hkv, pitch, D), 902 + Skv, dtype)
    o, lse = binding.attn_prefill_chunk(q.cuda(), kc.cuda(), vc.cuda(), Skv, rope=rope,
                                        rope_theta=10000.0, want_lse=True)
    status_ok()
    ro, rl = oracle.prefill_chunk(f64(q), f64(kc), f64(vc), Skv, rope=rope, theta=10000.0)
    if dtype == "fp8":
        check(o.cpu(), ro, FP8_MAX, 1e-2, what="O chunk fp8")
    else:
        check(o.cpu(), ro, what="O chunk")
    check(lse.cpu(), rl, 2e-2 if dtype == "fp8" else LSE_TOL, None, what="LSE chunk")


def test_prefill_chunk_rejects_bad_lengths():
    q = torch.zeros((1, 4, 8, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 4, 16, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.AttnError):
        binding.attn_prefill_chunk(q, kc, kc, 7)      # Sq > Skv
    with pytest.raises(binding.AttnError):
        binding.attn_prefill_chunk(q, kc, kc, 17)     # Skv > cache rows


# --------------------------------------------------------------------------------------------
# growing decode: the current token joins the cache
# --------------------------------------------------------------------------------------------

def _append_inputs(B, Hq, Hkv, Lmax, D, lens, seed):
    q, kc, vc, cl = synthetic.decode_inputs(B, Hq, Hkv, Lmax, D, lens, seed=seed)
    kn = synthetic.normal((B, Hkv, D), 1000 * seed + 77)
    vn = synthetic.normal((B, Hkv, D), 1000 * seed + 78)
    return q, kc, vc, cl, kn, vn


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,D,lens", [
    (3, 32, 8, 2048, 128, [2047, 1, 700]),   # last free row, a one-key history, a middle one
    (2, 8, 2, 300, 64, [5, 256]),
    (5, 16, 1, 600, 128, [599, 129, 128, 1, 300]),   # group of 16
    (40, 32, 8, 520, 128, 400),
])
def test_decode_append(B, Hq, Hkv, Lmax, D, lens):
    q, kc, vc, cl, kn, vn = _append_inputs(B, Hq, Hkv, Lmax, D, lens, seed=B + D)
    gk, gv, gl = kc.cuda(), vc.cuda(), cl.cuda()
    o, lse = binding.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), gk, gv, gl,
                                        want_lse=True, rope=True, rope_theta=10000.0)
    status_ok()
    ro, rl, krow = oracle.decode_append(f64(q), f64(kc), f64(vc), cl.numpy(), f64(kn), f64(vn),
                                        rope=True, theta=10000.0)
    check(o.cpu(), ro, what="O append")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE append")
    assert torch.equal(gl.cpu(), cl + 1)
    gk, gv = gk.cpu(), gv.cpu()
    for b in range(B):
        L = int(cl[b])
        # the new row: the rotated key rounded to bf16, the value as given
        np.testing.assert_allclose(f64(gk[b, :, L]), krow[b], rtol=0, atol=1.6e-2)
        assert torch.equal(gv[b, :, L], vn[b])
        # every other row is untouched
        assert torch.equal(gk[b, :, :L], kc[b, :, :L])
        assert torch.equal(gk[b, :, L + 1:], kc[b, :, L + 1:])


def test_decode_append_graph_replays_grow_the_cache():
    """One captured step replayed three times: each replay reads the length it left behind."""
    B, Hq, Hkv, Lmax, D, steps = 4, 32, 8, 1100, 128, 3
    q, kc, vc, cl, kn, vn = _append_inputs(B, Hq, Hkv, Lmax, D, [1000, 7, 511, 1024], seed=5)
    dq, dkn, dvn = q.cuda(), kn.cuda(), vn.cuda()
    gk, gv, gl = kc.cuda(), vc.cuda(), cl.cuda()
    o = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(binding.attn_decode_append_workspace_size(B, Hq, Hkv, D, Lmax),
                     dtype=torch.uint8, device="cuda")
    binding.attn_rope_table_reserve(D, 10000.0, Lmax + 1)
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            binding.attn_decode_append(dq, dkn, dvn, gk, gv, gl, o=o, workspace=ws, stream=st)
    torch.cuda.synchronize()
    assert torch.equal(gl.cpu(), cl)  # capturing ran nothing
    for _ in range(steps):
        g.replay()
    torch.cuda.synchronize()
    status_ok()
    k_ref, v_ref, lens = f64(kc), f64(vc), cl.numpy().copy()
    for _ in range(steps):
        ro, _, krow = oracle.decode_append(f64(q), k_ref, v_ref, lens, f64(kn), f64(vn),
                                           rope=True, theta=10000.0)
        for b in range(B):
            k_ref[b, :, lens[b]] = f64(torch.from_numpy(krow[b]).to(torch.bfloat16))
            v_ref[b, :, lens[b]] = f64(vn[b])
        lens = lens + 1
    assert np.array_equal(gl.cpu().numpy(), lens)
    check(o.cpu(), ro, what="O after replays")


def test_decode_append_full_cache_sets_status():
    B, Hq, Hkv, Lmax, D = 2, 8, 2, 64, 128
    q, kc, vc, cl, kn, vn = _append_inputs(B, Hq, Hkv, Lmax, D, [64, 10], seed=9)
    gk, gl = kc.cuda(), cl.cuda()
    o = binding.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), gk, vc.cuda(), gl)
    assert binding.attn_get_device_status() == 7  # no row left for sequence 0
    assert binding.attn_get_device_status() == 0
    assert gl.cpu().tolist() == [64, 11]
    ro, _, _ = oracle.decode_append(f64(q[1:]), f64(kc[1:]), f64(vc[1:]), cl[1:].numpy(),
                                    f64(kn[1:]), f64(vn[1:]), rope=True, theta=10000.0)
    check(o[1:].cpu(), ro, what="valid row")
    assert torch.equal(gk[0].cpu(), kc[0])


# --------------------------------------------------------------------------------------------
# latent decode
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("B,H,Lmax,lens", [
    (4, 16, 2048, [2048, 1, 1000, 64]),
    (1, 16, 2048, [2048]),                 # one sequence spread over many SMs
    (2, 5, 200, [200, 37]),
    (160, 16, 256, [256 - (i % 7) * 33 for i in range(160)]),  # more sequences than SMs
    # one whole sequence per CTA, ragged lengths, Lmax = 200: the last tile's copy runs past the
    # cache's key extent (zero fill) and past each length (masked)
    (128, 16, 200, [200 - (i % 5) * 37 for i in range(128)]),
])
def test_latent_decode(B, H, Lmax, lens):
    q, c, cl = synthetic.latent_inputs(B, H, Lmax, lens, seed=B)
    o, lse = binding.attn_decode_latent(q.cuda(), c.cuda(), cl.cuda(), want_lse=True)
    status_ok()
    ro, rl = oracle.latent_decode(f64(q), f64(c), cl.numpy(), rope=True, theta=10000.0)
    check(o.cpu(), ro, what="O")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE")


@pytest.mark.parametrize("B,H,Lmax,lens", [
    (4, 16, 2048, [2048, 1, 1000, 64]),
    (128, 16, 2048, 2048),                 # one whole sequence per CTA
    (2, 5, 200, [200, 37]),
    (160, 16, 256, [256 - (i % 7) * 33 for i in range(160)]),
    (128, 16, 200, [200 - (i % 5) * 37 for i in range(128)]),
])
def test_latent_decode_fp8_cache(B, H, Lmax, lens):
    """e5m2 latent cache (q bf16): widened exactly to f16 in the MMAs, so the bf16 bounds apply."""
    q, c, cl = synthetic.latent_inputs(B, H, Lmax, lens, seed=B + 7, cache_dtype="fp8")
    o, lse = binding.attn_decode_latent(q.cuda(), c.cuda(), cl.cuda(), want_lse=True)
    status_ok()
    ro, rl = oracle.latent_decode(f64(q), f64(c), cl.numpy(), rope=True, theta=10000.0)
    check(o.cpu(), ro, what="O fp8 latent")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE fp8 latent")


def test_latent_bad_cache_len_sets_status():
    q, c, cl = synthetic.latent_inputs(3, 16, 128, [128, 128, 50], seed=6)
    cl[1] = 0  # out of range
    o = binding.attn_decode_latent(q.cuda(), c.cuda(), cl.cuda())
    assert binding.attn_get_device_status() == 7
    assert binding.attn_get_device_status() == 0
    keep = [0, 2]
    ro, _ = oracle.latent_decode(f64(q[keep]), f64(c[keep]), cl[keep].numpy())
    check(o[keep].cpu(), ro, what="valid rows")
    assert torch.all(o[1].cpu() == 0)


# --------------------------------------------------------------------------------------------
# the interleaved RoPE pairing (2i, 2i+1) through every entry point that rotates
# --------------------------------------------------------------------------------------------

IL = "interleaved"


@pytest.mark.parametrize("shape,pos0,dtype", [
    ((2, 3, 37, 64), 5, "bf16"),      # per-row kernel (3 heads), whole chunks
    ((1, 8, 300, 128), 16000, "bf16"),  # per-position kernel, far positions
    ((1, 1, 3, 6), 11, "bf16"),       # D = 6: one thread per pair
    ((2, 7, 70, 128), 9, "fp8"),
    ((1, 2, 5, 10), 0, "fp8"),        # D = 10: one thread per pair
])
def test_rope_apply_interleaved(shape, pos0, dtype):
    x = synthetic.rope_input(*shape, dtype=dtype, seed=shape[2])
    y = binding.rope_apply(x.cuda(), pos0=pos0, theta=10000.0, rope_style=IL)
    torch.cuda.synchronize()
    ref = oracle.rope_rotate_interleaved(f64(x), pos0 + np.arange(shape[2]), 10000.0)
    if dtype == "bf16":
        check(y.cpu(), ref, what="rope interleaved bf16")
        assert (y.cpu() == torch.from_numpy(ref).to(torch.bfloat16)).float().mean() > 0.99
    else:
        r = f64(torch.from_numpy(ref).to(torch.float8_e5m2))
        g = f64(y.cpu())
        step = np.maximum(np.abs(r), 2.0 ** -14) * 0.25
        assert np.all(np.abs(g - r) <= step * 1.0001)
        assert (g == r).mean() > 0.99


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,pos0", [
    (1, 4, 1, 128, 64, True, 0),       # the tiny config with interleaved pairs
    (2, 8, 2, 700, 128, True, 3),      # below the pass threshold of the half-split form
    (1, 4, 1, 1100, 128, True, 0),
    (1, 2, 2, 300, 64, False, 5000),
])
def test_prefill_rope_interleaved(B, Hq, Hkv, S, D, causal, pos0):
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=S + 7)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, rope=True,
                                  rope_theta=10000.0, pos0=pos0, want_lse=True, rope_style=IL)
    status_ok()
    ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=causal, rope=True, theta=10000.0,
                            pos0=pos0, rope_style=IL)
    check(o.cpu(), ro, what="O prefill interleaved")
    check(lse.cpu(), rl, ROPE_LSE_TOL, None, what="LSE prefill interleaved")


def test_prefill_chunk_rope_interleaved():
    B, Hq, Hkv, Sq, Skv, pitch, D = 2, 8, 2, 96, 700, 704, 128
    q = synthetic.normal((B, Hq, Sq, D), 930, "bf16")
    kc = synthetic.normal((B, Hkv, pitch, D), 931, "bf16")
    vc = synthetic.normal((B, Hkv, pitch, D), 932, "bf16")
    o, lse = binding.attn_prefill_chunk(q.cuda(), kc.cuda(), vc.cuda(), Skv, rope=True,
                                        rope_theta=10000.0, pos0=4, want_lse=True, rope_style=IL)
    status_ok()
    ro, rl = oracle.prefill_chunk(f64(q), f64(kc), f64(vc), Skv, rope=True, theta=10000.0, pos0=4,
                                  rope_style=IL)
    check(o.cpu(), ro, what="O chunk interleaved")
    check(lse.cpu(), rl, ROPE_LSE_TOL, None, what="LSE chunk interleaved")


@pytest.mark.parametrize("cache_dtype,B,Hq,Hkv,D,lens", [
    ("bf16", 3, 32, 8, 128, [2048, 1, 777]),
    ("bf16", 2, 8, 1, 64, [300, 129]),
    ("fp8", 3, 24, 2, 128, [1999, 65, 2048]),
])
def test_decode_rope_interleaved(cache_dtype, B, Hq, Hkv, D, lens):
    Lmax = max(lens)
    q, kc, vc, cl = synthetic.decode_inputs(B, Hq, Hkv, Lmax, D, lens, seed=B + 70,
                                            cache_dtype=None if cache_dtype == "bf16" else "fp8")
    o, lse = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda(), want_lse=True,
                                 rope_style=IL)
    status_ok()
    ro, rl = oracle.decode(f64(q), f64(kc), f64(vc), cl.numpy(), rope=True, theta=10000.0,
                           rope_style=IL)
    check(o.cpu(), ro, what="O decode interleaved")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE decode interleaved")


def test_decode_append_rope_interleaved():
    B, Hq, Hkv, Lmax, D, lens = 3, 32, 8, 600, 128, [599, 1, 300]
    q, kc, vc, cl, kn, vn = _append_inputs(B, Hq, Hkv, Lmax, D, lens, seed=77)
    gk, gv, gl = kc.cuda(), vc.cuda(), cl.cuda()
    o, lse = binding.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), gk, gv, gl, want_lse=True,
                                        rope=True, rope_theta=10000.0, rope_style=IL)
    status_ok()
    ro, rl, krow = oracle.decode_append(f64(q), f64(kc), f64(vc), cl.numpy(), f64(kn), f64(vn),
                                        rope=True, theta=10000.0, rope_style=IL)
    check(o.cpu(), ro, what="O append interleaved")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE append interleaved")
    gk, gv = gk.cpu(), gv.cpu()
    for b in range(B):
        L = int(cl[b])
        np.testing.assert_allclose(f64(gk[b, :, L]), krow[b], rtol=0, atol=1.6e-2)
        assert torch.equal(gv[b, :, L], vn[b])


@pytest.mark.parametrize("cache_dtype", ["bf16", "fp8"])
def test_latent_decode_rope_interleaved(cache_dtype):
    B, H, Lmax, lens = 4, 16, 1024, [1024, 1, 500, 64]
    q, c, cl = synthetic.latent_inputs(B, H, Lmax, lens, seed=91,
                                       cache_dtype=None if cache_dtype == "bf16" else "fp8")
    o, lse = binding.attn_decode_latent(q.cuda(), c.cuda(), cl.cuda(), want_lse=True,
                                        rope_style=IL)
    status_ok()
    ro, rl = oracle.latent_decode(f64(q), f64(c), cl.numpy(), rope=True, theta=10000.0,
                                  rope_style=IL)
    check(o.cpu(), ro, what="O latent interleaved")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE latent interleaved")


def test_rope_styles_differ_on_device():
    """The two pairings really produce different rotations (D > 2), and the flag reaches the
    decode kernel: swapping the style changes the result."""
    q, kc, vc, cl = synthetic.decode_inputs(2, 8, 2, 256, 128, [256, 100], seed=5)
    a = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda())
    b = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda(), rope_style=IL)
    assert (a.float() - b.float()).abs().max().item() > 1e-2


# --------------------------------------------------------------------------------------------
# head dim 256 (bf16 caches): decode and append
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens,style", [
    (1, 32, 8, 2048, [2048], "half"),           # split KV over many CTAs
    (3, 32, 8, 2048, [2048, 1, 777], "half"),   # ragged, one single-key sequence
    (2, 16, 1, 300, [300, 129], "half"),        # group of 16, Lmax not a tile multiple
    (2, 8, 2, 512, [512, 65], IL),
])
def test_decode_d256(B, Hq, Hkv, Lmax, lens, style):
    q, kc, vc, cl = synthetic.decode_inputs(B, Hq, Hkv, Lmax, 256, lens, seed=B + Hq + 256)
    o, lse = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda(), want_lse=True,
                                 rope_style=style)
    status_ok()
    ro, rl = oracle.decode(f64(q), f64(kc), f64(vc), cl.numpy(), rope=True, theta=10000.0,
                           rope_style=style)
    check(o.cpu(), ro, what="O decode D=256")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE decode D=256")


def test_decode_append_d256():
    B, Hq, Hkv, Lmax, D, lens = 3, 16, 4, 400, 256, [399, 1, 200]
    q, kc, vc, cl, kn, vn = _append_inputs(B, Hq, Hkv, Lmax, D, lens, seed=256)
    gk, gv, gl = kc.cuda(), vc.cuda(), cl.cuda()
    o, lse = binding.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), gk, gv, gl, want_lse=True,
                                        rope=True, rope_theta=10000.0)
    status_ok()
    ro, rl, krow = oracle.decode_append(f64(q), f64(kc), f64(vc), cl.numpy(), f64(kn), f64(vn),
                                        rope=True, theta=10000.0)
    check(o.cpu(), ro, what="O append D=256")
    check(lse.cpu(), rl, LSE_TOL, None, what="LSE append D=256")
    assert torch.equal(gl.cpu(), cl + 1)
    gk, gv = gk.cpu(), gv.cpu()
    for b in range(B):
        L = int(cl[b])
        np.testing.assert_allclose(f64(gk[b, :, L]), krow[b], rtol=0, atol=1.6e-2)
        assert torch.equal(gv[b, :, L], vn[b])


# --------------------------------------------------------------------------------------------
# backward: dQ, dK, dV of the prefill attention
# --------------------------------------------------------------------------------------------

def check_grad(gpu, ref, what):
    """P and dS are rounded to bf16 (2^-9 relative) before their products and Delta uses the
    bf16 forward output, so each gradient carries ~0.2-0.5 % relative error: max-abs within
    2e-2 of the tensor's largest entry, mean-abs within 5e-3 of its mean magnitude."""
    g = f64(gpu)
    d = np.abs(g - ref)
    assert np.all(np.isfinite(g)), f"{what}: non-finite"
    big, mean = np.abs(ref).max(), np.abs(ref).mean()
    assert d.max() <= 2e-2 * big, f"{what}: max-abs {d.max():.3e} > 2e-2 * {big:.3e}"
    assert d.mean() <= 5e-3 * mean, f"{what}: mean-abs {d.mean():.3e} > 5e-3 * {mean:.3e}"


@pytest.fixture(params=[2, 1], ids=["tcgen05", "mma_sync"])
def bwd_path(request):
    """Runs a backward test on each of the two kernel paths, then restores the default."""
    binding.attn_set_backward_path(request.param)
    yield request.param
    binding.attn_set_backward_path(0)


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal", [
    (1, 4, 1, 128, 64, True),      # the tiny config's shape
    (2, 4, 2, 300, 128, True),     # GQA, ragged tail (several key tiles, partial last)
    (1, 2, 2, 200, 64, False),
    (1, 8, 2, 513, 128, True),     # group of 4, one row past whole tiles
    (1, 2, 1, 77, 128, False),     # shorter than one tile
    (1, 1, 1, 1, 64, True),        # S = 1
    (1, 8, 1, 640, 128, False),    # group of 8, five whole tiles: long step rings, no mask
    (2, 6, 3, 1000, 64, True),     # group of 2 at D = 64, eight tiles, ragged
])
def test_prefill_backward(B, Hq, Hkv, S, D, causal, bwd_path):
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=S + 11)
    do = synthetic.normal((B, Hq, S, D), 5000 + S, "bf16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = binding.attn_prefill(qd, kd, vd, causal=causal, want_lse=True)
    dq, dk, dv = binding.attn_prefill_backward(qd, kd, vd, o, lse, do.cuda(), causal=causal)
    status_ok()
    rq, rk, rv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), causal)
    check_grad(dq.cpu(), rq, "dQ")
    check_grad(dk.cpu(), rk, "dK")
    check_grad(dv.cpu(), rv, "dV")


@pytest.mark.parametrize("B,Hq,Hkv,S,D,causal,scale", [
    (1, 16, 1, 300, 128, True, 0.0),     # a group of 16 query heads on one KV head
    (2, 4, 4, 257, 64, False, 0.05),     # a softmax scale other than 1/sqrt(D), ragged
    (1, 2, 1, 129, 128, True, 0.2),      # one row past a whole tile, larger scale
])
def test_prefill_backward_groups_and_scales(B, Hq, Hkv, S, D, causal, scale, bwd_path):
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=S + 37)
    do = synthetic.normal((B, Hq, S, D), 6000 + S, "bf16")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = binding.attn_prefill(qd, kd, vd, causal=causal, softmax_scale=scale, want_lse=True)
    dq, dk, dv = binding.attn_prefill_backward(qd, kd, vd, o, lse, do.cuda(), causal=causal,
                                               softmax_scale=scale)
    status_ok()
    rq, rk, rv = oracle.attention_backward(f64(q), f64(k), f64(v), f64(do), causal,
                                           scale=scale if scale > 0 else None)
    check_grad(dq.cpu(), rq, "dQ")
    check_grad(dk.cpu(), rk, "dK")
    check_grad(dv.cpu(), rv, "dV")


def test_prefill_backward_equals_finite_difference_direction(bwd_path):
    """A directional derivative of sum(O * W) on the device (forward at q +- h u) agrees with
    <dQ, u> from the backward, independently of the oracle."""
    B, Hq, Hkv, S, D = 1, 2, 1, 96, 64
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=3)
    w = synthetic.normal((B, Hq, S, D), 31, "bf16").cuda().float()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = binding.attn_prefill(qd, kd, vd, causal=True, want_lse=True)
    dq, _, _ = binding.attn_prefill_backward(qd, kd, vd, o, lse, w.bfloat16(), causal=True)
    # the oracle's float64 forward gives the finite difference at float64 precision
    u = np.asarray(synthetic.normal((B, Hq, S, D), 32, "bf16").float())
    h = 1e-4
    lp = np.sum(oracle.attention(f64(q) + h * u, f64(k), f64(v), True)[0] * f64(w.cpu()))
    lm = np.sum(oracle.attention(f64(q) - h * u, f64(k), f64(v), True)[0] * f64(w.cpu()))
    fd = (lp - lm) / (2 * h)
    an = float(np.sum(f64(dq.cpu()) * u))
    assert abs(fd - an) <= 2e-2 * max(1.0, abs(fd)), (fd, an)


@pytest.mark.parametrize("style,dtype,shape", [
    ("half", "bf16", (2, 4, 70, 128)), ("interleaved", "bf16", (1, 3, 37, 64)),
    ("half", "fp8", (1, 2, 50, 64)), ("interleaved", "bf16", (1, 1, 3, 6)),
])
def test_rope_apply_inverse(style, dtype, shape):
    x = synthetic.rope_input(*shape, dtype=dtype, seed=shape[2] + 5)
    y = binding.rope_apply(x.cuda(), pos0=7, theta=10000.0, rope_style=style, inverse=True)
    torch.cuda.synchronize()
    ref = oracle.rope_rotate(f64(x), 7 + np.arange(shape[2]), 10000.0, style, inverse=True)
    if dtype == "bf16":
        check(y.cpu(), ref, what="inverse rope")
    else:
        r = f64(torch.from_numpy(ref).to(torch.float8_e5m2))
        g = f64(y.cpu())
        assert np.all(np.abs(g - r) <= np.maximum(np.abs(r), 2.0 ** -14) * 0.25 * 1.0001)


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_backward_through_rope(style, bwd_path):
    """RoPE applied by rope_apply, attention, its backward, and the inverse rotation of dQ / dK:
    the gradients with respect to the un-rotated Q and K."""
    B, Hq, Hkv, S, D = 1, 4, 2, 200, 128
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=41)
    do = synthetic.normal((B, Hq, S, D), 42, "bf16")
    qr = binding.rope_apply(q.cuda(), pos0=3, rope_style=style)
    kr = binding.rope_apply(k.cuda(), pos0=3, rope_style=style)
    o, lse = binding.attn_prefill(qr, kr, v.cuda(), causal=True, want_lse=True)
    dqr, dkr, dv = binding.attn_prefill_backward(qr, kr, v.cuda(), o, lse, do.cuda(), causal=True)
    dq = binding.rope_apply(dqr, pos0=3, rope_style=style, inverse=True)
    dk = binding.rope_apply(dkr, pos0=3, rope_style=style, inverse=True)
    status_ok()
    pos = 3 + np.arange(S)
    rq_r, rk_r, rv = oracle.attention_backward(oracle.rope_rotate(f64(q), pos, 10000.0, style),
                                               oracle.rope_rotate(f64(k), pos, 10000.0, style),
                                               f64(v), f64(do), True)
    check_grad(dq.cpu(), oracle.rope_rotate(rq_r, pos, 10000.0, style, inverse=True), "dQ")
    check_grad(dk.cpu(), oracle.rope_rotate(rk_r, pos, 10000.0, style, inverse=True), "dK")
    check_grad(dv.cpu(), rv, "dV")


# --------------------------------------------------------------------------------------------
# head dim 256 prefill: one Q tile per work item
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("B,Hq,Hkv,S,causal,rope", [
    (1, 4, 1, 128, True, False),
    (2, 8, 2, 300, True, True),      # ragged tail, RoPE through the rotation passes, GQA
    (1, 2, 2, 200, False, False),
    (1, 4, 4, 513, True, True),
    (2, 32, 8, 1024, True, False),   # 256 items, more than the SMs: CTAs run several items, so
                                     # the chunk ring, both S buffers and the Q/O phases carry over
    (1, 2, 1, 1, True, False),       # one query row, one masked key tile
    (1, 16, 1, 257, True, False),    # 16 query heads per KV head, ragged tail
    (1, 4, 2, 640, False, False),    # five KV tiles per item: the 8-chunk ring wraps every step
])
def test_prefill_d256(B, Hq, Hkv, S, causal, rope):
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, 256, "bf16", seed=S + 256)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, rope=rope,
                                  rope_theta=10000.0, want_lse=True)
    status_ok()
    ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=causal, rope=rope, theta=10000.0)
    check(o.cpu(), ro, what="O prefill D=256")
    check(lse.cpu(), rl, ROPE_LSE_TOL if rope else LSE_TOL, None, what="LSE prefill D=256")


@pytest.mark.parametrize("B,Hq,Hkv,S,causal", [
    (1, 4, 1, 128, True),
    (2, 8, 2, 300, True),      # ragged tail, GQA
    (1, 2, 2, 200, False),
    (1, 16, 1, 257, True),     # 16 query heads per KV head
    (2, 32, 8, 1024, True),    # 256 items: the chunk ring and the phases carry over between items
])
def test_prefill_fp8_d256(B, Hq, Hkv, S, causal):
    """fp8 e5m2 Q/K/V at head dim 256 (no RoPE): 256-byte rows as two 128-byte column boxes,
    64-key V chunks, P rounded to e4m3; the oracle runs on the dequantised values."""
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, 256, "fp8", seed=S + 11)
    o, lse = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, want_lse=True)
    status_ok()
    ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=causal)
    check(o.cpu(), ro, FP8_MAX, 1e-2, what="O fp8 D=256")
    check(lse.cpu(), rl, 2e-2, None, what="LSE fp8 D=256")


def test_prefill_fp8_d256_scales_and_chunk():
    """fp8 at head dim 256: the dequantisation scales (q stored halved with q_scale = 2, v
    quartered with v_scale = 4 give the same attention), and a chunk against a cache of pitch
    320 whose queries start mid-tile, against the oracle."""
    B, H, S, D = 1, 2, 200, 256
    q, k, v = synthetic.prefill_inputs(B, H, H, S, D, "fp8", seed=6)
    o1 = binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=True)
    qh = (q.float() / 2).to(torch.float8_e5m2)
    o2 = binding.attn_prefill(qh.cuda(), k.cuda(), v.cuda(), causal=True, q_scale=2.0)
    vh = (v.float() / 4).to(torch.float8_e5m2)
    o3 = binding.attn_prefill(q.cuda(), k.cuda(), vh.cuda(), causal=True, v_scale=4.0)
    status_ok()
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (o1.float() - o3.float()).abs().max().item() <= 1e-2
    Bc, Hq, Hkv, Sq, Skv, pitch = 2, 8, 2, 70, 300, 320
    qc = synthetic.normal((Bc, Hq, Sq, D), 980, "fp8")
    kc = synthetic.normal((Bc, Hkv, pitch, D), 981, "fp8")
    vc = synthetic.normal((Bc, Hkv, pitch, D), 982, "fp8")
    o, lse = binding.attn_prefill_chunk(qc.cuda(), kc.cuda(), vc.cuda(), Skv, rope=False,
                                        want_lse=True)
    status_ok()
    ro, rl = oracle.prefill_chunk(f64(qc), f64(kc), f64(vc), Skv)
    check(o.cpu(), ro, FP8_MAX, 1e-2, what="O chunk fp8 D=256")
    check(lse.cpu(), rl, 2e-2, None, what="LSE chunk fp8 D=256")


@pytest.mark.parametrize("Sq,Skv,pitch", [(64, 300, 320), (200, 1000, 1000), (1, 129, 160)])
def test_prefill_chunk_d256(Sq, Skv, pitch):
    B, Hq, Hkv, D = 2, 8, 2, 256
    q = synthetic.normal((B, Hq, Sq, D), 960, "bf16")
    kc = synthetic.normal((B, Hkv, pitch, D), 961, "bf16")
    vc = synthetic.normal((B, Hkv, pitch, D), 962, "bf16")
    o, lse = binding.attn_prefill_chunk(q.cuda(), kc.cuda(), vc.cuda(), Skv, rope=True,
                                        rope_theta=10000.0, want_lse=True)
    status_ok()
    ro, rl = oracle.prefill_chunk(f64(q), f64(kc), f64(vc), Skv, rope=True, theta=10000.0)
    check(o.cpu(), ro, what="O chunk D=256")
    check(lse.cpu(), rl, ROPE_LSE_TOL, None, what="LSE chunk D=256")
