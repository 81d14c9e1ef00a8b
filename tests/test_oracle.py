"""Pins for the float64 CPU oracle: checks against things other than the oracle itself.

Each check uses a closed form, an invariant the mathematics fixes, an independent library
routine (torch's scaled_dot_product_attention in float64), brute force over tiny enumerated
inputs with a separately written scalar loop, or a number printed on the pages
(tests/golden/page_facts.json).  The last tests plant typical mistakes in copies of the oracle
and check that the pins catch every one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention_fp64 as O
from attention_attn_prefill_02_gb300 import synthetic, workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FACTS = json.load(open(os.path.join(GOLDEN, "page_facts.json")))
RNG = np.random.default_rng(1234)


def rnd(*shape):
    return RNG.standard_normal(shape)


# ---------------------------------------------------------------------------------------------
# pin functions: each takes the functions under test, so planted mistakes can be fed in
# ---------------------------------------------------------------------------------------------

def pin_softmax_sums_to_one(probs=O.attention_probs):
    q, k = rnd(1, 2, 7, 4), rnd(1, 2, 7, 4)
    for causal in (False, True):
        P = probs(q, k, causal)
        np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-12)
        assert np.all(P >= 0)


def pin_zero_query_is_causal_mean(attn=O.attention):
    """q = 0: all logits equal, so causal row i is the plain mean of v_0..v_i, LSE = ln(i+1)."""
    S, D = 9, 5
    q = np.zeros((1, 1, S, D))
    k, v = rnd(1, 1, S, D), rnd(1, 1, S, 3)
    o, lse = attn(q, k, v, True, 0.37)
    for i in range(S):
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, : i + 1].mean(0), rtol=0, atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(i + 1)) < 1e-13


def pin_hand_two_key_case(attn=O.attention):
    """logits (0, ln 3) give weights (1/4, 3/4): O = (1, 6) for v0 = (4, 0), v1 = (0, 8)."""
    q = np.array([[[[math.log(3.0), 0.0]]]])
    k = np.array([[[[0.0, 0.0], [1.0, 0.0]]]])
    v = np.array([[[[4.0, 0.0], [0.0, 8.0]]]])
    o, lse = attn(q, k, v, False, 1.0)
    np.testing.assert_allclose(o[0, 0, 0], [1.0, 6.0], rtol=0, atol=1e-13)
    assert abs(lse[0, 0, 0] - math.log(4.0)) < 1e-13


def pin_one_hot_and_single_key(attn=O.attention):
    S, D = 6, 4
    k, v = rnd(1, 1, S, D), rnd(1, 1, S, D)
    # one large logit on key 3 -> output is v_3 (other keys are orthogonal to q)
    k[0, 0, :, 0] = 0.0
    k[0, 0, 3] = [1.0, 0.0, 0.0, 0.0]
    q = np.array([[[[60.0, 0.0, 0.0, 0.0]]]])
    o, _ = attn(q, k, v, False, 1.0)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 3], rtol=0, atol=1e-12)
    # a single key -> output is v_0 whatever q is
    o1, lse1 = attn(rnd(1, 1, 1, D), k[:, :, :1], v[:, :, :1], True, 0.5)
    np.testing.assert_allclose(o1[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-15)


def pin_causal_ignores_future(attn=O.attention):
    S, D = 8, 4
    q, k, v = rnd(1, 2, S, D), rnd(1, 2, S, D), rnd(1, 2, S, D)
    o, lse = attn(q, k, v, True, 0.5)
    for i in range(S - 1):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, i + 1:] = rnd(1, 2, S - i - 1, D) * 10
        v2[:, :, i + 1:] = rnd(1, 2, S - i - 1, D) * 10
        o2, lse2 = attn(q, k2, v2, True, 0.5)
        assert np.array_equal(o2[:, :, : i + 1], o[:, :, : i + 1])
        assert np.array_equal(lse2[:, :, : i + 1], lse[:, :, : i + 1])


def pin_matches_torch_sdpa(attn=O.attention):
    """Independent library routine: torch SDPA in float64 on the CPU (KV heads repeated)."""
    for causal, (B, Hq, Hkv, S, D) in itertools.product(
            (False, True), [(2, 4, 1, 13, 8), (1, 6, 3, 20, 16), (1, 2, 2, 5, 64)]):
        q, k, v = rnd(B, Hq, S, D), rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
        scale = 1 / math.sqrt(D)
        o, _ = attn(q, k, v, causal, scale)
        G = Hq // Hkv
        tq = torch.from_numpy(q)
        tk = torch.from_numpy(k).repeat_interleave(G, dim=1)
        tv = torch.from_numpy(v).repeat_interleave(G, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                               scale=scale)
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def scalar_attention_row(qi, keys, vals, scale):
    """Separately written scalar loop: softmax-weighted average with math.exp."""
    logits = [scale * sum(a * b for a, b in zip(qi, kj)) for kj in keys]
    z = sum(math.exp(t) for t in logits)
    out = [0.0] * len(vals[0])
    for t, vj in zip(logits, vals):
        w = math.exp(t) / z
        for d in range(len(out)):
            out[d] += w * vj[d]
    return out, math.log(z)


def pin_bruteforce_enumeration(attn=O.attention):
    """Every q, k in {-1,0,1}^2 for S = 2 plus random v; S = 3, 4 on a sample of grids."""
    vals3 = (-1.0, 0.0, 1.0)
    vecs = list(itertools.product(vals3, repeat=2))
    for S in (1, 2, 3, 4):
        combos = list(itertools.product(vecs, repeat=S))
        if len(combos) > 200:
            idx = np.random.default_rng(S).choice(len(combos), 200, replace=False)
            combos = [combos[i] for i in idx]
        for kq in combos:
            k = np.array(kq, dtype=np.float64)[None, None]
            q = k[:, :, ::-1].copy()  # queries: the keys with rows reversed
            v = np.arange(S * 2, dtype=np.float64).reshape(1, 1, S, 2) - 2.5
            for causal in (False, True):
                o, lse = attn(q, k, v, causal, 0.75)
                for i in range(S):
                    n = i + 1 if causal else S
                    ref_o, ref_l = scalar_attention_row(q[0, 0, i], k[0, 0, :n], v[0, 0, :n], 0.75)
                    np.testing.assert_allclose(o[0, 0, i], ref_o, rtol=0, atol=1e-13)
                    assert abs(lse[0, 0, i] - ref_l) < 1e-13


def pin_gqa_equals_repeated_mha(attn=O.attention):
    B, Hq, Hkv, S, D = 2, 8, 2, 6, 4
    q, k, v = rnd(B, Hq, S, D), rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    o, lse = attn(q, k, v, True, 0.5)
    o2, lse2 = attn(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), True, 0.5)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-14)
    # and each query head really uses head hq // G (contiguous grouping)
    o3, _ = attn(q[:, 5:6], k[:, 1:2], v[:, 1:2], True, 0.5)
    np.testing.assert_allclose(o[:, 5:6], o3, rtol=0, atol=1e-14)


def pin_rope(rope=O.rope_rotate_half):
    D, n = 16, 11
    x = rnd(3, n, D)
    pos = np.arange(n) * 37 + 5
    y = rope(x, pos, 10000.0)
    # norm preserved
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    # position 0 is the identity
    np.testing.assert_allclose(rope(x, np.zeros(n), 10000.0), x, rtol=0, atol=0)
    # <R(m) q, R(n) k> depends only on m - n
    q, k = rnd(1, 1, D), rnd(1, 1, D)
    for (m, nn, t) in [(3, 1, 100), (0, 7, 2048), (16000, 5, 123)]:
        a = np.sum(rope(q, [m], 500.0) * rope(k, [nn], 500.0))
        b = np.sum(rope(q, [m + t], 500.0) * rope(k, [nn + t], 500.0))
        assert abs(a - b) < 1e-9
    # D = 2: a plain 2x2 rotation by angle pos (inverse frequency theta^0 = 1)
    for p in (0.0, 1.0, 2.0, 7.5, 2048.0):
        out = rope(np.array([[[0.3, -1.2]]]), [p], 10000.0)[0, 0]
        c, s = math.cos(p), math.sin(p)
        np.testing.assert_allclose(out, [0.3 * c + 1.2 * s, -1.2 * c + 0.3 * s], atol=1e-12)
    # D = 4, theta = 100: pairs (0,2) at angle p and (1,3) at angle p/10
    p = 10.0
    out = rope(np.array([[[1.0, 2.0, 3.0, 4.0]]]), [p], 100.0)[0, 0]
    c0, s0, c1, s1 = math.cos(p), math.sin(p), math.cos(p / 10), math.sin(p / 10)
    np.testing.assert_allclose(out, [c0 - 3 * s0, 2 * c1 - 4 * s1, 3 * c0 + s0, 4 * c1 + 2 * s1],
                               atol=1e-12)


def _il_to_half(D):
    """Index map taking the interleaved layout to the rotate-half one: dims 0, 2, 4, .. then
    1, 3, 5, ..  (pair (2i, 2i+1) lands on (i, i + D/2))."""
    return np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])


def pin_rope_interleaved(rope=O.rope_rotate_interleaved, rope_half=O.rope_rotate_half):
    D, n = 16, 11
    x = rnd(3, n, D)
    pos = np.arange(n) * 37 + 5
    y = rope(x, pos, 10000.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    np.testing.assert_allclose(rope(x, np.zeros(n), 10000.0), x, rtol=0, atol=0)
    q, k = rnd(1, 1, D), rnd(1, 1, D)
    for (m, nn, t) in [(3, 1, 100), (0, 7, 2048), (16000, 5, 123)]:
        a = np.sum(rope(q, [m], 500.0) * rope(k, [nn], 500.0))
        b = np.sum(rope(q, [m + t], 500.0) * rope(k, [nn + t], 500.0))
        assert abs(a - b) < 1e-9
    # D = 4, theta = 100: adjacent pairs (0,1) at angle p and (2,3) at angle p/10
    p = 10.0
    out = rope(np.array([[[1.0, 2.0, 3.0, 4.0]]]), [p], 100.0)[0, 0]
    c0, s0, c1, s1 = math.cos(p), math.sin(p), math.cos(p / 10), math.sin(p / 10)
    np.testing.assert_allclose(out, [c0 - 2 * s0, 2 * c0 + s0, 3 * c1 - 4 * s1, 4 * c1 + 3 * s1],
                               atol=1e-12)
    # the same rotation as the (separately pinned) rotate-half form on re-ordered dims
    perm = _il_to_half(D)
    np.testing.assert_allclose(rope(x, pos, 10000.0)[..., perm], rope_half(x[..., perm], pos, 10000.0),
                               atol=1e-12)


def pin_rope_style_through_entry_points(prefill=O.prefill, decode=O.decode,
                                        latent=O.latent_decode, append=O.decode_append,
                                        chunk=O.prefill_chunk):
    """With interleaved RoPE every entry point equals the half-split one on inputs whose q/k
    dims are re-ordered the same way (scores are invariant under a common permutation)."""
    D = 8
    perm = _il_to_half(D)
    q, k, v = rnd(1, 4, 6, D), rnd(1, 2, 6, D), rnd(1, 2, 6, D)
    a = prefill(q, k, v, causal=True, rope=True, theta=50.0, pos0=3, rope_style="interleaved")
    b = prefill(q[..., perm], k[..., perm], v, causal=True, rope=True, theta=50.0, pos0=3)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)
    a = chunk(q[:, :, :2], k, v, 5, rope=True, theta=50.0, pos0=1, rope_style="interleaved")
    b = chunk(q[:, :, :2][..., perm], k[..., perm], v, 5, rope=True, theta=50.0, pos0=1)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)
    qd, lens = rnd(2, 4, D), np.array([3, 6])
    kc, vc = rnd(2, 2, 7, D), rnd(2, 2, 7, D)
    a = decode(qd, kc, vc, lens, theta=50.0, rope_style="interleaved")
    b = decode(qd[..., perm], kc[..., perm], vc, lens, theta=50.0)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)
    kn, vn = rnd(2, 2, D), rnd(2, 2, D)
    a = append(qd, kc, vc, lens, kn, vn, theta=50.0, rope_style="interleaved")
    b = append(qd[..., perm], kc[..., perm], vc, lens, kn[..., perm], vn, theta=50.0)
    np.testing.assert_allclose(a[0], b[0], atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], atol=1e-12)
    np.testing.assert_allclose(a[2][..., perm], b[2], atol=1e-12)  # the stored key, re-ordered
    dl, dr = 6, 8  # latent: only the last dr dims rotate; re-order those
    pl = np.concatenate([np.arange(dl), dl + _il_to_half(dr)])
    ql, cl = rnd(2, 3, dl + dr), rnd(2, 5, dl + dr)
    a = latent(ql, cl, np.array([2, 5]), theta=50.0, d_latent=dl, d_rope=dr,
               rope_style="interleaved")
    b = latent(ql[..., pl], cl[..., pl], np.array([2, 5]), theta=50.0, d_latent=dl, d_rope=dr)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)


def pin_backward_finite_differences(bwd=O.attention_backward):
    """Central differences of L = sum(O * W) in float64 against the analytic gradients."""
    for causal in (True, False):
        q, k, v = rnd(1, 2, 5, 3), rnd(1, 1, 5, 3), rnd(1, 1, 5, 3)
        W = rnd(1, 2, 5, 3)

        def loss(qq, kk, vv):
            return float(np.sum(O.attention(qq, kk, vv, causal)[0] * W))

        dq, dk, dv = bwd(q, k, v, W, causal)
        h = 1e-5
        for x, g in ((q, dq), (k, dk), (v, dv)):
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = loss(q, k, v)
                x[idx] = old - h
                lm = loss(q, k, v)
                x[idx] = old
                assert abs((lp - lm) / (2 * h) - g[idx]) < 1e-7, (causal, idx)


def pin_backward_gqa_equals_repeated(bwd=O.attention_backward):
    """GQA gradients equal those of MHA on repeated K/V, the K/V ones summed over each group."""
    q, k, v, do = rnd(2, 4, 6, 8), rnd(2, 2, 6, 8), rnd(2, 2, 6, 8), rnd(2, 4, 6, 8)
    dq, dk, dv = bwd(q, k, v, do, True)
    rq, rk, rv = bwd(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), do, True)
    np.testing.assert_allclose(dq, rq, atol=1e-12)
    np.testing.assert_allclose(dk, rk.reshape(2, 2, 2, 6, 8).sum(2), atol=1e-12)
    np.testing.assert_allclose(dv, rv.reshape(2, 2, 2, 6, 8).sum(2), atol=1e-12)


def pin_backward_invariants(bwd=O.attention_backward):
    """Shifting every key by one vector adds a constant to each row of scores, which the
    softmax ignores: the key gradients of a head sum to zero.  A zero query attends uniformly,
    so dV_j is the mean of the dO rows that see key j (causal: row i sees i + 1 keys)."""
    for causal in (True, False):
        q, k, v, do = rnd(1, 3, 7, 4), rnd(1, 3, 7, 4), rnd(1, 3, 7, 4), rnd(1, 3, 7, 4)
        _, dk, _ = bwd(q, k, v, do, causal)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    S = 6
    do = rnd(1, 1, S, 4)
    _, _, dv = bwd(np.zeros((1, 1, S, 4)), rnd(1, 1, S, 4), rnd(1, 1, S, 4), do, True)
    for j in range(S):
        want = sum(do[0, 0, i] / (i + 1) for i in range(j, S))
        np.testing.assert_allclose(dv[0, 0, j], want, atol=1e-12)


def pin_rope_inverse_and_backward_chain(rope=O.rope_rotate, bwd=O.attention_backward):
    """The inverse rotation undoes the rotation, and it carries gradients back through RoPE:
    for L = sum(attention(R q, R k, v) * W), dL/dq = R^-1 dQ_rot (central differences)."""
    for style in O.ROPE_STYLES:
        x = rnd(2, 9, 8)
        pos = np.arange(9) * 13 + 2
        np.testing.assert_allclose(rope(rope(x, pos, 100.0, style), pos, 100.0, style, inverse=True),
                                   x, atol=1e-12)
        q, k, v, W = rnd(1, 2, 5, 4), rnd(1, 1, 5, 4), rnd(1, 1, 5, 4), rnd(1, 2, 5, 4)
        p5 = np.arange(5) + 3

        def loss(qq, kk):
            return float(np.sum(O.attention(rope(qq, p5, 50.0, style), rope(kk, p5, 50.0, style),
                                            v, True)[0] * W))

        dq_r, dk_r, _ = bwd(rope(q, p5, 50.0, style), rope(k, p5, 50.0, style), v, W, True)
        dq = rope(dq_r, p5, 50.0, style, inverse=True)
        dk = rope(dk_r, p5, 50.0, style, inverse=True)
        h = 1e-5
        for x, g in ((q, dq), (k, dk)):
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = loss(q, k)
                x[idx] = old - h
                lm = loss(q, k)
                x[idx] = old
                assert abs((lp - lm) / (2 * h) - g[idx]) < 1e-7, (style, idx)


def pin_latent_absorbed_equals_explicit(latent=O.latent_decode):
    """Absorbed attention over the shared latent equals the explicit up-projected form.

    Explicit: k_h = [W_UK,h c || k_rope], v_h = W_UV,h c, q_h = [q_nope,h || q_rope,h].
    Absorbed: q_lat,h = [W_UK,h^T q_nope,h || q_rope,h] attends C directly, then W_UV,h is
    applied to the latent output.  (Fixed-budget decode audit — 2026-09-11, "Which
    implementation was tested": MLA with eager absorption, 448 latent + 64 RoPE dims.)
    """
    dl, dr = FACTS["mla_latent_dims"]["value"], FACTS["mla_rope_dims"]["value"]
    B, H, L, d_nope, d_v = 2, 3, 17, 128, 128
    c = rnd(B, L, dl + dr)
    W_UK, W_UV = rnd(H, d_nope, dl) * 0.05, rnd(H, d_v, dl) * 0.05
    q_nope, q_rope = rnd(B, H, d_nope), rnd(B, H, dr)
    lens = np.array([L, 9])
    scale = 1.0 / math.sqrt(d_nope + dr)
    q_lat = np.concatenate([np.einsum("hnl,bhn->bhl", W_UK, q_nope), q_rope], axis=-1)
    o_lat, _ = latent(q_lat, c, lens, scale=scale, rope=False)
    o_abs = np.einsum("hvl,bhl->bhv", W_UV, o_lat)
    for b in range(B):
        Lb = lens[b]
        cb = c[b, :Lb]
        for h in range(H):
            kh = np.concatenate([cb[:, :dl] @ W_UK[h].T, cb[:, dl:]], axis=-1)
            vh = cb[:, :dl] @ W_UV[h].T
            qh = np.concatenate([q_nope[b, h], q_rope[b, h]])
            ref, _ = scalar_attention_row(qh, kh, vh, scale)
            np.testing.assert_allclose(o_abs[b, h], ref, rtol=0, atol=1e-10)


def pin_latent_rope_by_hand(latent=O.latent_decode):
    """The latent decode's RoPE branch: rotating the last 64 query dims at position
    L = cache_len[b] by hand, then float64 SDPA over the cache rows with V = the first 448 dims.

    The rotation is written out pair by pair with math.cos / math.sin at the angle
    L * theta^(-2i/64): pairs (i, i + 32) of the 64 RoPE dims for the half-split form, (2i, 2i+1)
    for the interleaved one (Fixed-budget decode audit — 2026-09-11, "Which implementation was
    tested": 448 latent dims + 64 RoPE dims; only the RoPE part rotates).  The default scale is
    1/sqrt(512), the dims the scores use.  Ragged lengths, including 1.
    """
    dl, dr = FACTS["mla_latent_dims"]["value"], FACTS["mla_rope_dims"]["value"]
    B, H, Lmax, theta = 3, 4, 21, 10000.0
    q, c = rnd(B, H, dl + dr), rnd(B, Lmax, dl + dr)
    lens = np.array([21, 1, 8])
    for style in ("half", "interleaved"):
        o, lse = latent(q, c, lens, rope=True, theta=theta, rope_style=style)
        for b in range(B):
            L = int(lens[b])
            qr = q[b].copy()
            for i in range(dr // 2):
                a = L * theta ** (-2.0 * i / dr)
                i1, i2 = (dl + i, dl + i + dr // 2) if style == "half" else (dl + 2 * i, dl + 2 * i + 1)
                x1, x2 = q[b, :, i1].copy(), q[b, :, i2].copy()
                qr[:, i1] = x1 * math.cos(a) - x2 * math.sin(a)
                qr[:, i2] = x2 * math.cos(a) + x1 * math.sin(a)
            keys = torch.from_numpy(c[b, :L])[None].expand(H, L, dl + dr)
            vals = torch.from_numpy(c[b, :L, :dl])[None].expand(H, L, dl)
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(qr)[:, None], keys, vals, scale=1 / math.sqrt(dl + dr))
            np.testing.assert_allclose(o[b], ref[:, 0].numpy(), rtol=0, atol=1e-12)
            s = (qr @ c[b, :L].T) / math.sqrt(dl + dr)
            ref_l = s.max(-1) + np.log(np.exp(s - s.max(-1, keepdims=True)).sum(-1))
            np.testing.assert_allclose(lse[b], ref_l, rtol=0, atol=1e-12)


def pin_merge_identity(merge=O.merge_one_key, combine=O.combine_partials):
    tol = FACTS["merge_identity_tolerance"]["value"]
    L, D = 37, 8
    q, k, v = rnd(D), rnd(L + 1, D), rnd(L + 1, D)
    s = k @ q * 0.4
    o_hist, lse_hist = O.attention(q[None, None, None], k[None, None, :L], v[None, None, :L],
                                   False, 0.4)
    o_m, lse_m = merge(o_hist[0, 0, 0], lse_hist[0, 0, 0], s[L], v[L])
    ref_o, ref_l = scalar_attention_row(q, k, v, 0.4)
    np.testing.assert_allclose(o_m, ref_o, rtol=0, atol=tol)
    assert abs(lse_m - ref_l) < tol
    # split into chunks of the audit's split size (and ragged ones), combine == whole
    for split in (FACTS["decode_split_size"]["value"], 5, 1, 64):
        kk, vv = rnd(300, D), rnd(300, D)
        op, lp = O.split_decode_partials(q, kk, vv, split, 0.4)
        o_c, l_c = combine(op, lp)
        ref_o, ref_l = scalar_attention_row(q, kk, vv, 0.4)
        np.testing.assert_allclose(o_c, ref_o, rtol=0, atol=1e-12)
        assert abs(l_c - ref_l) < 1e-11
    # an empty split (lse = -inf) contributes nothing
    o_c, l_c = combine(np.stack([op[0], np.full(D, 7.0)]), np.array([lp[0], -np.inf]))
    np.testing.assert_allclose(o_c, op[0], atol=0)


def pin_chunk_equals_prompt_rows(chunk=O.prefill_chunk):
    """A chunk of queries against a cache equals the same rows of the whole-prompt prefill.

    The cache holds the keys rotated at their positions, as a decode cache stores them; rows
    past ``skv`` hold huge values that no chunk may touch.  Chunks of 1 and 32 rows (the audit's
    chunk size), ragged ones, and the whole prompt as one chunk.
    """
    B, Hq, Hkv, S, D, theta = 2, 4, 2, 45, 8, 500.0
    q, k, v = rnd(B, Hq, S, D), rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    full_o, full_l = O.prefill(q, k, v, causal=True, rope=True, theta=theta)
    kc = np.full((B, Hkv, S + 7, D), 1e6)
    vc = np.full((B, Hkv, S + 7, D), -1e6)
    kc[:, :, :S] = O.rope_rotate_half(k, np.arange(S), theta)
    vc[:, :, :S] = v
    for sq, skv in [(32, 32), (32, 45), (1, 45), (13, 20), (45, 45), (1, 1)]:
        o, l = chunk(q[:, :, skv - sq: skv], kc, vc, skv, rope=True, theta=theta)
        np.testing.assert_allclose(o, full_o[:, :, skv - sq: skv], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, full_l[:, :, skv - sq: skv], rtol=0, atol=1e-12)


def pin_append_equals_longer_prompt(append=O.decode_append, merge=O.merge_one_key):
    """A decode step that appends its token equals the last row of a prefill over the L + 1
    tokens, and equals the cached-history decode with the new key merged in by the sigmoid
    identity (Fixed-budget decode audit — 2026-09-11, "A: group-entry queries and one joint
    history scan")."""
    B, Hq, Hkv, Lmax, D, theta = 3, 4, 2, 30, 8, 10000.0
    G = Hq // Hkv
    lens = np.array([29, 1, 12])
    q, k_raw, v = rnd(B, Hq, D), rnd(B, Hkv, Lmax, D), rnd(B, Hkv, Lmax, D)
    k_new, v_new = rnd(B, Hkv, D), rnd(B, Hkv, D)
    kc = O.rope_rotate_half(k_raw, np.arange(Lmax), theta)
    o, lse, krow = append(q, kc, v, lens, k_new, v_new, rope=True, theta=theta)
    o_h, lse_h = O.decode(q, kc, v, lens, rope=True, theta=theta)
    for b in range(B):
        L = int(lens[b])
        qp = np.zeros((1, Hq, L + 1, D))
        qp[0, :, L] = q[b]
        kp = np.concatenate([k_raw[b, :, :L], k_new[b][:, None]], axis=1)[None]
        vp = np.concatenate([v[b, :, :L], v_new[b][:, None]], axis=1)[None]
        ref_o, ref_l = O.prefill(qp, kp, vp, causal=True, rope=True, theta=theta)
        np.testing.assert_allclose(o[b], ref_o[0, :, L], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_l[0, :, L], rtol=0, atol=1e-12)
        for hq in range(Hq):
            qr = O.rope_rotate_half(q[b, hq][None], np.array([L]), theta)[0]
            s_cur = float(qr @ krow[b, hq // G]) / math.sqrt(D)
            mo, ml = merge(o_h[b, hq], lse_h[b, hq], s_cur, v_new[b, hq // G])
            np.testing.assert_allclose(o[b, hq], mo, rtol=0, atol=1e-12)
            assert abs(lse[b, hq] - ml) < 1e-12


ALL_PINS = [pin_softmax_sums_to_one, pin_zero_query_is_causal_mean, pin_hand_two_key_case,
            pin_one_hot_and_single_key, pin_causal_ignores_future, pin_matches_torch_sdpa,
            pin_bruteforce_enumeration, pin_gqa_equals_repeated_mha, pin_rope,
            pin_latent_absorbed_equals_explicit, pin_latent_rope_by_hand, pin_merge_identity,
            pin_chunk_equals_prompt_rows, pin_append_equals_longer_prompt, pin_rope_interleaved,
            pin_rope_style_through_entry_points, pin_backward_finite_differences,
            pin_backward_gqa_equals_repeated, pin_backward_invariants,
            pin_rope_inverse_and_backward_chain]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------------------------
# entry-point level checks of the oracle (decode / latent / prefill wrappers)
# ---------------------------------------------------------------------------------------------

def test_decode_matches_sdpa_and_rotation():
    """Decode = one query row at position L attending the L cached (pre-rotated) keys."""
    B, Hq, Hkv, Lmax, D = 3, 8, 2, 40, 16
    q, kc, vc = rnd(B, Hq, D), rnd(B, Hkv, Lmax, D), rnd(B, Hkv, Lmax, D)
    lens = np.array([40, 1, 23])
    o, lse = O.decode(q, kc, vc, lens, rope=True, theta=10000.0)
    for b in range(B):
        L = lens[b]
        # rotate q by hand per pair at angle L * theta^(-2i/D)
        qr = q[b].copy()
        for i in range(D // 2):
            a = L * 10000.0 ** (-2 * i / D)
            x1, x2 = q[b, :, i].copy(), q[b, :, i + D // 2].copy()
            qr[:, i] = x1 * math.cos(a) - x2 * math.sin(a)
            qr[:, i + D // 2] = x2 * math.cos(a) + x1 * math.sin(a)
        tk = torch.from_numpy(kc[b, :, :L]).repeat_interleave(4, 0)
        tv = torch.from_numpy(vc[b, :, :L]).repeat_interleave(4, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qr)[:, None], tk, tv, scale=1 / math.sqrt(D))
        np.testing.assert_allclose(o[b], ref[:, 0].numpy(), atol=1e-12)


def test_prefill_rows_equals_full_prefill():
    q, k, v = rnd(2, 4, 33, 8), rnd(2, 2, 33, 8), rnd(2, 2, 33, 8)
    full_o, full_l = O.prefill(q, k, v, causal=True, rope=True, theta=50.0)
    rows = [(0, 0, 0), (1, 3, 32), (0, 2, 17), (1, 1, 5)]
    ro, rl = O.prefill_rows(q, k, v, rows, causal=True, rope=True, theta=50.0)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(ro[n], full_o[b, h, i], atol=1e-13)
        assert abs(rl[n] - full_l[b, h, i]) < 1e-13


def test_prefill_rope_equals_rotated_sdpa():
    """Prefill with RoPE = SDPA on Q, K rotated at 0..S-1 (rotation written out here)."""
    B, H, S, D, theta = 1, 2, 12, 8, 10000.0
    q, k, v = rnd(B, H, S, D), rnd(B, H, S, D), rnd(B, H, S, D)

    def rot(x):
        y = x.copy()
        for s in range(S):
            for i in range(D // 2):
                a = s * theta ** (-2 * i / D)
                x1, x2 = x[..., s, i], x[..., s, i + D // 2]
                y[..., s, i] = x1 * math.cos(a) - x2 * math.sin(a)
                y[..., s, i + D // 2] = x2 * math.cos(a) + x1 * math.sin(a)
        return y

    o, _ = O.prefill(q, k, v, causal=True, rope=True, theta=theta)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(rot(q)), torch.from_numpy(rot(k)), torch.from_numpy(v), is_causal=True)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)


def test_fp8_inputs_dequantise_exactly():
    """The oracle sees the stored e5m2 values exactly (per-tensor scale 1)."""
    x = synthetic.normal((4, 64), 3, "fp8")
    f = oracle.as_f64(x)
    # e5m2 has 2 mantissa bits: every finite value is m * 2^e with |m| < 8 an integer
    nz = f[f != 0]
    e = np.floor(np.log2(np.abs(nz)))
    mant = np.abs(nz) / 2.0 ** (e - 2)
    assert np.allclose(mant, np.round(mant))
    assert np.array_equal(f, x.float().double().numpy())


# ---------------------------------------------------------------------------------------------
# the pages' printed numbers pin the workload counts the bench divides by
# ---------------------------------------------------------------------------------------------

def test_golden_page_volumes():
    f = FACTS
    assert 4 * 2 * 4 * 64 == f["gqa_history_elements_per_token_per_group"]["value"]
    # decode config: Hkv = 8, D = 128 -> 2 * 8 * 128 = 2048 elements/token, the audit's figure
    assert 2 * 8 * 128 == f["gqa_history_elements_per_token_per_group"]["value"]
    hist = workload.decode_bytes(128, 32, 8, 2048, 128) - 128 * 32 * 128 * 4
    assert hist == f["gqa_history_bytes_batch128_ctx2048"]["value"]
    assert workload.latent_bytes(128, 16, 2048) - 128 * 16 * (512 + 448) * 2 == 128 * 2048 * 512 * 2
    assert f["mla_latent_dims"]["value"] + f["mla_rope_dims"]["value"] == 512
    assert (oracle.LATENT_DIM, oracle.LATENT_ROPE_DIM) == (448, 64)


def test_flop_counts_match_enumeration():
    """Causal FLOPs count exactly the scored pairs: enumerate them for a small S."""
    S, D = 37, 8
    pairs = sum(1 for i in range(S) for j in range(S) if j <= i)
    assert workload.prefill_flops(1, 1, S, D, True) == 2 * pairs * 2 * D
    assert workload.prefill_flops(2, 3, S, D, False) == 2 * 3 * 4 * S * S * D
    assert workload.decode_flops(2, 4, 10, 8) == 2 * 4 * 10 * 8 * 4


# ---------------------------------------------------------------------------------------------
# planted mistakes: each mutant of the oracle must fail at least one pin
# ---------------------------------------------------------------------------------------------

def _mutant_attention(kind):
    def attn(q, k, v, causal, scale=None, q_pos=None):
        q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
        B, Hq, Sq, D = q.shape
        G = Hq // k.shape[1]
        scale = 1 / np.sqrt(D) if scale is None else scale
        Ov = np.empty((B, Hq, Sq, v.shape[-1]))
        L = np.empty((B, Hq, Sq))
        for b in range(B):
            for hq in range(Hq):
                h = hq % k.shape[1] if kind == "gqa_modulo" else hq // G
                kk = k[b, h]
                s = (1.0 if kind == "no_scale" else scale) * (q[b, hq] @ kk.T)
                if causal:
                    j = np.arange(kk.shape[0])[None, :]
                    i = np.arange(Sq)[:, None] + (kk.shape[0] - Sq)
                    s = np.where((j >= i) if kind == "mask_diag" else (j > i), -np.inf, s)
                m = s.max(-1, keepdims=True)
                # the mask_diag mutant leaves row 0 with no key: NaN there is part of the mistake
                with np.errstate(invalid="ignore"):
                    e = np.exp(s - m)
                l = e.sum(-1, keepdims=True)
                if kind == "no_norm":
                    l = np.ones_like(l)
                vv = v[b, h]
                Ov[b, hq] = (e / l) @ (vv[::-1] if kind == "v_reversed" else vv)
                L[b, hq] = (m + (0 if kind == "lse_no_log" else np.log(l)))[:, 0]
        return Ov, L
    return attn


def _mutant_rope(kind):
    def rope(x, positions, theta):
        x = np.asarray(x, np.float64)
        D = x.shape[-1]
        i = np.arange(D // 2)
        inv = theta ** (-(2.0 if kind != "freq_no2" else 1.0) * i / D)
        a = np.asarray(positions, np.float64)[:, None] * inv[None]
        c, s = np.cos(a), np.sin(a)
        x1, x2 = x[..., : D // 2], x[..., D // 2:]
        if kind == "sign":
            return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], -1)
        if kind == "interleaved_swap":
            return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], -1)[..., ::-1]
        return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], -1)
    return rope


def _mutant_rope_interleaved(kind):
    def rope(x, positions, theta):
        x = np.asarray(x, np.float64)
        D = x.shape[-1]
        i = np.arange(D // 2)
        if kind == "pair_freq_index":  # pair i at the frequency of dim 2i's own index
            inv = theta ** (-2.0 * (2 * i) / D)
        else:
            inv = theta ** (-2.0 * i / D)
        a = np.asarray(positions, np.float64)[:, None] * inv[None]
        c, s = np.cos(a), np.sin(a)
        out = np.empty_like(x)
        e, o = x[..., 0::2], x[..., 1::2]
        if kind == "half_pairs":  # the rotate-half pairing under the interleaved name
            return O.rope_rotate_half(x, positions, theta)
        if kind == "sign":
            out[..., 0::2], out[..., 1::2] = e * c + o * s, o * c - e * s
        else:
            out[..., 0::2], out[..., 1::2] = e * c - o * s, o * c + e * s
        return out
    return rope


@pytest.mark.parametrize("kind", ["pair_freq_index", "half_pairs", "sign"])
def test_planted_interleaved_rope_mistake_is_caught(kind):
    assert _fails_some([pin_rope_interleaved], rope=_mutant_rope_interleaved(kind))


def test_planted_inverse_rotation_mistake_is_caught():
    """An 'inverse' that rotates forwards again (sign kept) fails the round trip."""
    def rope_no_inverse(x, positions, theta, style="half", inverse=False):
        return O.rope_rotate(x, positions, theta, style)
    assert _fails_some([pin_rope_inverse_and_backward_chain], rope=rope_no_inverse)


def test_planted_style_plumbing_mistake_is_caught():
    """A decode that ignores the requested style fails the entry-point pin."""
    def decode_ignoring_style(q, k_cache, v_cache, cache_len, scale=None, rope=True,
                              theta=10000.0, rope_style="half"):
        return O.decode(q, k_cache, v_cache, cache_len, scale, rope, theta)
    assert _fails_some([pin_rope_style_through_entry_points], decode=decode_ignoring_style)


def _mutant_backward(kind):
    def bwd(q, k, v, do, causal, scale=None):
        q, k, v, do = (np.asarray(t, np.float64) for t in (q, k, v, do))
        B, Hq, S, D = q.shape
        G = Hq // k.shape[1]
        scale = 1 / np.sqrt(D) if scale is None else scale
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(B):
            for hq in range(Hq):
                h = hq // G
                s = O.scores(q[b, hq], k[b, h], scale, causal)
                e = np.exp(s - s.max(-1, keepdims=True))
                p = e / e.sum(-1, keepdims=True)
                dv[b, h] += (p @ do[b, hq]) if kind == "dv_no_transpose" else (p.T @ do[b, hq])
                dp = do[b, hq] @ v[b, h].T
                ds = p * dp if kind == "no_delta" else p * (dp - np.sum(dp * p, -1, keepdims=True))
                dq[b, hq] = scale * ((ds.T if kind == "dq_transposed" else ds) @ k[b, h])
                dk[b, h] += (1.0 if kind == "dk_no_scale" else scale) * (ds.T @ q[b, hq])
        return dq, dk, dv
    return bwd


BWD_PINS = [pin_backward_finite_differences, pin_backward_gqa_equals_repeated,
            pin_backward_invariants]


@pytest.mark.parametrize("kind", ["dv_no_transpose", "no_delta", "dq_transposed", "dk_no_scale"])
def test_planted_backward_mistake_is_caught(kind):
    assert _fails_some(BWD_PINS, bwd=_mutant_backward(kind))


def _fails_some(pins, **kw):
    for p in pins:
        try:
            p(**kw)
        except AssertionError:
            return True
    return False


ATTN_PINS = [pin_zero_query_is_causal_mean, pin_hand_two_key_case, pin_one_hot_and_single_key,
             pin_causal_ignores_future, pin_matches_torch_sdpa, pin_bruteforce_enumeration,
             pin_gqa_equals_repeated_mha]


@pytest.mark.parametrize("kind", ["gqa_modulo", "no_scale", "mask_diag", "no_norm", "v_reversed",
                                  "lse_no_log"])
def test_planted_attention_mistake_is_caught(kind):
    assert _fails_some(ATTN_PINS, attn=_mutant_attention(kind))


@pytest.mark.parametrize("kind", ["sign", "freq_no2", "interleaved_swap"])
def test_planted_rope_mistake_is_caught(kind):
    assert _fails_some([pin_rope], rope=_mutant_rope(kind))


def test_planted_merge_mistake_is_caught():
    def bad_merge(o_hist, lse_hist, s_cur, v_cur):
        alpha = 1.0 / (1.0 + np.exp(s_cur - lse_hist))  # sign flipped
        return (1 - alpha) * o_hist + alpha * v_cur, np.logaddexp(lse_hist, s_cur)

    def bad_combine(o_parts, lse_parts):
        w = np.exp(lse_parts - lse_parts.max())
        return (w[:, None] * o_parts).sum(0), np.log(w.sum())  # not normalised

    assert _fails_some([pin_merge_identity], merge=bad_merge)
    assert _fails_some([pin_merge_identity], combine=bad_combine)


def _mutant_latent(kind):
    """Copies of the latent decode with one planted mistake in its RoPE branch."""
    def f(q, c_cache, cache_len, scale=None, rope=True, theta=10000.0, d_latent=448, d_rope=64,
          rope_style="half"):
        q, c = np.asarray(q, np.float64), np.asarray(c_cache, np.float64)
        B, H, dqk = q.shape
        scale = 1.0 / np.sqrt(dqk) if scale is None else scale
        O_, L_ = np.empty((B, H, d_latent)), np.empty((B, H))
        for b in range(B):
            L = int(cache_len[b])
            pos = L - 1 if kind == "pos_L_minus_1" else L
            qb = q[b].copy()
            if rope:
                lo = 0 if kind == "first_dims" else d_latent
                part = qb[:, None, lo: lo + d_rope]
                if kind == "freq_no2":
                    ang = pos * np.power(theta, -np.arange(d_rope // 2) / d_rope)
                    cs, sn = np.cos(ang), np.sin(ang)
                    x1, x2 = part[..., : d_rope // 2], part[..., d_rope // 2:]
                    rot = np.concatenate([x1 * cs - x2 * sn, x2 * cs + x1 * sn], -1)
                else:
                    rot = O.rope_rotate(part, np.array([pos]), theta, rope_style)
                qb[:, lo: lo + d_rope] = rot[:, 0]
            cb = c[b, :L]
            o, l = O.attention(qb[None, :, None, :], cb[None, None], cb[None, None, :, :d_latent],
                               causal=False, scale=scale)
            O_[b], L_[b] = o[0, :, 0], l[0, :, 0]
        return O_, L_
    return f


@pytest.mark.parametrize("kind", ["pos_L_minus_1", "first_dims", "freq_no2"])
def test_planted_latent_rope_mistake_is_caught(kind):
    assert _fails_some([pin_latent_rope_by_hand], latent=_mutant_latent(kind))


def test_latent_mutant_harness_is_faithful():
    """With no mistake planted the mutant copy passes the pin (so the failures above come from
    the planted mistakes, not from the copy)."""
    pin_latent_rope_by_hand(latent=_mutant_latent("none"))


def test_planted_chunk_and_append_mistakes_are_caught():
    """Queries rotated from position 0 instead of their place after the cache, a mask aligned
    top-left, and an appended key left unrotated all fail the pins."""
    def chunk_pos0(q, k, v, skv, scale=None, rope=False, theta=10000.0, pos0=0):
        qq = O.rope_rotate_half(np.asarray(q, np.float64), pos0 + np.arange(q.shape[2]), theta)
        return O.attention(qq, k[:, :, :skv], v[:, :, :skv], causal=True, scale=scale)

    def chunk_topleft(q, k, v, skv, scale=None, rope=False, theta=10000.0, pos0=0):
        sq = q.shape[2]
        qq = O.rope_rotate_half(np.asarray(q, np.float64), pos0 + skv - sq + np.arange(sq), theta)
        return O.attention(qq, k[:, :, :skv], v[:, :, :skv], causal=True, scale=scale,
                           q_pos=np.arange(sq))

    def append_unrotated(q, k_cache, v_cache, cache_len, k_new, v_new, scale=None, rope=True,
                         theta=10000.0):
        # the new key joins the cache as given instead of rotated at position L
        B, Hq, D = q.shape
        o_all, l_all = np.empty((B, Hq, D)), np.empty((B, Hq))
        for b in range(B):
            L = int(cache_len[b])
            qb = O.rope_rotate_half(np.asarray(q[b])[:, None], np.array([L]), theta)
            keys = np.concatenate([k_cache[b, :, :L], np.asarray(k_new[b])[:, None]], 1)
            vals = np.concatenate([v_cache[b, :, :L], np.asarray(v_new[b])[:, None]], 1)
            o, l = O.attention(qb[None], keys[None], vals[None], causal=False, scale=scale)
            o_all[b], l_all[b] = o[0, :, 0], l[0, :, 0]
        return o_all, l_all, np.asarray(k_new)

    assert _fails_some([pin_chunk_equals_prompt_rows], chunk=chunk_pos0)
    assert _fails_some([pin_chunk_equals_prompt_rows], chunk=chunk_topleft)
    assert _fails_some([pin_append_equals_longer_prompt], append=append_unrotated)
