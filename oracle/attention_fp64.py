"""CPU oracle for causal grouped-query attention with RoPE, split-KV decode and latent decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg may import this module.  The product path (the CUDA library and its Python binding)
never calls it, and this module never calls the CUDA path: the two share no code.

Everything here is plain NumPy in float64, written as the textbook definition: materialise the
full score matrix, mask it, subtract the row maximum, exponentiate, normalise, multiply by V.  No
blocking, no online softmax, no fusion.  The only library primitives used are ``@`` (matmul),
``np.exp``/``np.log``/``np.cos``/``np.sin`` and reductions.

Where the pages are silent, the readings used are (each is repeated in the design notes):

* RoPE is the rotate-half pairing (i, i + D/2) with inverse frequency theta^(-2i/D).  The pages
  only name "RoPE-attention fusion" (Lesson: shape adaptive attention negative 20260722, rows
  "해본 것" / "당시 조건").  The other common convention, adjacent pairs (2i, 2i + 1) rotated by
  the same angles ("interleaved"), is available as ``rope_style="interleaved"``; the pages do not
  name a convention, so both are offered and the half-split one is the default.
* Query head hq reads KV head hq // G with G = Hq / Hkv (contiguous grouping).
* Causal masking hides key j from query i when j > i + (Skv - Sq) (bottom-right alignment; the
  workloads only use Sq == Skv, where this is the usual j > i).
* Decode: the single query sits at position L = cache_len[b] and attends the L cached keys
  0..L-1, which are stored already rotated; only the query is rotated.
* Latent decode: the query and every cache row have 448 latent dims followed by 64 RoPE dims;
  scores use all 512 dims, values are the first 448 dims of the cache row (Fixed-budget decode
  audit — 2026-09-11, "Which implementation was tested": 448-dimensional latent + 64-dimensional
  RoPE).  RoPE is applied to the last 64 query dims only.
"""
from __future__ import annotations

import numpy as np

LATENT_DIM = 448
LATENT_ROPE_DIM = 64


def as_f64(x) -> np.ndarray:
    """Exact float64 copy of a torch tensor (any storage dtype) or array-like."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------------------------

def rope_inv_freq(D: int, theta: float) -> np.ndarray:
    """theta^(-2i/D) for i < D/2, in float64."""
    i = np.arange(D // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / D)


def rope_rotate_half(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate each pair (x_i, x_{i+D/2}) of the last axis by angle pos * theta^(-2i/D).

    ``x`` has shape [..., n, D]; ``positions`` has shape [n] (one position per row).
    Returns x'_i = x_i cos a - x_{i+D/2} sin a and x'_{i+D/2} = x_{i+D/2} cos a + x_i sin a.
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    assert D % 2 == 0
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(D, theta)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1 = x[..., : D // 2]
    x2 = x[..., D // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_rotate_interleaved(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate each adjacent pair (x_{2i}, x_{2i+1}) of the last axis by pos * theta^(-2i/D).

    The interleaved convention: x'_{2i} = x_{2i} cos a - x_{2i+1} sin a and
    x'_{2i+1} = x_{2i+1} cos a + x_{2i} sin a, with the same angle a for pair i as the
    rotate-half form uses for its pair (i, i + D/2).
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    assert D % 2 == 0
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(D, theta)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    even, odd = x[..., 0::2], x[..., 1::2]
    out[..., 0::2] = even * c - odd * s
    out[..., 1::2] = odd * c + even * s
    return out


ROPE_STYLES = ("half", "interleaved")


def rope_rotate(x: np.ndarray, positions: np.ndarray, theta: float, style: str = "half",
                inverse: bool = False):
    """RoPE in the given pairing convention ("half": (i, i + D/2); "interleaved": (2i, 2i+1)).

    ``inverse`` rotates by the opposite angles: the transpose of the rotation, which is also
    the gradient map from rotated to un-rotated vectors (backward through RoPE).
    """
    pos = -np.asarray(positions, dtype=np.float64) if inverse else positions
    if style == "half":
        return rope_rotate_half(x, pos, theta)
    if style == "interleaved":
        return rope_rotate_interleaved(x, pos, theta)
    raise ValueError(f"unknown RoPE style {style!r}")


# --------------------------------------------------------------------------------------------
# Attention by its definition
# --------------------------------------------------------------------------------------------

def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax with max subtraction; rows that are entirely -inf are not allowed."""
    m = np.max(s, axis=-1, keepdims=True)
    assert np.all(np.isfinite(m)), "fully masked row"
    p = np.exp(s - m)
    return p / np.sum(p, axis=-1, keepdims=True)


def scores(q: np.ndarray, k: np.ndarray, scale: float, causal: bool, q_pos=None) -> np.ndarray:
    """Masked score matrix scale * q k^T for one head: q [Sq,D], k [Skv,D] -> [Sq,Skv].

    ``q_pos`` gives each query row's position in key coordinates (default: bottom-right aligned
    positions Skv - Sq + i).  Key j is hidden from a row at position p when j > p.
    """
    Sq, Skv = q.shape[0], k.shape[0]
    s = scale * (q @ k.T)
    if causal:
        if q_pos is None:
            q_pos = np.arange(Sq) + (Skv - Sq)
        j = np.arange(Skv)[None, :]
        s = np.where(j > np.asarray(q_pos)[:, None], -np.inf, s)
    return s


def attention(q, k, v, causal: bool, scale: float | None = None, q_pos=None):
    """O = softmax(scale * Q K^T + mask) V and LSE = log sum_j exp(S_ij), per (b, hq).

    q [B,Hq,Sq,D], k [B,Hkv,Skv,D], v [B,Hkv,Skv,Dv] (float64).  Query head hq uses KV head
    hq // (Hq / Hkv).  Returns (O [B,Hq,Sq,Dv], LSE [B,Hq,Sq]) in float64.
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O = np.empty((B, Hq, Sq, v.shape[-1]))
    LSE = np.empty((B, Hq, Sq))
    for b in range(B):
        for hq in range(Hq):
            h = hq // G
            s = scores(q[b, hq], k[b, h], scale, causal, q_pos)
            m = np.max(s, axis=-1, keepdims=True)
            e = np.exp(s - m)
            l = np.sum(e, axis=-1, keepdims=True)
            O[b, hq] = (e / l) @ v[b, h]
            LSE[b, hq] = (m + np.log(l))[:, 0]
    return O, LSE


def attention_backward(q, k, v, do, causal: bool, scale: float | None = None):
    """Gradients of the loss L with dL/dO = ``do`` through O = softmax(scale Q K^T + mask) V.

    Inputs as ``attention`` (RoPE, when used, is applied to q and k before this call; its own
    gradient is the inverse rotation).  Per (b, hq) with KV head h = hq // G, by the chain rule
    on the definition: P = softmax(S); dV_h += P^T dO; dP = dO V^T; dS = P * (dP - rowsum(dP * P))
    (the softmax Jacobian); dQ = scale dS K; dK_h += scale dS^T Q.  The KV gradients of a group
    are summed over its G query heads.  Returns (dQ, dK, dV) in float64.
    """
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for hq in range(Hq):
            h = hq // G
            s = scores(q[b, hq], k[b, h], scale, causal)
            m = np.max(s, axis=-1, keepdims=True)
            e = np.exp(s - m)
            p = e / np.sum(e, axis=-1, keepdims=True)
            dv[b, h] += p.T @ do[b, hq]
            dp = do[b, hq] @ v[b, h].T
            ds = p * (dp - np.sum(dp * p, axis=-1, keepdims=True))
            dq[b, hq] = scale * (ds @ k[b, h])
            dk[b, h] += scale * (ds.T @ q[b, hq])
    return dq, dk, dv


def attention_probs(q, k, causal: bool, scale: float | None = None):
    """The normalised probability matrices P [B,Hq,Sq,Skv] (for invariant checks)."""
    q, k = np.asarray(q, np.float64), np.asarray(k, np.float64)
    B, Hq, Sq, D = q.shape
    G = Hq // k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    P = np.empty((B, Hq, Sq, k.shape[2]))
    for b in range(B):
        for hq in range(Hq):
            P[b, hq] = softmax_rows(scores(q[b, hq], k[b, hq // G], scale, causal))
    return P


def prefill(q, k, v, causal=True, scale=None, rope=False, theta=10000.0, pos0=0,
            rope_style="half"):
    """Prefill: optionally rotate Q and K at positions pos0 .. pos0+S-1, then attention.

    Positions follow the reading that prefill tokens sit at 0..S-1 (pos0 = 0) on a fresh
    sequence.  Returns (O, LSE) in float64.
    """
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    if rope:
        pos_q = pos0 + np.arange(q.shape[2])
        pos_k = pos0 + np.arange(k.shape[2])
        q = rope_rotate(q, pos_q, theta, rope_style)
        k = rope_rotate(k, pos_k, theta, rope_style)
    return attention(q, k, v, causal, scale)


def prefill_rows(q, k, v, rows, causal=True, scale=None, rope=False, theta=10000.0, pos0=0,
                 rope_style="half"):
    """Selected output rows of ``prefill`` (for sizes where the full oracle is too slow).

    ``rows`` is a list of (b, hq, i).  Each row is computed by the same definition: rotate the
    query row at position pos0+i and all keys, form the row of scores, mask keys j > i (causal,
    Sq == Skv), softmax, multiply by V.  Returns (O [n,Dv], LSE [n]).
    """
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    B, Hq, S, D = q.shape
    G = Hq // k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cache = {}
    out_o, out_l = [], []
    for (b, hq, i) in rows:
        h = hq // G
        key = (b, h)
        if key not in cache:
            kk = k[b, h]
            if rope:
                kk = rope_rotate(kk, pos0 + np.arange(kk.shape[0]), theta, rope_style)
            cache[key] = kk
        kk = cache[key]
        qi = q[b, hq, i][None, :]
        if rope:
            qi = rope_rotate(qi, np.array([pos0 + i]), theta, rope_style)
        s = scores(qi, kk, scale, causal, q_pos=np.array([i + (kk.shape[0] - S)]))
        m = np.max(s)
        e = np.exp(s - m)
        l = np.sum(e)
        out_o.append(((e / l) @ v[b, h])[0])
        out_l.append(m + np.log(l))
    return np.array(out_o), np.array(out_l)


def decode(q, k_cache, v_cache, cache_len, scale=None, rope=True, theta=10000.0,
           rope_style="half"):
    """Single-token decode against a static cache.

    q [B,Hq,D]; k_cache/v_cache [B,Hkv,Lmax,D] (keys stored already rotated); cache_len [B].
    Sequence b's query sits at position L = cache_len[b]; it is rotated there when ``rope``;
    it attends keys 0..L-1.  Returns (O [B,Hq,D], LSE [B,Hq]).
    """
    q, kc, vc = (np.asarray(t, np.float64) for t in (q, k_cache, v_cache))
    lens = np.asarray(cache_len).astype(np.int64)
    B, Hq, D = q.shape
    Dv = vc.shape[-1]
    O = np.empty((B, Hq, Dv))
    LSE = np.empty((B, Hq))
    for b in range(B):
        L = int(lens[b])
        assert 1 <= L <= kc.shape[2]
        qb = q[b][:, None, :]  # [Hq, 1, D]
        if rope:
            qb = rope_rotate(qb, np.array([L]), theta, rope_style)
        o, lse = attention(qb[None], kc[b: b + 1, :, :L], vc[b: b + 1, :, :L], causal=False,
                           scale=scale)
        O[b] = o[0, :, 0]
        LSE[b] = lse[0, :, 0]
    return O, LSE


def prefill_chunk(q, k, v, skv, scale=None, rope=False, theta=10000.0, pos0=0,
                  rope_style="half"):
    """One chunk of a prompt against the keys before it and its own (chunked prefill).

    The prompt is prefilled a chunk at a time into a static cache before decoding (Fixed-budget
    decode audit — 2026-09-11, "Setup and interpretation").  q [B,Hq,Sq,D]; k, v
    [B,Hkv,>=skv,D] whose first ``skv`` rows are the keys before the chunk followed by the
    chunk's own, stored already rotated.  Query row i sits at position skv - Sq + i (rotated at
    pos0 plus that when ``rope``) and attends keys 0..skv - Sq + i.  Returns (O, LSE).
    """
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    Sq = q.shape[2]
    assert 1 <= Sq <= skv <= k.shape[2]
    if rope:
        q = rope_rotate(q, pos0 + skv - Sq + np.arange(Sq), theta, rope_style)
    return attention(q, k[:, :, :skv], v[:, :, :skv], causal=True, scale=scale)


def decode_append(q, k_cache, v_cache, cache_len, k_new, v_new, scale=None, rope=True,
                  theta=10000.0, rope_style="half"):
    """Decode step that also attends the current token, whose key/value join the cache.

    Sequence b's query and new key sit at position L = cache_len[b]; both are rotated there when
    ``rope``.  The query attends the L cached keys plus the new one: the plain definition over
    L + 1 keys (the kernel reaches it by merging the new key into the cached-history result, the
    merge of ``merge_one_key``).  k_new, v_new [B,Hkv,D].  Returns (O [B,Hq,D], LSE [B,Hq],
    K_ROW [B,Hkv,D]: the new key as the cache stores it, i.e. rotated).
    """
    q, kc, vc, kn, vn = (np.asarray(t, np.float64) for t in (q, k_cache, v_cache, k_new, v_new))
    lens = np.asarray(cache_len).astype(np.int64)
    B, Hq, D = q.shape
    O = np.empty((B, Hq, vc.shape[-1]))
    LSE = np.empty((B, Hq))
    K_ROW = np.empty(kn.shape)
    for b in range(B):
        L = int(lens[b])
        assert 0 <= L < kc.shape[2]
        kr = kn[b][:, None, :]  # [Hkv, 1, D]
        qb = q[b][:, None, :]
        if rope:
            kr = rope_rotate(kr, np.array([L]), theta, rope_style)
            qb = rope_rotate(qb, np.array([L]), theta, rope_style)
        K_ROW[b] = kr[:, 0]
        keys = np.concatenate([kc[b, :, :L], kr], axis=1)
        vals = np.concatenate([vc[b, :, :L], vn[b][:, None, :]], axis=1)
        o, lse = attention(qb[None], keys[None], vals[None], causal=False, scale=scale)
        O[b] = o[0, :, 0]
        LSE[b] = lse[0, :, 0]
    return O, LSE, K_ROW


def latent_decode(q, c_cache, cache_len, scale=None, rope=True, theta=10000.0,
                  d_latent=LATENT_DIM, d_rope=LATENT_ROPE_DIM, rope_style="half"):
    """Absorbed latent (MLA-style) decode.

    q [B,H,d_latent+d_rope]; c_cache [B,Lmax,d_latent+d_rope] (rope part stored rotated);
    every head attends the same latent rows: S = scale * q C^T over all dims, V = C[:, :d_latent].
    The last ``d_rope`` query dims are rotated at position L = cache_len[b] when ``rope``.
    Returns (O [B,H,d_latent], LSE [B,H]).
    """
    q, c = np.asarray(q, np.float64), np.asarray(c_cache, np.float64)
    lens = np.asarray(cache_len).astype(np.int64)
    B, H, dqk = q.shape
    assert dqk == d_latent + d_rope == c.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(dqk)
    O = np.empty((B, H, d_latent))
    LSE = np.empty((B, H))
    for b in range(B):
        L = int(lens[b])
        assert 1 <= L <= c.shape[1]
        qb = q[b].copy()
        if rope:
            qb[:, d_latent:] = rope_rotate(qb[:, None, d_latent:], np.array([L]), theta,
                                           rope_style)[:, 0]
        cb = c[b, :L]
        o, lse = attention(qb[None, :, None, :], cb[None, None], cb[None, None, :, :d_latent],
                           causal=False, scale=scale)
        O[b] = o[0, :, 0]
        LSE[b] = lse[0, :, 0]
    return O, LSE


# --------------------------------------------------------------------------------------------
# Merging partial attention results
# --------------------------------------------------------------------------------------------

def merge_one_key(o_hist, lse_hist, s_cur, v_cur):
    """Merge one extra key into an already normalised partial attention.

    Fixed-budget decode audit — 2026-09-11, "A: group-entry queries and one joint history scan":
    with alpha = sigmoid(s_cur - lse_hist), the merged output is (1-alpha) o_hist + alpha v_cur.
    The merged log-sum-exp is log(exp(lse_hist) + exp(s_cur)).
    """
    o_hist, v_cur = np.asarray(o_hist, np.float64), np.asarray(v_cur, np.float64)
    lse_hist, s_cur = np.asarray(lse_hist, np.float64), np.asarray(s_cur, np.float64)
    alpha = 1.0 / (1.0 + np.exp(-(s_cur - lse_hist)))
    out = (1.0 - alpha)[..., None] * o_hist + alpha[..., None] * v_cur
    return out, np.logaddexp(lse_hist, s_cur)


def combine_partials(o_parts, lse_parts):
    """Combine split partials: LSE = log sum_s exp(lse_s), O = sum_s exp(lse_s - LSE) o_s.

    o_parts [..., n, D], lse_parts [..., n]; a split with lse = -inf contributes nothing.
    """
    o_parts, lse_parts = np.asarray(o_parts, np.float64), np.asarray(lse_parts, np.float64)
    m = np.max(lse_parts, axis=-1, keepdims=True)
    w = np.exp(lse_parts - m)
    tot = np.sum(w, axis=-1, keepdims=True)
    lse = (m + np.log(tot))[..., 0]
    o = np.sum((w / tot)[..., None] * o_parts, axis=-2)
    return o, lse


def split_decode_partials(q_row, k, v, split: int, scale: float):
    """Attention of one query row over k/v [L,D] computed split by split (partials + LSE).

    Each split of ``split`` keys is attention restricted to that split; returns
    (o_parts [n, Dv], lse_parts [n]).  Used to check that combining splits equals the whole.
    """
    q_row, k, v = (np.asarray(t, np.float64) for t in (q_row, k, v))
    L = k.shape[0]
    o_parts, lse_parts = [], []
    for s0 in range(0, L, split):
        o, lse = attention(q_row[None, None, None, :], k[None, None, s0:s0 + split],
                           v[None, None, s0:s0 + split], causal=False, scale=scale)
        o_parts.append(o[0, 0, 0])
        lse_parts.append(lse[0, 0, 0])
    return np.array(o_parts), np.array(lse_parts)
