"""Thin ctypes binding over the C ABI in ``include/attn.h``.

Every function here only marshals arguments (tensor -> device pointer, sizes, the current CUDA
stream) and turns a non-OK status into ``AttnError``.  All arithmetic runs in the library's CUDA
kernels; there is no CPU fallback.  The names match the C entry points.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

ATTN_OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA",
                5: "TIMEOUT", 6: "NO_DEVICE", 7: "DEVICE_ARG"}
DTYPE_CODES = {torch.bfloat16: 0, torch.float8_e5m2: 1}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({lib().attn_status_string(status).decode()})")


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first when needed) the in-tree shared library."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing:
        path = _build.build_library()
    if not os.path.exists(path):
        raise RuntimeError(f"attention library not built: {path} is missing")
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_status_string.argtypes = [i]
    L.attn_version.restype = i
    L.attn_version.argtypes = []
    L.rope_apply.restype = i
    L.rope_apply.argtypes = [vp, vp, i, i, i, i, i, i, f, vp]
    L.rope_apply_style.restype = i
    L.rope_apply_style.argtypes = [vp, vp, i, i, i, i, i, i, f, i, vp]
    L.attn_prefill.restype = i
    L.attn_prefill.argtypes = [vp, vp, vp, vp, vp, i, f, f, f, i, i, i, i, i, i, f, i, f, i, vp,
                               sz, vp]
    L.attn_prefill_workspace_size.restype = sz
    L.attn_prefill_workspace_size.argtypes = [i, i, i, i, i, i, i]
    L.attn_prefill_chunk_workspace_size.restype = sz
    L.attn_prefill_chunk_workspace_size.argtypes = [i, i, i, i, i, i]
    L.attn_prefill_backward_workspace_size.restype = sz
    L.attn_prefill_backward_workspace_size.argtypes = [i, i, i, i]
    L.attn_prefill_backward.restype = i
    L.attn_prefill_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f,
                                        vp, sz, vp]
    L.attn_prefill_chunk.restype = i
    L.attn_prefill_chunk.argtypes = [vp, vp, vp, vp, vp, i, f, f, f, i, i, i, i, i, i, i, f, i, f,
                                     i, vp, sz, vp]
    L.attn_decode_workspace_size.restype = sz
    L.attn_decode_workspace_size.argtypes = [i, i, i, i, i]
    L.attn_decode.restype = i
    L.attn_decode.argtypes = [vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, f, i, f, vp, sz, vp]
    L.attn_decode_noalloc.restype = i
    L.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, f, i, f, vp]
    L.attn_set_prefill_tiles.restype = i
    L.attn_set_prefill_tiles.argtypes = [i]
    L.attn_set_backward_path.restype = i
    L.attn_set_backward_path.argtypes = [i]
    L.attn_set_prefill_events.restype = i
    L.attn_set_prefill_events.argtypes = [vp, vp]
    L.attn_set_decode_splits.restype = i
    L.attn_set_decode_splits.argtypes = [i]
    L.attn_decode_append_workspace_size.restype = sz
    L.attn_decode_append_workspace_size.argtypes = [i, i, i, i, i]
    L.attn_decode_append.restype = i
    L.attn_decode_append.argtypes = [vp, vp, vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, f, i, f,
                                     vp, sz, vp]
    L.attn_decode_latent_workspace_size.restype = sz
    L.attn_decode_latent_workspace_size.argtypes = [i, i, i]
    L.attn_decode_latent.restype = i
    L.attn_decode_latent.argtypes = [vp, vp, vp, i, vp, vp, i, i, i, f, i, f, vp, sz, vp]
    L.attn_rope_table_reserve.restype = i
    L.attn_rope_table_reserve.argtypes = [i, f, i]
    L.attn_selftest_wait_timeout.restype = i
    L.attn_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
    L.attn_get_device_status.restype = i
    L.attn_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    _lib = L
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def _require_cuda(*tensors):
    for t in tensors:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# RoPE pairing: "half" pairs dims (i, i + D/2), "interleaved" pairs (2i, 2i+1); same angles.
ROPE_STYLES = {"half": 0, "interleaved": 1}
ROPE_FLAG_INTERLEAVED = 16  # ATTN_ROPE_FLAG_INTERLEAVED, OR'd into the attention calls' rope


def rope_apply(x, y=None, pos0=0, theta=10000.0, stream=None, rope_style="half", inverse=False):
    """Rotate x [B,H,S,D] at positions pos0 + s into y (new tensor when None; may be x);
    `inverse` rotates by the opposite angles (gradients back through RoPE)."""
    _require_cuda(x)
    if y is None:
        y = torch.empty_like(x)
    B, H, S, D = x.shape
    _check(lib().rope_apply_style(_ptr(x), _ptr(y), DTYPE_CODES[x.dtype], B, H, S, D, int(pos0),
                                  float(theta), ROPE_STYLES[rope_style] | (2 if inverse else 0),
                                  _stream(stream)),
           "rope_apply")
    return y


def _rope_mode(rope, rope_style="half"):
    """False/0: none; True/1: the library's choice; 2: Q and K both rotated inside the kernel;
    with the interleaved pairing the flag is OR'd in."""
    mode = 2 if (not isinstance(rope, bool) and rope == 2) else int(bool(rope))
    return mode | (ROPE_FLAG_INTERLEAVED if (mode and ROPE_STYLES[rope_style]) else 0)


def attn_prefill_workspace_size(B, Hq, Hkv, S, D, dtype=torch.bfloat16, rope=False,
                                rope_style="half"):
    """Bytes of workspace attn_prefill needs (nonzero when RoPE runs as rotation passes)."""
    return int(lib().attn_prefill_workspace_size(B, Hq, Hkv, S, D, DTYPE_CODES[dtype],
                                                 _rope_mode(rope, rope_style)))


def _workspace(workspace, need, device):
    """The caller's workspace, or a fresh one of `need` bytes (None when nothing is needed)."""
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace, (0 if workspace is None else workspace.numel() * workspace.element_size())


def attn_prefill(q, k, v, causal=True, softmax_scale=0.0, rope=False, rope_theta=10000.0,
                 pos0=0, o=None, lse=None, want_lse=False, q_scale=1.0, k_scale=1.0,
                 v_scale=1.0, stream=None, rope_style="half", workspace=None):
    """O [B,Hq,S,D] bf16 (and LSE [B,Hq,S] fp32 when requested) for q [B,Hq,S,D], k/v [B,Hkv,S,D].
    `workspace`: a uint8 CUDA tensor of at least attn_prefill_workspace_size() bytes (allocated
    here when None and needed)."""
    _require_cuda(q, k, v, o, lse, workspace)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    if o is None:
        o = torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    mode = _rope_mode(rope, rope_style)
    workspace, wbytes = _workspace(
        workspace, int(lib().attn_prefill_workspace_size(B, Hq, Hkv, S, D, DTYPE_CODES[q.dtype],
                                                         mode)), q.device)
    _check(lib().attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                              DTYPE_CODES[q.dtype], float(q_scale), float(k_scale),
                              float(v_scale), B, Hq, Hkv, S, D, int(bool(causal)),
                              float(softmax_scale), mode, float(rope_theta), int(pos0),
                              _ptr(workspace), wbytes, _stream(stream)), "attn_prefill")
    return (o, lse) if (want_lse or lse is not None) else o


def attn_prefill_backward_workspace_size(B, Hq, S, D):
    return int(lib().attn_prefill_backward_workspace_size(B, Hq, S, D))


def attn_prefill_backward(q, k, v, o, lse, dout, causal=True, softmax_scale=0.0, dq=None,
                          dk=None, dv=None, workspace=None, stream=None):
    """(dQ, dK, dV) bf16 of attn_prefill's attention for q [B,Hq,S,D], k/v [B,Hkv,S,D] (as the
    forward used them), its output o and LSE, and dout = dL/dO."""
    _require_cuda(q, k, v, o, lse, dout, dq, dk, dv, workspace)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(attn_prefill_backward_workspace_size(B, Hq, S, D),
                                dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    _check(lib().attn_prefill_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
                                       _ptr(dq), _ptr(dk), _ptr(dv), DTYPE_CODES[q.dtype], B, Hq,
                                       Hkv, S, D, int(bool(causal)), float(softmax_scale),
                                       _ptr(workspace), wbytes, _stream(stream)),
           "attn_prefill_backward")
    return dq, dk, dv


def attn_prefill_chunk_workspace_size(B, Hq, Sq, D, dtype=torch.bfloat16, rope=True,
                                      rope_style="half"):
    return int(lib().attn_prefill_chunk_workspace_size(B, Hq, Sq, D, DTYPE_CODES[dtype],
                                                       _rope_mode(bool(rope), rope_style)))


def attn_prefill_chunk(q, k_cache, v_cache, skv, softmax_scale=0.0, rope=True,
                       rope_theta=10000.0, pos0=0, o=None, lse=None, want_lse=False, q_scale=1.0,
                       k_scale=1.0, v_scale=1.0, stream=None, rope_style="half", workspace=None):
    """O [B,Hq,Sq,D] bf16 for a chunk q [B,Hq,Sq,D] whose rows are the last Sq of `skv` tokens,
    against the first `skv` rows of the caches [B,Hkv,Lmax,D] (keys stored rotated)."""
    _require_cuda(q, k_cache, v_cache, o, lse, workspace)
    B, Hq, Sq, D = q.shape
    Hkv, pitch = k_cache.shape[1], k_cache.shape[2]
    if o is None:
        o = torch.empty((B, Hq, Sq, D), dtype=torch.bfloat16, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    mode = _rope_mode(bool(rope), rope_style)
    workspace, wbytes = _workspace(
        workspace, int(lib().attn_prefill_chunk_workspace_size(B, Hq, Sq, D,
                                                               DTYPE_CODES[q.dtype], mode)),
        q.device)
    _check(lib().attn_prefill_chunk(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse),
                                    DTYPE_CODES[q.dtype], float(q_scale), float(k_scale),
                                    float(v_scale), B, Hq, Hkv, Sq, int(skv), pitch, D,
                                    float(softmax_scale), mode, float(rope_theta), int(pos0),
                                    _ptr(workspace), wbytes, _stream(stream)),
           "attn_prefill_chunk")
    return (o, lse) if (want_lse or lse is not None) else o


def attn_decode_workspace_size(B, Hq, Hkv, D, Lmax):
    return int(lib().attn_decode_workspace_size(B, Hq, Hkv, D, Lmax))


def attn_decode(q, k_cache, v_cache, cache_len, o=None, lse=None, want_lse=False,
                softmax_scale=0.0, rope=True, rope_theta=10000.0, workspace=None, stream=None,
                rope_style="half"):
    """O [B,Hq,D] for q [B,Hq,D] (bf16) against caches [B,Hkv,Lmax,D] (bf16 or fp8 e5m2) with
    device cache_len [B]."""
    _require_cuda(q, k_cache, v_cache, cache_len, o, lse, workspace)
    B, Hq, D = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = attn_decode_workspace_size(B, Hq, Hkv, D, Lmax)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_len), Lmax,
                             _ptr(o), _ptr(lse), DTYPE_CODES[k_cache.dtype], B, Hq, Hkv, D,
                             float(softmax_scale), _rope_mode(bool(rope), rope_style),
                             float(rope_theta), _ptr(workspace), wbytes, _stream(stream)),
           "attn_decode")
    return (o, lse) if (want_lse or lse is not None) else o


def attn_decode_noalloc(q, k_cache, v_cache, cache_len, o=None, lse=None, want_lse=False,
                        softmax_scale=0.0, rope=True, rope_theta=10000.0, stream=None,
                        rope_style="half"):
    """attn_decode without a workspace: its split partials use the library's fixed 2 MiB
    device array (for callers that cannot allocate at call time)."""
    _require_cuda(q, k_cache, v_cache, cache_len, o, lse)
    B, Hq, D = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(lib().attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_len),
                                     Lmax, _ptr(o), _ptr(lse), DTYPE_CODES[k_cache.dtype], B, Hq, Hkv,
                                     D, float(softmax_scale), _rope_mode(bool(rope), rope_style),
                                     float(rope_theta), _stream(stream)), "attn_decode_noalloc")
    return (o, lse) if (want_lse or lse is not None) else o


def attn_set_prefill_tiles(q_tiles):
    """1 or 2 Q tiles per prefill work item for later calls at D <= 128; 0: the default (2)."""
    _check(lib().attn_set_prefill_tiles(int(q_tiles)), "attn_set_prefill_tiles")


def attn_set_backward_path(path):
    """Kernels of later attn_prefill_backward calls: 1 = warp-level mma.sync, 2 = tcgen05,
    0 = the default (tcgen05)."""
    _check(lib().attn_set_backward_path(int(path)), "attn_set_backward_path")


def attn_set_prefill_events(begin=None, end=None):
    """Record the torch.cuda.Event pair `begin`/`end` around the attention kernel of every later
    prefill call (both None: stop).  The events must have been recorded once (torch creates the
    CUDA event on first use)."""
    h = [None if e is None else ctypes.c_void_p(e.cuda_event) for e in (begin, end)]
    _check(lib().attn_set_prefill_events(*h), "attn_set_prefill_events")


def attn_set_decode_splits(nsplit):
    """nsplit > 0: force that split count for later decode calls; 0: the per-shape planner."""
    _check(lib().attn_set_decode_splits(int(nsplit)), "attn_set_decode_splits")


def attn_decode_append_workspace_size(B, Hq, Hkv, D, Lmax):
    return int(lib().attn_decode_append_workspace_size(B, Hq, Hkv, D, Lmax))


def attn_decode_append(q, k_new, v_new, k_cache, v_cache, cache_len, o=None, lse=None,
                       want_lse=False, softmax_scale=0.0, rope=True, rope_theta=10000.0,
                       workspace=None, stream=None, rope_style="half"):
    """One growing-decode step: O [B,Hq,D] over the cache rows 0..L-1 plus the current token,
    whose key/value are written to row L = cache_len[b]; cache_len is incremented on device."""
    _require_cuda(q, k_new, v_new, k_cache, v_cache, cache_len, o, lse, workspace)
    B, Hq, D = q.shape
    Hkv, Lmax = k_cache.shape[1], k_cache.shape[2]
    if o is None:
        o = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(attn_decode_append_workspace_size(B, Hq, Hkv, D, Lmax),
                                dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    _check(lib().attn_decode_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                    _ptr(v_cache), _ptr(cache_len), Lmax, _ptr(o), _ptr(lse),
                                    DTYPE_CODES[k_cache.dtype], B, Hq, Hkv, D,
                                    float(softmax_scale), _rope_mode(bool(rope), rope_style),
                                    float(rope_theta), _ptr(workspace), wbytes, _stream(stream)),
           "attn_decode_append")
    return (o, lse) if (want_lse or lse is not None) else o


def attn_decode_latent_workspace_size(B, H, Lmax):
    return int(lib().attn_decode_latent_workspace_size(B, H, Lmax))


def attn_decode_latent(q, c_cache, cache_len, o=None, lse=None, want_lse=False,
                       softmax_scale=0.0, rope=True, rope_theta=10000.0, workspace=None,
                       stream=None, rope_style="half"):
    """O [B,H,448] for q [B,H,512] against the latent cache [B,Lmax,512]."""
    _require_cuda(q, c_cache, cache_len, o, lse, workspace)
    B, H, _ = q.shape
    Lmax = c_cache.shape[1]
    if o is None:
        o = torch.empty((B, H, 448), dtype=torch.bfloat16, device=q.device)
    if want_lse and lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    need = attn_decode_latent_workspace_size(B, H, Lmax)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().attn_decode_latent(_ptr(q), _ptr(c_cache), _ptr(cache_len), Lmax, _ptr(o),
                                    _ptr(lse), DTYPE_CODES[c_cache.dtype], B, H,
                                    float(softmax_scale), _rope_mode(bool(rope), rope_style),
                                    float(rope_theta), _ptr(workspace), wbytes,
                                    _stream(stream)), "attn_decode_latent")
    return (o, lse) if (want_lse or lse is not None) else o


def attn_rope_table_reserve(D, theta, max_pos):
    _check(lib().attn_rope_table_reserve(int(D), float(theta), int(max_pos)),
           "attn_rope_table_reserve")


def attn_selftest_wait_timeout(timeout_us, stream=None):
    """Run one bounded wait that must time out after `timeout_us` (sets TIMEOUT in the status
    word; the kernel returns on its own)."""
    _check(lib().attn_selftest_wait_timeout(int(timeout_us), _stream(stream)),
           "attn_selftest_wait_timeout")


def attn_get_device_status(stream=None) -> int:
    out = ctypes.c_int(-1)
    _check(lib().attn_get_device_status(_stream(stream), ctypes.byref(out)),
           "attn_get_device_status")
    return out.value


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def attn_version() -> int:
    return int(lib().attn_version())
