"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports every
entry point include/attn.h declares, and rejects invalid arguments before touching a device.

Only invalid calls are made here (or valid ones when no device is visible), so nothing is ever
launched with the fake pointers these tests pass.
"""
import ctypes
import os
import re

import pytest
import torch

from attention_attn_prefill_02_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA, TIMEOUT, NO_DEVICE, DEVICE_ARG = range(8)
FAKE = ctypes.c_void_p(0x7F0000000000)  # 16-byte aligned, never dereferenced
FAKE2 = ctypes.c_void_p(0x7F0000100000)
MIS = ctypes.c_void_p(0x7F0000000008)   # misaligned


@pytest.fixture(scope="module")
def L():
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_four_operations():
    names = declared_functions()
    for fn in ("rope_apply", "attn_prefill", "attn_decode", "attn_decode_latent"):
        assert fn in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    # and nothing of the internal namespace leaks as a dynamic symbol
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", binding._build.LIB], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(names) <= exported
    assert not any("attn4" in e or "_ZN4attn" in e for e in exported)


def test_status_strings(L):
    for s in range(8):
        assert len(binding.attn_status_string(s)) > 0
    assert binding.attn_status_string(99) == "unknown status"
    assert binding.attn_version() >= 100


def _stream():
    return ctypes.c_void_p(0)


def test_rope_apply_rejects_bad_arguments(L):
    bad = [
        (None, FAKE, 0, 1, 1, 1, 8, 0, 1e4),     # null input
        (FAKE, MIS, 0, 1, 1, 1, 8, 0, 1e4),      # misaligned output
        (FAKE, FAKE2, 5, 1, 1, 1, 8, 0, 1e4),    # bad dtype
        (FAKE, FAKE2, 0, 0, 1, 1, 8, 0, 1e4),    # B = 0
        (FAKE, FAKE2, 0, 1, 1, 1, 7, 0, 1e4),    # odd D
        (FAKE, FAKE2, 0, 1, 1, 1, 8, -1, 1e4),   # negative pos0
        (FAKE, FAKE2, 0, 1, 1, 1, 8, 0, 0.0),    # theta 0
        (FAKE, FAKE2, 0, 1, 1, 1, 8, 0, float("nan")),
        (FAKE, ctypes.c_void_p(0x7F0000000010), 0, 1, 1, 4, 8, 0, 1e4),  # partial overlap
    ]
    for a in bad:
        assert L.rope_apply(*a, _stream()) == INVALID, a


IL = binding.ROPE_FLAG_INTERLEAVED


def test_rope_style_arguments(L):
    """rope_apply_style takes the two pairings only; the attention calls take the interleaved
    flag only together with a rotation mode, and refuse the forms that have no kernel."""
    for style in (-1, 4, 7):
        assert L.rope_apply_style(FAKE, FAKE2, 0, 1, 1, 1, 8, 0, 1e4, style, _stream()) == INVALID
    assert L.rope_apply_style(None, FAKE2, 0, 1, 1, 1, 8, 0, 1e4, 1, _stream()) == INVALID
    assert _prefill(L, rope=IL) == INVALID                    # a pairing without a rotation
    assert _prefill(L, rope=1 | 32) == INVALID                # an unknown bit
    assert _prefill(L, rope=-1) == INVALID
    assert _prefill(L, rope=2 | IL) == UNSUPPORTED            # the kernel rotates half-split only
    assert _prefill(L, rope=1 | IL, dt=1, D=128) == UNSUPPORTED  # fp8 rotates in the kernel
    assert _chunk(L, rope=1 | IL, dt=1) == UNSUPPORTED
    assert _chunk(L, rope=2 | IL) == INVALID
    assert _decode(L, rope=IL) == INVALID
    assert _decode(L, rope=2 | IL) == INVALID
    assert _append(L, rope=IL) == INVALID
    assert _latent(L, rope=IL) == INVALID
    assert _latent(L, rope=1 | 64) == INVALID
    # the binding composes the flag from rope_style
    assert binding._rope_mode(True, "interleaved") == 1 | IL
    assert binding._rope_mode(2, "interleaved") == 2 | IL
    assert binding._rope_mode(False, "interleaved") == 0
    assert binding._rope_mode(True) == 1


def _bwd(L, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE2, do=FAKE, dq=FAKE2, dk=FAKE2, dv=FAKE2,
                dt=0, B=1, Hq=4, Hkv=1, S=128, D=64, causal=1, scale=0.0, ws=FAKE2, wsb=1 << 30)
    args.update(kw)
    return L.attn_prefill_backward(*args.values(), _stream())


def test_prefill_backward_validation(L):
    assert _bwd(L, lse=None) == INVALID
    assert _bwd(L, ws=None) == INVALID
    assert _bwd(L, dq=MIS) == INVALID
    assert _bwd(L, lse=ctypes.c_void_p(0x7F0000000002)) == INVALID
    assert _bwd(L, Hq=6, Hkv=4) == INVALID
    assert _bwd(L, causal=2) == INVALID
    assert _bwd(L, S=0) == INVALID
    assert _bwd(L, dt=1) == UNSUPPORTED                # bf16 only
    assert _bwd(L, D=256) == UNSUPPORTED
    assert _bwd(L, wsb=16) == WORKSPACE
    n = binding.attn_prefill_backward_workspace_size(2, 8, 300, 128)
    rows = 2 * 8 * 300
    assert n == ((rows * 4 + 255) // 256) * 256 + rows * 128 * 4
    assert binding.attn_prefill_backward_workspace_size(1, 1, 1, 96) == 0


def _prefill(L, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE2, lse=None, dt=0, qs=1.0, ks=1.0, vs=1.0, B=1,
                Hq=4, Hkv=1, S=128, D=64, causal=1, scale=0.0, rope=1, theta=1e4, pos0=0,
                ws=FAKE, wsb=1 << 30)
    args.update(kw)
    return L.attn_prefill(*args.values(), _stream())


def test_prefill_validation(L):
    assert _prefill(L, q=None) == INVALID
    assert _prefill(L, o=MIS) == INVALID
    assert _prefill(L, Hq=6, Hkv=4) == INVALID          # Hq % Hkv
    assert _prefill(L, S=0) == INVALID
    assert _prefill(L, causal=2) == INVALID
    assert _prefill(L, rope=1, theta=-1.0) == INVALID
    assert _prefill(L, rope=3) == INVALID
    assert _prefill(L, qs=0.0) == INVALID
    assert _prefill(L, lse=ctypes.c_void_p(0x7F0000000002)) == INVALID
    assert _prefill(L, D=96) == UNSUPPORTED
    assert _prefill(L, D=512) == UNSUPPORTED
    assert _prefill(L, D=256, dt=1) == UNSUPPORTED     # D = 256: fp8 without RoPE only
    assert _prefill(L, D=256, rope=2) == UNSUPPORTED   # ... and RoPE through the passes
    assert _chunk(L, D=256, dt=1, rope=1) == UNSUPPORTED


def _chunk(L, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE2, lse=None, dt=0, qs=1.0, ks=1.0, vs=1.0, B=1,
                Hq=4, Hkv=1, Sq=32, Skv=300, pitch=320, D=128, scale=0.0, rope=1, theta=1e4,
                pos0=0, ws=FAKE, wsb=1 << 30)
    args.update(kw)
    return L.attn_prefill_chunk(*args.values(), _stream())


def test_prefill_chunk_validation(L):
    assert _chunk(L, Sq=0) == INVALID
    assert _chunk(L, Sq=301) == INVALID               # more queries than keys
    assert _chunk(L, pitch=299) == INVALID            # keys past the cache rows
    assert _chunk(L, Hq=6, Hkv=4) == INVALID
    assert _chunk(L, v=MIS) == INVALID
    assert _chunk(L, D=96) == UNSUPPORTED
    assert _chunk(L, dt=1, D=64) == UNSUPPORTED       # fp8 with q RoPE: D = 128 only
    assert _chunk(L, ws=None, wsb=0) == WORKSPACE     # bf16 with RoPE rotates q into it
    assert _chunk(L, wsb=32 * 4 * 128 * 2 - 1) == WORKSPACE
    assert _chunk(L, ws=MIS) == WORKSPACE


def test_prefill_workspace_sizes(L):
    """The caller's workspace holds the rotated Q (rounded up to 256 bytes) then the rotated K
    exactly when RoPE runs as rotation passes: bf16, rope = 1 and S >= 1024, or the interleaved
    pairing, or D = 256.  Everything else needs none."""
    bf16, fp8, il = 0, 1, 16
    q_bytes = 4 * 32 * 16384 * 128 * 2
    assert L.attn_prefill_workspace_size(4, 32, 8, 16384, 128, bf16, 1) == \
        q_bytes + 4 * 8 * 16384 * 128 * 2
    assert L.attn_prefill_workspace_size(4, 32, 8, 16384, 128, bf16, 2) == 0   # in the kernel
    assert L.attn_prefill_workspace_size(4, 32, 8, 16384, 128, bf16, 0) == 0
    assert L.attn_prefill_workspace_size(4, 32, 8, 16384, 128, fp8, 1) == 0    # fp8: in-kernel
    assert L.attn_prefill_workspace_size(1, 4, 1, 1023, 64, bf16, 1) == 0      # short prompt
    assert L.attn_prefill_workspace_size(1, 3, 1, 5, 64, bf16, 1 | il) == \
        ((3 * 5 * 64 * 2 + 255) // 256) * 256 + 5 * 64 * 2
    assert L.attn_prefill_workspace_size(1, 2, 1, 8, 256, bf16, 1) == 2 * 8 * 256 * 2 + 8 * 256 * 2
    assert L.attn_prefill_workspace_size(1, 2, 1, 8, 96, bf16, 1) == 0         # invalid -> 0
    assert L.attn_prefill_workspace_size(1, 2, 1, 8, 64, bf16, 3) == 0
    assert L.attn_prefill_chunk_workspace_size(2, 8, 33, 128, bf16, 1) == \
        ((2 * 8 * 33 * 128 * 2 + 255) // 256) * 256
    assert L.attn_prefill_chunk_workspace_size(2, 8, 33, 128, fp8, 1) == 0
    assert L.attn_prefill_chunk_workspace_size(2, 8, 33, 128, bf16, 0) == 0
    # a call that needs it refuses a missing, short or misaligned workspace before any launch
    assert _prefill(L, S=1024, ws=None, wsb=0) == WORKSPACE
    assert _prefill(L, S=1024, wsb=L.attn_prefill_workspace_size(1, 4, 1, 1024, 64, bf16, 1) - 1) \
        == WORKSPACE
    assert _prefill(L, S=1024, ws=MIS) == WORKSPACE


def _decode(L, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, lens=FAKE2, Lmax=2048, o=FAKE2, lse=None, dt=0, B=1,
                Hq=32, Hkv=8, D=128, scale=0.0, rope=1, theta=1e4, ws=FAKE2, wsb=1 << 30)
    args.update(kw)
    return L.attn_decode(*args.values(), _stream())


def test_forced_decode_splits_change_the_plan(L):
    """The global-split hook: the workspace follows the forced split, 0 restores the planner."""
    planned = binding.attn_decode_workspace_size(1, 32, 8, 128, 2048)
    assert L.attn_set_decode_splits(-1) == INVALID
    assert L.attn_set_decode_splits(1025) == INVALID
    try:
        binding.attn_set_decode_splits(1)
        assert binding.attn_decode_workspace_size(1, 32, 8, 128, 2048) == 0
        binding.attn_set_decode_splits(4)
        assert binding.attn_decode_workspace_size(1, 32, 8, 128, 2048) == 1 * 32 * 4 * 129 * 4
        binding.attn_set_decode_splits(5000 // 64)  # more than one split per tile is capped
        assert binding.attn_decode_workspace_size(1, 32, 8, 128, 640) == 1 * 32 * 10 * 129 * 4
    finally:
        binding.attn_set_decode_splits(0)
    assert binding.attn_decode_workspace_size(1, 32, 8, 128, 2048) == planned


def test_decode_validation(L):
    assert _decode(L, lens=None) == INVALID
    assert _decode(L, Lmax=0) == INVALID
    assert _decode(L, Hq=30) == INVALID
    assert _decode(L, D=80) == UNSUPPORTED
    assert _decode(L, Hq=64, Hkv=2) == UNSUPPORTED      # group of 32 > 16
    assert _decode(L, dt=1, D=64) == UNSUPPORTED        # fp8 cache only for D = 128
    assert _decode(L, rope=3) == INVALID
    assert _decode(L, D=256, dt=1) == UNSUPPORTED        # fp8 cache: D = 128 only
    assert _decode(L, D=512) == UNSUPPORTED
    # D = 256 (bf16) is a decode head dim: it has a plan (and a workspace when it splits)
    assert binding.attn_decode_workspace_size(1, 32, 8, 256, 2048) > 0
    assert binding.attn_decode_append_workspace_size(1, 32, 8, 256, 2048) > 0


def _append(L, **kw):
    args = dict(q=FAKE, kn=FAKE, vn=FAKE, kc=FAKE, vc=FAKE, lens=FAKE2, Lmax=2048, o=FAKE2,
                lse=None, dt=0, B=2, Hq=32, Hkv=8, D=128, scale=0.0, rope=1, theta=1e4, ws=FAKE2,
                wsb=1 << 20)
    args.update(kw)
    return L.attn_decode_append(*args.values(), _stream())


def test_decode_append_validation(L):
    assert _append(L, ws=None) == INVALID                # the history LSE always needs room
    assert _append(L, kn=None) == INVALID
    assert _append(L, vc=MIS) == INVALID
    assert _append(L, Lmax=1) == INVALID                 # no row for the new token
    assert _append(L, Hq=30) == INVALID
    assert _append(L, D=80) == UNSUPPORTED
    assert _append(L, dt=1) == UNSUPPORTED               # bf16 caches only
    assert _append(L, Hq=64, Hkv=2) == UNSUPPORTED
    # history workspace (rounded to 256 bytes) plus one float per query row
    assert binding.attn_decode_append_workspace_size(128, 32, 8, 128, 2048) == 128 * 32 * 4
    w1 = binding.attn_decode_append_workspace_size(1, 32, 8, 128, 2048)
    d1 = binding.attn_decode_workspace_size(1, 32, 8, 128, 2048)
    assert w1 == ((d1 + 255) // 256) * 256 + 32 * 4
    assert binding.attn_decode_append_workspace_size(1, 30, 8, 128, 2048) == 0


def _latent(L, **kw):
    args = dict(q=FAKE, c=FAKE, lens=FAKE2, Lmax=2048, o=FAKE2, lse=None, dt=0, B=128, H=16,
                scale=0.0, rope=1, theta=1e4, ws=FAKE2, wsb=1 << 30)
    args.update(kw)
    return L.attn_decode_latent(*args.values(), _stream())


def test_latent_validation(L):
    assert _latent(L, c=None) == INVALID
    assert _latent(L, H=0) == INVALID
    assert _latent(L, H=17) == UNSUPPORTED
    assert _latent(L, q=MIS) == INVALID
    assert _latent(L, dt=7) == INVALID


def test_workspace_sizes_are_consistent(L):
    # sizes that split the key range need workspace; the batch-128 decode config needs none
    assert binding.attn_decode_workspace_size(1, 32, 8, 128, 2048) > 0
    assert binding.attn_decode_workspace_size(128, 32, 8, 128, 2048) == 0
    assert binding.attn_decode_workspace_size(1, 30, 8, 128, 2048) == 0  # invalid -> 0
    # latent decode: 128 CTAs; with B = 128 each takes one whole sequence (no workspace),
    # otherwise the key tiles are split evenly over the CTAs and the pieces (B + 127 slots,
    # 449 floats per head) are merged afterwards, with the tile prefix sums (B + 1 ints)
    assert binding.attn_decode_latent_workspace_size(128, 16, 2048) == 0
    assert binding.attn_decode_latent_workspace_size(8, 16, 2048) == \
        (8 + 128 - 1) * 16 * 449 * 4 + (8 + 1) * 4
    assert binding.attn_decode_latent_workspace_size(1, 16, 2048) > 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_calls_report_no_device_without_gpu(L):
    assert _prefill(L) == NO_DEVICE
    assert _prefill(L, rope=2) == NO_DEVICE
    assert _prefill(L, S=16384) == NO_DEVICE
    assert _prefill(L, ws=None, wsb=0) == NO_DEVICE   # S = 128: the kernel rotates, no workspace
    assert _chunk(L) == NO_DEVICE
    assert _prefill(L, D=256, dt=1, rope=0) == NO_DEVICE   # fp8 at D = 256 without RoPE
    assert _chunk(L, D=256, dt=1, rope=0) == NO_DEVICE
    assert _decode(L) == NO_DEVICE
    assert _append(L) == NO_DEVICE
    assert _decode(L, ws=None, wsb=0) in (NO_DEVICE, WORKSPACE)
    assert _latent(L) == NO_DEVICE
    assert L.rope_apply(FAKE, FAKE, 0, 1, 1, 4, 8, 0, 1e4, _stream()) == NO_DEVICE
    st = ctypes.c_int(-1)
    assert L.attn_get_device_status(_stream(), ctypes.byref(st)) == NO_DEVICE
    assert L.attn_rope_table_reserve(64, 1e4, 100) == NO_DEVICE


def test_product_path_does_not_import_the_oracle():
    """The CUDA path's Python package never refers to the oracle package."""
    pkg = os.path.join(ROOT, "attention_attn_prefill_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_selftest_and_event_hook_validation(L):
    """The bounded-wait self-test takes a limit of 1 us .. 2 s; the measurement hook takes both
    events or neither.  Both answer on the host before touching a device."""
    assert L.attn_selftest_wait_timeout(0, _stream()) == INVALID
    assert L.attn_selftest_wait_timeout(2000001, _stream()) == INVALID
    assert L.attn_set_prefill_events(FAKE, None) == INVALID
    assert L.attn_set_prefill_events(None, FAKE) == INVALID
    assert L.attn_set_prefill_events(None, None) == OK
    assert L.attn_set_prefill_tiles(3) == INVALID
    assert L.attn_set_prefill_tiles(-1) == INVALID
    assert L.attn_set_prefill_tiles(0) == OK
    assert L.attn_set_backward_path(3) == INVALID
    assert L.attn_set_backward_path(-1) == INVALID
    assert L.attn_set_backward_path(0) == OK
    if not torch.cuda.is_available():
        assert L.attn_selftest_wait_timeout(10000, _stream()) == NO_DEVICE
