"""GPU checks of the boundary's contracts: caller-owned workspaces (two prefills at once on two
streams), outputs written only where the call says (guard bytes around every output), the
bounded-wait failure path (a wait that must time out reports TIMEOUT and leaves the context
usable), and the measurement hook that brackets the attention kernel with events.

Numerical results are compared with the float64 oracle at the bf16 bounds (max-abs 2e-2,
mean-abs 2e-3).
"""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_prefill_02_gb300 import binding, synthetic

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3
TIMEOUT, DEVICE_ARG = 5, 7


def f64(t):
    return oracle.as_f64(t)


def check(gpu, ref, max_abs=BF16_MAX, mean_abs=BF16_MEAN, what=""):
    d = np.abs(f64(gpu) - ref)
    assert np.all(np.isfinite(f64(gpu))), what
    assert d.max() <= max_abs, f"{what}: max-abs {d.max():.3e}"
    assert d.mean() <= mean_abs, f"{what}: mean-abs {d.mean():.3e}"


def guarded(shape, dtype, guard_elems=4096, fill=None):
    """A view of `shape` inside a larger buffer whose guard regions before and after hold a
    sentinel; returns (view, buffer, sentinel).  The view starts 16-byte aligned."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 2 * guard_elems, dtype=dtype, device="cuda")
    sentinel = -12345.0 if fill is None else fill
    buf.fill_(sentinel)
    return buf[guard_elems: guard_elems + n].view(shape), buf, guard_elems


def guards_intact(buf, g, n, sentinel=-12345.0):
    head, tail = buf[:g], buf[g + n:]
    return bool(torch.all(head == sentinel)) and bool(torch.all(tail == sentinel))


# --------------------------------------------------------------------------------------------
# caller-owned workspaces
# --------------------------------------------------------------------------------------------

def test_prefill_two_streams_own_workspaces():
    """Two RoPE prefills run at the same time on two streams, each rotating its Q and K into a
    workspace of its own: both match the oracle (a shared scratch would let one call's rotated
    inputs overwrite the other's)."""
    shapes = [(1, 4, 2, 1100, 128, 21), (1, 4, 2, 1100, 128, 22)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ins, outs, wss = [], [], []
    for (B, Hq, Hkv, S, D, seed) in shapes:
        q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=seed)
        ins.append((q, k, v))
        need = binding.attn_prefill_workspace_size(B, Hq, Hkv, S, D, rope=1)
        assert need == (B * Hq * S * D * 2 + 255) // 256 * 256 + B * Hkv * S * D * 2
        wss.append(torch.empty(need, dtype=torch.uint8, device="cuda"))
    dev = [(q.cuda(), k.cuda(), v.cuda()) for q, k, v in ins]
    torch.cuda.synchronize()
    for rep in range(3):  # several overlapping rounds
        outs = []
        for (qd, kd, vd), ws, st in zip(dev, wss, streams):
            with torch.cuda.stream(st):
                outs.append(binding.attn_prefill(qd, kd, vd, causal=True, rope=1,
                                                 rope_theta=10000.0, workspace=ws, stream=st,
                                                 want_lse=True))
        torch.cuda.synchronize()
    assert binding.attn_get_device_status() == 0
    for (q, k, v), (o, lse) in zip(ins, outs):
        ro, rl = oracle.prefill(f64(q), f64(k), f64(v), causal=True, rope=True, theta=10000.0)
        check(o.cpu(), ro, what="O")
        assert np.abs(f64(lse.cpu()) - rl).max() <= 1e-2


def test_prefill_chunk_caller_workspace():
    """A bf16 RoPE chunk rotates its queries into the caller's workspace; too small a workspace
    is refused before any launch."""
    B, Hq, Hkv, Sq, Skv, D = 2, 8, 2, 40, 300, 128
    q = synthetic.normal((B, Hq, Sq, D), 31, "bf16")
    kc = synthetic.normal((B, Hkv, 320, D), 32, "bf16")
    vc = synthetic.normal((B, Hkv, 320, D), 33, "bf16")
    need = binding.attn_prefill_chunk_workspace_size(B, Hq, Sq, D, rope=True)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = binding.attn_prefill_chunk(q.cuda(), kc.cuda(), vc.cuda(), Skv, rope=True, workspace=ws)
    with pytest.raises(binding.AttnError):
        binding.attn_prefill_chunk(q.cuda(), kc.cuda(), vc.cuda(), Skv, rope=True,
                                   workspace=ws[: need - 16])
    assert binding.attn_get_device_status() == 0
    ro, _ = oracle.prefill_chunk(f64(q), f64(kc), f64(vc), Skv, rope=True, theta=10000.0)
    check(o.cpu(), ro, what="O chunk")


# --------------------------------------------------------------------------------------------
# outputs are written only inside their bounds (guard bytes around each)
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("S,D,rope", [(300, 128, 1), (1025, 64, 1), (77, 64, 0), (130, 256, 0)])
def test_prefill_writes_only_its_output(S, D, rope):
    """Ragged prompt lengths: O and LSE rows past S (the padded tail of the last tile) are never
    stored, so guard regions around both stay intact."""
    B, Hq, Hkv = 1, 4, 2
    q, k, v = synthetic.prefill_inputs(B, Hq, Hkv, S, D, "bf16", seed=S + D)
    o, obuf, g = guarded((B, Hq, S, D), torch.bfloat16)
    lse, lbuf, gl = guarded((B, Hq, S), torch.float32)
    binding.attn_prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, rope=rope, o=o, lse=lse)
    torch.cuda.synchronize()
    assert binding.attn_get_device_status() == 0
    assert guards_intact(obuf, g, o.numel()) and guards_intact(lbuf, gl, lse.numel())
    ro, _ = oracle.prefill(f64(q), f64(k), f64(v), causal=True, rope=bool(rope), theta=10000.0)
    check(o.cpu(), ro, what="O")


def test_chunk_decode_latent_write_only_their_outputs():
    # a chunk of 33 rows after 260 cached ones
    B, Hq, Hkv, D = 2, 4, 2, 128
    q = synthetic.normal((B, Hq, 33, D), 41, "bf16")
    kc = synthetic.normal((B, Hkv, 320, D), 42, "bf16")
    vc = synthetic.normal((B, Hkv, 320, D), 43, "bf16")
    o, obuf, g = guarded((B, Hq, 33, D), torch.bfloat16)
    binding.attn_prefill_chunk(q.cuda(), kc.cuda(), vc.cuda(), 293, rope=True, o=o)
    torch.cuda.synchronize()
    assert guards_intact(obuf, g, o.numel())
    # decode with ragged lengths and a split plan
    q, kc, vc, cl = synthetic.decode_inputs(3, 32, 8, 2048, 128, [2048, 1, 700], seed=44)
    o, obuf, g = guarded((3, 32, 128), torch.bfloat16)
    lse, lbuf, gl = guarded((3, 32), torch.float32)
    binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda(), o=o, lse=lse)
    torch.cuda.synchronize()
    assert guards_intact(obuf, g, o.numel()) and guards_intact(lbuf, gl, lse.numel())
    # latent decode, stream-K split over the SMs
    q, c, cl = synthetic.latent_inputs(3, 16, 2048, [2048, 5, 1000], seed=45)
    o, obuf, g = guarded((3, 16, 448), torch.bfloat16)
    binding.attn_decode_latent(q.cuda(), c.cuda(), cl.cuda(), o=o)
    torch.cuda.synchronize()
    assert guards_intact(obuf, g, o.numel())
    assert binding.attn_get_device_status() == 0


def test_append_writes_only_row_L():
    """The growing-decode step writes the new key and value to row L = cache_len[b] of each
    sequence and nothing else of the caches."""
    B, Hq, Hkv, Lmax, D = 3, 16, 4, 96, 128
    lens = [10, 95, 1]
    q, kc, vc, cl = synthetic.decode_inputs(B, Hq, Hkv, Lmax, D, lens, seed=46)
    kn = synthetic.normal((B, Hkv, D), 47)
    vn = synthetic.normal((B, Hkv, D), 48)
    kd, vd, cl_d = kc.cuda(), vc.cuda(), cl.cuda()
    binding.attn_decode_append(q.cuda(), kn.cuda(), vn.cuda(), kd, vd, cl_d)
    torch.cuda.synchronize()
    assert binding.attn_get_device_status() == 0
    kd, vd = kd.cpu(), vd.cpu()
    for b, L in enumerate(lens):
        keep = [r for r in range(Lmax) if r != L]
        assert torch.equal(kd[b][:, keep], kc[b][:, keep])
        assert torch.equal(vd[b][:, keep], vc[b][:, keep])
        assert torch.equal(vd[b][:, L], vn[b])
    assert cl_d.cpu().tolist() == [L + 1 for L in lens]


# --------------------------------------------------------------------------------------------
# bounded waits and the device status word
# --------------------------------------------------------------------------------------------

def test_bounded_wait_times_out_and_context_survives():
    """A wait on an mbarrier that nothing arrives at gives up after its limit (10 ms here),
    reports TIMEOUT once through the status word and returns; the next calls on the same context
    are correct."""
    assert binding.attn_get_device_status() == 0
    binding.attn_selftest_wait_timeout(10_000)
    assert binding.attn_get_device_status() == TIMEOUT
    assert binding.attn_get_device_status() == 0      # reported once, then cleared
    q, kc, vc, cl = synthetic.decode_inputs(2, 32, 8, 2048, 128, [2048, 300], seed=49)
    o = binding.attn_decode(q.cuda(), kc.cuda(), vc.cuda(), cl.cuda())
    assert binding.attn_get_device_status() == 0
    ro, _ = oracle.decode(f64(q), f64(kc), f64(vc), cl.numpy())
    check(o.cpu(), ro, what="decode after a timeout")
    with pytest.raises(binding.AttnError):
        binding.attn_selftest_wait_timeout(0)           # limit outside 1 us .. 2 s


def test_prefill_event_hook_brackets_the_attention_kernel():
    """The measurement hook records its events around the attention kernel only: with the two
    rotation passes in front, the bracketed time is shorter than the whole call's."""
    q, k, v = synthetic.prefill_inputs(2, 16, 4, 4096, 128, "bf16", seed=50)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.empty(binding.attn_prefill_workspace_size(2, 16, 4, 4096, 128, rope=1),
                     dtype=torch.uint8, device="cuda")
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for x in e:
        x.record()
    binding.attn_prefill(qd, kd, vd, causal=True, rope=1, workspace=ws)  # warm-up
    torch.cuda.synchronize()
    binding.attn_set_prefill_events(e[1], e[2])
    try:
        e[0].record()
        binding.attn_prefill(qd, kd, vd, causal=True, rope=1, workspace=ws)
        e[3].record()
    finally:
        binding.attn_set_prefill_events(None, None)
    torch.cuda.synchronize()
    kernel, call = e[1].elapsed_time(e[2]), e[0].elapsed_time(e[3])
    assert 0 < kernel < call
    assert binding.attn_get_device_status() == 0
