"""attn_decode_noalloc: the decode entry point for callers that cannot allocate device memory
when they call (plugin-style enqueue paths, processes whose memory another allocator owns,
latency-bound serving loops).  It keeps its split partials in the library's fixed 2 MiB device
array instead of a caller workspace.

Checked through the C ABI against attn_decode (same inputs, the tolerance the other parity tests
use) and against the float64 oracle, on two calls in a row with different inputs, so the second
call runs over the first call's leftover scratch.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_attn_prefill_02_gb300 import binding, synthetic

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
SCRATCH = 2 << 20


def _close(a, b):
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS, (d.max(), d.mean())


@pytest.mark.parametrize("B,Hq,Hkv,D,Lmax,lens", [
    (1, 32, 8, 128, 2048, [2048]),          # decode config at batch 1: 32 splits of the cache
    (3, 32, 8, 128, 2048, [2048, 1, 700]),  # ragged lengths, still split
    (2, 16, 4, 256, 2048, [2048, 300]),     # D = 256: one CTA per SM, larger partials
])
def test_noalloc_matches_workspace_decode_twice(B, Hq, Hkv, D, Lmax, lens):
    assert 0 < binding.attn_decode_workspace_size(B, Hq, Hkv, D, Lmax) <= SCRATCH
    binding.attn_rope_table_reserve(D, 10000.0, Lmax)
    for call in range(2):
        q, kc, vc, cl = synthetic.decode_inputs(B, Hq, Hkv, Lmax, D, lens, seed=40 + call)
        q, kc, vc, cl = q.cuda(), kc.cuda(), vc.cuda(), cl.cuda()
        ref, ref_lse = binding.attn_decode(q, kc, vc, cl, want_lse=True, rope=True)
        out, out_lse = binding.attn_decode_noalloc(q, kc, vc, cl, want_lse=True, rope=True)
        torch.cuda.synchronize()
        assert binding.attn_get_device_status() == 0
        _close(out, ref)
        np.testing.assert_allclose(out_lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=5e-3)
        # and directly against the oracle, at the same bounds
        ro, rl = oracle.decode(*(oracle.as_f64(t.cpu()) for t in (q, kc, vc)), cl.cpu().numpy(),
                               rope=True, theta=10000.0)
        d = np.abs(oracle.as_f64(out.cpu()) - ro)
        assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (d.max(), d.mean())
        assert np.abs(out_lse.cpu().numpy() - rl).max() <= 5e-3


def test_noalloc_rejects_what_it_cannot_do_without_allocating():
    q, kc, vc, cl = synthetic.decode_inputs(1, 16, 1, 64, 128, 64, seed=3)
    q, kc, vc, cl = q.cuda(), kc.cuda(), vc.cuda(), cl.cuda()
    # fp8 e5m2 caches are not built for this entry point: UNSUPPORTED, nothing launched
    with pytest.raises(binding.AttnError) as e:
        binding.attn_decode_noalloc(q, kc.to(torch.float8_e5m2), vc.to(torch.float8_e5m2), cl,
                                    rope=False)
    assert e.value.status == 2
    # a RoPE table that was never built would need an allocation: refused before any launch
    with pytest.raises(binding.AttnError) as e:
        binding.attn_decode_noalloc(q, kc, vc, cl, rope=True, rope_theta=12345.5)
    assert e.value.status == 3
    # sizes whose split partials exceed the fixed scratch are refused before any launch
    # (the size check runs on the host before anything is launched, so the small buffers
    # passed here are never read)
    big = dict(B=1, Hq=128, Hkv=8, D=128, Lmax=1 << 18)
    assert binding.attn_decode_workspace_size(*big.values()) > SCRATCH
    L = binding.lib()
    import ctypes
    st = L.attn_decode_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
                               ctypes.c_void_p(vc.data_ptr()), ctypes.c_void_p(cl.data_ptr()),
                               big["Lmax"], ctypes.c_void_p(q.data_ptr()), None, 0, big["B"],
                               big["Hq"], big["Hkv"], big["D"], 0.0, 0, 10000.0,
                               ctypes.c_void_p(0))
    assert st == 3
