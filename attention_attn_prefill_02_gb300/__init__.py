"""GB300 (sm_103a) attention library: causal GQA prefill with fused RoPE, split-KV decode,
absorbed-latent decode and rope_apply, exposed through a C ABI (include/attn.h).

The Python names below are a ctypes binding of that ABI; every computation runs in the
library's CUDA kernels.
"""
from .binding import (  # noqa: F401
    AttnError, attn_decode, attn_decode_latent, attn_decode_noalloc, attn_decode_latent_workspace_size,
    attn_decode_workspace_size, attn_get_device_status, attn_prefill, attn_rope_table_reserve,
    attn_status_string, attn_version, lib, rope_apply,
)
