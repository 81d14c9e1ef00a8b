// api.cpp — the C ABI: argument validation, workspace planning and dispatch to the kernels.
// Validation happens entirely on the host before anything is enqueued, so an invalid call
// returns its status without touching the GPU (this is what the CPU-only tests exercise).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"

using namespace attn;

namespace {

cudaStream_t as_stream(attn_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

bool finite_pos(float x) { return std::isfinite(x) && x > 0.f; }

bool overlap_partial(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  if (x == y) return false;
  return x < y + bytes && y < x + bytes;
}

size_t dtype_bytes(attn_dtype_t dt) { return dt == ATTN_BF16 ? 2 : 1; }

bool valid_dtype(int dt) { return dt == ATTN_BF16 || dt == ATTN_FP8_E5M2; }

// Events recorded around the attention kernel of attn_prefill / attn_prefill_chunk (diagnostics,
// see attn_set_prefill_events); both null when unset.
std::atomic<cudaEvent_t> g_ev_begin{nullptr}, g_ev_end{nullptr};

attn_status_t timed_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                            attn_dtype_t dt, float q_scale, float k_scale, float v_scale, int B,
                            int Hq, int Hkv, int S, int Skv, int kv_pitch, int D, int causal,
                            float scale, const float2* table, int rope_k, int pos0,
                            cudaStream_t st) {
  cudaEvent_t e0 = g_ev_begin.load(), e1 = g_ev_end.load();
  if (e0 && cudaEventRecord(e0, st) != cudaSuccess) return ATTN_ERR_CUDA;
  const attn_status_t r = launch_prefill(q, k, v, o, lse, dt, q_scale, k_scale, v_scale, B, Hq,
                                         Hkv, S, Skv, kv_pitch, D, causal, scale, table, rope_k,
                                         pos0, st);
  if (r == ATTN_OK && e1 && cudaEventRecord(e1, st) != cudaSuccess) return ATTN_ERR_CUDA;
  return r;
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA runtime or launch error";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    case ATTN_ERR_NO_DEVICE: return "no usable sm_100-family CUDA device";
    case ATTN_ERR_DEVICE_ARG: return "device-resident argument out of range";
  }
  return "unknown status";
}

int attn_version(void) { return 200; }

// Head dims of the single-token decode paths (bf16 caches; the fp8 cache is D = 128 only).
static bool decode_head_dim(int D) { return D == 64 || D == 128 || D == 256; }

attn_status_t rope_apply(const void* x, void* y, attn_dtype_t dtype, int B, int H, int S, int D,
                         int pos0, float theta, attn_stream_t stream) {
  return rope_apply_style(x, y, dtype, B, H, S, D, pos0, theta, ATTN_ROPE_HALF_SPLIT, stream);
}

attn_status_t rope_apply_style(const void* x, void* y, attn_dtype_t dtype, int B, int H, int S,
                               int D, int pos0, float theta, attn_rope_style_t style,
                               attn_stream_t stream) {
  if (static_cast<int>(style) < 0 || static_cast<int>(style) > 3) return ATTN_ERR_INVALID_ARG;
  if (!x || !y || !aligned16(x) || !aligned16(y)) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1 || D < 2 || D > 256 || (D & 1) || pos0 < 0) return ATTN_ERR_INVALID_ARG;
  if (!finite_pos(theta)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(pos0) + S > (1LL << 30)) return ATTN_ERR_INVALID_ARG;
  const size_t bytes = static_cast<size_t>(B) * H * S * D * dtype_bytes(dtype);
  if (overlap_partial(x, y, bytes)) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  const float2* tab = rope_table(D, theta, pos0 + S, &st);
  if (!tab) return st;
  const int st_bits = static_cast<int>(style);
  return launch_rope(x, y, dtype, B, H, S, D, pos0, tab, st_bits & 1, as_stream(stream),
                     (st_bits >> 1) & 1);
}

size_t attn_prefill_workspace_size(int B, int Hq, int Hkv, int S, int D, attn_dtype_t dtype,
                                   int rope) {
  int mode = 0, il = 0;
  if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || !valid_dtype(dtype)) return 0;
  if (D != 64 && D != 128 && D != 256) return 0;
  if (!split_rope_arg(rope, 2, &mode, &il)) return 0;
  return prefill_ws_bytes(B, Hq, Hkv, S, D, dtype, mode, il);
}

attn_status_t attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                           attn_dtype_t dtype, float q_scale, float k_scale, float v_scale,
                           int B, int Hq, int Hkv, int S, int D, int causal, float softmax_scale,
                           int rope, float rope_theta, int pos0, void* workspace,
                           size_t workspace_bytes, attn_stream_t stream) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  int il = 0;
  if (!split_rope_arg(rope, 2, &rope, &il)) return ATTN_ERR_INVALID_ARG;
  if (rope && (!finite_pos(rope_theta) || pos0 < 0)) return ATTN_ERR_INVALID_ARG;
  if (!finite_pos(q_scale) || !finite_pos(k_scale) || !finite_pos(v_scale))
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(S) > (1LL << 30) || static_cast<long long>(B) * Hq > (1LL << 24))
    return ATTN_ERR_UNSUPPORTED;
  // the interleaved pairing runs only as rope_apply passes (bf16; the kernel's in-tile rotation
  // is the half-split form); so does every rotation at D = 256, which therefore takes fp8 only
  // without RoPE (rotated fp8 tiles would have to stay bf16)
  if (il && (rope == 2 || dtype != ATTN_BF16)) return ATTN_ERR_UNSUPPORTED;
  if (D == 256 && (rope == 2 || (rope && dtype != ATTN_BF16))) return ATTN_ERR_UNSUPPORTED;
  const size_t ws_need = prefill_ws_bytes(B, Hq, Hkv, S, D, dtype, rope, il);
  if (ws_need > 0 && (!workspace || workspace_bytes < ws_need || !aligned16(workspace)))
    return ATTN_ERR_WORKSPACE;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  const float2* tab = nullptr;
  if (rope) {
    // the fused K rotation starts every thread's recurrence from rows pos0 .. pos0 + 31
    tab = rope_table(D, rope_theta, pos0 + std::max(S, 128), &st);
    if (!tab) return st;
  }
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (ws_need > 0) {
    // Q and K rotated once each into the caller's workspace, then attention without RoPE
    const size_t qb = prefill_ws_q_bytes(B, Hq, S, D);
    uint8_t* sc = static_cast<uint8_t*>(workspace);
    st = launch_rope(q, sc, dtype, B, Hq, S, D, pos0, tab, il, as_stream(stream));
    if (st != ATTN_OK) return st;
    st = launch_rope(k, sc + qb, dtype, B, Hkv, S, D, pos0, tab, il, as_stream(stream));
    if (st != ATTN_OK) return st;
    return timed_prefill(sc, sc + qb, v, o, lse, dtype, q_scale, k_scale, v_scale, B, Hq, Hkv,
                          S, S, S, D, causal, scale, nullptr, 0, pos0, as_stream(stream));
  }
  return timed_prefill(q, k, v, o, lse, dtype, q_scale, k_scale, v_scale, B, Hq, Hkv, S, S, S,
                        D, causal, scale, tab, rope ? 1 : 0, pos0, as_stream(stream));
}

size_t attn_prefill_backward_workspace_size(int B, int Hq, int S, int D) {
  if (B < 1 || Hq < 1 || S < 1 || (D != 64 && D != 128)) return 0;
  return bwd_workspace_bytes(B, Hq, S, D);
}

attn_status_t attn_prefill_backward(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dout, void* dq, void* dk,
                                    void* dv, attn_dtype_t dtype, int B, int Hq, int Hkv, int S,
                                    int D, int causal, float softmax_scale, void* workspace,
                                    size_t workspace_bytes, attn_stream_t stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(S) > (1LL << 30) ||
      static_cast<long long>(B) * Hq * S > (1LL << 31) / 128)
    return ATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < bwd_workspace_bytes(B, Hq, S, D)) return ATTN_ERR_WORKSPACE;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  return launch_prefill_backward(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, causal,
                                 scale, workspace, as_stream(stream));
}

size_t attn_prefill_chunk_workspace_size(int B, int Hq, int Sq, int D, attn_dtype_t dtype,
                                         int rope) {
  int mode = 0, il = 0;
  if (B < 1 || Hq < 1 || Sq < 1 || !valid_dtype(dtype)) return 0;
  if (D != 64 && D != 128 && D != 256) return 0;
  if (!split_rope_arg(rope, 1, &mode, &il)) return 0;
  return chunk_ws_bytes(B, Hq, Sq, D, dtype, mode);
}

attn_status_t attn_prefill_chunk(const void* q, const void* k, const void* v, void* o, float* lse,
                                 attn_dtype_t dtype, float q_scale, float k_scale, float v_scale,
                                 int B, int Hq, int Hkv, int Sq, int Skv, int kv_pitch, int D,
                                 float softmax_scale, int rope, float rope_theta, int pos0,
                                 void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (Sq < 1 || Skv < Sq || kv_pitch < Skv) return ATTN_ERR_INVALID_ARG;
  int il = 0;
  if (!split_rope_arg(rope, 1, &rope, &il)) return ATTN_ERR_INVALID_ARG;
  if (rope && (!finite_pos(rope_theta) || pos0 < 0)) return ATTN_ERR_INVALID_ARG;
  if (!finite_pos(q_scale) || !finite_pos(k_scale) || !finite_pos(v_scale))
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(kv_pitch) > (1LL << 30) || static_cast<long long>(B) * Hq > (1LL << 24))
    return ATTN_ERR_UNSUPPORTED;
  if (rope && dtype == ATTN_FP8_E5M2 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (il && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  const size_t ws_need = chunk_ws_bytes(B, Hq, Sq, D, dtype, rope);
  if (ws_need > 0 && (!workspace || workspace_bytes < ws_need || !aligned16(workspace)))
    return ATTN_ERR_WORKSPACE;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  const float2* tab = nullptr;
  if (rope) {
    tab = rope_table(D, rope_theta, pos0 + std::max(Skv, 128), &st);
    if (!tab) return st;
  }
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (ws_need > 0) {
    // the chunk's queries rotated once at their absolute positions into the caller's
    // workspace, then attention without RoPE
    void* sq = workspace;
    st = launch_rope(q, sq, dtype, B, Hq, Sq, D, pos0 + Skv - Sq, tab, il, as_stream(stream));
    if (st != ATTN_OK) return st;
    return timed_prefill(sq, k, v, o, lse, dtype, q_scale, k_scale, v_scale, B, Hq, Hkv, Sq,
                          Skv, kv_pitch, D, 1, scale, nullptr, 0, pos0, as_stream(stream));
  }
  // fp8: q rotated into bf16 inside the kernel; the staged keys are widened as stored
  return timed_prefill(q, k, v, o, lse, dtype, q_scale, k_scale, v_scale, B, Hq, Hkv, Sq, Skv,
                        kv_pitch, D, 1, scale, tab, 0, pos0, as_stream(stream));
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int D, int Lmax) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || (!decode_head_dim(D)) || Hq % Hkv) return 0;
  return plan_decode(B, Hq, Hkv, D, Lmax).ws_bytes;
}

attn_status_t attn_decode(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* cache_len, int Lmax, void* o, float* lse,
                          attn_dtype_t dtype, int B, int Hq, int Hkv, int D, float softmax_scale,
                          int rope, float rope_theta, void* workspace, size_t workspace_bytes,
                          attn_stream_t stream) {
  if (!q || !k_cache || !v_cache || !cache_len || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cache_len) & 3u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  int il = 0;
  if (!split_rope_arg(rope, 1, &rope, &il)) return ATTN_ERR_INVALID_ARG;
  if (rope && !finite_pos(rope_theta)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return ATTN_ERR_INVALID_ARG;
  if (!decode_head_dim(D)) return ATTN_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16) return ATTN_ERR_UNSUPPORTED;
  if (dtype == ATTN_FP8_E5M2 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(Lmax) > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  const DecodePlan plan = plan_decode(B, Hq, Hkv, D, Lmax);
  if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes ||
                            !aligned16(workspace)))
    return ATTN_ERR_WORKSPACE;
  const float2* tab = nullptr;
  if (rope) {
    tab = rope_table(D, rope_theta, Lmax + 1, &st);
    if (!tab) return st;
  }
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  if (dtype == ATTN_FP8_E5M2)
    return launch_decode_fp8(q, k_cache, v_cache, cache_len, Lmax, o, lse, B, Hq, Hkv, scale,
                             tab, il, workspace, plan, as_stream(stream));
  return launch_decode(q, k_cache, v_cache, cache_len, Lmax, o, lse, B, Hq, Hkv, D, scale, tab,
                       il, workspace, plan, as_stream(stream));
}

attn_status_t attn_set_prefill_events(void* begin_event, void* end_event) {
  if ((begin_event == nullptr) != (end_event == nullptr)) return ATTN_ERR_INVALID_ARG;
  g_ev_begin.store(static_cast<cudaEvent_t>(begin_event));
  g_ev_end.store(static_cast<cudaEvent_t>(end_event));
  return ATTN_OK;
}

attn_status_t attn_set_prefill_tiles(int q_tiles) {
  if (q_tiles < 0 || q_tiles > 2) return ATTN_ERR_INVALID_ARG;
  force_prefill_tiles(q_tiles);
  return ATTN_OK;
}

attn_status_t attn_set_backward_path(int path) {
  if (path < 0 || path > 2) return ATTN_ERR_INVALID_ARG;
  force_backward_path(path);
  return ATTN_OK;
}

attn_status_t attn_set_decode_splits(int nsplit) {
  if (nsplit < 0 || nsplit > 1024) return ATTN_ERR_INVALID_ARG;
  force_decode_splits(nsplit);
  return ATTN_OK;
}

size_t attn_decode_append_workspace_size(int B, int Hq, int Hkv, int D, int Lmax) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 2 || (!decode_head_dim(D)) || Hq % Hkv) return 0;
  return append_ws_bytes(plan_decode(B, Hq, Hkv, D, Lmax), B, Hq);
}

attn_status_t attn_decode_append(const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, int32_t* cache_len, int Lmax,
                                 void* o, float* lse, attn_dtype_t dtype, int B, int Hq, int Hkv,
                                 int D, float softmax_scale, int rope, float rope_theta,
                                 void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !cache_len || !o || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(o) || !aligned16(workspace))
    return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cache_len) & 3u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 2 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  int il = 0;
  if (!split_rope_arg(rope, 1, &rope, &il)) return ATTN_ERR_INVALID_ARG;
  if (rope && !finite_pos(rope_theta)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return ATTN_ERR_INVALID_ARG;
  if (!decode_head_dim(D)) return ATTN_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(Lmax) > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  const DecodePlan plan = plan_decode(B, Hq, Hkv, D, Lmax);
  if (workspace_bytes < append_ws_bytes(plan, B, Hq)) return ATTN_ERR_WORKSPACE;
  const float2* tab = nullptr;
  if (rope) {
    tab = rope_table(D, rope_theta, Lmax + 1, &st);
    if (!tab) return st;
  }
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  return launch_decode_append(q, k_new, v_new, k_cache, v_cache, cache_len, Lmax, o, lse, B, Hq,
                              Hkv, D, scale, tab, il, workspace, plan, as_stream(stream));
}

size_t attn_decode_latent_workspace_size(int B, int H, int Lmax) {
  if (B < 1 || H < 1 || H > 16 || Lmax < 1) return 0;
  return plan_latent(B, H, Lmax).ws_bytes;
}

attn_status_t attn_decode_latent(const void* q, const void* c_cache, const int32_t* cache_len,
                                 int Lmax, void* o, float* lse, attn_dtype_t dtype, int B, int H,
                                 float softmax_scale, int rope, float rope_theta,
                                 void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  if (!q || !c_cache || !cache_len || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(c_cache) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cache_len) & 3u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Lmax < 1) return ATTN_ERR_INVALID_ARG;
  int il = 0;
  if (!split_rope_arg(rope, 1, &rope, &il)) return ATTN_ERR_INVALID_ARG;
  if (rope && !finite_pos(rope_theta)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return ATTN_ERR_INVALID_ARG;
  if (H > 16) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(Lmax) > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  const DecodePlan plan = plan_latent(B, H, Lmax);
  if (plan.ws_bytes > 0 && (!workspace || workspace_bytes < plan.ws_bytes ||
                            !aligned16(workspace)))
    return ATTN_ERR_WORKSPACE;
  const float2* tab = nullptr;
  if (rope) {
    tab = rope_table(64, rope_theta, Lmax + 1, &st);
    if (!tab) return st;
  }
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(512.0f);
  return launch_latent(q, c_cache, cache_len, Lmax, o, lse, dtype, B, H, scale, tab, il,
                       workspace, plan, as_stream(stream));
}

attn_status_t attn_rope_table_reserve(int D, float theta, int max_pos) {
  if (D < 2 || D > 512 || (D & 1) || !finite_pos(theta) || max_pos < 0 || max_pos >= (1 << 30))
    return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  return rope_table(D, theta, max_pos + 1, &st) ? ATTN_OK : st;
}

attn_status_t attn_get_device_status(attn_stream_t stream, int* status_out) {
  if (!status_out) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int* p = device_status_ptr();
  if (!p) return ATTN_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaMemset(p, 0, sizeof(word)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  *status_out = (word & (1u << ATTN_ERR_TIMEOUT))      ? ATTN_ERR_TIMEOUT
                : (word & (1u << ATTN_ERR_DEVICE_ARG)) ? ATTN_ERR_DEVICE_ARG
                                                       : ATTN_OK;
  return ATTN_OK;
}

}  // extern "C"
