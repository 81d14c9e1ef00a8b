// internal.h — declarations shared by the library's translation units (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

// Device status word (an unsigned int in device global memory, one per device).  Kernels OR
// in (1 << attn_status_t).  Returns nullptr if it could not be resolved.
unsigned int* device_status_ptr();

// Number of SMs of the current device (152 if no device is visible).
int sm_count();

// True when the current device is an sm_100-family part this library was built for.
attn_status_t check_device();

// Cos/sin table for (D, theta) covering positions [0, npos): float2 {cos, sin} laid out
// [pos][D/2].  Builds or grows it on the current device on first use (synchronous cudaMalloc +
// copy).  Returns nullptr on failure and sets *err.
const float2* rope_table(int D, float theta, int npos, attn_status_t* err);

// The cached table for (D, theta) if it already covers [0, npos) on the current device, else
// nullptr.  Never allocates.
const float2* rope_table_find(int D, float theta, int npos);

// Prompt length from which a bf16 RoPE prefill rotates Q and K once per call (rope_apply passes
// into the caller's workspace, then attention without RoPE) instead of inside the attention
// kernel, where every query block re-rotates the K tiles it reads.
constexpr int kRopePassMinS = 1024;
inline size_t prefill_ws_q_bytes(int B, int Hq, int S, int D) {
  return (static_cast<size_t>(B) * Hq * S * D * 2 + 255) & ~size_t(255);
}
// Workspace of attn_prefill (rope: the mode without the flag, il: the interleaved flag): the
// rotated Q (256-byte rounded) then the rotated K, when RoPE runs as rotation passes.
inline size_t prefill_ws_bytes(int B, int Hq, int Hkv, int S, int D, attn_dtype_t dt, int rope,
                               int il) {
  if (rope != 1 || dt != ATTN_BF16 || !(S >= kRopePassMinS || il || D == 256)) return 0;
  return prefill_ws_q_bytes(B, Hq, S, D) + static_cast<size_t>(B) * Hkv * S * D * 2;
}
// Workspace of attn_prefill_chunk: the chunk's rotated queries (bf16 with RoPE).
inline size_t chunk_ws_bytes(int B, int Hq, int Sq, int D, attn_dtype_t dt, int rope) {
  return (rope && dt == ATTN_BF16) ? prefill_ws_q_bytes(B, Hq, Sq, D) : 0;
}

// Encode a 3-D tiled TMA descriptor for a dense row-major tensor of `elem_bytes`-byte elements
// with logical sizes {inner, mid, outer} (innermost first), box {box_inner, box_mid, 1} and
// `swizzle_bytes` swizzling.  Returns false on failure.
// mid_pitch: rows between consecutive outer indices (0: mid, a dense tensor).
bool make_tmap_3d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner,
                  uint64_t mid, uint64_t outer, uint32_t box_inner, uint32_t box_mid,
                  int swizzle_bytes, uint64_t mid_pitch = 0);

// Encode a 4-D tiled TMA descriptor over sizes dims[0..3] (innermost first, dims[0] contiguous)
// with byte strides strides[0..2] for dims 1..3 (any order of magnitude: a view may step through
// a row in chunks), box box[0..3] and 128-byte swizzling.  Returns false on failure.
bool make_tmap_4d(CUtensorMap* map, const void* base, int elem_bytes, const uint64_t dims[4],
                  const uint64_t strides[3], const uint32_t box[4]);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize), done once per (kernel, device, size).
bool set_smem_attr(const void* kernel, int bytes);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch-status helper: map the last launch error to a status.
// The `rope` argument of the attention calls: the mode (0 .. max_mode) in the low bits, optionally
// OR'd with ATTN_ROPE_FLAG_INTERLEAVED.  False for anything else (and for the flag without a mode).
inline bool split_rope_arg(int rope, int max_mode, int* mode, int* interleaved) {
  const int m = rope & ~ATTN_ROPE_FLAG_INTERLEAVED;
  const int il = (rope & ATTN_ROPE_FLAG_INTERLEAVED) ? 1 : 0;
  if (m < 0 || m > max_mode || (il && m == 0)) return false;
  *mode = m;
  *interleaved = il;
  return true;
}

inline attn_status_t launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ------------------------------------------------------------------------------------------
// entry points implemented per translation unit (called from api.cpp after validation)
// ------------------------------------------------------------------------------------------
// interleaved: pairs (2i, 2i+1) instead of (i, i + D/2), same table; inverse: rotate by the
// opposite angles (the transpose).
attn_status_t launch_rope(const void* x, void* y, attn_dtype_t dt, int B, int H, int S, int D,
                          int pos0, const float2* table, int interleaved, cudaStream_t st,
                          int inverse = 0);

struct DecodePlan {
  int nsplit;      // splits of the key range per (b, kv head)
  int chunk;       // keys per split (multiple of the key tile)
  int grid;        // persistent CTAs
  size_t ws_bytes; // partial O (fp32) + partial LSE (fp32)
};
DecodePlan plan_decode(int B, int Hq, int Hkv, int D, int Lmax);
// nsplit > 0: every later GQA decode plan uses that split count; 0: the per-shape planner.
void force_decode_splits(int nsplit);

// Append decode workspace: the decode's own (rounded up to 256 bytes), then B*Hq floats.
inline size_t append_ws_offset(const DecodePlan& pl) { return (pl.ws_bytes + 255) & ~size_t(255); }
inline size_t append_ws_bytes(const DecodePlan& pl, int B, int Hq) {
  return append_ws_offset(pl) + static_cast<size_t>(B) * Hq * sizeof(float);
}
attn_status_t launch_decode_append(const void* q, const void* k_new, const void* v_new,
                                   void* k_cache, void* v_cache, int32_t* lens, int Lmax,
                                   void* o, float* lse, int B, int Hq, int Hkv, int D,
                                   float scale, const float2* table, int rope_il, void* ws,
                                   const DecodePlan& plan, cudaStream_t st);
DecodePlan plan_latent(int B, int H, int Lmax);

attn_status_t launch_decode(const void* q, const void* k, const void* v, const int32_t* lens,
                            int Lmax, void* o, float* lse, int B, int Hq, int Hkv, int D,
                            float scale, const float2* table, int rope_il, void* ws,
                            const DecodePlan& plan, cudaStream_t st);

attn_status_t launch_decode_fp8(const void* q, const void* k, const void* v,
                                const int32_t* lens, int Lmax, void* o, float* lse, int B, int Hq,
                                int Hkv, float scale, const float2* table, int rope_il, void* ws,
                                const DecodePlan& plan, cudaStream_t st);

attn_status_t launch_latent(const void* q, const void* c, const int32_t* lens, int Lmax, void* o,
                            float* lse, attn_dtype_t dt, int B, int H, float scale,
                            const float2* table, int rope_il, void* ws, const DecodePlan& plan,
                            cudaStream_t st);

// Attention backward (bf16): workspace = Delta [B*Hq*S] fp32 (256-byte rounded) + the fp32 dQ
// accumulator [B*Hq*S*D].
size_t bwd_workspace_bytes(int B, int Hq, int S, int D);
attn_status_t launch_prefill_backward(const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, int B, int Hq, int Hkv, int S, int D, int causal,
                                      float scale, void* ws, cudaStream_t st);

// The tcgen05 form of the backward (a dK/dV kernel over key tiles and a dQ kernel over query
// tiles, no atomics); uses the first Delta part of the backward workspace only.
attn_status_t launch_prefill_backward_tc(const void* q, const void* k, const void* v,
                                         const void* o, const float* lse, const void* dout,
                                         void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                         int S, int D, int causal, float scale, void* ws,
                                         cudaStream_t st);

// 0: the default backward (tcgen05), 1: the warp-level mma.sync kernels, 2: tcgen05.
void force_backward_path(int path);

// q_tiles 1 or 2: every later prefill at D <= 128 runs that many 128-row Q tiles per work item;
// 0: the default (two).
void force_prefill_tiles(int q_tiles);

// S query rows at positions Skv - S .. Skv - 1 against Skv keys (rows kv_pitch apart per head);
// rope_k: the fused RoPE rotates the keys too (else only the queries).
attn_status_t launch_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                             attn_dtype_t dt, float q_scale, float k_scale, float v_scale, int B,
                             int Hq, int Hkv, int S, int Skv, int kv_pitch, int D, int causal,
                             float scale, const float2* table, int rope_k, int pos0,
                             cudaStream_t st);

}  // namespace attn
