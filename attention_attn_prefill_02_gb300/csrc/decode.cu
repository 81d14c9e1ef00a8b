// decode.cu — single-token decode against a static cache: grouped-query split-KV decode, the
// absorbed-latent (MLA-style) decode, and the log-sum-exp combine of split partials.
//
// Both decode kernels are HBM-bound (4 and 30 useful flop per cache byte), so the design goal is
// to keep enough cache bytes in flight: a persistent grid, one TMA producer warp per CTA
// streaming 64-key tiles of the cache through a multi-stage mbarrier ring (128-byte swizzled, so
// ldmatrix reads are bank-conflict free), and four compute warps that consume each tile with
// warp-level bf16 MMAs.  The GQA group's query heads (G = Hq/Hkv <= 16) share one 16-row MMA
// tile, so every K/V byte is read from HBM once for the whole group (Fixed-budget decode audit —
// 2026-09-11, "What theory can and cannot establish": once-per-KV-head reuse; the padded row
// tile is the same observation).  Work items are (sequence, KV head, split of the key range);
// splits are merged by their log-sum-exp ("A: group-entry queries and one joint history scan").
#include <algorithm>
#include <atomic>
#include <cmath>
#include <type_traits>

#include "common.cuh"

namespace attn {
namespace {

constexpr int kTileKeys = 64;
constexpr int kComputeWarps = 4;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ void compute_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kComputeWarps * 32) : "memory");
}

struct GqaParams {
  const __nv_bfloat16* q;
  const int32_t* lens;
  __nv_bfloat16* o;
  float* lse;
  float* ws_o;    // [B*Hq, nsplit, D] fp32 partial outputs (normalised)
  float* ws_lse;  // [B*Hq, nsplit] fp32 partial log2-sum-exp (scaled-log2 domain)
  const float2* table;
  int rope_il;    // RoPE pairs (2i, 2i+1) instead of (i, i + D/2)
  unsigned int* status;
  int B, Hq, Hkv, G, Lmax, nsplit, chunk;
  float scale_log2;  // softmax_scale * log2(e)
};

// The query tile of one (sequence, KV head) item: rows r < G of `q_rows` (the group's first
// query row; bf16, D dims each) into `qs` (row pitch `pitch` bytes) as T_OUT, rows G .. rows-1
// zero; then, with a table, each pair (i, i + D/2) (or (2i, 2i+1) when `il`) rotated at
// position len in float32 and rounded once.  The 16-byte loads all go out before any store.  Ends before the final barrier:
// the caller synchronises before reading the tile.
template <int D, typename T_OUT>
__device__ __forceinline__ void fill_query_tile(uint8_t* qs, int pitch, int rows,
                                                const __nv_bfloat16* __restrict__ q_rows, int G,
                                                bool valid, const float2* __restrict__ table,
                                                int len, int tid, bool il) {
  constexpr int kChunks = D / 8;  // 8-dim chunks per row
  constexpr int kMaxPer = 16 * kChunks / (kComputeWarps * 32);
  uint4 v[kMaxPer];
#pragma unroll
  for (int k = 0; k < kMaxPer; ++k) {
    const int idx = tid + k * kComputeWarps * 32, r = idx / kChunks, c = idx % kChunks;
    v[k] = (r < G && valid)
               ? __ldg(reinterpret_cast<const uint4*>(q_rows + static_cast<size_t>(r) * D + c * 8))
               : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int k = 0; k < kMaxPer; ++k) {
    const int idx = tid + k * kComputeWarps * 32, r = idx / kChunks, c = idx % kChunks;
    if (r >= rows) continue;
    uint4 w = v[k];
    if constexpr (sizeof(T_OUT) == 2 && !std::is_same<T_OUT, __nv_bfloat16>::value) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[k]);
      __half2* o = reinterpret_cast<__half2*>(&w);
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = __float22half2_rn(__bfloat1622float2(h[j]));
    }
    *reinterpret_cast<uint4*>(qs + r * pitch + c * 16) = w;
  }
  if (!table || !valid) return;
  compute_bar_sync();
  for (int idx = tid; idx < G * (D / 2); idx += kComputeWarps * 32) {
    const int r = idx / (D / 2), i = idx % (D / 2);
    const int ia = il ? 2 * i : i, ib = il ? 2 * i + 1 : i + D / 2;
    T_OUT* row = reinterpret_cast<T_OUT*>(qs + r * pitch);
    const float x1 = static_cast<float>(row[ia]), x2 = static_cast<float>(row[ib]);
    const float2 cs = table[static_cast<size_t>(len) * (D / 2) + i];
    row[ia] = static_cast<T_OUT>(x1 * cs.x - x2 * cs.y);
    row[ib] = static_cast<T_OUT>(x2 * cs.x + x1 * cs.y);
  }
}

template <int D, int NST>
struct GqaSmem {
  static constexpr int kTileBytes = kTileKeys * D * 2;  // one K (or V) tile
  static constexpr int kQPitch = D * 2 + 16;            // padded row pitch of the query tile
  static constexpr int kStageOff = 0;
  static constexpr int kQOff = NST * 2 * kTileBytes;
  static constexpr int kRedOff = kQOff + 16 * kQPitch;      // m, l per warp per row
  static constexpr int kOOff = kRedOff + 2 * kComputeWarps * 16 * 4;
  static int bytes(int G) { return kOOff + kComputeWarps * G * D * 4 + 2 * NST * 8 + 1024; }
};

// CTAs per SM of the bf16 decode: two up to D = 128; one at D = 256, whose 64 KB stages, 64 KB
// cross-warp reduction and ~230 registers per thread (query fragments and 32 accumulator tiles)
// leave room for a single CTA.
__host__ __device__ constexpr int gqa_ctas_per_sm(int D) { return D >= 256 ? 1 : 2; }
__host__ __device__ constexpr int gqa_stages(int D) { return D >= 256 ? 2 : 3; }

// Grouped-query split-KV decode.  Grid: persistent; items (b, kv head, split) in row-major
// order, CTA c takes items c, c + grid, ...
template <int D, int NST>
__global__ void __launch_bounds__(kThreads, gqa_ctas_per_sm(D))
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const GqaParams p) {
  using L = GqaSmem<D, NST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int G = p.G;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOOff + kComputeWarps * G * D * 4);
  uint64_t* empty = full + NST;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_items = p.B * p.Hkv * p.nsplit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kComputeWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // ---------------- producer warp: stream K/V tiles of every item of this CTA ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int stage = 0;
      uint32_t phase = 0;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int sp = it % p.nsplit;
        const int bh = it / p.nsplit;  // b * Hkv + kv head
        const int b = bh / p.Hkv;
        int len = p.lens[b];
        if (len < 1 || len > p.Lmax) len = 0;
        const int k0 = sp * p.chunk;
        const int k1 = min(k0 + p.chunk, len);
        for (int t0 = k0; t0 < k1; t0 += kTileKeys) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status)) return;
          mbar_arrive_expect_tx(&full[stage], 2 * L::kTileBytes);
          uint8_t* kt = smem + L::kStageOff + stage * 2 * L::kTileBytes;
          uint8_t* vt = kt + L::kTileBytes;
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx) {
            tma_load_3d(kt + bx * kTileKeys * 128, &tmK, &full[stage], bx * 64, t0, bh);
            tma_load_3d(vt + bx * kTileKeys * 128, &tmV, &full[stage], bx * 64, t0, bh);
          }
          if (++stage == NST) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    return;
  }

  // ---------------- compute warps ----------------
  const int tid = threadIdx.x;  // 0..127
  const int g = lane >> 2, tq = lane & 3;
  uint8_t* qs = smem + L::kQOff;
  float* red_m = reinterpret_cast<float*>(smem + L::kRedOff);
  float* red_l = red_m + kComputeWarps * 16;
  float* red_o = reinterpret_cast<float*>(smem + L::kOOff);
  const uint32_t qs_addr = smem_u32(qs);
  int stage = 0;
  uint32_t phase = 0;
  bool alive = true;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int sp = it % p.nsplit;
    const int bh = it / p.nsplit;
    const int b = bh / p.Hkv, kvh = bh % p.Hkv;
    int len = p.lens[b];
    const bool valid = len >= 1 && len <= p.Lmax;
    if (!valid) {
      if (tid == 0 && sp == 0) report_status(p.status, ATTN_ERR_DEVICE_ARG);
      len = 0;
    }
    const int k0 = sp * p.chunk;
    const int k1 = min(k0 + p.chunk, len);

    // query tile: G rows (rotated at position len), zero-padded to 16 rows
    compute_bar_sync();
    fill_query_tile<D, __nv_bfloat16>(qs, L::kQPitch, 16,
                                      p.q + (static_cast<size_t>(b) * p.Hq + kvh * G) * D, G,
                                      valid, p.table, len, tid, p.rope_il != 0);
    compute_bar_sync();
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ldsm_x4(qs_addr + (lane & 15) * L::kQPitch + (kk * 16 + (lane >> 4) * 8) * 2, qa[kk][0],
              qa[kk][1], qa[kk][2], qa[kk][3]);

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

    for (int t0 = k0; t0 < k1 && alive; t0 += kTileKeys) {
      if (!mbar_wait(&full[stage], phase, p.status)) {
        alive = false;
        break;
      }
      const uint8_t* kt = smem + L::kStageOff + stage * 2 * L::kTileBytes;
      const uint32_t kt_addr = smem_u32(kt);
      const uint32_t vt_addr = kt_addr + L::kTileBytes;
      // S (16 query rows x this warp's 16 keys)
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int m = lane >> 3;
        const int key = warp * 16 + (m >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = kk * 2 + (m & 1);  // 16-byte chunk index along d
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kt_addr + (c >> 3) * kTileKeys * 128 + sw128_offset(key, c & 7), b0, b1, b2,
                  b3);
          mma_bf16_16816(s[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          mma_bf16_16816(s[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
      }
      // scale, mask keys >= k1, online softmax (rows g and g + 8)
      float rm0 = -INFINITY, rm1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int key = t0 + warp * 16 + nt * 8 + tq * 2 + (j & 1);
          const float v = key < k1 ? s[nt][j] * p.scale_log2 : -INFINITY;
          s[nt][j] = v;
          if (j < 2)
            rm0 = fmaxf(rm0, v);
          else
            rm1 = fmaxf(rm1, v);
        }
      rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, 1));
      rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, 2));
      rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, 1));
      rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, 2));
      const float mn0 = fmaxf(m0, rm0), mn1 = fmaxf(m1, rm1);
      const float base0 = mn0 == -INFINITY ? 0.f : mn0;
      const float base1 = mn1 == -INFINITY ? 0.f : mn1;
      const float c0 = fast_exp2(m0 - base0), c1 = fast_exp2(m1 - base1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        s[nt][0] = fast_exp2(s[nt][0] - base0);
        s[nt][1] = fast_exp2(s[nt][1] - base0);
        s[nt][2] = fast_exp2(s[nt][2] - base1);
        s[nt][3] = fast_exp2(s[nt][3] - base1);
        ps0 += s[nt][0] + s[nt][1];
        ps1 += s[nt][2] + s[nt][3];
      }
      l0 = l0 * c0 + ps0;
      l1 = l1 * c1 + ps1;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        acc[n][0] *= c0;
        acc[n][1] *= c0;
        acc[n][2] *= c1;
        acc[n][3] *= c1;
      }
      const uint32_t pa0 = pack_bf16(s[0][0], s[0][1]);
      const uint32_t pa1 = pack_bf16(s[0][2], s[0][3]);
      const uint32_t pa2 = pack_bf16(s[1][0], s[1][1]);
      const uint32_t pa3 = pack_bf16(s[1][2], s[1][3]);
      // O += P V over this warp's 16 keys
      {
        const int m = lane >> 3;
        const int key = warp * 16 + (m & 1) * 8 + (lane & 7);
#pragma unroll
        for (int n2 = 0; n2 < D / 16; ++n2) {
          const int c = n2 * 2 + (m >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vt_addr + (c >> 3) * kTileKeys * 128 + sw128_offset(key, c & 7), b0, b1, b2,
                    b3);
          mma_bf16_16816(acc[2 * n2], pa0, pa1, pa2, pa3, b0, b1);
          mma_bf16_16816(acc[2 * n2 + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == NST) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (!alive) return;

    // merge the four warps' partial states (each covered a quarter of every tile's keys)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (tq == 0) {
      red_m[warp * 16 + g] = m0;
      red_m[warp * 16 + g + 8] = m1;
      red_l[warp * 16 + g] = l0;
      red_l[warp * 16 + g + 8] = l1;
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int d = n * 8 + tq * 2;
      if (g < G) {
        red_o[(warp * G + g) * D + d] = acc[n][0];
        red_o[(warp * G + g) * D + d + 1] = acc[n][1];
      }
      if (g + 8 < G) {
        red_o[(warp * G + g + 8) * D + d] = acc[n][2];
        red_o[(warp * G + g + 8) * D + d + 1] = acc[n][3];
      }
    }
    compute_bar_sync();
    for (int idx = tid; idx < G * D; idx += kComputeWarps * 32) {
      const int r = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, red_m[w * 16 + r]);
      float lsum = 0.f, osum = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) {
          const float mw = red_m[w * 16 + r];
          const float wgt = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
          lsum += wgt * red_l[w * 16 + r];
          osum += wgt * red_o[(w * G + r) * D + d];
        }
      }
      const float o = lsum > 0.f ? osum / lsum : 0.f;
      const float lse2 = lsum > 0.f ? M + log2f(lsum) : -INFINITY;
      const size_t row = static_cast<size_t>(b) * p.Hq + kvh * G + r;
      if (p.nsplit == 1) {
        p.o[row * D + d] = __float2bfloat16_rn(o);
        if (p.lse && d == 0) p.lse[row] = lse2 * kLn2;
      } else {
        p.ws_o[(row * p.nsplit + sp) * D + d] = o;
        if (d == 0) p.ws_lse[row * p.nsplit + sp] = lse2;
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// GQA decode with an fp8 (e5m2) cache: the same streaming structure at half the bytes.  Every
// e5m2 value is exactly an f16 value (its bits are the top byte of the f16), so the MMAs run in
// f16 on values widened in registers by byte permutes.
//
// The MMAs are transposed with respect to the bf16 kernel: S^T = K Q^T and O^T = V^T P^T.  Keys
// (and, for PV, head dimensions) take the 16-row side of m16n8k16 and the group's query heads the
// 8-column side, so a group of up to 8 heads wastes no MMA rows on padding (NT = 2 column tiles
// for groups of 9..16).  K fragments are 4-byte reads of the swizzled tile (4 consecutive dims;
// the query fragments use the same dimension order, which leaves every dot product unchanged).
// V^T fragments come from ldmatrix.trans on the fp8 tile read as 16-bit pairs: one register holds
// dims (2c, 2c+1) of keys (2t, 2t+1), and the two byte permutes split it into the rows of dims 2c
// and 2c+1, so MMA row r of a 16-dim chunk is dim 2r (r < 8) or dim 2(r-8)+1.  The probabilities
// go from the S^T accumulator layout to the P^T operand layout with movmatrix.trans.  The query
// stays bf16 in memory and is converted to f16 (values beyond f16 range are not supported).
// ------------------------------------------------------------------------------------------------

constexpr int kF8D = 128;
constexpr int kF8TileBytes = kTileKeys * kF8D;  // 8 KB: 64 keys x 128 fp8
// 5 stages for groups of up to 8 heads, 4 for larger groups (two CTAs per SM either way)
constexpr int f8_stages(int nt) { return nt == 1 ? 5 : 4; }

template <int NST>
struct GqaF8Smem {
  static constexpr int kQOff = NST * 2 * kF8TileBytes;
  static constexpr int kQPitch = kF8D * 2 + 16;
  static constexpr int kRedOff = kQOff + 16 * kQPitch;
  static constexpr int kOOff = kRedOff + 2 * kComputeWarps * 16 * 4;
  static int bytes(int G) { return kOOff + kComputeWarps * G * kF8D * 4 + 2 * NST * 8 + 1024; }
};

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 8x8 16-bit matrix held one row pair per lane -> its transpose in the same layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// e5m2 bytes -> f16x2 holding them exactly: bytes 0,1 / 2,3 (consecutive dims of one key), or
// bytes 0,2 / 1,3 (one dim of two keys, as ldmatrix.trans delivers V).
__device__ __forceinline__ uint32_t e5m2x2_lo(uint32_t w) { return __byte_perm(w, 0u, 0x1404); }
__device__ __forceinline__ uint32_t e5m2x2_hi(uint32_t w) { return __byte_perm(w, 0u, 0x3424); }
__device__ __forceinline__ uint32_t e5m2x2_even(uint32_t w) { return __byte_perm(w, 0u, 0x2404); }
__device__ __forceinline__ uint32_t e5m2x2_odd(uint32_t w) { return __byte_perm(w, 0u, 0x3414); }

template <int NST, int NT>
__global__ void __launch_bounds__(kThreads, 2)
    gqa_decode_fp8_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const GqaParams p) {
  constexpr int D = kF8D;
  constexpr int NC = D / 16;  // 16-dim chunks
  using L = GqaF8Smem<NST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int G = p.G;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOOff + kComputeWarps * G * D * 4);
  uint64_t* empty = full + NST;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_items = p.B * p.Hkv * p.nsplit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kComputeWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int stage = 0;
      uint32_t phase = 0;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int sp = it % p.nsplit;
        const int bh = it / p.nsplit;
        const int b = bh / p.Hkv;
        int len = p.lens[b];
        if (len < 1 || len > p.Lmax) len = 0;
        const int k0 = sp * p.chunk;
        const int k1 = min(k0 + p.chunk, len);
        for (int t0 = k0; t0 < k1; t0 += kTileKeys) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.status)) return;
          mbar_arrive_expect_tx(&full[stage], 2 * kF8TileBytes);
          uint8_t* kt = smem + stage * 2 * kF8TileBytes;
          tma_load_3d(kt, &tmK, &full[stage], 0, t0, bh);
          tma_load_3d(kt + kF8TileBytes, &tmV, &full[stage], 0, t0, bh);
          if (++stage == NST) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    return;
  }

  const int tid = threadIdx.x;
  const int g = lane >> 2, tq = lane & 3;
  uint8_t* qs = smem + L::kQOff;
  float* red_m = reinterpret_cast<float*>(smem + L::kRedOff);
  float* red_l = red_m + kComputeWarps * 16;
  float* red_o = reinterpret_cast<float*>(smem + L::kOOff);
  // this warp's 16 keys: S^T rows g and g + 8
  const int key_a = warp * 16 + g;
  // ldmatrix.trans row of this lane: matrices (keys 0-7 | 8-15) x (chunk 2c | 2c + 1)
  const int v_key = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
  const int v_chunk = lane >> 4;
  int stage = 0;
  uint32_t phase = 0;
  bool alive = true;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int sp = it % p.nsplit;
    const int bh = it / p.nsplit;
    const int b = bh / p.Hkv, kvh = bh % p.Hkv;
    int len = p.lens[b];
    const bool valid = len >= 1 && len <= p.Lmax;
    if (!valid) {
      if (tid == 0 && sp == 0) report_status(p.status, ATTN_ERR_DEVICE_ARG);
      len = 0;
    }
    const int k0 = sp * p.chunk;
    const int k1 = min(k0 + p.chunk, len);

    // query rows as f16 (rotated at position len), zero-padded to 8 NT rows
    compute_bar_sync();
    fill_query_tile<D, __half>(qs, L::kQPitch, 8 * NT,
                               p.q + (static_cast<size_t>(b) * p.Hq + kvh * G) * D, G, valid,
                               p.table, len, tid, p.rope_il != 0);
    compute_bar_sync();
    // Q^T operand: column g is query 8 nt + g; logical k = 2t+e -> dim 16kk+4t+e and
    // k = 8+2t+e -> dim 16kk+4t+2+e, the order the K reads deliver
    uint32_t qb[NT][NC][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int kk = 0; kk < NC; ++kk) {
        const uint8_t* src = qs + (nt * 8 + g) * L::kQPitch + (16 * kk + 4 * tq) * 2;
        qb[nt][kk][0] = *reinterpret_cast<const uint32_t*>(src);
        qb[nt][kk][1] = *reinterpret_cast<const uint32_t*>(src + 4);
      }

    // softmax state of queries 8 nt + 2 tq + e; l is this lane's partial sum over its keys
    float m[NT][2], l[NT][2];
    float acc[NT][NC][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[nt][c][0] = acc[nt][c][1] = acc[nt][c][2] = acc[nt][c][3] = 0.f;
    }

    for (int t0 = k0; t0 < k1 && alive; t0 += kTileKeys) {
      if (!mbar_wait(&full[stage], phase, p.status)) {
        alive = false;
        break;
      }
      const uint8_t* kt = smem + stage * 2 * kF8TileBytes;
      const uint32_t vt_addr = smem_u32(kt + kF8TileBytes);
      uint32_t kw[NC][2];
#pragma unroll
      for (int kk = 0; kk < NC; ++kk) {
        kw[kk][0] = *reinterpret_cast<const uint32_t*>(kt + sw128_offset(key_a, kk) + 4 * tq);
        kw[kk][1] = *reinterpret_cast<const uint32_t*>(kt + sw128_offset(key_a + 8, kk) + 4 * tq);
      }
      uint32_t vw[NC / 2][4];
#pragma unroll
      for (int c2 = 0; c2 < NC / 2; ++c2)
        ldsm_x4_t(vt_addr + sw128_offset(v_key, 2 * c2 + v_chunk), vw[c2][0], vw[c2][1],
                  vw[c2][2], vw[c2][3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);  // the stage is no longer read
      if (++stage == NST) {
        stage = 0;
        phase ^= 1;
      }

      // S^T: two accumulation chains (even / odd dim chunks) per column tile
      float s[NT][2][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) s[nt][h][0] = s[nt][h][1] = s[nt][h][2] = s[nt][h][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < NC; ++kk) {
        const uint32_t a0 = e5m2x2_lo(kw[kk][0]), a1 = e5m2x2_lo(kw[kk][1]);
        const uint32_t a2 = e5m2x2_hi(kw[kk][0]), a3 = e5m2x2_hi(kw[kk][1]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_f16_16816(s[nt][kk & 1], a0, a1, a2, a3, qb[nt][kk][0], qb[nt][kk][1]);
      }

      const bool in0 = t0 + key_a < k1, in1 = t0 + key_a + 8 < k1;
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // rows: key_a (j = 0, 1) and key_a + 8 (j = 2, 3); columns: queries 2 tq + (j & 1)
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool in = j < 2 ? in0 : in1;
          v[j] = in ? (s[nt][0][j] + s[nt][1][j]) * p.scale_log2 : -INFINITY;
        }
        float rm0 = fmaxf(v[0], v[2]), rm1 = fmaxf(v[1], v[3]);
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
          rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, o2));
          rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, o2));
        }
        const float mn0 = fmaxf(m[nt][0], rm0), mn1 = fmaxf(m[nt][1], rm1);
        const float base0 = mn0 == -INFINITY ? 0.f : mn0;
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        const float c0 = fast_exp2(m[nt][0] - base0), c1 = fast_exp2(m[nt][1] - base1);
        m[nt][0] = mn0;
        m[nt][1] = mn1;
        v[0] = fast_exp2(v[0] - base0);
        v[2] = fast_exp2(v[2] - base0);
        v[1] = fast_exp2(v[1] - base1);
        v[3] = fast_exp2(v[3] - base1);
        l[nt][0] = l[nt][0] * c0 + v[0] + v[2];
        l[nt][1] = l[nt][1] * c1 + v[1] + v[3];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          acc[nt][c][0] *= c0;
          acc[nt][c][2] *= c0;
          acc[nt][c][1] *= c1;
          acc[nt][c][3] *= c1;
        }
        pb[nt][0] = movmatrix_t(pack_f16(v[0], v[1]));  // keys 2 tq, 2 tq + 1 of query g
        pb[nt][1] = movmatrix_t(pack_f16(v[2], v[3]));  // keys 8 + 2 tq, 9 + 2 tq
      }

      // O^T += V^T P^T
#pragma unroll
      for (int c2 = 0; c2 < NC / 2; ++c2) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t lo = vw[c2][2 * h], hi = vw[c2][2 * h + 1];  // keys 0-7, 8-15
          const uint32_t a0 = e5m2x2_even(lo), a1 = e5m2x2_odd(lo);
          const uint32_t a2 = e5m2x2_even(hi), a3 = e5m2x2_odd(hi);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_f16_16816(acc[nt][2 * c2 + h], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
        }
      }
    }
    if (!alive) return;

#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], o2);
      if (g == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          red_m[warp * 16 + nt * 8 + 2 * tq + e] = m[nt][e];
          red_l[warp * 16 + nt * 8 + 2 * tq + e] = l[nt][e];
        }
      }
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int qr = nt * 8 + 2 * tq + (j & 1);
          const int d = 16 * c + 2 * g + (j >> 1);
          if (qr < G) red_o[(warp * G + qr) * D + d] = acc[nt][c][j];
        }
    }
    compute_bar_sync();
    for (int idx = tid; idx < G * D; idx += kComputeWarps * 32) {
      const int r = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, red_m[w * 16 + r]);
      float lsum = 0.f, osum = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) {
          const float mw = red_m[w * 16 + r];
          const float wgt = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
          lsum += wgt * red_l[w * 16 + r];
          osum += wgt * red_o[(w * G + r) * D + d];
        }
      }
      const float o = lsum > 0.f ? osum / lsum : 0.f;
      const float lse2 = lsum > 0.f ? M + log2f(lsum) : -INFINITY;
      const size_t row = static_cast<size_t>(b) * p.Hq + kvh * G + r;
      if (p.nsplit == 1) {
        p.o[row * D + d] = __float2bfloat16_rn(o);
        if (p.lse && d == 0) p.lse[row] = lse2 * kLn2;
      } else {
        p.ws_o[(row * p.nsplit + sp) * D + d] = o;
        if (d == 0) p.ws_lse[row * p.nsplit + sp] = lse2;
      }
    }
  }
}

// Merge the split partials of one (sequence, query head) row per block: weights first (one
// warp), then every output column reads its partials eight at a time.
constexpr int kMaxSplits = 1024;

__global__ void __launch_bounds__(128)
    combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse, int nsplit,
                   int D, __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  __shared__ float wgt[kMaxSplits];
  __shared__ float inv_s, lse_s;
  const size_t row = blockIdx.x;
  const float* lp = ws_lse + row * nsplit;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float M = -INFINITY;
    for (int s2 = lane; s2 < nsplit; s2 += 32) {
      const float l = lp[s2];
      wgt[s2] = l;
      M = fmaxf(M, l);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    float wsum = 0.f;
    for (int s2 = lane; s2 < nsplit; s2 += 32) {
      const float l = wgt[s2];
      const float w = l == -INFINITY ? 0.f : exp2f(l - M);
      wgt[s2] = w;
      wsum += w;
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o2);
    if (lane == 0) {
      inv_s = wsum > 0.f ? 1.f / wsum : 0.f;
      lse_s = wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
    }
  }
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int i = 0;
    for (; i + 8 <= nsplit; i += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = ws_o[(row * nsplit + i + u) * D + d];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] += wgt[i + u] * v[u];
    }
    for (; i < nsplit; ++i) acc[0] += wgt[i] * ws_o[(row * nsplit + i) * D + d];
    const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    o[row * D + d] = __float2bfloat16_rn(sum * inv_s);
  }
  if (lse && threadIdx.x == 0) lse[row] = lse_s;
}

// ------------------------------------------------------------------------------------------------
// Absorbed latent decode: all H (<= 16) heads of a sequence share each 512-dim cache row.
// ------------------------------------------------------------------------------------------------

constexpr int kLatQK = 512;
constexpr int kLatV = 448;
constexpr int kLatRope = 64;
constexpr int kLatStages = 3;
constexpr int kLatWarps = 8;                              // compute warps (no separate producer:
constexpr int kLatThreads = kLatWarps * 32;               // warp 0, lane 0 issues the TMA loads)
constexpr int kLatTileBytes = kTileKeys * kLatQK * 2;     // 64 KB: 64 keys x 512 dims
constexpr int kLatQPitch = kLatQK * 2 + 16;
constexpr int kLatColsPerWarp = kLatV / kLatWarps;        // 56 = 7 n-tiles of the 448 outputs

__device__ __forceinline__ void lat_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kLatWarps * 32) : "memory");
}

__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

constexpr int kLatMaxB = 2048;  // sequences per call (the tile prefix sums live in smem)
#ifndef ATTN_LAT_MAX_CTAS
#define ATTN_LAT_MAX_CTAS 128
#endif
constexpr int kLatMaxCtas = ATTN_LAT_MAX_CTAS;

// Cache tile geometry: bf16 tiles of 64 keys x 512 dims or e5m2 tiles of 128 keys x 512 bytes,
// 64 KB either way, three stages (192 KB).  The per-tile work that does not grow with the keys
// (two block barriers, the maximum exchange, the refill) is spread over twice the keys in the
// e5m2 tiles.  A tile lands as its 128-byte column chunks, each kKeys rows x 128 bytes with the
// 128-byte swizzle, in ONE TMA copy: the tensor map views the cache as {128 bytes of a row, key,
// chunk, sequence}, so the box {128 B, kKeys keys, all chunks, 1} is laid out chunk-major.
// Issued as one box per chunk, the copies held the issuing thread (and with it its warp, and the
// next block barrier) ~700 cycles per tile.
template <bool F8>
struct LatGeo {
  static constexpr int kKeys = F8 ? 2 * kTileKeys : kTileKeys;  // keys per tile
  static constexpr int kTileBytes = kKeys * kLatQK * (F8 ? 1 : 2);
  static constexpr int kStages = kLatStages;
  static constexpr int kKeysPerWarp = kKeys / kLatWarps;  // keys scored per warp per tile
  static constexpr int kNS = kKeysPerWarp / 8;            // n8 score tiles per warp
  static constexpr int kPPitch = kKeys * 2 + 16;          // P row pitch in shared memory
  static_assert(kTileBytes == kLatTileBytes, "64 KB tiles");
};
constexpr int kLatMaxStages = 6;

struct LatSmem {
  static constexpr int kQOff = kLatStages * kLatTileBytes;  // 192 KB of stages for both dtypes
  // P [2][16][pitch] reuses the query tile's bytes: the query sits in registers while the tiles
  // of a segment run (loaded after, and overwritten before, block barriers that P's use is
  // between)
  static constexpr int kPOff = kQOff;
  static constexpr int kRedOff = kQOff + 16 * kLatQPitch;            // [2][warps][16] row max
  static constexpr int kLOff = kRedOff + 2 * kLatWarps * 16 * 4;      // [warps][16] row sums
  static constexpr int kScanOff = kLOff + kLatWarps * 16 * 4;         // [warps] scan scratch
  static constexpr int kPrefOff = kScanOff + 64;                      // [B + 1] tile prefix
  static constexpr int kBarOff = kPrefOff + (kLatMaxB + 1) * 4 + 60;
  static constexpr int kBytes = kBarOff + 2 * kLatMaxStages * 8 + 1024;
};
static_assert(LatGeo<true>::kStages * LatGeo<true>::kTileBytes == LatSmem::kQOff, "ring size");
static_assert(2 * 16 * LatGeo<true>::kPPitch <= 16 * kLatQPitch &&
                  2 * 16 * LatGeo<false>::kPPitch <= 16 * kLatQPitch,
              "P fits in the query tile's bytes");

struct LatParams {
  const __nv_bfloat16* q;
  const int32_t* lens;
  __nv_bfloat16* o;
  float* lse;
  float* ws_o;    // [B + grid - 1][H][448] partial outputs of sequences split between CTAs
  float* ws_lse;  // [B + grid - 1][H]
  int* ws_pref;   // [B + 1] tile prefix sums (stream-K; written by CTA 0 for the merge)
  const float2* table;  // D = 64 table for the RoPE dims
  int rope_il;          // RoPE pairs (2i, 2i+1) of the RoPE dims instead of (i, i + 32)
  unsigned int* status;
  int B, H, Lmax;
  int streamk;  // 1: split all key tiles evenly over the CTAs; 0: whole sequences c, c+grid, ...
  float scale_log2;
};

// Key tiles (KEYS keys) of sequence b; 0 for an out-of-range length.
template <int KEYS>
__device__ __forceinline__ int lat_tiles(const int32_t* lens, int b, int Lmax) {
  const int len = lens[b];
  return (len >= 1 && len <= Lmax) ? (len + KEYS - 1) / KEYS : 0;
}

// Stream-K split: the T key tiles of all sequences, in order, are cut into gridDim.x equal
// contiguous ranges, one per CTA; tile range of CTA c is [T c / G, T (c+1) / G).
__device__ __forceinline__ long long lat_range_lo(long long T, int c, int G) {
  return T * c / G;
}

// One contiguous run of a sequence's keys inside a CTA's share of the work.
struct LatSeg {
  int b, k0, k1;
  bool whole;    // the CTA covers every key of sequence b: it writes the final output
  bool invalid;  // sequence b has an out-of-range length (whole-sequence mode only)
};

template <int KEYS>
struct LatSegIter {
  long long lo, hi;
  int b, stride;
  bool streamk;
  // whole-sequence mode: sequences first, first + stride, ...
  __device__ void init_whole(int first, int stride_) {
    streamk = false;
    b = first;
    stride = stride_;
  }
  __device__ void init(const int* pref, int B, long long lo_, long long hi_) {
    streamk = true;
    lo = lo_;
    hi = hi_;
    int a = 0, z = B - 1;  // largest b with pref[b] <= lo
    while (a < z) {
      const int mid = (a + z + 1) >> 1;
      if (pref[mid] <= lo) a = mid; else z = mid - 1;
    }
    b = a;
  }
  __device__ bool next(const int* pref, int B, const int32_t* lens, LatSeg& sg) {
    if (!streamk) {
      if (b >= B) return false;
      const int len = lens[b];
      sg.b = b;
      sg.k0 = 0;
      sg.invalid = !(len >= 1 && len <= 0x40000000);
      sg.k1 = sg.invalid ? 0 : len;
      sg.whole = true;
      b += stride;
      return true;
    }
    while (b < B && pref[b] < hi) {
      const long long tb = pref[b], te = pref[b + 1];
      const int cur = b++;
      const long long s0 = lo > tb ? lo : tb, s1 = hi < te ? hi : te;
      if (s0 >= s1) continue;
      sg.b = cur;
      sg.k0 = static_cast<int>(s0 - tb) * KEYS;
      sg.k1 = min(static_cast<int>(s1 - tb) * KEYS, static_cast<int>(lens[cur]));
      sg.whole = (s0 == tb && s1 == te);
      sg.invalid = false;
      return true;
    }
    return false;
  }
};

// Issues this CTA's tiles, in order, into the stage ring.  Run by one thread.
template <bool F8>
struct LatLoader {
  using G = LatGeo<F8>;
  LatSegIter<G::kKeys> seg;
  LatSeg cur;
  int t0, stage;
  uint32_t phase;
  bool done;
  __device__ void advance(const int* pref, int B, const int32_t* lens, int Lmax) {
    while (true) {
      done = !seg.next(pref, B, lens, cur);
      if (done) return;
      if (cur.k1 > Lmax) cur.k1 = 0;  // out-of-range length: nothing to load
      if (cur.k0 < cur.k1) break;
    }
    t0 = cur.k0;
  }
  __device__ bool next(const LatParams& p, const int* pref, uint8_t* smem, uint64_t* full,
                       uint64_t* empty, const CUtensorMap* tm) {
    if (done) return true;
    if (!mbar_wait(&empty[stage], phase ^ 1, p.status)) return false;
    mbar_arrive_expect_tx(&full[stage], G::kTileBytes);
    uint8_t* ct = smem + stage * G::kTileBytes;
    tma_load_4d(ct, tm, &full[stage], 0, t0, 0, cur.b);
    if (++stage == G::kStages) {
      stage = 0;
      phase ^= 1;
    }
    t0 += G::kKeys;
    if (t0 >= cur.k1) advance(pref, p.B, p.lens, p.Lmax);
    return true;
  }
};

// Absorbed latent decode, stream-K over all sequences' key tiles.  Per tile (64 keys for a bf16
// cache, 128 for e5m2): warp w scores its kKeysPerWarp keys (8 or 16: one or two n8 key tiles)
// against the 16 query rows over all 512 dims (query fragments held in registers, four
// independent MMA chains in all), the tile's row maximum and P go through shared memory, then
// warp w accumulates its output columns over all the tile's keys.  Thread 0 refills each stage
// as soon as all warps released it.
//
// F8: an e5m2 cache.  Every e5m2 value is exactly an f16 value, so the MMAs run in f16 on values
// widened in registers: key fragments are 4-byte reads of the swizzled tile (4 consecutive
// dims, with the query fragments in the same dimension order), value fragments come from
// ldmatrix.trans on the fp8 tile read as 16-bit pairs, split by byte permutes into an even-dim
// and an odd-dim column tile of each 16-dim chunk; warp w owns chunks w, w + 8, w + 16, w + 24.
template <bool F8>
__global__ void __launch_bounds__(kLatThreads, 1)
    latent_decode_kernel(const __grid_constant__ CUtensorMap tmC, const LatParams p) {
  using G = LatGeo<F8>;
  constexpr int kNT = F8 ? 8 : kLatColsPerWarp / 8;  // output column tiles per warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + LatSmem::kBarOff);
  uint64_t* empty = full + kLatMaxStages;
  int* pref = reinterpret_cast<int*>(smem + LatSmem::kPrefOff);
  int* scan = reinterpret_cast<int*>(smem + LatSmem::kScanOff);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kLatWarps);
    }
    fence_barrier_init();
  }
  // stream-K mode: prefix sums of the tiles per sequence (each thread owns a contiguous chunk)
  if (p.streamk) {
    const int per = (p.B + kLatThreads - 1) / kLatThreads;
    const int b0 = tid * per, b1 = min(b0 + per, p.B);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += lat_tiles<G::kKeys>(p.lens, b, p.Lmax);
    int x = sum;  // inclusive scan over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) scan[warp] = x;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += scan[w];
    int run = base + x - sum;  // exclusive prefix of this thread's chunk
    for (int b = b0; b < b1; ++b) {
      pref[b] = run;
      run += lat_tiles<G::kKeys>(p.lens, b, p.Lmax);
    }
    if (tid == kLatThreads - 1) pref[p.B] = base + x;
  }
  __syncthreads();
  if (p.streamk && blockIdx.x == 0)  // the merge reads the same prefix sums
    for (int b = tid; b <= p.B; b += kLatThreads) p.ws_pref[b] = pref[b];
  long long lo = 0, hi = 0;
  if (p.streamk) {
    const long long T = pref[p.B];
    lo = lat_range_lo(T, blockIdx.x, gridDim.x);
    hi = lat_range_lo(T, blockIdx.x + 1, gridDim.x);
  }

  LatLoader<F8> loader;
  if (tid == 0) {
    tma_prefetch_desc(&tmC);
    if (p.streamk)
      loader.seg.init(pref, p.B, lo, hi);
    else
      loader.seg.init_whole(blockIdx.x, gridDim.x);
    loader.stage = 0;
    loader.phase = 0;
    loader.advance(pref, p.B, p.lens, p.Lmax);
    for (int s = 0; s < G::kStages; ++s) loader.next(p, pref, smem, full, empty, &tmC);
  }
  bool alive = true;

  const int g = lane >> 2, tq = lane & 3;
  uint8_t* qs = smem + LatSmem::kQOff;
  const uint32_t qs_addr = smem_u32(qs);
  const uint32_t ps_addr0 = smem_u32(smem + LatSmem::kPOff);
  float* red = reinterpret_cast<float*>(smem + LatSmem::kRedOff);
  float* lred = reinterpret_cast<float*>(smem + LatSmem::kLOff);
  int stage = 0;
  uint32_t phase = 0;
  int tcount = 0;
  const int H = p.H;

  LatSegIter<G::kKeys> segs;
  if (p.streamk)
    segs.init(pref, p.B, lo, hi);
  else
    segs.init_whole(blockIdx.x, gridDim.x);
  LatSeg sg;
  while (segs.next(pref, p.B, p.lens, sg)) {
    const int b = sg.b, k0 = sg.k0;
    const int len = p.lens[b];
    if (sg.invalid || len > p.Lmax) {  // whole-sequence mode: out-of-range length
      if (tid == 0) report_status(p.status, ATTN_ERR_DEVICE_ARG);
      for (int i = tid; i < H * kLatV; i += kLatThreads)
        p.o[static_cast<size_t>(b) * H * kLatV + i] = __float2bfloat16_rn(0.f);
      if (p.lse && tid < H) p.lse[static_cast<size_t>(b) * H + tid] = -INFINITY;
      continue;
    }
    const int k1 = sg.k1;

    lat_bar_sync();
    // query rows: 16-byte loads, all in flight before any store (rows >= H are zero) ...
    {
      constexpr int kChunks = kLatQK / 8;  // 8-dim chunks per row
      constexpr int kPer = 16 * kChunks / kLatThreads;
      uint4 v[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int idx = tid + k * kLatThreads, r = idx / kChunks, c = idx % kChunks;
        v[k] = r < H ? __ldg(reinterpret_cast<const uint4*>(
                           p.q + (static_cast<size_t>(b) * H + r) * kLatQK + c * 8))
                     : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int idx = tid + k * kLatThreads, r = idx / kChunks, c = idx % kChunks;
        uint4 w = v[k];
        if constexpr (F8) {  // the query in f16 (values beyond f16 range are not supported)
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[k]);
          __half2* o = reinterpret_cast<__half2*>(&w);
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] = __float22half2_rn(__bfloat1622float2(h[j]));
        }
        *reinterpret_cast<uint4*>(qs + r * kLatQPitch + c * 16) = w;
      }
    }
    lat_bar_sync();
    // ... then the 64 RoPE dims rotated at position len, pairs (i, i + 32) or (2i, 2i+1)
    if (p.table) {
      using QT = typename std::conditional<F8, __half, __nv_bfloat16>::type;
      for (int idx = tid; idx < 16 * (kLatRope / 2); idx += kLatThreads) {
        const int r = idx / (kLatRope / 2), i = idx % (kLatRope / 2);
        const int ia = kLatV + (p.rope_il ? 2 * i : i);
        const int ib = kLatV + (p.rope_il ? 2 * i + 1 : i + kLatRope / 2);
        QT* row = reinterpret_cast<QT*>(qs + r * kLatQPitch);
        const float x1 = static_cast<float>(row[ia]);
        const float x2 = static_cast<float>(row[ib]);
        const float2 cs = p.table[static_cast<size_t>(len) * (kLatRope / 2) + i];
        row[ia] = static_cast<QT>(x1 * cs.x - x2 * cs.y);
        row[ib] = static_cast<QT>(x2 * cs.x + x1 * cs.y);
      }
    }
    lat_bar_sync();
    uint32_t qa[kLatQK / 16][4];  // the 16 x 512 query tile as A fragments, for the segment
    if constexpr (F8) {
      // logical k = 2t+e -> dim 16kk+4t+e, k = 8+2t+e -> dim 16kk+4t+2+e (the key reads' order)
#pragma unroll
      for (int kk = 0; kk < kLatQK / 16; ++kk) {
        const uint8_t* r0 = qs + (lane >> 2) * kLatQPitch + (16 * kk + 4 * (lane & 3)) * 2;
        qa[kk][0] = *reinterpret_cast<const uint32_t*>(r0);
        qa[kk][1] = *reinterpret_cast<const uint32_t*>(r0 + 8 * kLatQPitch);
        qa[kk][2] = *reinterpret_cast<const uint32_t*>(r0 + 4);
        qa[kk][3] = *reinterpret_cast<const uint32_t*>(r0 + 8 * kLatQPitch + 4);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < kLatQK / 16; ++kk)
        ldsm_x4(qs_addr + (lane & 15) * kLatQPitch + (kk * 16 + (lane >> 4) * 8) * 2, qa[kk][0],
                qa[kk][1], qa[kk][2], qa[kk][3]);
    }

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc[kNT][4];
#pragma unroll
    for (int n = 0; n < kNT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

    constexpr int kNS = G::kNS;         // n8 key tiles this warp scores per tile
    constexpr int kCh = 4 / kNS;        // independent MMA chains per key tile (four in all)
    for (int t0 = k0; t0 < k1; t0 += G::kKeys, ++tcount) {
      if (!mbar_wait(&full[stage], phase, p.status)) {
        alive = false;
        break;
      }
      const uint32_t ct = smem_u32(smem + stage * G::kTileBytes);
      const int par = tcount & 1;
      float s[kNS][4];  // rows g / g+8 x keys kKeysPerWarp w + 8 nt + 2 tq + {0,1}
      {
        float ch[kNS][kCh][4];
#pragma unroll
        for (int nt = 0; nt < kNS; ++nt)
#pragma unroll
          for (int c = 0; c < kCh; ++c) ch[nt][c][0] = ch[nt][c][1] = ch[nt][c][2] = ch[nt][c][3] = 0.f;
        if constexpr (F8) {
          const uint8_t* kt = smem + stage * G::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kLatQK / 16; ++kk) {
#pragma unroll
            for (int nt = 0; nt < kNS; ++nt) {
              const int key = warp * G::kKeysPerWarp + nt * 8 + g;
              const uint32_t w = *reinterpret_cast<const uint32_t*>(
                  kt + (kk >> 3) * G::kKeys * 128 + sw128_offset(key, kk & 7) + 4 * tq);
              mma_f16_16816(ch[nt][kk % kCh], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3],
                            e5m2x2_lo(w), e5m2x2_hi(w));
            }
          }
        } else {
          static_assert(F8 || kNS == 1, "bf16 tiles: one key tile per warp");
          const int key = warp * G::kKeysPerWarp + (lane & 7);
          const int mi = lane >> 3;  // matrix index: 16-byte dim chunk within a pair of k-steps
#pragma unroll
          for (int kk = 0; kk < kLatQK / 16; kk += 2) {
            const int c = kk * 2 + mi;  // dims 8c .. 8c+7
            uint32_t b0, b1, b2, b3;
            ldsm_x4(ct + (c >> 3) * G::kKeys * 128 + sw128_offset(key, c & 7), b0, b1, b2, b3);
            mma_bf16_16816(ch[0][kk & 3], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
            mma_bf16_16816(ch[0][(kk + 1) & 3], qa[kk + 1][0], qa[kk + 1][1], qa[kk + 1][2],
                           qa[kk + 1][3], b2, b3);
          }
        }
#pragma unroll
        for (int nt = 0; nt < kNS; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v = ch[nt][0][e];
#pragma unroll
            for (int c = 1; c < kCh; ++c) v += ch[nt][c][e];
            s[nt][e] = v;
          }
      }
      float rm0 = -INFINITY, rm1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < kNS; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = t0 + warp * G::kKeysPerWarp + nt * 8 + tq * 2 + (e & 1);
          const float v = key < k1 ? s[nt][e] * p.scale_log2 : -INFINITY;
          s[nt][e] = v;
          if (e < 2)
            rm0 = fmaxf(rm0, v);
          else
            rm1 = fmaxf(rm1, v);
        }
      rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, 1));
      rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, 2));
      rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, 1));
      rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, 2));
      if (tq == 0) {
        red[(par * kLatWarps + warp) * 16 + g] = rm0;
        red[(par * kLatWarps + warp) * 16 + g + 8] = rm1;
      }
      lat_bar_sync();
      float tm0 = -INFINITY, tm1 = -INFINITY;
#pragma unroll
      for (int w = 0; w < kLatWarps; ++w) {
        tm0 = fmaxf(tm0, red[(par * kLatWarps + w) * 16 + g]);
        tm1 = fmaxf(tm1, red[(par * kLatWarps + w) * 16 + g + 8]);
      }
      const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);
      const float base0 = mn0 == -INFINITY ? 0.f : mn0;
      const float base1 = mn1 == -INFINITY ? 0.f : mn1;
      const float c0 = fast_exp2(m0 - base0), c1 = fast_exp2(m1 - base1);
      m0 = mn0;
      m1 = mn1;
      uint8_t* pw = smem + LatSmem::kPOff + par * 16 * G::kPPitch;
      l0 *= c0;
      l1 *= c1;
#pragma unroll
      for (int nt = 0; nt < kNS; ++nt) {
        const float e0 = fast_exp2(s[nt][0] - base0), e1 = fast_exp2(s[nt][1] - base0);
        const float e2 = fast_exp2(s[nt][2] - base1), e3 = fast_exp2(s[nt][3] - base1);
        const int col = warp * G::kKeysPerWarp + nt * 8 + tq * 2;
        *reinterpret_cast<uint32_t*>(pw + g * G::kPPitch + col * 2) =
            F8 ? pack_f16(e0, e1) : pack_bf16(e0, e1);
        *reinterpret_cast<uint32_t*>(pw + (g + 8) * G::kPPitch + col * 2) =
            F8 ? pack_f16(e2, e3) : pack_bf16(e2, e3);
        l0 += e0 + e1;
        l1 += e2 + e3;
      }
#pragma unroll
      for (int n = 0; n < kNT; ++n) {
        acc[n][0] *= c0;
        acc[n][1] *= c0;
        acc[n][2] *= c1;
        acc[n][3] *= c1;
      }
      lat_bar_sync();
      // O[:, this warp's columns] += P (16 x kKeys) * C[:, cols]
      const uint32_t ps_addr = ps_addr0 + par * 16 * G::kPPitch;
      const int cbase = (warp * kLatColsPerWarp) / 8;  // first 8-column chunk of this warp
#pragma unroll
      for (int kk = 0; kk < G::kKeys / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ps_addr + (lane & 15) * G::kPPitch + (kk * 16 + (lane >> 4) * 8) * 2, a0, a1, a2,
                a3);
        if constexpr (F8) {
          // chunk c = warp + 8 ci; matrices keys 0-7 / 8-15 of this step (lanes 0-15 address)
          const int keyr = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int ci = 0; ci < 4; ++ci) {
            const int c = warp + 8 * ci;
            if (c >= kLatV / 16) continue;  // warp-uniform: warps 4-7 own three chunks
            uint32_t r0, r1;
            ldsm_x2_t(ct + (c >> 3) * G::kKeys * 128 + sw128_offset(keyr, c & 7), r0, r1);
            mma_f16_16816(acc[2 * ci], a0, a1, a2, a3, e5m2x2_even(r0), e5m2x2_even(r1));
            mma_f16_16816(acc[2 * ci + 1], a0, a1, a2, a3, e5m2x2_odd(r0), e5m2x2_odd(r1));
          }
          continue;
        }
        const int mi = lane >> 3;
        const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int n2 = 0; n2 < 3; ++n2) {  // n-tiles 2*n2, 2*n2+1
          const int c = cbase + n2 * 2 + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(ct + (c >> 3) * G::kKeys * 128 + sw128_offset(key, c & 7), b0, b1, b2, b3);
          mma_bf16_16816(acc[2 * n2], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(acc[2 * n2 + 1], a0, a1, a2, a3, b2, b3);
        }
        {  // n-tile 6 (two 8x8 matrices: keys 0-7 and 8-15 of this step)
          const int c = cbase + 6;
          uint32_t b0, b1;
          ldsm_x2_t(ct + (c >> 3) * G::kKeys * 128 + sw128_offset(key, c & 7), b0, b1);
          mma_bf16_16816(acc[6], a0, a1, a2, a3, b0, b1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (tid == 0) alive = loader.next(p, pref, smem, full, empty, &tmC);
      __syncwarp();
      if (++stage == G::kStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (!__all_sync(0xffffffffu, alive)) return;

    // every warp used the same running max; row sums are split by key slice
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (tq == 0) {
      lred[warp * 16 + g] = l0;
      lred[warp * 16 + g + 8] = l1;
    }
    lat_bar_sync();
    float lt0 = 0.f, lt1 = 0.f;
#pragma unroll
    for (int w = 0; w < kLatWarps; ++w) {
      lt0 += lred[w * 16 + g];
      lt1 += lred[w * 16 + g + 8];
    }
    const float inv0 = lt0 > 0.f ? 1.f / lt0 : 0.f, inv1 = lt1 > 0.f ? 1.f / lt1 : 0.f;
    const float lse0 = lt0 > 0.f ? m0 + log2f(lt0) : -INFINITY;
    const float lse1 = lt1 > 0.f ? m1 + log2f(lt1) : -INFINITY;
    const size_t slot = static_cast<size_t>(blockIdx.x) + b;  // unique per (CTA, sequence)
    if constexpr (F8) {
      // slot (ci, e) holds dims 16c + 4tq + e and 16c + 4tq + 2 + e: four consecutive dims per row
#pragma unroll
      for (int ci = 0; ci < 4; ++ci) {
        const int c = warp + 8 * ci;
        if (c >= kLatV / 16) continue;
        const int d = 16 * c + 4 * tq;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = g + hh * 8;
          if (r >= H) continue;
          const float inv = hh ? inv1 : inv0;
          const float o0 = acc[2 * ci][hh * 2] * inv, o1 = acc[2 * ci + 1][hh * 2] * inv;
          const float o2 = acc[2 * ci][hh * 2 + 1] * inv, o3 = acc[2 * ci + 1][hh * 2 + 1] * inv;
          if (sg.whole) {
            const size_t row = static_cast<size_t>(b) * H + r;
            *reinterpret_cast<uint2*>(p.o + row * kLatV + d) =
                make_uint2(pack_bf16(o0, o1), pack_bf16(o2, o3));
          } else {
            *reinterpret_cast<float4*>(p.ws_o + (slot * H + r) * kLatV + d) =
                make_float4(o0, o1, o2, o3);
          }
        }
      }
    }
#pragma unroll
    for (int n = 0; n < (F8 ? 0 : kLatColsPerWarp / 8); ++n) {
      const int d = warp * kLatColsPerWarp + n * 8 + tq * 2;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = g + hh * 8;
        if (r >= H) continue;
        const float inv = hh ? inv1 : inv0;
        const float o0 = acc[n][hh * 2] * inv, o1 = acc[n][hh * 2 + 1] * inv;
        if (sg.whole) {
          const size_t row = static_cast<size_t>(b) * H + r;
          *reinterpret_cast<uint32_t*>(p.o + row * kLatV + d) = pack_bf16(o0, o1);
        } else {
          float* wo = p.ws_o + (slot * H + r) * kLatV + d;
          wo[0] = o0;
          wo[1] = o1;
        }
      }
    }
    if (tq == 0 && warp == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = g + hh * 8;
        if (r >= H) continue;
        const float l2 = hh ? lse1 : lse0;
        if (sg.whole) {
          if (p.lse) p.lse[static_cast<size_t>(b) * H + r] = l2 * kLn2;
        } else {
          p.ws_lse[slot * H + r] = l2;
        }
      }
    }
  }
}

// Finish the sequences that were split between CTAs (merge their partials by log-sum-exp) and
// the sequences with an out-of-range length (O = 0, LSE = -inf, status DEVICE_ARG).  One block
// per (sequence, head); sequences a single CTA covered were written directly and are skipped.
constexpr int kFinishThreads = 448;  // one thread per output column
constexpr int kMaxParts = 256;  // CTAs one sequence may be spread over (>= the SM count)

__global__ void __launch_bounds__(kFinishThreads)
    latent_finish_kernel(const int* __restrict__ pref, int B, int H, int G,
                         const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                         __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                         unsigned int* status) {
  const int b = blockIdx.x, h = blockIdx.y;
  __shared__ int parts[kMaxParts];
  __shared__ float wgt[kMaxParts];
  __shared__ float inv_s, lse_s;
  const long long T = pref[B], tb = pref[b];  // all tiles, and tiles of the sequences before b
  const int tiles = pref[b + 1] - pref[b];
  const size_t orow = static_cast<size_t>(b) * H + h;
  if (tiles == 0) {
    if (threadIdx.x == 0 && h == 0) report_status(status, ATTN_ERR_DEVICE_ARG);
    for (int d = threadIdx.x; d < kLatV; d += blockDim.x) o[orow * kLatV + d] = __float2bfloat16_rn(0.f);
    if (lse && threadIdx.x == 0) lse[orow] = -INFINITY;
    return;
  }
  // The CTA whose range [T c / G, T (c+1) / G) holds tile t is the largest c with
  // T c < (t + 1) G, i.e. ((t + 1) G - 1) / T.
  auto cta_of = [&](long long t) { return ((t + 1) * G - 1) / T; };
  const long long c_first = cta_of(tb), c_last = cta_of(tb + tiles - 1);
  if (c_first == c_last) return;  // one CTA covered the whole sequence: already final
  // With T >= G every CTA owns at least one tile, so the pieces come from c_first..c_last; with
  // T < G every CTA owns at most one tile, so piece i is the CTA of tile tb + i.
  const bool dense = T >= G;
  const int np = static_cast<int>(dense ? c_last - c_first + 1 : tiles);
  if (np > kMaxParts) {
    if (threadIdx.x == 0) report_status(status, ATTN_ERR_UNSUPPORTED);
    return;
  }
  for (int i = threadIdx.x; i < np; i += blockDim.x)
    parts[i] = static_cast<int>(dense ? c_first + i : cta_of(tb + i));
  __syncthreads();
  if (threadIdx.x < 32) {  // one warp: partial log-sum-exps -> weights, in parallel
    const int lane = threadIdx.x;
    float M = -INFINITY;
    for (int i = lane; i < np; i += 32) {
      const float l = ws_lse[(static_cast<size_t>(parts[i]) + b) * H + h];
      wgt[i] = l;
      M = fmaxf(M, l);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    float wsum = 0.f;
    for (int i = lane; i < np; i += 32) {
      const float l = wgt[i];
      const float w = l == -INFINITY ? 0.f : exp2f(l - M);
      wgt[i] = w;
      wsum += w;
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o2);
    if (lane == 0) {
      inv_s = wsum > 0.f ? 1.f / wsum : 0.f;
      lse_s = wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
    }
  }
  __syncthreads();
  for (int d = threadIdx.x; d < kLatV; d += blockDim.x) {
    // sixteen pieces per step, loads issued before any use (in-order issue would otherwise
    // wait for each load in turn)
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int i = 0;
    for (; i + 16 <= np; i += 16) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u)
        v[u] = ws_o[((static_cast<size_t>(parts[i + u]) + b) * H + h) * kLatV + d];
#pragma unroll
      for (int u = 0; u < 16; ++u) acc[u & 7] += wgt[i + u] * v[u];
    }
    for (; i < np; ++i) acc[0] += wgt[i] * ws_o[((static_cast<size_t>(parts[i]) + b) * H + h) * kLatV + d];
    const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    o[orow * kLatV + d] = __float2bfloat16_rn(sum * inv_s);
  }
  if (lse && threadIdx.x == 0) lse[orow] = lse_s;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Pick the number of key-range splits.  Cost model in bytes of HBM traffic (the kernels are
// bandwidth bound): a CTA streams at most twice its fair share of the bandwidth, so the time is
// max(busiest CTA's bytes * ctas / 2, all cache bytes) plus the split partials written and read
// back by the combine.
DecodePlan plan_common(int units, int Lmax, int ctas, double key_bytes, int rows_per_unit,
                       int out_dim, int forced_split) {
  const int max_split = std::min(kMaxSplits, std::max(1, (Lmax + kTileKeys - 1) / kTileKeys));
  int best = 1;
  double best_cost = 1e300;
  for (int ns = 1; ns <= max_split && forced_split <= 0; ns *= 2) {
    const int chunk = round_up((Lmax + ns - 1) / ns, kTileKeys);
    const int nsp = (Lmax + chunk - 1) / chunk;
    const double items = static_cast<double>(units) * nsp;
    const double waves = std::ceil(items / ctas);
    const double part = nsp > 1 ? static_cast<double>(rows_per_unit) * (out_dim + 1) * 4 : 0.0;
    const double busiest = waves * (chunk * key_bytes + part);
    const double total = static_cast<double>(units) * Lmax * key_bytes;
    const double cost = std::max(busiest * ctas / 2.0, total) + 2.0 * items * part;
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = nsp;
    }
  }
  if (forced_split > 0) best = std::min(forced_split, max_split);
  DecodePlan pl;
  pl.chunk = round_up((Lmax + best - 1) / best, kTileKeys);
  pl.nsplit = (Lmax + pl.chunk - 1) / pl.chunk;
  pl.grid = ctas;
  pl.ws_bytes = pl.nsplit > 1
                    ? static_cast<size_t>(units) * rows_per_unit * pl.nsplit * (out_dim + 1) * 4
                    : 0;
  return pl;
}

template <int D>
attn_status_t launch_gqa_typed(const void* q, const void* k, const void* v, const int32_t* lens,
                               int Lmax, void* o, float* lse, int B, int Hq, int Hkv, float scale,
                               const float2* table, int rope_il, void* ws, const DecodePlan& plan,
                               cudaStream_t st) {
  constexpr int NST = gqa_stages(D);
  using L = GqaSmem<D, NST>;
  CUtensorMap tk, tv;
  if (!make_tmap_3d(&tk, k, 2, D, Lmax, static_cast<uint64_t>(B) * Hkv, 64, kTileKeys, 128) ||
      !make_tmap_3d(&tv, v, 2, D, Lmax, static_cast<uint64_t>(B) * Hkv, 64, kTileKeys, 128))
    return ATTN_ERR_CUDA;
  GqaParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.lens = lens;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  const size_t rows = static_cast<size_t>(B) * Hq;
  p.ws_o = plan.nsplit > 1 ? static_cast<float*>(ws) : nullptr;
  p.ws_lse = plan.nsplit > 1 ? static_cast<float*>(ws) + rows * plan.nsplit * D : nullptr;
  p.table = table;
  p.rope_il = rope_il;
  p.status = device_status_ptr();
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.Lmax = Lmax;
  p.nsplit = plan.nsplit;
  p.chunk = plan.chunk;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int smem = L::bytes(p.G);
  auto kern = gqa_decode_kernel<D, NST>;
  if (!set_smem_attr(reinterpret_cast<const void*>(kern), smem)) return ATTN_ERR_CUDA;
  const int items = B * Hkv * plan.nsplit;
  const int grid = std::min(items, plan.grid);
  kern<<<grid, kThreads, smem, st>>>(tk, tv, p);
  if (launch_status() != ATTN_OK) return ATTN_ERR_CUDA;
  if (plan.nsplit > 1) {
    combine_kernel<<<static_cast<unsigned>(rows), 128, 0, st>>>(p.ws_o, p.ws_lse, plan.nsplit, D,
                                                              p.o, lse);
    return launch_status();
  }
  return ATTN_OK;
}

}  // namespace

std::atomic<int> g_forced_decode_splits{0};

DecodePlan plan_decode(int B, int Hq, int Hkv, int D, int Lmax) {
  return plan_common(B * Hkv, Lmax, gqa_ctas_per_sm(D) * sm_count(), 2.0 * D * 2, Hq / Hkv, D,
                     g_forced_decode_splits.load());
}

void force_decode_splits(int nsplit) { g_forced_decode_splits.store(nsplit); }

DecodePlan plan_latent(int B, int H, int Lmax) {
  (void)Lmax;
  DecodePlan pl;
  // At most 128 CTAs: at B = 128 one CTA per sequence on 128 SMs ran 0.047 ms under graph
  // replay, the stream-K split over 152 SMs 0.068 ms (0.053 ms for its main kernel alone: each
  // CTA then switches sequence mid-stream).  B equal to the CTA count: one CTA per sequence, no
  // merge.  Otherwise the key tiles of all sequences are spread
  // evenly over the CTAs and the pieces of split sequences merged afterwards.
  const int ctas = std::min(sm_count(), kLatMaxCtas);
  const bool streamk = B != ctas;
  pl.grid = ctas;
  pl.nsplit = streamk ? 1 : 0;  // 1 = stream-K mode (nsplit doubles as the mode flag here)
  pl.chunk = 0;
  // stream-K: partial outputs of sequences split between CTAs, slot (CTA + sequence)
  // and the tile prefix sums [B + 1] for the merge
  pl.ws_bytes = streamk ? static_cast<size_t>(B + pl.grid - 1) * H * (kLatV + 1) * 4 +
                              static_cast<size_t>(B + 1) * 4
                        : 0;
  return pl;
}

template <int NT>
attn_status_t launch_decode_fp8_nt(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const GqaParams& p, size_t rows, const DecodePlan& plan,
                                   float* lse, cudaStream_t st) {
  constexpr int NST = f8_stages(NT);
  const int smem = GqaF8Smem<NST>::bytes(p.G);
  auto kern = gqa_decode_fp8_kernel<NST, NT>;
  if (!set_smem_attr(reinterpret_cast<const void*>(kern), smem)) return ATTN_ERR_CUDA;
  const int items = p.B * p.Hkv * plan.nsplit;
  kern<<<std::min(items, plan.grid), kThreads, smem, st>>>(tk, tv, p);
  if (launch_status() != ATTN_OK) return ATTN_ERR_CUDA;
  if (plan.nsplit > 1) {
    combine_kernel<<<static_cast<unsigned>(rows), 128, 0, st>>>(p.ws_o, p.ws_lse, plan.nsplit,
                                                              kF8D, p.o, lse);
    return launch_status();
  }
  return ATTN_OK;
}

attn_status_t launch_decode_fp8(const void* q, const void* k, const void* v,
                                const int32_t* lens, int Lmax, void* o, float* lse, int B, int Hq,
                                int Hkv, float scale, const float2* table, int rope_il, void* ws,
                                const DecodePlan& plan, cudaStream_t st) {
  constexpr int D = kF8D;
  CUtensorMap tk, tv;
  if (!make_tmap_3d(&tk, k, 1, D, Lmax, static_cast<uint64_t>(B) * Hkv, D, kTileKeys, 128) ||
      !make_tmap_3d(&tv, v, 1, D, Lmax, static_cast<uint64_t>(B) * Hkv, D, kTileKeys, 128))
    return ATTN_ERR_CUDA;
  GqaParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.lens = lens;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  const size_t rows = static_cast<size_t>(B) * Hq;
  p.ws_o = plan.nsplit > 1 ? static_cast<float*>(ws) : nullptr;
  p.ws_lse = plan.nsplit > 1 ? static_cast<float*>(ws) + rows * plan.nsplit * D : nullptr;
  p.table = table;
  p.rope_il = rope_il;
  p.status = device_status_ptr();
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.Lmax = Lmax;
  p.nsplit = plan.nsplit;
  p.chunk = plan.chunk;
  p.scale_log2 = scale * 1.4426950408889634f;
  if (p.G <= 8) return launch_decode_fp8_nt<1>(tk, tv, p, rows, plan, lse, st);
  return launch_decode_fp8_nt<2>(tk, tv, p, rows, plan, lse, st);
}

// ------------------------------------------------------------------------------------------------
// Decode with the current token appended: after the history decode (keys 0..L-1), the current
// token's key (rotated at position L) and value are written to cache row L, and every query row
// of the group merges that one key into its history result (Fixed-budget decode audit —
// 2026-09-11, "A: group-entry queries and one joint history scan": the weight of the current
// token is the logistic function of its score minus the history's log-sum-exp, the history
// output takes the rest).  The query and the new key are rounded to bf16 after rotation, as the
// history decode and the cache hold them.  One block per (sequence, KV head).
// ------------------------------------------------------------------------------------------------

// One block per (sequence, KV head), one warp per query head of the group.  Lane l owns the
// rotation pairs i = 2l, 2l+1 (D = 128; i = l for D = 64), i.e. dims i and i + D/2 (dims 2i
// and 2i+1 when `il`), for the key, the query and the merge.  The group's first warp writes the
// cache row.
template <int D>
__global__ void __launch_bounds__(16 * 32)
    append_merge_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_new,
                        const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* k_cache,
                        __nv_bfloat16* v_cache, const int32_t* __restrict__ lens, int Lmax,
                        __nv_bfloat16* o, const float* __restrict__ lse_hist, float* lse_out,
                        int Hq, int Hkv, float scale, const float2* __restrict__ table,
                        int il, unsigned int* status) {
  constexpr int P = D / 64;  // pairs per lane
  const int b = blockIdx.x, kvh = blockIdx.y;
  const int g = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = Hq / Hkv;
  const int L = lens[b];
  if (L < 1 || L >= Lmax) {  // no history, or no row left for the new token
    if (threadIdx.x == 0 && kvh == 0) report_status(status, ATTN_ERR_DEVICE_ARG);
    return;
  }
  const size_t kv = static_cast<size_t>(b) * Hkv + kvh;
  const size_t crow = (kv * Lmax + L) * D;
  const size_t row = static_cast<size_t>(b) * Hq + kvh * G + g;
  const int i0 = lane * P;
  int da[P], db[P];  // the two dims of pair i0 + j
#pragma unroll
  for (int j = 0; j < P; ++j) {
    da[j] = il ? 2 * (i0 + j) : i0 + j;
    db[j] = il ? 2 * (i0 + j) + 1 : i0 + j + D / 2;
  }
  float k1[P], k2[P], q1[P], q2[P], v1[P], v2[P];
#pragma unroll
  for (int j = 0; j < P; ++j) {
    k1[j] = __bfloat162float(k_new[kv * D + da[j]]);
    k2[j] = __bfloat162float(k_new[kv * D + db[j]]);
    q1[j] = __bfloat162float(q[row * D + da[j]]);
    q2[j] = __bfloat162float(q[row * D + db[j]]);
    v1[j] = __bfloat162float(v_new[kv * D + da[j]]);
    v2[j] = __bfloat162float(v_new[kv * D + db[j]]);
  }
  float part = 0.f;
#pragma unroll
  for (int j = 0; j < P; ++j) {
    float c = 1.f, sn = 0.f;
    if (table) {
      const float2 cs = table[static_cast<size_t>(L) * (D / 2) + i0 + j];
      c = cs.x;
      sn = cs.y;
    }
    // key and query rotated at L and rounded to bf16, as the cache and the history hold them
    const float kr1 = __bfloat162float(__float2bfloat16_rn(k1[j] * c - k2[j] * sn));
    const float kr2 = __bfloat162float(__float2bfloat16_rn(k2[j] * c + k1[j] * sn));
    const float qr1 = __bfloat162float(__float2bfloat16_rn(q1[j] * c - q2[j] * sn));
    const float qr2 = __bfloat162float(__float2bfloat16_rn(q2[j] * c + q1[j] * sn));
    part = fmaf(qr1, kr1, fmaf(qr2, kr2, part));
    if (g == 0) {
      k_cache[crow + da[j]] = __float2bfloat16_rn(kr1);
      k_cache[crow + db[j]] = __float2bfloat16_rn(kr2);
      v_cache[crow + da[j]] = v_new[kv * D + da[j]];
      v_cache[crow + db[j]] = v_new[kv * D + db[j]];
    }
  }
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
  const float sc = part * scale;
  const float lh = lse_hist[row];
  const float a = 1.f / (1.f + expf(lh - sc));  // weight of the current token
#pragma unroll
  for (int j = 0; j < P; ++j) {
    __nv_bfloat16* orow = o + row * D;
    const float oh1 = __bfloat162float(orow[da[j]]), oh2 = __bfloat162float(orow[db[j]]);
    orow[da[j]] = __float2bfloat16_rn(fmaf(a, v1[j] - oh1, oh1));
    orow[db[j]] = __float2bfloat16_rn(fmaf(a, v2[j] - oh2, oh2));
  }
  if (lse_out && lane == 0) lse_out[row] = fmaxf(lh, sc) + log1pf(expf(-fabsf(sc - lh)));
}

// cache_len[b] += 1 where the append wrote a row (after every block of the merge has read it).
__global__ void append_len_kernel(int32_t* lens, int B, int Lmax) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int L = lens[b];
    if (L >= 1 && L < Lmax) lens[b] = L + 1;
  }
}

attn_status_t launch_decode_append(const void* q, const void* k_new, const void* v_new,
                                   void* k_cache, void* v_cache, int32_t* lens, int Lmax,
                                   void* o, float* lse, int B, int Hq, int Hkv, int D,
                                   float scale, const float2* table, int rope_il, void* ws,
                                   const DecodePlan& plan, cudaStream_t st) {
  // workspace: the history decode's own part, then the history LSE [B*Hq] (natural log)
  float* lse_hist = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + append_ws_offset(plan));
  attn_status_t r = launch_decode(q, k_cache, v_cache, lens, Lmax, o, lse_hist, B, Hq, Hkv, D,
                                  scale, table, rope_il, plan.ws_bytes ? ws : nullptr, plan, st);
  if (r != ATTN_OK) return r;
  const dim3 grid(B, Hkv);
  const int threads = 32 * (Hq / Hkv);  // one warp per query head of the group (<= 16)
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  const auto* kn = static_cast<const __nv_bfloat16*>(k_new);
  const auto* vn = static_cast<const __nv_bfloat16*>(v_new);
  auto* kc = static_cast<__nv_bfloat16*>(k_cache);
  auto* vc = static_cast<__nv_bfloat16*>(v_cache);
  auto* oo = static_cast<__nv_bfloat16*>(o);
  if (D == 256)
    append_merge_kernel<256><<<grid, threads, 0, st>>>(qq, kn, vn, kc, vc, lens, Lmax, oo,
                                                              lse_hist, lse, Hq, Hkv, scale,
                                                              table, rope_il, device_status_ptr());
  else if (D == 128)
    append_merge_kernel<128><<<grid, threads, 0, st>>>(qq, kn, vn, kc, vc, lens, Lmax, oo,
                                                              lse_hist, lse, Hq, Hkv, scale,
                                                              table, rope_il, device_status_ptr());
  else
    append_merge_kernel<64><<<grid, threads, 0, st>>>(qq, kn, vn, kc, vc, lens, Lmax, oo,
                                                             lse_hist, lse, Hq, Hkv, scale,
                                                             table, rope_il, device_status_ptr());
  if (launch_status() != ATTN_OK) return ATTN_ERR_CUDA;
  append_len_kernel<<<(B + 255) / 256, 256, 0, st>>>(lens, B, Lmax);
  return launch_status();
}

attn_status_t launch_decode(const void* q, const void* k, const void* v, const int32_t* lens,
                            int Lmax, void* o, float* lse, int B, int Hq, int Hkv, int D,
                            float scale, const float2* table, int rope_il, void* ws,
                            const DecodePlan& plan, cudaStream_t st) {
  if (D == 256)
    return launch_gqa_typed<256>(q, k, v, lens, Lmax, o, lse, B, Hq, Hkv, scale, table, rope_il,
                                 ws, plan, st);
  if (D == 128)
    return launch_gqa_typed<128>(q, k, v, lens, Lmax, o, lse, B, Hq, Hkv, scale, table, rope_il,
                                 ws, plan, st);
  return launch_gqa_typed<64>(q, k, v, lens, Lmax, o, lse, B, Hq, Hkv, scale, table, rope_il, ws,
                              plan, st);
}

attn_status_t launch_latent(const void* q, const void* c, const int32_t* lens, int Lmax, void* o,
                            float* lse, attn_dtype_t dt, int B, int H, float scale,
                            const float2* table, int rope_il, void* ws, const DecodePlan& plan,
                            cudaStream_t st) {
  if (B > kLatMaxB) return ATTN_ERR_UNSUPPORTED;
  const bool f8 = dt == ATTN_FP8_E5M2;
  CUtensorMap tc;
  const int esz = f8 ? 1 : 2;
  const uint32_t chunk = 128 / esz;  // elements per 128-byte column chunk of a cache row
  const uint64_t dims[4] = {chunk, static_cast<uint64_t>(Lmax), kLatQK / chunk,
                            static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {static_cast<uint64_t>(kLatQK) * esz, 128,
                               static_cast<uint64_t>(Lmax) * kLatQK * esz};
  const uint32_t box[4] = {chunk, static_cast<uint32_t>(f8 ? LatGeo<true>::kKeys
                                                         : LatGeo<false>::kKeys),
                           kLatQK / chunk, 1};
  if (!make_tmap_4d(&tc, c, esz, dims, strides, box)) return ATTN_ERR_CUDA;
  LatParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.lens = lens;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.ws_o = ws ? static_cast<float*>(ws) : nullptr;
  p.ws_lse = ws ? static_cast<float*>(ws) + static_cast<size_t>(B + plan.grid - 1) * H * kLatV
                : nullptr;
  p.ws_pref = ws ? reinterpret_cast<int*>(p.ws_lse + static_cast<size_t>(B + plan.grid - 1) * H)
                 : nullptr;
  p.table = table;
  p.rope_il = rope_il;
  p.status = device_status_ptr();
  p.B = B;
  p.H = H;
  p.Lmax = Lmax;
  p.streamk = plan.nsplit;  // the plan marks stream-K mode with nsplit = 1
  p.scale_log2 = scale * 1.4426950408889634f;
  auto kern = f8 ? latent_decode_kernel<true> : latent_decode_kernel<false>;
  if (!set_smem_attr(reinterpret_cast<const void*>(kern), LatSmem::kBytes)) return ATTN_ERR_CUDA;
  kern<<<plan.grid, kLatThreads, LatSmem::kBytes, st>>>(tc, p);
  if (launch_status() != ATTN_OK) return ATTN_ERR_CUDA;
  if (!p.streamk) return ATTN_OK;
  latent_finish_kernel<<<dim3(B, H), kFinishThreads, 0, st>>>(p.ws_pref, B, H, plan.grid, p.ws_o,
                                                              p.ws_lse, p.o, lse, p.status);
  return launch_status();
}

}  // namespace attn
