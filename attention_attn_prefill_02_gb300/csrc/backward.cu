// backward.cu — gradients of grouped-query attention: dQ, dK, dV for bf16 Q/K/V (D = 64 / 128).
//
// With P = softmax(scale Q K^T + mask) recomputed from the forward's log-sum-exp, the chain rule
// gives dV = P^T dO, dP = dO V^T, dS = P * (dP - Delta) with Delta_i = sum_d dO_id O_id (the
// softmax Jacobian, rowsum(dP * P) = rowsum(dO * O)), dQ = scale dS K and dK = scale dS^T Q; the
// K/V gradients of a KV head sum over the G query heads that read it.  Q and K are taken as the
// forward used them (already rotated when RoPE is on; the rotation's own gradient is the inverse
// rotation).
//
//   bwd_delta_kernel       Delta per query row, and zeroes the fp32 dQ accumulator
//   bwd_dkdv_kernel        one CTA per (batch, KV head, 64-key tile), four warps of 16 keys.
//                          For each query head of the group and each 64-row query tile that
//                          sees the keys: S^T = K Q^T, P^T, dV += P^T dO, dP^T = V dO^T,
//                          dS^T, dK += dS^T Q in registers (mma.sync m16n8k16, ldmatrix from
//                          128-byte-swizzled shared tiles); dS^T goes through shared memory and
//                          the warps add dQ += dS K into the fp32 accumulator (2-wide atomics).
//   bwd_dq_convert_kernel  dQ = scale * accumulator -> bf16.
//
// These warp-level kernels are the second path; the default runs every product on tcgen05
// (backward_tc.cu) and attn_set_backward_path selects between them.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "common.cuh"

namespace attn {
namespace {

constexpr int kBwdKeys = 64;  // keys per CTA (4 warps x 16)
constexpr int kBwdRows = 64;  // query rows per inner tile
constexpr int kBwdWarps = 4;
constexpr int kBwdThreads = kBwdWarps * 32;
constexpr int kDsPitch = kBwdRows * 2 + 16;  // bytes per key row of the dS^T tile (padded)
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;  // [B*Hq*S], natural log
  float* delta;      // [B*Hq*S]
  float* dq_acc;     // [B*Hq*S*D], unscaled dS K
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int B, Hq, Hkv, G, S, causal;
  float scale;
};

// Byte offset of (row, 16-byte chunk c) in a [rows x D] bf16 tile stored as 64-column boxes of
// 128-byte rows, 128-byte swizzled (conflict-free ldmatrix).
__device__ __forceinline__ uint32_t tile_off(int row, int c) {
  return static_cast<uint32_t>((c >> 3) * (kBwdKeys * 128)) + sw128_offset(row, c & 7);
}

// rows [0, valid) of a [64 x D] row-major global tile into shared memory, zeros past `valid`
template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const __nv_bfloat16* __restrict__ src,
                                          int valid, int tid) {
  constexpr int kChunks = D / 8;
#pragma unroll 4
  for (int idx = tid; idx < kBwdKeys * kChunks; idx += kBwdThreads) {
    const int r = idx / kChunks, c = idx % kChunks;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < valid) val = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * D + c * 8));
    *reinterpret_cast<uint4*>(dst + tile_off(r, c)) = val;
  }
}

// The same tile copy as cp.async (16-byte, L2 only), zero-filled past `valid`; the caller
// commits and waits.
template <int D>
__device__ __forceinline__ void prefetch_tile(uint8_t* dst, const __nv_bfloat16* __restrict__ src,
                                              int valid, int tid) {
  constexpr int kChunks = D / 8;
#pragma unroll 4
  for (int idx = tid; idx < kBwdKeys * kChunks; idx += kBwdThreads) {
    const int r = idx / kChunks, c = idx % kChunks;
    const bool in = r < valid;
    const __nv_bfloat16* g = src + (in ? static_cast<size_t>(r) * D + c * 8 : 0);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst + tile_off(r, c))),
                 "l"(g), "r"(in ? 16 : 0)
                 : "memory");
  }
}

template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const BwdParams p) {
  constexpr int E = D / 32;  // elements per lane
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.S;
  const int lane = threadIdx.x & 31;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < rows;
       r += warps) {
    const __nv_bfloat16* orow = p.o + r * D + lane * E;
    const __nv_bfloat16* drow = p.dout + r * D + lane * E;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(orow + e));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(drow + e));
      acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2);
    if (lane == 0) p.delta[r] = acc;
    float* z = p.dq_acc + r * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) *reinterpret_cast<float2*>(z + e) = make_float2(0.f, 0.f);
  }
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 2) bwd_dkdv_kernel(const BwdParams p) {
  constexpr int kTile = kBwdKeys * D * 2;
  constexpr int NT = D / 8;  // 8-column output tiles along d
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kTile;
  uint8_t* sQb = sV + kTile;      // two Q tiles, then two dO tiles (double-buffered)
  uint8_t* sOb = sQb + 2 * kTile;
  uint8_t* sDs = sOb + 2 * kTile;
  float* sLse = reinterpret_cast<float*>(sDs + kBwdKeys * kDsPitch);
  float* sDel = sLse + kBwdRows;
  const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aDs = smem_u32(sDs);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3, m8 = lane >> 3;
  const int bhkv = p.B * p.Hkv;
  const int tile = blockIdx.x / bhkv;  // heaviest key tiles first when causal
  const int bh = blockIdx.x - tile * bhkv;
  const int b = bh / p.Hkv, kvh = bh - b * p.Hkv;
  const int kv0 = tile * kBwdKeys;
  const float sl2 = p.scale * kLog2e;

  load_tile<D>(sK, p.k + (static_cast<size_t>(bh) * p.S + kv0) * D, p.S - kv0, tid);
  load_tile<D>(sV, p.v + (static_cast<size_t>(bh) * p.S + kv0) * D, p.S - kv0, tid);

  float dk[NT][4], dv[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int j = 0; j < 4; ++j) dk[n][j] = dv[n][j] = 0.f;

  const int key_lo = kv0 + warp * 16 + g;  // this thread's key rows: key_lo and key_lo + 8
  const int q_first = p.causal ? kv0 : 0;   // earlier query rows see none of these keys
  // the (query head, query tile) steps of this CTA, flattened so the next tile's Q and dO can be
  // fetched while the current one is processed
  const int per_head = (p.S - q_first + kBwdRows - 1) / kBwdRows;
  const int steps = p.G * per_head;
  auto step_rows = [&](int st, size_t& row0, int& q0) {
    const int gi = st / per_head;
    q0 = q_first + (st - gi * per_head) * kBwdRows;
    row0 = (static_cast<size_t>(b) * p.Hq + kvh * p.G + gi) * p.S;
  };
  {
    size_t r0;
    int q0;
    step_rows(0, r0, q0);
    prefetch_tile<D>(sQb, p.q + (r0 + q0) * D, p.S - q0, tid);
    prefetch_tile<D>(sOb, p.dout + (r0 + q0) * D, p.S - q0, tid);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int st = 0; st < steps; ++st) {
    size_t row0;
    int q0;
    step_rows(st, row0, q0);
    const int buf = st & 1;
    const uint32_t aQ = smem_u32(sQb + buf * kTile), aO = smem_u32(sOb + buf * kTile);
    {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      __syncthreads();  // this step's tiles have landed; every warp is done with the last step
      if (tid < kBwdRows) {
        const bool ok = q0 + tid < p.S;
        sLse[tid] = ok ? p.lse[row0 + q0 + tid] * kLog2e : INFINITY;
        sDel[tid] = ok ? p.delta[row0 + q0 + tid] : 0.f;
      }
      if (st + 1 < steps) {  // the next step's tiles into the other buffers
        size_t r1;
        int q1;
        step_rows(st + 1, r1, q1);
        prefetch_tile<D>(sQb + (buf ^ 1) * kTile, p.q + (r1 + q1) * D, p.S - q1, tid);
        prefetch_tile<D>(sOb + (buf ^ 1) * kTile, p.dout + (r1 + q1) * D, p.S - q1, tid);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      __syncthreads();
      // S^T (this warp's 16 keys x 64 query rows) = K_w Q^T, and dP^T = V_w dO^T
      float s[8][4], dp[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[n][j] = dp[n][j] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t ka0, ka1, ka2, ka3, va0, va1, va2, va3;
        ldsm_x4(aK + tile_off(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), ka0, ka1, ka2, ka3);
        ldsm_x4(aV + tile_off(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), va0, va1, va2, va3);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int qr = np * 16 + (m8 >> 1) * 8 + (lane & 7);
          const int c = kk * 2 + (m8 & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(aQ + tile_off(qr, c), b0, b1, b2, b3);
          mma_bf16_16816(s[2 * np], ka0, ka1, ka2, ka3, b0, b1);
          mma_bf16_16816(s[2 * np + 1], ka0, ka1, ka2, ka3, b2, b3);
          ldsm_x4(aO + tile_off(qr, c), b0, b1, b2, b3);
          mma_bf16_16816(dp[2 * np], va0, va1, va2, va3, b0, b1);
          mma_bf16_16816(dp[2 * np + 1], va0, va1, va2, va3, b2, b3);
        }
      }
      // P^T = exp2(S^T scale log2e - LSE log2e) on visible (key, query) pairs; dS^T = P^T (dP^T - Delta)
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int key = key_lo + (j >= 2 ? 8 : 0);
          const int ql = n * 8 + t4 * 2 + (j & 1);
          const int qq = q0 + ql;
          const bool vis = key < p.S && qq < p.S && (!p.causal || key <= qq);
          const float pv = vis ? fast_exp2(s[n][j] * sl2 - sLse[ql]) : 0.f;
          s[n][j] = pv;
          dp[n][j] = pv * (dp[n][j] - sDel[ql]);
        }
      // dV += P^T dO and dK += dS^T Q (A operands straight from the accumulators)
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        const uint32_t pa0 = pack_bf16(s[2 * kq][0], s[2 * kq][1]);
        const uint32_t pa1 = pack_bf16(s[2 * kq][2], s[2 * kq][3]);
        const uint32_t pa2 = pack_bf16(s[2 * kq + 1][0], s[2 * kq + 1][1]);
        const uint32_t pa3 = pack_bf16(s[2 * kq + 1][2], s[2 * kq + 1][3]);
        const uint32_t da0 = pack_bf16(dp[2 * kq][0], dp[2 * kq][1]);
        const uint32_t da1 = pack_bf16(dp[2 * kq][2], dp[2 * kq][3]);
        const uint32_t da2 = pack_bf16(dp[2 * kq + 1][0], dp[2 * kq + 1][1]);
        const uint32_t da3 = pack_bf16(dp[2 * kq + 1][2], dp[2 * kq + 1][3]);
#pragma unroll
        for (int n2 = 0; n2 < D / 16; ++n2) {
          const int qr = kq * 16 + (m8 & 1) * 8 + (lane & 7);
          const int c = n2 * 2 + (m8 >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(aO + tile_off(qr, c), b0, b1, b2, b3);
          mma_bf16_16816(dv[2 * n2], pa0, pa1, pa2, pa3, b0, b1);
          mma_bf16_16816(dv[2 * n2 + 1], pa0, pa1, pa2, pa3, b2, b3);
          ldsm_x4_t(aQ + tile_off(qr, c), b0, b1, b2, b3);
          mma_bf16_16816(dk[2 * n2], da0, da1, da2, da3, b0, b1);
          mma_bf16_16816(dk[2 * n2 + 1], da0, da1, da2, da3, b2, b3);
        }
      }
      // dS^T (bf16) to shared memory: key rows, query columns
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int col = n * 8 + t4 * 2;
        *reinterpret_cast<uint32_t*>(sDs + (warp * 16 + g) * kDsPitch + col * 2) =
            pack_bf16(dp[n][0], dp[n][1]);
        *reinterpret_cast<uint32_t*>(sDs + (warp * 16 + g + 8) * kDsPitch + col * 2) =
            pack_bf16(dp[n][2], dp[n][3]);
      }
      __syncthreads();
      // dQ rows q0 + 16 warp .. + 15 += dS K over the 64 keys
      uint32_t qa[4][4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int keyrow = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int qcol = warp * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4_t(aDs + keyrow * kDsPitch + qcol * 2, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
      const int qrow_lo = q0 + warp * 16 + g;
      float* dqa = p.dq_acc + (row0 + qrow_lo) * D;
#pragma unroll
      for (int n2 = 0; n2 < D / 16; ++n2) {
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int kr = kk * 16 + (m8 & 1) * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(aK + tile_off(kr, n2 * 2 + (m8 >> 1)), b0, b1, b2, b3);
          mma_bf16_16816(acc[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          mma_bf16_16816(acc[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int d = (2 * n2 + h) * 8 + t4 * 2;
          if (qrow_lo < p.S) atomicAdd(reinterpret_cast<float2*>(dqa + d), make_float2(acc[h][0], acc[h][1]));
          if (qrow_lo + 8 < p.S)
            atomicAdd(reinterpret_cast<float2*>(dqa + 8 * D + d), make_float2(acc[h][2], acc[h][3]));
        }
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  // dK = scale * sum dS^T Q and dV, bf16, rows key_lo and key_lo + 8
  __nv_bfloat16* dkr = p.dk + (static_cast<size_t>(bh) * p.S + key_lo) * D;
  __nv_bfloat16* dvr = p.dv + (static_cast<size_t>(bh) * p.S + key_lo) * D;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int d = n * 8 + t4 * 2;
    if (key_lo < p.S) {
      *reinterpret_cast<uint32_t*>(dkr + d) = pack_bf16(dk[n][0] * p.scale, dk[n][1] * p.scale);
      *reinterpret_cast<uint32_t*>(dvr + d) = pack_bf16(dv[n][0], dv[n][1]);
    }
    if (key_lo + 8 < p.S) {
      *reinterpret_cast<uint32_t*>(dkr + 8 * D + d) = pack_bf16(dk[n][2] * p.scale, dk[n][3] * p.scale);
      *reinterpret_cast<uint32_t*>(dvr + 8 * D + d) = pack_bf16(dv[n][2], dv[n][3]);
    }
  }
}

__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                            __nv_bfloat16* dq, long long n4,
                                                            float scale) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(acc) + i);
    uint2 w;
    w.x = pack_bf16(a.x * scale, a.y * scale);
    w.y = pack_bf16(a.z * scale, a.w * scale);
    reinterpret_cast<uint2*>(dq)[i] = w;
  }
}

template <int D>
attn_status_t launch_bwd_typed(BwdParams p, cudaStream_t st) {
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.S;
  const int sms = sm_count();
  {
    const long long blocks = std::min<long long>((rows * 32 + 255) / 256, static_cast<long long>(sms) * 16);
    bwd_delta_kernel<D><<<static_cast<int>(blocks), 256, 0, st>>>(p);
    if (launch_status() != ATTN_OK) return ATTN_ERR_CUDA;
  }
  {
    constexpr int kSmem = 6 * kBwdKeys * D * 2 + kBwdKeys * kDsPitch + 2 * kBwdRows * 4 + 1024;
    auto kern = bwd_dkdv_kernel<D>;
    if (!set_smem_attr(reinterpret_cast<const void*>(kern), kSmem)) return ATTN_ERR_CUDA;
    const int tiles = (p.S + kBwdKeys - 1) / kBwdKeys;
    kern<<<tiles * p.B * p.Hkv, kBwdThreads, kSmem, st>>>(p);
    if (launch_status() != ATTN_OK) return ATTN_ERR_CUDA;
  }
  {
    const long long n4 = rows * D / 4;
    const long long blocks = std::min<long long>((n4 + 255) / 256, static_cast<long long>(sms) * 16);
    bwd_dq_convert_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(p.dq_acc, p.dq, n4, p.scale);
  }
  return launch_status();
}

}  // namespace

size_t bwd_workspace_bytes(int B, int Hq, int S, int D) {
  const size_t rows = static_cast<size_t>(B) * Hq * S;
  const size_t delta = (rows * 4 + 255) / 256 * 256;
  return delta + rows * D * 4;
}

namespace {
std::atomic<int> g_bwd_path{0};
}  // namespace

void force_backward_path(int path) { g_bwd_path.store(path); }

attn_status_t launch_prefill_backward(const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, int B, int Hq, int Hkv, int S, int D, int causal,
                                      float scale, void* ws, cudaStream_t st) {
  if (g_bwd_path.load() != 1)
    return launch_prefill_backward_tc(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, S, D, causal,
                                      scale, ws, st);
  BwdParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  const size_t rows = static_cast<size_t>(B) * Hq * S;
  p.delta = static_cast<float*>(ws);
  p.dq_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + (rows * 4 + 255) / 256 * 256);
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.S = S;
  p.causal = causal;
  p.scale = scale;
  if (D == 128) return launch_bwd_typed<128>(p, st);
  return launch_bwd_typed<64>(p, st);
}

}  // namespace attn
