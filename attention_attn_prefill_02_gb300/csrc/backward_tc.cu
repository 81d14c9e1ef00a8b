// backward_tc.cu — gradients of grouped-query attention on the 5th-generation tensor cores:
// dQ, dK, dV for bf16 Q/K/V at D = 64 / 128, every product on tcgen05 with TMEM accumulators.
//
// With P = softmax(scale Q K^T + mask) recomputed from the forward's log-sum-exp, the chain rule
// gives dV = P^T dO, dP = dO V^T, dS = P * (dP - Delta) with Delta_i = sum_d dO_id O_id,
// dQ = scale dS K and dK = scale dS^T Q; a KV head's dK and dV sum over the G query heads that
// read it.  Two kernels, neither with atomics:
//
//   bwd_tc_kv_kernel  one CTA per (128-key tile, batch, KV head).  Per step (one 128-row query
//                     tile of one query head of the group): S^T = K Q^T and dP^T = V dO^T into
//                     TMEM; four warps (one key row per thread) turn them into P^T and dS^T,
//                     written back as bf16 over the columns they were read from; then
//                     dV += P^T dO and dK += dS^T Q with P^T / dS^T as the TMEM A operand.
//                     TMEM: S^T 128 | dP^T 128 | dV D | dK D columns.
//   bwd_tc_q_kernel   one CTA per (128-row query tile, batch, query head).  Per key tile:
//                     S = Q K^T and dP = dO V^T into TMEM, dS (bf16) over S, dQ += dS K.
//                     TMEM: S 128 | dP 128 | dQ D columns.
//
// Each step runs in two halves of 64 columns (query columns in the first kernel, key columns in
// the second): the score warps turn half 0 into P / dS while the tensor core computes the
// scores of half 1, and half 1 while the gradient products of half 0 (and the next step's
// half-0 scores) run.  Each of the two score warpgroups takes one 32-column chunk of every half.
//
// Tiles move by TMA in 128-row boxes of 64 bf16 with the 128-byte swizzle; one shared tile
// serves as a K-major operand (the Q K^T style products) and an MN-major one (the P V style).
// Warps 0-7 turn scores into P / dS and write the result (warp w reads TMEM lanes
// 32 (w % 4)..), warp 8 loads (TMA, plus the per-row log-sum-exp and Delta of each query tile),
// warp 9 issues the MMAs (the whole warp in the loop, one elected lane issuing).  Every wait is
// bounded, and warp-uniform where the warp goes on to a .sync.aligned TMEM access.
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace attn {
namespace {

constexpr int kTcRows = 128;     // keys per key tile, query rows per query tile (TMEM lanes)
constexpr int kTcHalf = 64;      // columns per half step
constexpr int kTcThreads = 320;  // 8 score warps (two warpgroups), the load warp, the MMA warp
constexpr int kTcLoader = 8, kTcMma = 9;
constexpr float kTcLog2e = 1.4426950408889634f;

struct TcParams {
  const __nv_bfloat16* q;     // [B*Hq*S, D]
  const __nv_bfloat16* dout;  // [B*Hq*S, D]
  const float* lse;           // [B*Hq*S] natural log
  const float* delta;         // [B*Hq*S]
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  unsigned int* status;
  int B, Hq, Hkv, G, S, causal, nT;  // nT: 128-row tiles along S
  float scale;                      // softmax scale
};

// A [128 x D] bf16 tile as D/64 boxes of [128 rows x 128 bytes] (128-byte swizzle).
template <int D>
struct TcTile {
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = kTcRows * 128;
  static constexpr int kBytes = kBoxes * kBoxBytes;
};

// Loads a [128 x D] tile (rows r0.., outer index z) into `dst` through TMA, completing on `bar`.
template <int D>
__device__ __forceinline__ void tc_load_tile(uint8_t* dst, const CUtensorMap* tm, uint64_t* bar,
                                             int r0, int z) {
#pragma unroll
  for (int bx = 0; bx < TcTile<D>::kBoxes; ++bx)
    tma_load_3d(dst + bx * TcTile<D>::kBoxBytes, tm, bar, bx * 64, r0, z);
}

// D[tmem] = A B^T over the head dim for the 64 B rows b_row0..: A [128 x D] and B [128 x D]
// K-major tiles in shared memory; the result fills 64 TMEM columns.
template <int D>
__device__ __forceinline__ void tc_mma_scores(uint32_t d, uint64_t a0, uint64_t b0, int b_row0,
                                              uint32_t idesc) {
  const uint64_t b1 = b0 + static_cast<uint64_t>((b_row0 * 128) >> 4);  // 8-row groups stay whole
  // one 64-column box (four K steps of 32 bytes) per batch of four MMAs
#pragma unroll
  for (int bx = 0; bx < TcTile<D>::kBoxes; ++bx) {
    const uint64_t o = static_cast<uint64_t>((bx * TcTile<D>::kBoxBytes) >> 4);
    umma_ss_x4(d, a0 + o, b1 + o, a0 + o + 2, b1 + o + 2, a0 + o + 4, b1 + o + 4, a0 + o + 6,
               b1 + o + 6, idesc, bx > 0);
  }
}

// D[tmem] = A B^T over the head dim for the 64 B rows b_row0..: A [128 x D] bf16 in TMEM
// (a_tmem.., two elements per column, 8 columns per K step of 16), B a [128 x D] K-major tile
// in shared memory; the result fills 64 TMEM columns.
template <int D>
__device__ __forceinline__ void tc_mma_scores_ta(uint32_t d, uint32_t a_tmem, uint64_t b0, int b_row0,
                                                 uint32_t idesc) {
  const uint64_t b1 = b0 + static_cast<uint64_t>((b_row0 * 128) >> 4);
#pragma unroll
  for (int bx = 0; bx < TcTile<D>::kBoxes; ++bx) {
    const uint64_t o = static_cast<uint64_t>((bx * TcTile<D>::kBoxBytes) >> 4);
    const uint32_t a = a_tmem + bx * 32;
    umma_ts_x4(d, a, b1 + o, a + 8, b1 + o + 2, a + 16, b1 + o + 4, a + 24, b1 + o + 6, idesc,
               bx > 0);
  }
}

// D[tmem] (+)= A X over 64 rows r0..r0+63: A [128 x 64] bf16 packed two per TMEM column (rows
// 0..31 at a_tmem.., rows 32..63 at a_tmem + 32..), X rows r0.. of a [128 x D] tile in shared
// memory read MN-major (D contiguous).
template <int D>
__device__ __forceinline__ void tc_mma_grad(uint32_t d, uint32_t a_tmem, uint64_t x0, int r0,
                                            uint32_t idesc, bool acc) {
  // four K steps of 16 rows (2048 bytes of the tile, 8 TMEM columns of A each), one batch; the
  // half's two 32-column chunks hold their 16 packed columns at the chunk's start (columns
  // 0..15 and 32..47 of the half)
  const uint64_t x = x0 + static_cast<uint64_t>((r0 * 128) >> 4);
  umma_ts_x4(d, a_tmem, x, a_tmem + 8, x + 128, a_tmem + 32, x + 256, a_tmem + 40, x + 384, idesc,
             acc ? 1u : 0u);
}

// Columns 32 c0 .. 32 c1 - 1 of one TMEM lane's accumulator, times `mul`, as bf16 at the same
// columns of the row dst (written only when `store`).  Every lane of the warp runs the TMEM
// loads, which are warp-collective (.sync.aligned): rows past S skip only the global store.
__device__ __forceinline__ void tc_store_row(__nv_bfloat16* dst, uint32_t taddr, float mul,
                                             bool store, int c0, int c1) {
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + c * 32, v);
    if (store) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 w;
        w.x = pack_bf16(__uint_as_float(v[q4 * 8 + 0]) * mul, __uint_as_float(v[q4 * 8 + 1]) * mul);
        w.y = pack_bf16(__uint_as_float(v[q4 * 8 + 2]) * mul, __uint_as_float(v[q4 * 8 + 3]) * mul);
        w.z = pack_bf16(__uint_as_float(v[q4 * 8 + 4]) * mul, __uint_as_float(v[q4 * 8 + 5]) * mul);
        w.w = pack_bf16(__uint_as_float(v[q4 * 8 + 6]) * mul, __uint_as_float(v[q4 * 8 + 7]) * mul);
        reinterpret_cast<uint4*>(dst + c * 32)[q4] = w;
      }
    }
  }
}

// P^T and dS^T of one key row over 32 query columns (the dK / dV kernel): p = 2^(s scale log2e -
// lse log2e) and ds = p (dp - Delta), packed as bf16 pairs, in paired f32x2 arithmetic.  nl_s /
// nd_s: -lse log2e and -Delta of the 32 queries.  MASK: zero p where the query is past S or
// (causal) before the key; without it the body has no branch.
template <bool MASK>
__device__ __forceinline__ void kv_scores_chunk(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                                const float* nl_s, const float* nd_s, float sl2,
                                                int key, int q_first, int S, int causal,
                                                uint32_t (&pp)[16], uint32_t (&dd)[16]) {
  const float2 c2 = make_float2(sl2, sl2);
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 l4 = *reinterpret_cast<const float4*>(nl_s + e);
    const float4 d4 = *reinterpret_cast<const float4*>(nd_s + e);
    float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2,
                           make_float2(l4.x, l4.y));
    float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])), c2,
                           make_float2(l4.z, l4.w));
    x0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
    x1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
    if constexpr (MASK) {
      const int q = q_first + e;
      const bool kin = key < S;
      if (!(kin && q < S && (!causal || key <= q))) x0.x = 0.f;
      if (!(kin && q + 1 < S && (!causal || key <= q + 1))) x0.y = 0.f;
      if (!(kin && q + 2 < S && (!causal || key <= q + 2))) x1.x = 0.f;
      if (!(kin && q + 3 < S && (!causal || key <= q + 3))) x1.y = 0.f;
    }
    const float2 g0 = __fmul2_rn(x0, __fadd2_rn(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                                make_float2(d4.x, d4.y)));
    const float2 g1 = __fmul2_rn(x1, __fadd2_rn(make_float2(__uint_as_float(dv[e + 2]), __uint_as_float(dv[e + 3])),
                                                make_float2(d4.z, d4.w)));
    pp[e / 2] = pack_bf16(x0.x, x0.y);
    pp[e / 2 + 1] = pack_bf16(x1.x, x1.y);
    dd[e / 2] = pack_bf16(g0.x, g0.y);
    dd[e / 2 + 1] = pack_bf16(g1.x, g1.y);
  }
}

// dS of one query row over 32 key columns (the dQ kernel), packed as bf16 pairs.  nl2 / nde:
// -lse log2e and -Delta of the row.  MASK as above with the roles of query and key exchanged.
template <bool MASK>
__device__ __forceinline__ void q_scores_chunk(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                               float sl2, float nl2, float nde, int q, int k_first,
                                               int S, int causal, uint32_t (&dd)[16]) {
  const float2 c2 = make_float2(sl2, sl2), l2 = make_float2(nl2, nl2), d2 = make_float2(nde, nde);
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, l2);
    x = make_float2(fast_exp2(x.x), fast_exp2(x.y));
    if constexpr (MASK) {
      const int k = k_first + e;
      if (!(q < S && k < S && (!causal || k <= q))) x.x = 0.f;
      if (!(q < S && k + 1 < S && (!causal || k + 1 <= q))) x.y = 0.f;
    }
    const float2 g = __fmul2_rn(x, __fadd2_rn(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), d2));
    dd[e / 2] = pack_bf16(g.x, g.y);
  }
}

// ------------------------------------------------------------------------------------------
// dK, dV
// ------------------------------------------------------------------------------------------

template <int D>
struct KvSmem {
  using T = TcTile<D>;
  static constexpr int kK = 0;
  static constexpr int kV = kK + T::kBytes;
  static constexpr int kQ = kV + T::kBytes;            // two stages
  static constexpr int kO = kQ + 2 * T::kBytes;        // two stages (dO)
  static constexpr int kLse = kO + 2 * T::kBytes;      // [2][128] -LSE * log2e
  static constexpr int kDel = kLse + 2 * kTcRows * 4;  // [2][128] -Delta
  static constexpr int kBar = kDel + 2 * kTcRows * 4;
  // at least 120 KB so that one CTA (and one 512-column TMEM allocation) runs per SM
  static constexpr int kBytes = std::max(kBar + 256 + 1024, 120 * 1024);
  static_assert(kBytes <= 232448, "shared memory per CTA");
};

struct KvBars {
  uint64_t kv_full, q_full[2], q_empty[2], row_full[2], s_full[2], p_full[2], done;
  uint32_t tmem_slot;
};
static_assert(sizeof(KvBars) <= 256, "barrier block");

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    bwd_tc_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const TcParams p) {
  using L = KvSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  KvBars* bars = reinterpret_cast<KvBars*>(smem + L::kBar);
  float* s_lse = reinterpret_cast<float*>(smem + L::kLse);
  float* s_del = reinterpret_cast<float*>(smem + L::kDel);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bhkv = p.B * p.Hkv;
  const int tile = blockIdx.x / bhkv;  // key tile 0 first: it meets the most query rows
  const int bh = blockIdx.x - tile * bhkv;
  const int b = bh / p.Hkv, kvh = bh - b * p.Hkv;
  const int kv0 = tile * kTcRows;
  const int qt0 = p.causal ? tile : 0;  // earlier query tiles see none of these keys
  const int per_head = p.nT - qt0;
  const int steps = p.G * per_head;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->q_empty[t], 1);
      mbar_init(&bars->row_full[t], 32);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 256);  // both score warpgroups
    }
    mbar_init(&bars->done, 1);
    fence_barrier_init();
  }
  if (warp == kTcMma) tmem_alloc(&bars->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  // step st: query head kvh * G + st / per_head, query tile qt0 + st % per_head
  auto step_q = [&](int st, int& hq, int& qt) {
    const int gi = st / per_head;
    qt = qt0 + (st - gi * per_head);
    hq = kvh * p.G + gi;
  };

  if (warp == kTcLoader) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * TcTile<D>::kBytes);
      tc_load_tile<D>(smem + L::kK, &tmK, &bars->kv_full, kv0, bh);
      tc_load_tile<D>(smem + L::kV, &tmV, &bars->kv_full, kv0, bh);
    }
    for (int st = 0; st < steps; ++st) {
      const int sg = st & 1;
      // stage sg is free once the gradient products of step st - 2 completed (they follow the
      // score warps' last read of its log-sum-exp and Delta)
      if (st >= 2 && !mbar_wait_warp_sleep(&bars->q_empty[sg], ((st >> 1) & 1) ^ 1, p.status)) break;
      int hq, qt;
      step_q(st, hq, qt);
      const int z = b * p.Hq + hq;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full[sg], 2 * TcTile<D>::kBytes);
        tc_load_tile<D>(smem + L::kQ + sg * TcTile<D>::kBytes, &tmQ, &bars->q_full[sg],
                        qt * kTcRows, z);
        tc_load_tile<D>(smem + L::kO + sg * TcTile<D>::kBytes, &tmO, &bars->q_full[sg],
                        qt * kTcRows, z);
      }
      const size_t rbase = static_cast<size_t>(z) * p.S;
#pragma unroll
      for (int i = 0; i < kTcRows / 32; ++i) {
        const int r = i * 32 + lane, q = qt * kTcRows + r;
        // stored negated (-lse log2e, -Delta); rows past S: P = 0 through an infinite
        // log-sum-exp (their scores are masked as well)
        s_lse[sg * kTcRows + r] = q < p.S ? -__ldg(p.lse + rbase + q) * kTcLog2e : -INFINITY;
        s_del[sg * kTcRows + r] = q < p.S ? -__ldg(p.delta + rbase + q) : 0.f;
      }
      mbar_arrive(&bars->row_full[sg]);
    }
  } else if (warp == kTcMma) {
    const uint32_t idesc_s = make_idesc(1, 1, false, false, kTcHalf, kTcRows);
    const uint32_t idesc_g = make_idesc(1, 1, false, true, D, kTcRows);  // B MN-major
    const uint64_t k_desc = smem_desc(smem_u32(smem + L::kK), 16, 1024, 2);
    const uint64_t v_desc = smem_desc(smem_u32(smem + L::kV), 16, 1024, 2);
    const uint64_t q_desc0 = smem_desc(smem_u32(smem + L::kQ), 16, 1024, 2);
    const uint64_t o_desc0 = smem_desc(smem_u32(smem + L::kO), 16, 1024, 2);
    const uint64_t qg_desc0 = smem_desc(smem_u32(smem + L::kQ), TcTile<D>::kBoxBytes, 1024, 2);
    const uint64_t og_desc0 = smem_desc(smem_u32(smem + L::kO), TcTile<D>::kBoxBytes, 1024, 2);
    auto stage_off = [](int st) {
      return static_cast<uint64_t>(((st & 1) * TcTile<D>::kBytes) >> 4);
    };
    // S^T = K Q^T and dP^T = V dO^T of half h (query columns 64h..) of step st
    auto issue_scores = [&](int st, int h) {
      const uint64_t so = stage_off(st);
      tc_mma_scores<D>(tmem + kColS + h * kTcHalf, k_desc, q_desc0 + so, h * kTcHalf, idesc_s);
      tc_mma_scores<D>(tmem + kColDP + h * kTcHalf, v_desc, o_desc0 + so, h * kTcHalf, idesc_s);
      umma_commit_e(&bars->s_full[h]);
    };
    // dV += P^T dO, dK += dS^T Q over the 64 query rows of half h; P^T / dS^T of half h sit in
    // columns 64h..64h+15 and 64h+32..64h+47 (bf16 pairs, one block per 32-column chunk)
    auto issue_grads = [&](int st, int h) {
      const uint64_t so = stage_off(st);
      const bool acc = st > 0 || h > 0;
      tc_mma_grad<D>(tmem + kColDV, tmem + kColS + kTcHalf * h, og_desc0 + so, h * kTcHalf, idesc_g, acc);
      tc_mma_grad<D>(tmem + kColDK, tmem + kColDP + kTcHalf * h, qg_desc0 + so, h * kTcHalf, idesc_g, acc);
    };
    // Pipelined order: ... grads h0 (st), scores h0 (st + 1), grads h1 (st), scores h1 (st + 1)
    // ...: the next step's half-0 scores run while warpgroup 1 works on half 1.  Scores of half
    // h overwrite the columns the grads of half h read, issued before them (the tensor core
    // runs one CTA's MMAs in issue order), and only after warpgroup h released them.
    bool ok = mbar_wait_warp_sleep(&bars->kv_full, 0, p.status) &&
              mbar_wait_warp_sleep(&bars->q_full[0], 0, p.status);
    if (ok) {
      tc_fence_after();
      issue_scores(0, 0);
      issue_scores(0, 1);
    }
    for (int st = 0; st < steps && ok; ++st) {
      const bool next = st + 1 < steps;
      if (!(ok = mbar_wait_warp_sleep(&bars->p_full[0], st & 1, p.status))) break;
      tc_fence_after();
      issue_grads(st, 0);
      if (next) {
        if (!(ok = mbar_wait_warp_sleep(&bars->q_full[(st + 1) & 1], ((st + 1) >> 1) & 1, p.status)))
          break;
        tc_fence_after();
        issue_scores(st + 1, 0);
      }
      if (!(ok = mbar_wait_warp_sleep(&bars->p_full[1], st & 1, p.status))) break;
      tc_fence_after();
      issue_grads(st, 1);
      umma_commit_e(&bars->q_empty[st & 1]);
      if (next) issue_scores(st + 1, 1);
    }
    if (ok) umma_commit_e(&bars->done);
  } else {
    // ---------------------------------------------------------------- P^T and dS^T, one key row
    // Warpgroup c takes the 32-column chunk c of both halves of every step, so a half is done
    // by both warpgroups at once.
    const int c = warp >> 2;
    const int kr = (warp & 3) * 32 + lane;  // TMEM lane quarter warp % 4
    const int key = kv0 + kr;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS, tDP = tmem + lane_off + kColDP;
    const float sl2 = p.scale * kTcLog2e;
    bool ok = true;
    for (int st = 0; st < steps && ok; ++st) {
      const int sg = st & 1;
      int hq, qt;
      step_q(st, hq, qt);
      const int q0 = qt * kTcRows;
      // masks: the diagonal tile, and the last query or key tile when S is ragged
      const bool need_mask = (p.causal && qt == tile) || q0 + kTcRows > p.S || kv0 + kTcRows > p.S;
      if (!(ok = mbar_wait_warp_sleep(&bars->row_full[sg], (st >> 1) & 1, p.status))) break;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (!(ok = mbar_wait_warp_sleep(&bars->s_full[h], st & 1, p.status))) break;
        tc_fence_after();
        const int col = h * kTcHalf + c * 32;  // this chunk's query columns in the tile
        uint32_t sv[32], dv[32];
        tmem_ld32x2(tS + col, sv, tDP + col, dv);
        uint32_t pp[16], dd[16];
        const float* lse_s = s_lse + sg * kTcRows + col;
        const float* del_s = s_del + sg * kTcRows + col;
        if (need_mask)
          kv_scores_chunk<true>(sv, dv, lse_s, del_s, sl2, key, q0 + col, p.S, p.causal, pp, dd);
        else
          kv_scores_chunk<false>(sv, dv, lse_s, del_s, sl2, key, q0 + col, p.S, p.causal, pp, dd);
        // bf16 pairs into the chunk's own first 16 columns, which this thread already read (the
        // other warpgroup reads only its own chunk's columns)
        tmem_st16(tS + col, pp);
        tmem_st16(tDP + col, dd);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[h]);
      }
    }
    // warpgroup 0: dK = scale * sum dS^T Q; warpgroup 1: dV; bf16, this thread's key row
    if (ok && (ok = mbar_wait_warp_sleep(&bars->done, 0, p.status))) {
      tc_fence_after();
      const size_t row = static_cast<size_t>(bh) * p.S + key;
      if (c == 0)
        tc_store_row(p.dk + row * D, tmem + lane_off + kColDK, p.scale, key < p.S, 0, D / 32);
      else
        tc_store_row(p.dv + row * D, tmem + lane_off + kColDV, 1.f, key < p.S, 0, D / 32);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// dQ
// ------------------------------------------------------------------------------------------

template <int D>
struct QSmem {
  using T = TcTile<D>;
  // Q and dO live in TMEM (the A operand of the score products).  K is read by the scores and
  // the dQ products, V by the scores only.
  static constexpr int kKStages = 4, kVStages = 3;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKStages * T::kBytes;
  static constexpr int kBar = kV + kVStages * T::kBytes;
  static constexpr int kBytes = std::max(kBar + 256 + 1024, 120 * 1024);
  static_assert(kBytes <= 232448, "shared memory per CTA");
};

struct QBars {
  uint64_t qd_full, k_full[4], k_empty[4], v_full[3], v_empty[3], s_full[2], p_full[2], done;
  uint32_t tmem_slot;
};
static_assert(sizeof(QBars) <= 256, "barrier block");

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    bwd_tc_q_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const TcParams p) {
  using L = QSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  QBars* bars = reinterpret_cast<QBars*>(smem + L::kBar);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bhq = p.B * p.Hq;
  const int lvl = blockIdx.x / bhq;
  const int qt = p.causal ? p.nT - 1 - lvl : lvl;  // causal: the longest query tiles first
  const int bh = blockIdx.x - lvl * bhq;
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int kvz = b * p.Hkv + hq / p.G;
  const int q0 = qt * kTcRows;
  const int steps = p.causal ? qt + 1 : p.nT;  // key tiles this query tile meets
  // TMEM: S 128 | dP 128 | dQ D | Q D/2 | dO D/2 columns (bf16 Q and dO rows packed in pairs)
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColQ = 256 + D, kColO = kColQ + D / 2;
  static_assert(kColO + D / 2 <= 512, "TMEM columns");

  if (threadIdx.x == 0) {
    mbar_init(&bars->qd_full, 256);  // both score warpgroups store their operand rows
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 256);  // both score warpgroups
    }
    for (int t = 0; t < L::kVStages; ++t) {
      mbar_init(&bars->v_full[t], 1);
      mbar_init(&bars->v_empty[t], 1);
    }
    for (int t = 0; t < L::kKStages; ++t) {
      mbar_init(&bars->k_full[t], 1);
      mbar_init(&bars->k_empty[t], 1);
    }
    mbar_init(&bars->done, 1);
    fence_barrier_init();
  }
  if (warp == kTcMma) tmem_alloc(&bars->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  if (warp == kTcLoader) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      for (int st = 0; st < steps; ++st) {
        // K stage st % 4 (free once the dQ products of step st - 4 completed), V stage st % 3
        // (free once the scores of step st - 3 completed)
        const int ks = st % L::kKStages, vs = st % L::kVStages;
        if (st >= L::kKStages &&
            !mbar_wait_sleep(&bars->k_empty[ks], ((st / L::kKStages) & 1) ^ 1, p.status))
          break;
        mbar_arrive_expect_tx(&bars->k_full[ks], TcTile<D>::kBytes);
        tc_load_tile<D>(smem + L::kK + ks * TcTile<D>::kBytes, &tmK, &bars->k_full[ks],
                        st * kTcRows, kvz);
        if (st >= L::kVStages &&
            !mbar_wait_sleep(&bars->v_empty[vs], ((st / L::kVStages) & 1) ^ 1, p.status))
          break;
        mbar_arrive_expect_tx(&bars->v_full[vs], TcTile<D>::kBytes);
        tc_load_tile<D>(smem + L::kV + vs * TcTile<D>::kBytes, &tmV, &bars->v_full[vs],
                        st * kTcRows, kvz);
      }
    }
  } else if (warp == kTcMma) {
    const uint32_t idesc_s = make_idesc(1, 1, false, false, kTcHalf, kTcRows);
    const uint32_t idesc_g = make_idesc(1, 1, false, true, D, kTcRows);  // B MN-major
    const uint64_t k_desc0 = smem_desc(smem_u32(smem + L::kK), 16, 1024, 2);
    const uint64_t v_desc0 = smem_desc(smem_u32(smem + L::kV), 16, 1024, 2);
    const uint64_t kg_desc0 = smem_desc(smem_u32(smem + L::kK), TcTile<D>::kBoxBytes, 1024, 2);
    auto k_off = [](int st) {
      return static_cast<uint64_t>(((st % L::kKStages) * TcTile<D>::kBytes) >> 4);
    };
    auto v_off = [](int st) {
      return static_cast<uint64_t>(((st % L::kVStages) * TcTile<D>::kBytes) >> 4);
    };
    // S = Q K^T and dP = dO V^T of half h (key columns 64h..) of key tile st, Q and dO from TMEM
    auto issue_scores = [&](int st, int h) {
      tc_mma_scores_ta<D>(tmem + kColS + h * kTcHalf, tmem + kColQ, k_desc0 + k_off(st), h * kTcHalf,
                          idesc_s);
      tc_mma_scores_ta<D>(tmem + kColDP + h * kTcHalf, tmem + kColO, v_desc0 + v_off(st),
                          h * kTcHalf, idesc_s);
      umma_commit_e(&bars->s_full[h]);
    };
    // dQ += dS K over the 64 keys of half h (dS of half h in S columns 64h..64h+15 and
    // 64h+32..64h+47)
    auto issue_grads = [&](int st, int h) {
      tc_mma_grad<D>(tmem + kColDQ, tmem + kColS + kTcHalf * h, kg_desc0 + k_off(st),
                     h * kTcHalf, idesc_g, st > 0 || h > 0);
    };
    // K and V of key tile st landed
    auto wait_kv = [&](int st) {
      return mbar_wait_warp_sleep(&bars->k_full[st % L::kKStages], (st / L::kKStages) & 1, p.status) &&
             mbar_wait_warp_sleep(&bars->v_full[st % L::kVStages], (st / L::kVStages) & 1, p.status);
    };
    // the pipelined order of the dK / dV kernel; V stage of step st is released once both
    // halves of its scores completed, the K stage once its dQ products did.  qd_full: the score
    // warps stored Q and dO into TMEM.
    bool ok = mbar_wait_warp_sleep(&bars->qd_full, 0, p.status) && wait_kv(0);
    if (ok) {
      tc_fence_after();
      issue_scores(0, 0);
      issue_scores(0, 1);
      umma_commit_e(&bars->v_empty[0]);
    }
    for (int st = 0; st < steps && ok; ++st) {
      const bool next = st + 1 < steps;
      if (!(ok = mbar_wait_warp_sleep(&bars->p_full[0], st & 1, p.status))) break;
      tc_fence_after();
      issue_grads(st, 0);
      if (next) {
        if (!(ok = wait_kv(st + 1))) break;
        tc_fence_after();
        issue_scores(st + 1, 0);
      }
      if (!(ok = mbar_wait_warp_sleep(&bars->p_full[1], st & 1, p.status))) break;
      tc_fence_after();
      issue_grads(st, 1);
      umma_commit_e(&bars->k_empty[st % L::kKStages]);
      if (next) {
        issue_scores(st + 1, 1);
        umma_commit_e(&bars->v_empty[(st + 1) % L::kVStages]);
      }
    }
    if (ok) umma_commit_e(&bars->done);
  } else {
    // ---------------------------------------------------------------- dS, one query row
    // Warpgroup c takes the 32-column chunk c of both halves of every key tile.
    const int c = warp >> 2;
    const int qr = (warp & 3) * 32 + lane;  // TMEM lane quarter warp % 4
    const int q = q0 + qr;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS, tDP = tmem + lane_off + kColDP;
    const float sl2 = p.scale * kTcLog2e;
    const size_t row = static_cast<size_t>(bh) * p.S + q;
    const float nl2 = q < p.S ? -__ldg(p.lse + row) * kTcLog2e : -INFINITY;
    const float nde = q < p.S ? -__ldg(p.delta + row) : 0.f;
    {
      // this thread's row of Q (warpgroup 0) or dO (warpgroup 1) into its TMEM lane as the A
      // operand of the score products: dims 2i, 2i+1 in column i (zeros past S)
      const uint4* src = reinterpret_cast<const uint4*>((c == 0 ? p.q : p.dout) + row * D);
      uint32_t v[D / 2];
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const uint4 x = q < p.S ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
        v[4 * i] = x.x;
        v[4 * i + 1] = x.y;
        v[4 * i + 2] = x.z;
        v[4 * i + 3] = x.w;
      }
      const uint32_t ta = tmem + lane_off + (c == 0 ? kColQ : kColO);
      if constexpr (D == 128) {
        tmem_st64(ta, v);
      } else {
        tmem_st32(ta, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->qd_full);
    }
    bool ok = true;
    for (int st = 0; st < steps && ok; ++st) {
      const int k0 = st * kTcRows;
      const bool need_mask = (p.causal && st == qt) || k0 + kTcRows > p.S || q0 + kTcRows > p.S;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (!(ok = mbar_wait_warp_sleep(&bars->s_full[h], st & 1, p.status))) break;
        tc_fence_after();
        const int col = h * kTcHalf + c * 32;  // this chunk's key columns in the tile
        uint32_t sv[32], dv[32];
        tmem_ld32x2(tS + col, sv, tDP + col, dv);
        uint32_t dd[16];
        if (need_mask)
          q_scores_chunk<true>(sv, dv, sl2, nl2, nde, q, k0 + col, p.S, p.causal, dd);
        else
          q_scores_chunk<false>(sv, dv, sl2, nl2, nde, q, k0 + col, p.S, p.causal, dd);
        // bf16 pairs into the chunk's own first 16 S columns, already read by this thread
        tmem_st16(tS + col, dd);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[h]);
      }
    }
    // dQ = scale * sum dS K, bf16, this thread's query row; warpgroup c writes columns
    // c D / 2 .. (c + 1) D / 2 - 1
    if (ok && (ok = mbar_wait_warp_sleep(&bars->done, 0, p.status))) {
      tc_fence_after();
      tc_store_row(p.dq + row * D, tmem + lane_off + kColDQ, p.scale, q < p.S, c * (D / 64),
                   (c + 1) * (D / 64));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Delta_i = sum_d dO_id O_id, one warp per query row.
template <int D>
__global__ void __launch_bounds__(256) bwd_tc_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                           const __nv_bfloat16* __restrict__ dout,
                                                           float* __restrict__ delta,
                                                           long long rows) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < rows;
       r += warps) {
    const __nv_bfloat16* orow = o + r * D + lane * E;
    const __nv_bfloat16* drow = dout + r * D + lane * E;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(orow + e));
      const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(drow + e));
      acc = fmaf(a.x, c.x, fmaf(a.y, c.y, acc));
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2);
    if (lane == 0) delta[r] = acc;
  }
}

template <int D>
attn_status_t launch_bwd_tc_typed(const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                  int B, int Hq, int Hkv, int S, int causal, float scale,
                                  float* delta, cudaStream_t st) {
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_3d(&tq, q, 2, D, S, static_cast<uint64_t>(B) * Hq, 64, kTcRows, 128) ||
      !make_tmap_3d(&tk, k, 2, D, S, static_cast<uint64_t>(B) * Hkv, 64, kTcRows, 128) ||
      !make_tmap_3d(&tv, v, 2, D, S, static_cast<uint64_t>(B) * Hkv, 64, kTcRows, 128) ||
      !make_tmap_3d(&to, dout, 2, D, S, static_cast<uint64_t>(B) * Hq, 64, kTcRows, 128))
    return ATTN_ERR_CUDA;
  const long long rows = static_cast<long long>(B) * Hq * S;
  {
    const long long blocks =
        std::min<long long>((rows * 32 + 255) / 256, static_cast<long long>(sm_count()) * 16);
    bwd_tc_delta_kernel<D><<<static_cast<int>(blocks), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), delta,
        rows);
    if (launch_status() != ATTN_OK) return ATTN_ERR_CUDA;
  }
  TcParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.delta = delta;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.status = device_status_ptr();
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.S = S;
  p.causal = causal;
  p.nT = (S + kTcRows - 1) / kTcRows;
  p.scale = scale;
  {
    auto kern = bwd_tc_kv_kernel<D>;
    if (!set_smem_attr(reinterpret_cast<const void*>(kern), KvSmem<D>::kBytes)) return ATTN_ERR_CUDA;
    kern<<<p.nT * B * Hkv, kTcThreads, KvSmem<D>::kBytes, st>>>(tq, tk, tv, to, p);
    if (launch_status() != ATTN_OK) return ATTN_ERR_CUDA;
  }
  {
    auto kern = bwd_tc_q_kernel<D>;
    if (!set_smem_attr(reinterpret_cast<const void*>(kern), QSmem<D>::kBytes)) return ATTN_ERR_CUDA;
    kern<<<p.nT * B * Hq, kTcThreads, QSmem<D>::kBytes, st>>>(tk, tv, p);
  }
  return launch_status();
}

}  // namespace

attn_status_t launch_prefill_backward_tc(const void* q, const void* k, const void* v,
                                         const void* o, const float* lse, const void* dout,
                                         void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                         int S, int D, int causal, float scale, void* ws,
                                         cudaStream_t st) {
  float* delta = static_cast<float*>(ws);
  if (D == 128)
    return launch_bwd_tc_typed<128>(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, S, causal,
                                    scale, delta, st);
  return launch_bwd_tc_typed<64>(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, S, causal, scale,
                                 delta, st);
}

}  // namespace attn
