// prefill.cu — grouped-query attention prefill on the 5th-generation tensor cores (tcgen05).
//
// One persistent CTA per SM.  (Head dim 256 runs prefill_d256_kernel, at the end of this file.)
// A work item is 256 query rows (two 128-row Q tiles) of one
// (batch, query head); items are ordered heaviest-first for causal attention and dealt to CTAs
// in a serpentine order (the persistent, causal-aware scheduling of the persistent-attention
// refactor page, "概要").  Inside a CTA the roles are warp-specialised:
//
//   warp 8      TMA producer: Q tiles, then K_j / V_j tiles through a shared-memory ring
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM, O_t += P_t V_j from TMEM
//   warps 0-7   two softmax warpgroups, one per Q tile; each thread owns one query row (one
//               TMEM lane): masks, online softmax in the exp2 domain, writes P (bf16) over its
//               S columns in TMEM, rescales O lazily, and runs the epilogue.
//
// The two Q tiles ping-pong: while the softmax of tile 0 runs, the tensor core works on tile 1
// (and the reverse), so the exponentials (the "softmax partition" the refactor page singles out
// as the slow part, "性能ベンチマーク") overlap the matrix products.  TMEM holds S0, S1 (128
// columns each) and O0, O1 (D columns each); P_t is written as packed bf16 into the first 64
// columns of S_t and consumed by the next MMA as its A operand straight from TMEM.
//
// Lazy rescaling: the running row maximum used for the exponentials is only raised when a tile's
// maximum exceeds it by more than 8 (log2 units); O and the row sum share that stale maximum, so
// the final O / l is exact.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <type_traits>

#include "common.cuh"

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per Q tile (TMEM lanes)
constexpr int BN = 128;  // keys per KV tile
// Q tiles per work item in the kernel below (D <= 128): two by default (the ping-pong of the two
// softmax warpgroups), or one (128-row items: twice as many, each without the ping-pong), the
// second tile configuration of the global-vs-per-shape comparison.  D = 256 has a kernel of its
// own at the end of this file.
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kRopeWarp0 = 10;  // fused RoPE: warps 10-13 rotate each K tile in shared memory
constexpr int kRopeThreads = 128;
// RoPE mode 1 adds the four K-rotation warps.
__host__ __device__ constexpr int threads_for(int rm) { return rm == 1 ? 448 : 320; }
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

// Tile geometry for head dim D and element size ESZ (2 = bf16, 1 = fp8 e5m2).  Rows of 128 (or,
// for 64-byte rows, 64) bytes are TMA-swizzled; the MMA advances 32 bytes per K step (16 bf16
// or 32 fp8 elements) and 16 / 32 keys per PV step.  STAGED (fp8 with fused RoPE): Q and K land
// as fp8 in staging tiles and are rotated into bf16 tiles, so QK^T runs in bf16 while V stays fp8.
template <int SWZ_BYTES_ROW>
struct Swz {
  static constexpr int kSwz = SWZ_BYTES_ROW >= 128 ? 128 : SWZ_BYTES_ROW;  // 128 or 64 bytes
  static constexpr uint32_t kCode = kSwz == 128 ? 2u : 4u;                  // descriptor mode
  static constexpr int kBoxBytes = 128 * kSwz;                               // one 128-row box
  static constexpr int kSBO = 8 * kSwz;                                      // 8-row group
};

template <int D, int ESZ, bool STAGED, int NT_>
struct Cfg {
  static_assert(D == 64 || D == 128, "the generic kernel's head dims");
  // Q / K tiles read by the QK^T MMA
  static constexpr int kQKE = STAGED ? 2 : ESZ;
  static constexpr int kRowBytes = D * kQKE;
  static constexpr int kSwz = Swz<kRowBytes>::kSwz;
  static constexpr int kBoxElems = kSwz / kQKE;
  static constexpr int kBoxes = kRowBytes / kSwz;
  static constexpr int kBoxBytes = Swz<kRowBytes>::kBoxBytes;
  static constexpr uint32_t kSwzCode = Swz<kRowBytes>::kCode;
  static constexpr int kSBO = Swz<kRowBytes>::kSBO;
  static constexpr int kKSteps = kRowBytes / 32;
  static constexpr int kQTileBytes = BM * kRowBytes;
  static constexpr int kKVTileBytes = BN * kRowBytes;  // K tile as the MMA reads it
  // V tiles (storage type)
  static constexpr int kVRowBytes = D * ESZ;
  static constexpr int kVSwz = Swz<kVRowBytes>::kSwz;
  static constexpr int kVBoxElems = kVSwz / ESZ;
  static constexpr int kVBoxes = kVRowBytes / kVSwz;
  static constexpr int kVBoxBytes = Swz<kVRowBytes>::kBoxBytes;
  static constexpr uint32_t kVSwzCode = Swz<kVRowBytes>::kCode;
  static constexpr int kVSBO = Swz<kVRowBytes>::kSBO;
  static constexpr int kVTileBytes = BN * kVRowBytes;
  static constexpr int kPVKeys = 32 / ESZ;  // keys per PV step
  static constexpr int kPVSteps = BN / kPVKeys;
  // staging tiles (STAGED only): fp8 Q / K as loaded, one 128-byte box per row for D = 128
  static constexpr int kStTileBytes = STAGED ? BM * D : 0;
  // Separate K and V rings; K is fetched one KV step ahead of V, so a K tile has about two KV
  // steps between landing and its first MMA (room for the TMA latency plus the fused RoPE).
  static constexpr int kKStages = STAGED ? 2 : ESZ == 2 ? (D == 128 ? 3 : 4) : (D == 128 ? 4 : 6);
  static constexpr int kVStages = STAGED ? 2 : ESZ == 2 ? (D == 128 ? 2 : 3) : (D == 128 ? 4 : 6);
  static constexpr int kNT = NT_;
  static_assert(NT_ == 1 || NT_ == 2, "one or two Q tiles per item");
  static constexpr int kQOff = 0;
  static constexpr int kQStOff = kQOff + kNT * kQTileBytes;
  static constexpr int kKVOff = kQStOff + 2 * kStTileBytes;
  static constexpr int kKStOff = kKVOff + kKStages * kKVTileBytes;
  static constexpr int kVOff = kKStOff + kKStages * kStTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kVTileBytes;
  // + the barrier block (under 1 KB) + slack for aligning the base to 1024 bytes
  static constexpr int kSmemBytes = kBarOff + 1024 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  static_assert(kKStages <= 8 && kVStages <= 8, "barrier arrays hold 8 stages");
  static_assert(kNT == 1 || kColO1 + D <= kTmemCols, "TMEM columns of O1 past the allocation");
  static_assert(!STAGED || D == 128, "fp8 with fused RoPE is built for D = 128");
};

struct Params {
  __nv_bfloat16* o;
  float* lse;
  unsigned int* status;
  int B, Hq, Hkv, G, S, causal;
  int Skv;    // keys (S for self-attention; a chunk's queries see Skv >= S keys)
  int off;    // absolute position of query row i is i + off (off = Skv - S: bottom-right causal)
  int rope_k;  // fused RoPE: rotate the K tiles too (0: keys arrive rotated, only q is rotated)
  int n_items, nM, nKV;
  int mblk;   // query-block levels per scheduling block (see item_coords)
  float c_log2;   // softmax_scale * q_scale * k_scale * log2(e)
  float v_scale;
  const float2* table;  // RoPE cos/sin [position][D/2] (fused RoPE only)
  int pos0;
};

struct Bars;
struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t k_full[8], k_empty[8], v_full[8], v_empty[8];
  uint64_t q_ready[2], k_ready[8];  // fused RoPE: tile rotated in shared memory
  uint64_t k_st_full[8], k_st_free[8];  // fp8 + RoPE: K staging tiles (loaded / consumed)
  uint64_t p_hi[2];  // P of keys 64..127 written (p_full: keys 0..63, or all of P with RoPE)
  uint64_t s_free[2];   // separate-P form: the softmax has read S_t (its columns may be reused)
  uint64_t pv_done[2];  // separate-P form: the P V products of the previous step completed
  uint32_t tmem_slot;
};
static_assert(sizeof(Bars) <= 1024, "barrier block");

// Item -> (query block m, batch b, query head hq).  Items are grouped so that the CTAs running
// at the same time read few K/V streams (one stream = the keys and values of one (batch, KV
// head)), which keeps the streams they share resident in L2: query blocks are taken in blocks of
// `mblk` levels (heaviest levels first when causal); inside a block, stream by stream, and for
// each stream level by level over the G query heads that read it.
__device__ __forceinline__ void item_coords(const Params& p, int it, int& m, int& b, int& hq) {
  const int per_blk = p.mblk * p.B * p.Hq;
  const int k = it / per_blk;
  const int nb = min(p.mblk, p.nM - k * p.mblk);  // levels in block k (the last may be short)
  const int idx = it - k * per_blk;
  const int s = idx / (nb * p.G);
  const int rem = idx - s * nb * p.G;
  const int li = k * p.mblk + rem / p.G;
  b = s / p.Hkv;
  hq = (s - b * p.Hkv) * p.G + rem % p.G;
  m = p.causal ? (p.nM - 1 - li) : li;
}

// KV tiles Q tile starting at row r0 must visit (0 when the tile is past the queries): causal
// tiles stop at the one holding the key at the tile's last row's position.
__device__ __forceinline__ int kv_tiles_for(const Params& p, int r0) {
  if (r0 >= p.S) return 0;
  if (!p.causal) return p.nKV;
  return min((min(r0 + BM - 1, p.S - 1) + p.off) / BN + 1, p.nKV);
}

// Serpentine assignment of items to persistent CTAs: round k visits CTAs forwards when k is even
// and backwards when odd, so heavy and light items pair up.
__device__ __forceinline__ int item_for(int round, int cta, int ncta) {
  return round * ncta + ((round & 1) ? (ncta - 1 - cta) : cta);
}

// Rotate one row of a 128-row tile held in shared memory as D/64 boxes of 128-byte swizzled
// rows: pairs (i, i + D/2) by the float32 cos/sin of this row's position (8 pairs per step).
template <int D>
__device__ __forceinline__ void rope_rotate_row(uint8_t* tile, int row,
                                                const float2* __restrict__ cs_row) {
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    const int c2 = c + D / 16;
    uint4* p1 = reinterpret_cast<uint4*>(tile + (c >> 3) * (128 * 128) + sw128_offset(row, c & 7));
    uint4* p2 =
        reinterpret_cast<uint4*>(tile + (c2 >> 3) * (128 * 128) + sw128_offset(row, c2 & 7));
    uint4 a = *p1, b = *p2;
    const float4* t4 = reinterpret_cast<const float4*>(cs_row + c * 8);
    uint32_t* aw = reinterpret_cast<uint32_t*>(&a);
    uint32_t* bw = reinterpret_cast<uint32_t*>(&b);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 t = __ldg(t4 + q);  // (cos, sin) of pairs 8c + 2q and 8c + 2q + 1
      const float2 x = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&aw[q]));
      const float2 y = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&bw[q]));
      aw[q] = pack_bf16(x.x * t.x - y.x * t.y, x.y * t.z - y.y * t.w);
      bw[q] = pack_bf16(y.x * t.x + x.x * t.y, y.y * t.z + x.y * t.w);
    }
    *p1 = a;
    *p2 = b;
  }
}

// fp8 (e5m2) Q row from a 128-byte-swizzled staging tile (D = 128: one box) -> rotated bf16 row
// in a two-box bf16 tile.  Pairs (i, i + 64) rotate by the row position's cos / sin.
__device__ __forceinline__ void rope_rotate_row_fp8_to_bf16(const uint8_t* st, uint8_t* bf, int row,
                                                           const float2* __restrict__ cs_row) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {  // 8 pairs per step: fp8 elements 8c..8c+7 and 64+8c..64+8c+7
    const uint2 a8 =
        *reinterpret_cast<const uint2*>(st + sw128_offset(row, c >> 1) + (c & 1) * 8);
    const uint2 b8 =
        *reinterpret_cast<const uint2*>(st + sw128_offset(row, 4 + (c >> 1)) + (c & 1) * 8);
    const __nv_fp8x2_storage_t* a2 = reinterpret_cast<const __nv_fp8x2_storage_t*>(&a8);
    const __nv_fp8x2_storage_t* b2 = reinterpret_cast<const __nv_fp8x2_storage_t*>(&b8);
    const float4* t4 = reinterpret_cast<const float4*>(cs_row + c * 8);
    uint4 oa, ob;
    uint32_t* aw = reinterpret_cast<uint32_t*>(&oa);
    uint32_t* bw = reinterpret_cast<uint32_t*>(&ob);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 t = __ldg(t4 + q);
      const float2 x = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(a2[q], __NV_E5M2)));
      const float2 y = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(b2[q], __NV_E5M2)));
      aw[q] = pack_bf16(x.x * t.x - y.x * t.y, x.y * t.z - y.y * t.w);
      bw[q] = pack_bf16(y.x * t.x + x.x * t.y, y.y * t.z + x.y * t.w);
    }
    *reinterpret_cast<uint4*>(bf + sw128_offset(row, c)) = oa;
    *reinterpret_cast<uint4*>(bf + 128 * 128 + sw128_offset(row, c)) = ob;
  }
}

// RM, the RoPE mode: 0 none; 1 Q and K rotated inside (the softmax warps rotate each Q tile as
// it lands, the RoPE warps every K tile).
// MMAs of K steps k0 .. K1 - 1 into D[d], issued in batches of four (then two, then one) under
// one elect each.  a(kk): the A operand of step kk (a shared-memory descriptor, or a TMEM address
// when TS); b(kk): the B descriptor.  The first MMA accumulates when `acc`, the rest always.
template <bool F8, bool TS, int K0, int K1, typename AF, typename BF>
__device__ __forceinline__ void issue_batched(uint32_t d, AF a, BF b, uint32_t idesc, bool acc) {
  constexpr int kN = K1 - K0;
  constexpr int k4 = K0 + kN / 4 * 4, k2 = k4 + (K1 - k4) / 2 * 2;
#pragma unroll
  for (int kk = K0; kk < k4; kk += 4) {
    const uint32_t ac = (acc || kk > K0) ? 1u : 0u;
    if constexpr (TS) {
      if constexpr (F8) umma_ts_f8_x4(d, a(kk), b(kk), a(kk + 1), b(kk + 1), a(kk + 2), b(kk + 2), a(kk + 3), b(kk + 3), idesc, ac);
      else umma_ts_x4(d, a(kk), b(kk), a(kk + 1), b(kk + 1), a(kk + 2), b(kk + 2), a(kk + 3), b(kk + 3), idesc, ac);
    } else {
      if constexpr (F8) umma_ss_f8_x4(d, a(kk), b(kk), a(kk + 1), b(kk + 1), a(kk + 2), b(kk + 2), a(kk + 3), b(kk + 3), idesc, ac);
      else umma_ss_x4(d, a(kk), b(kk), a(kk + 1), b(kk + 1), a(kk + 2), b(kk + 2), a(kk + 3), b(kk + 3), idesc, ac);
    }
  }
#pragma unroll
  for (int kk = k4; kk < k2; kk += 2) {
    const uint32_t ac = (acc || kk > K0) ? 1u : 0u;
    if constexpr (TS) {
      if constexpr (F8) umma_ts_f8_x2(d, a(kk), b(kk), a(kk + 1), b(kk + 1), idesc, ac);
      else umma_ts_x2(d, a(kk), b(kk), a(kk + 1), b(kk + 1), idesc, ac);
    } else {
      if constexpr (F8) umma_ss_f8_x2(d, a(kk), b(kk), a(kk + 1), b(kk + 1), idesc, ac);
      else umma_ss_x2(d, a(kk), b(kk), a(kk + 1), b(kk + 1), idesc, ac);
    }
  }
  if constexpr (k2 < K1) {
    const uint32_t ac = (acc || k2 > K0) ? 1u : 0u;
    if constexpr (TS) {
      if constexpr (F8) umma_ts_f8_e(d, a(k2), b(k2), idesc, ac);
      else umma_ts_e(d, a(k2), b(k2), idesc, ac);
    } else {
      if constexpr (F8) umma_ss_f8_e(d, a(k2), b(k2), idesc, ac);
      else umma_ss_e(d, a(k2), b(k2), idesc, ac);
    }
  }
}

template <int D, int RM, int ESZ, int NTT>
__global__ void __launch_bounds__(threads_for(RM), 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Params p) {
  constexpr bool FP8 = ESZ == 1;
  constexpr bool ROPE = RM == 1;  // Q and K rotated in shared memory
  constexpr bool STAGED = FP8 && ROPE;  // fp8 inputs, RoPE fused: rotate into bf16 Q/K tiles
  using C = Cfg<D, ESZ, STAGED, NTT>;
  constexpr int NT = C::kNT;             // Q tiles per item
  constexpr int kRowsPerItem = NT * BM;  // query rows per item
  // First TMEM column of P inside S_t.  The RoPE variants (four more warps, so fewer registers
  // per thread) run the softmax in two passes and write P over the upper half of S; the others
  // hold the whole S row in registers and write P over its first columns.
  constexpr uint32_t kPCol = ROPE ? (FP8 ? 96u : 64u) : 0u;
  // P released in two halves (keys 0..63, then 64..127) so that half of the P V products
  // overlap the softmax: measured faster at D >= 128, slower at D = 64, whose P V products are
  // short anyway (A/B on one GPU: bf16 / fp8 D=128 -1 to -2.4 %, D=64 +0.8 % / +5 %)
  constexpr bool kSplitP = D >= 128;
  // Separate P (D = 64 without in-kernel RoPE, where TMEM has room): P_t gets columns of its own
  // after O1 instead of S_t's, so that S_t(j+1) is issued as soon as the softmax has read S_t(j)
  // and runs during that softmax; the softmax then waits for the previous P V products
  // (pv_done) before it rescales O or overwrites P.
  constexpr uint32_t kPWidth = FP8 ? 32u : 64u;  // TMEM columns of one tile's P
  constexpr uint32_t kColP0 = C::kColO1 + D, kColP1 = kColP0 + kPWidth;
  constexpr bool kSepP = !ROPE && !kSplitP && kColP1 + kPWidth <= C::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->q_empty[t], 1);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128);
      if (kSplitP) mbar_init(&bars->p_hi[t], 128);
      mbar_init(&bars->o_full[t], 1);
      mbar_init(&bars->o_empty[t], 128);
    }
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->k_ready[s], kRopeThreads);
      mbar_init(&bars->k_st_full[s], 1);
      mbar_init(&bars->k_st_free[s], kRopeThreads);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->q_ready[0], 128);
    mbar_init(&bars->q_ready[1], 128);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_free[t], 128);
      mbar_init(&bars->pv_done[t], 1);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&bars->tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  const int rounds = (p.n_items + gridDim.x - 1) / gridDim.x;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t ph_qe[2] = {0, 0};
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      bool ok = true;
      for (int r = 0; r < rounds && ok; ++r) {
        const int it = item_for(r, blockIdx.x, gridDim.x);
        if (it >= p.n_items) continue;
        int m, b, hq;
        item_coords(p, it, m, b, hq);
        const int hkv = hq / p.G;
        int n[2] = {0, 0};
#pragma unroll
        for (int t = 0; t < NT; ++t) n[t] = kv_tiles_for(p, m * kRowsPerItem + t * BM);
        const int nkv = max(n[0], n[1]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (n[t] == 0 || !ok) continue;
          ok = mbar_wait(&bars->q_empty[t], ph_qe[t] ^ 1, p.status);
          ph_qe[t] ^= 1;
          if (!ok) continue;
          if constexpr (STAGED) {  // fp8 Q into its staging tile (one 128-byte box per row)
            mbar_arrive_expect_tx(&bars->q_full[t], C::kStTileBytes);
            tma_load_3d(smem + C::kQStOff + t * C::kStTileBytes, &tmQ, &bars->q_full[t], 0,
                        m * kRowsPerItem + t * BM, b * p.Hq + hq);
          } else {
            mbar_arrive_expect_tx(&bars->q_full[t], C::kQTileBytes);
            uint8_t* dst = smem + C::kQOff + t * C::kQTileBytes;
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_3d(dst + bx * C::kBoxBytes, &tmQ, &bars->q_full[t], bx * C::kBoxElems,
                          m * kRowsPerItem + t * BM, b * p.Hq + hq);
          }
        }
        // issue order K_0, K_1, V_0, K_2, V_1, ...: K runs one tile ahead of V
        auto load_k = [&](int j) {
          if constexpr (STAGED) {  // fp8 K into a staging tile; the RoPE warps convert it
            ok = mbar_wait(&bars->k_st_free[ks], kph ^ 1, p.status);
            if (!ok) return;
            mbar_arrive_expect_tx(&bars->k_st_full[ks], C::kStTileBytes);
            tma_load_3d(smem + C::kKStOff + ks * C::kStTileBytes, &tmK, &bars->k_st_full[ks], 0,
                        j * BN, b * p.Hkv + hkv);
            if (++ks == C::kKStages) { ks = 0; kph ^= 1; }
            return;
          }
          ok = mbar_wait(&bars->k_empty[ks], kph ^ 1, p.status);
          if (!ok) return;
          mbar_arrive_expect_tx(&bars->k_full[ks], C::kKVTileBytes);
          uint8_t* dst = smem + C::kKVOff + ks * C::kKVTileBytes;
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_3d(dst + bx * C::kBoxBytes, &tmK, &bars->k_full[ks], bx * C::kBoxElems,
                        j * BN, b * p.Hkv + hkv);
          if (++ks == C::kKStages) { ks = 0; kph ^= 1; }
        };
        auto load_v = [&](int j) {
          ok = mbar_wait(&bars->v_empty[vs], vph ^ 1, p.status);
          if (!ok) return;
          mbar_arrive_expect_tx(&bars->v_full[vs], C::kVTileBytes);
          uint8_t* dst = smem + C::kVOff + vs * C::kVTileBytes;
#pragma unroll
          for (int bx = 0; bx < C::kVBoxes; ++bx)
            tma_load_3d(dst + bx * C::kVBoxBytes, &tmV, &bars->v_full[vs], bx * C::kVBoxElems,
                        j * BN, b * p.Hkv + hkv);
          if (++vs == C::kVStages) { vs = 0; vph ^= 1; }
        };
        if (ok) load_k(0);
        for (int j = 0; j < nkv && ok; ++j) {
          if (j + 1 < nkv) load_k(j + 1);
          if (ok) load_v(j);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop in warp-uniform control flow and one elected lane
    // issues each MMA and commit: the descriptors then stay warp-uniform, and MMAs go out at
    // the tensor pipe's rate (a loop run by one lane alone issued them measurably slower).
    {
      // bf16 (format 1) x bf16, or e5m2 (1) x e5m2 for S and e4m3 (0) P x e5m2 V for PV
      const uint32_t idesc_s = make_idesc(1, 1, false, false, BN, BM);
      const uint32_t idesc_pv = make_idesc(FP8 ? 0u : 1u, 1, false, true, D, BM);  // V MN-major
      // descriptors of the first K step of Q tile 0 / ring slot 0; the address field (bits
      // 0-13, address / 16) of later tiles, slots and K steps is that plus a constant, with no
      // carry out of the field (shared memory ends below 256 KB)
      const uint64_t q_desc0 = smem_desc(smem_u32(smem + C::kQOff), 16, C::kSBO, C::kSwzCode);
      const uint64_t k_desc0 = smem_desc(smem_u32(smem + C::kKVOff), 16, C::kSBO, C::kSwzCode);
      const uint64_t v_desc0 =
          smem_desc(smem_u32(smem + C::kVOff), C::kVBoxBytes, C::kVSBO, C::kVSwzCode);
      uint32_t ph_qf[2] = {0, 0}, ph_pf[2] = {0, 0}, ph_oe[2] = {0, 0}, ph_sf[2] = {0, 0};
      int ks = 0, vs = 0;
      uint32_t kph = 0, vph = 0;
      bool ok = true;
      auto issue_s = [&](int t, int slot) {
        const uint64_t ad = q_desc0 + static_cast<uint64_t>((t * C::kQTileBytes) >> 4);
        const uint64_t bd = k_desc0 + static_cast<uint64_t>((slot * C::kKVTileBytes) >> 4);
        const uint32_t d = tmem + (t ? C::kColS1 : C::kColS0);
        constexpr int kPerBox = C::kSwz / 32;
        auto off = [](int kk) {
          return static_cast<uint64_t>(((kk / kPerBox) * C::kBoxBytes + (kk % kPerBox) * 32) >> 4);
        };
        issue_batched<C::kQKE == 1, false, 0, C::kKSteps>(
            d, [&](int kk) { return ad + off(kk); }, [&](int kk) { return bd + off(kk); }, idesc_s,
            false);
      };
      // the P V products of P columns [k0, k1) (k steps of 16 bf16 / 32 fp8 keys)
      auto issue_pv_part = [&](int t, int slot, bool acc, auto k0c, auto k1c) {
        constexpr int k0 = decltype(k0c)::value, k1 = decltype(k1c)::value;
        const uint64_t bd = v_desc0 + static_cast<uint64_t>((slot * C::kVTileBytes) >> 4);
        const uint32_t pcol =
            kSepP ? tmem + (t ? kColP1 : kColP0) : tmem + (t ? C::kColS1 : C::kColS0) + kPCol;
        const uint32_t d = tmem + (t ? C::kColO1 : C::kColO0);
        issue_batched<FP8, true, k0, k1>(
            d, [&](int kk) { return pcol + kk * 8; },
            [&](int kk) { return bd + static_cast<uint64_t>((kk * C::kPVKeys * C::kVSwz) >> 4); },
            idesc_pv, acc || k0 > 0);
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        // P: 8 TMEM columns per step (16 bf16 or 32 fp8 keys); V rows of kVSwz bytes per key
        issue_pv_part(t, slot, acc, std::integral_constant<int, 0>{},
                      std::integral_constant<int, C::kPVSteps>{});
      };
      for (int r = 0; r < rounds && ok; ++r) {
        const int it = item_for(r, blockIdx.x, gridDim.x);
        if (it >= p.n_items) continue;
        int m, b, hq;
        item_coords(p, it, m, b, hq);
        int n[2] = {0, 0};
#pragma unroll
        for (int t = 0; t < NT; ++t) n[t] = kv_tiles_for(p, m * kRowsPerItem + t * BM);
        const int nkv = max(n[0], n[1]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (n[t] == 0 || !ok) continue;
          ok = mbar_wait_warp(ROPE ? &bars->q_ready[t] : &bars->q_full[t], ph_qf[t], p.status);
          ph_qf[t] ^= 1;
        }
        if (!ok) break;
        // j = 0: S_t = Q_t K_0^T for both tiles
        const int kslot = ks;
        if (!(ok = mbar_wait_warp(ROPE ? &bars->k_ready[kslot] : &bars->k_full[kslot], kph,
                                  p.status)))
          break;
        if (++ks == C::kKStages) { ks = 0; kph ^= 1; }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (n[t] == 0) continue;
          issue_s(t, kslot);
          umma_commit_e(&bars->s_full[t]);
          if (n[t] == 1) umma_commit_e(&bars->q_empty[t]);
        }
        umma_commit_e(&bars->k_empty[kslot]);
        for (int j = 1; j <= nkv && ok; ++j) {
          const int vslot = vs;
          if (!(ok = mbar_wait_warp(&bars->v_full[vslot], vph, p.status))) break;
          if (++vs == C::kVStages) { vs = 0; vph ^= 1; }
          int kslot2 = -1;
          if (j < nkv) {
            kslot2 = ks;
            if (!(ok = mbar_wait_warp(ROPE ? &bars->k_ready[kslot2] : &bars->k_full[kslot2], kph,
                                      p.status)))
              break;
            if (++ks == C::kKStages) { ks = 0; kph ^= 1; }
          }
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (!ok) continue;
            if constexpr (kSepP) {
              // S_t(j) first, into the columns the softmax of step j - 1 has read (it runs while
              // that softmax computes), then P_t(j - 1) V from P's own columns
              if (j < n[t]) {
                if (!(ok = mbar_wait_warp(&bars->s_free[t], ph_sf[t], p.status))) continue;
                ph_sf[t] ^= 1;
                tc_fence_after();
                issue_s(t, kslot2);
                umma_commit_e(&bars->s_full[t]);
                if (j == n[t] - 1) umma_commit_e(&bars->q_empty[t]);
              }
              if (j - 1 < n[t]) {
                ok = mbar_wait_warp(&bars->p_full[t], ph_pf[t], p.status);
                ph_pf[t] ^= 1;
                if (ok && j == 1) {
                  ok = mbar_wait_warp(&bars->o_empty[t], ph_oe[t] ^ 1, p.status);
                  ph_oe[t] ^= 1;
                }
                if (!ok) continue;
                tc_fence_after();
                issue_pv(t, vslot, j > 1);
                umma_commit_e(&bars->pv_done[t]);
                if (j - 1 == n[t] - 1) umma_commit_e(&bars->o_full[t]);
              }
              if (t == NT - 1) umma_commit_e(&bars->v_empty[vslot]);
              continue;
            }
            if constexpr (kSplitP) {
              if (j - 1 < n[t]) {
                // each half of P goes to the tensor core as soon as the softmax has written it
                ok = mbar_wait_warp(&bars->p_full[t], ph_pf[t], p.status);
                if (ok && j == 1) {
                  ok = mbar_wait_warp(&bars->o_empty[t], ph_oe[t] ^ 1, p.status);
                  ph_oe[t] ^= 1;
                }
                if (!ok) continue;
                tc_fence_after();
                issue_pv_part(t, vslot, j > 1, std::integral_constant<int, 0>{},
                              std::integral_constant<int, C::kPVSteps / 2>{});
                ok = mbar_wait_warp(&bars->p_hi[t], ph_pf[t], p.status);
                ph_pf[t] ^= 1;
                if (!ok) continue;
                tc_fence_after();
                issue_pv_part(t, vslot, true, std::integral_constant<int, C::kPVSteps / 2>{},
                              std::integral_constant<int, C::kPVSteps>{});
                if (j - 1 == n[t] - 1) umma_commit_e(&bars->o_full[t]);
              }
            } else {
              if (j - 1 < n[t]) {
                ok = mbar_wait_warp(&bars->p_full[t], ph_pf[t], p.status);
                ph_pf[t] ^= 1;
                if (ok && j == 1) {
                  ok = mbar_wait_warp(&bars->o_empty[t], ph_oe[t] ^ 1, p.status);
                  ph_oe[t] ^= 1;
                }
                if (!ok) continue;
                tc_fence_after();
                issue_pv(t, vslot, j > 1);
                if (j - 1 == n[t] - 1) umma_commit_e(&bars->o_full[t]);
              }
            }
            // V stage free once the last tile's P V products completed (committed before that
            // tile's next QK^T, which the commit would otherwise also wait for)
            if (t == NT - 1) umma_commit_e(&bars->v_empty[vslot]);
            if (j < n[t]) {
              issue_s(t, kslot2);
              umma_commit_e(&bars->s_full[t]);
              if (j == n[t] - 1) umma_commit_e(&bars->q_empty[t]);
            }
          }
          if (kslot2 >= 0) umma_commit_e(&bars->k_empty[kslot2]);
        }
        if constexpr (kSepP) {
          // the softmax's last s_free of the item is not waited for (the item's next S needs
          // none): step over that phase
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (n[t] > 0) ph_sf[t] ^= 1;
        }
      }
    }
  } else if constexpr (ROPE) {
   if (warp >= kRopeWarp0) {
    // ------------------------------------------------------------------ K-tile RoPE warps
    // Thread rt owns 8 frequency pairs (chunk c) and the rows g, g + kGroups, ... of every K
    // tile.  The cos/sin of those rows come from a rotation recurrence in float32 instead of
    // table loads: one step advances the position by kGroups, one tile step by 128, and every
    // item restarts from the table value at position pos0 + g.
    constexpr int kChunks = D / 16;                 // 8-pair chunks in the first half of a row
    constexpr int kGroups = kRopeThreads / kChunks;  // row stride between a thread's rows
    constexpr int kRowsPer = BN / kGroups;
    const int rt = threadIdx.x - kRopeWarp0 * 32;
    const int c = rt % kChunks, g = rt / kChunks;
    // cos / sin of the 8 pairs as float2 over pairs (2q, 2q+1): anchor (position pos0 + g) and
    // row step (kGroups positions).  After a tile's kRowsPer steps the recurrence stands on row
    // g of the next tile, so it simply continues; each item restarts from the anchor.
    float2 anc_c[4], anc_s[4], stp_c[4], stp_s[4];
    {
      const float2* t0 = p.table + static_cast<size_t>(p.pos0 + g) * (D / 2) + c * 8;
      const float2* t1 = p.table + static_cast<size_t>(kGroups) * (D / 2) + c * 8;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 a = __ldg(t0 + 2 * q), a1 = __ldg(t0 + 2 * q + 1);
        const float2 b = __ldg(t1 + 2 * q), b1 = __ldg(t1 + 2 * q + 1);
        anc_c[q] = make_float2(a.x, a1.x);
        anc_s[q] = make_float2(a.y, a1.y);
        stp_c[q] = make_float2(b.x, b1.x);
        stp_s[q] = make_float2(-b.y, -b1.y);  // negated: see advance()
        if (!p.rope_k) {  // keys already rotated: the identity (the fp8 tiles still widen)
          anc_c[q] = stp_c[q] = make_float2(1.f, 1.f);
          anc_s[q] = stp_s[q] = make_float2(0.f, 0.f);
        }
      }
    }
    const int c2 = c + kChunks;
    const uint32_t off1 = (c >> 3) * (128 * 128) + ((c & 7) << 4);
    const uint32_t off2 = (c2 >> 3) * (128 * 128) + ((c2 & 7) << 4);
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int r = 0; r < rounds && ok; ++r) {
      const int it = item_for(r, blockIdx.x, gridDim.x);
      if (it >= p.n_items) continue;
      int m, b, hq;
      item_coords(p, it, m, b, hq);
      const int nkv = NT == 2 ? max(kv_tiles_for(p, m * kRowsPerItem),
                                    kv_tiles_for(p, m * kRowsPerItem + BM))
                              : kv_tiles_for(p, m * kRowsPerItem);
      float2 wc[4], ws[4];  // (cos, sin) at this thread's current row
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        wc[q] = anc_c[q];
        ws[q] = anc_s[q];
      }
      for (int j = 0; j < nkv && ok; ++j) {
        if constexpr (STAGED) {
          if (!(ok = mbar_wait(&bars->k_st_full[stage], ph, p.status))) break;
          if (!(ok = mbar_wait(&bars->k_empty[stage], ph ^ 1, p.status))) break;
        } else {
          if (!(ok = mbar_wait(&bars->k_full[stage], ph, p.status))) break;
        }
        uint8_t* tile = smem + C::kKVOff + stage * C::kKVTileBytes;
        const uint8_t* st = smem + C::kKStOff + stage * C::kStTileBytes;  // fp8 staging (STAGED)
        const int rows_valid = p.Skv - j * BN;  // rows >= this are past the keys (zeros)
#pragma unroll 2
        for (int k = 0; k < ((STAGED || p.rope_k) ? kRowsPer : 0); ++k) {
          const int row = g + k * kGroups;
          const uint32_t rsw = static_cast<uint32_t>((row & 7) << 4);
          uint4* p1 = reinterpret_cast<uint4*>(tile + row * 128 + (off1 ^ rsw));
          uint4* p2 = reinterpret_cast<uint4*>(tile + row * 128 + (off2 ^ rsw));
          if (STAGED || row < rows_valid) {  // staged tiles are always written (zeros past S)
            uint4 a, bq;
            if constexpr (STAGED) {  // fp8 elements 8c..8c+7 and 64+8c.. -> 4 + 4 packed pairs
              const uint2 a8 =
                  *reinterpret_cast<const uint2*>(st + sw128_offset(row, c >> 1) + (c & 1) * 8);
              const uint2 b8 = *reinterpret_cast<const uint2*>(
                  st + sw128_offset(row, 4 + (c >> 1)) + (c & 1) * 8);
              const __nv_fp8x2_storage_t* a2 = reinterpret_cast<const __nv_fp8x2_storage_t*>(&a8);
              const __nv_fp8x2_storage_t* b2 = reinterpret_cast<const __nv_fp8x2_storage_t*>(&b8);
              uint32_t* aw0 = reinterpret_cast<uint32_t*>(&a);
              uint32_t* bw0 = reinterpret_cast<uint32_t*>(&bq);
#pragma unroll
              for (int q = 0; q < 4; ++q) {  // widen to bf16 pairs (exact: e5m2 fits in bf16)
                const float2 xa = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(a2[q], __NV_E5M2)));
                const float2 xb = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(b2[q], __NV_E5M2)));
                aw0[q] = pack_bf16(xa.x, xa.y);
                bw0[q] = pack_bf16(xb.x, xb.y);
              }
            } else {
              a = *p1;
              bq = *p2;
            }
            uint32_t* aw = reinterpret_cast<uint32_t*>(&a);
            uint32_t* bw = reinterpret_cast<uint32_t*>(&bq);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 x = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&aw[q]));
              const float2 y = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&bw[q]));
              const float2 xn = __ffma2_rn(x, wc[q], __fmul2_rn(y, make_float2(-ws[q].x, -ws[q].y)));
              const float2 yn = __ffma2_rn(y, wc[q], __fmul2_rn(x, ws[q]));
              aw[q] = pack_bf16(xn.x, xn.y);
              bw[q] = pack_bf16(yn.x, yn.y);
            }
            *p1 = a;
            *p2 = bq;
          }
          // advance kGroups positions: c' = c dc - s ds, s' = s dc + c ds (stp_s holds -ds)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 c1 = __ffma2_rn(wc[q], stp_c[q], __fmul2_rn(ws[q], stp_s[q]));
            const float2 s1 = __ffma2_rn(ws[q], stp_c[q], __fmul2_rn(wc[q], make_float2(-stp_s[q].x, -stp_s[q].y)));
            wc[q] = c1;
            ws[q] = s1;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->k_ready[stage]);
        if constexpr (STAGED) mbar_arrive(&bars->k_st_free[stage]);
        if (++stage == C::kKStages) {
          stage = 0;
          ph ^= 1;
        }
      }
    }
   }
  }
  if (warp < 4 * NT) {  // (with one Q tile, warps 4-7 have no role)
    // ------------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;          // Q tile of this warpgroup
    const int quarter = warp & 3;     // TMEM lane quarter of this warp
    const int lrow = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + (t ? C::kColS1 : C::kColS0);
    const uint32_t tO = tmem + lane_off + (t ? C::kColO1 : C::kColO0);
    const uint32_t tP = tmem + lane_off + (t ? kColP1 : kColP0);  // separate-P form only
    uint32_t ph_s = 0, ph_o = 0, ph_q = 0, ph_pv = 0;
    bool ok = true;
    for (int r = 0; r < rounds && ok; ++r) {
      const int it = item_for(r, blockIdx.x, gridDim.x);
      if (it >= p.n_items) continue;
      int m, b, hq;
      item_coords(p, it, m, b, hq);
      const int r0 = m * kRowsPerItem + t * BM;
      const int n = kv_tiles_for(p, r0);
      if (n == 0) continue;
      const int row = r0 + lrow;
      if constexpr (ROPE) {
        if (!(ok = mbar_wait(&bars->q_full[t], ph_q, p.status))) break;
        ph_q ^= 1;
        if constexpr (STAGED) {
          // rows past S are zero in the staging tile; their table row may not exist: use row 0
          rope_rotate_row_fp8_to_bf16(smem + C::kQStOff + t * C::kStTileBytes,
                                      smem + C::kQOff + t * C::kQTileBytes, lrow,
                                      p.table + static_cast<size_t>(row < p.S ? p.pos0 + p.off + row : 0) * (D / 2));
        } else {
          if (row < p.S)
            rope_rotate_row<D>(smem + C::kQOff + t * C::kQTileBytes, lrow,
                               p.table + static_cast<size_t>(p.pos0 + p.off + row) * (D / 2));
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->q_ready[t]);
      }
      float m_run = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        if (!(ok = mbar_wait(&bars->s_full[t], ph_s, p.status))) break;
        ph_s ^= 1;
        tc_fence_after();
        // a tile is masked where it holds keys past the tile's first row's position, or past Skv
        const bool need_mask = (p.causal && j * BN + BN - 1 > r0 + p.off) || (j * BN + BN > p.Skv);
        const int lim = (p.causal ? min(row + p.off + 1, p.Skv) : p.Skv) - j * BN;  // keys >= lim hidden
        float f = 1.f;  // factor for O and l when the running maximum is raised
        if constexpr (ROPE) {
          // two passes over 64-column halves: max of both, then P of the upper half (kept in
          // registers) and of the lower half (loaded again); P goes to columns kPCol.. which
          // only hold scores already read
          float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
          uint32_t hb[64];
          {
            uint32_t ha[64];
            tmem_ld64(tS, ha);
            if (need_mask) {
#pragma unroll
              for (int e = 0; e < 64; ++e)
                if (e >= lim) ha[e] = __float_as_uint(-INFINITY);
            }
#pragma unroll
            for (int e = 0; e < 64; e += 8) {
              a0 = fmax3(a0, __uint_as_float(ha[e]), __uint_as_float(ha[e + 1]));
              a1 = fmax3(a1, __uint_as_float(ha[e + 2]), __uint_as_float(ha[e + 3]));
              a2 = fmax3(a2, __uint_as_float(ha[e + 4]), __uint_as_float(ha[e + 5]));
              a3 = fmax3(a3, __uint_as_float(ha[e + 6]), __uint_as_float(ha[e + 7]));
            }
          }
          tmem_ld64(tS + 64, hb);
          if (need_mask) {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (e + 64 >= lim) hb[e] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int e = 0; e < 64; e += 8) {
            a0 = fmax3(a0, __uint_as_float(hb[e]), __uint_as_float(hb[e + 1]));
            a1 = fmax3(a1, __uint_as_float(hb[e + 2]), __uint_as_float(hb[e + 3]));
            a2 = fmax3(a2, __uint_as_float(hb[e + 4]), __uint_as_float(hb[e + 5]));
            a3 = fmax3(a3, __uint_as_float(hb[e + 6]), __uint_as_float(hb[e + 7]));
          }
          const float m_tile = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * p.c_log2;
          if (j == 0) {
            m_run = m_tile;
          } else if (m_tile > m_run + kRescaleThreshold) {
            f = fast_exp2(m_run - m_tile);
            l *= f;
            m_run = m_tile;
          }
          const float2 c2 = make_float2(p.c_log2, p.c_log2);
          const float2 nm2 = make_float2(-m_run, -m_run);
          float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
          // 64 scores -> 32 packed bf16 pairs or 16 packed e4m3 quads, stored at column `col`
          auto emit = [&](const uint32_t (&h)[64], uint32_t col) {
            constexpr int kW = FP8 ? 16 : 32;
            uint32_t pk[kW];
#pragma unroll
            for (int e = 0; e < 64; e += 4) {
              float2 x0 = __ffma2_rn(make_float2(__uint_as_float(h[e]), __uint_as_float(h[e + 1])), c2, nm2);
              float2 x1 = __ffma2_rn(make_float2(__uint_as_float(h[e + 2]), __uint_as_float(h[e + 3])), c2, nm2);
              x0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
              x1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
              acc0 = __fadd2_rn(acc0, x0);
              acc1 = __fadd2_rn(acc1, x1);
              if constexpr (FP8) {
                pk[e / 4] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x0, __NV_SATFINITE, __NV_E4M3)) |
                            (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x1, __NV_SATFINITE, __NV_E4M3)) << 16);
              } else {
                pk[e / 2] = pack_bf16(x0.x, x0.y);
                pk[e / 2 + 1] = pack_bf16(x1.x, x1.y);
              }
            }
            if constexpr (FP8)
              tmem_st16(col, pk);
            else
              tmem_st32(col, pk);
          };
          emit(hb, tS + kPCol + (FP8 ? 16 : 32));  // keys 64..127
          {
            uint32_t ha[64];
            tmem_ld64(tS, ha);
            if (need_mask) {
#pragma unroll
              for (int e = 0; e < 64; ++e)
                if (e >= lim) ha[e] = __float_as_uint(-INFINITY);
            }
            emit(ha, tS + kPCol);  // keys 0..63
          }
          const float2 accs = __fadd2_rn(acc0, acc1);
          l += accs.x + accs.y;
        } else {
        uint32_t sr[128];
        tmem_ld128(tS, sr);
        if constexpr (kSepP) {
          // S_t(j) is in registers: its columns may take S_t(j + 1)
          tc_fence_before();
          mbar_arrive(&bars->s_free[t]);
        }
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 128; ++e)
            if (e >= lim) sr[e] = __float_as_uint(-INFINITY);
        }
        // row maximum: four independent 3-input max chains
        float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
        for (int e = 0; e < 128; e += 8) {
          a0 = fmax3(a0, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
          a1 = fmax3(a1, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
          a2 = fmax3(a2, __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
          a3 = fmax3(a3, __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
        }
        const float mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
        const float m_tile = mx * p.c_log2;
        if (j == 0) {
          m_run = m_tile;
        } else if (m_tile > m_run + kRescaleThreshold) {
          f = fast_exp2(m_run - m_tile);
          l *= f;
          m_run = m_tile;
        }
        // p = 2^(s * c - m): packed f32x2 FMA, one ex2 per element, four partial row sums
        const float2 c2 = make_float2(p.c_log2, p.c_log2);
        const float2 nm2 = make_float2(-m_run, -m_run);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
        if constexpr (kSplitP) {
          // O_t holds the tiles before j (their P V products completed before S_t(j) was
          // signalled); rescale it before this step's P V products accumulate onto it.
          // tcgen05.ld / st are warp-collective: rescale when any lane of the warp needs it
          // (lanes that do not have f == 1), eight columns at a time so that the scores stay
          // in registers meanwhile.
          if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < D / 8; ++c) {
              uint32_t ov[8];
              tmem_ld8(tO + c * 8, ov);
#pragma unroll
              for (int e = 0; e < 8; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
              tmem_st8(tO + c * 8, ov);
            }
          }
          // keys 0..63 first: their P is released to the MMA warp (p_full) before the
          // exponentials of keys 64..127 (p_hi), so half of the P V products overlap the softmax
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[FP8 ? 16 : 32];
#pragma unroll
            for (int e = 64 * h; e < 64 * h + 64; e += 8) {
              float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, nm2);
              float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), c2, nm2);
              float2 x2 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5])), c2, nm2);
              float2 x3 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7])), c2, nm2);
              x0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
              x1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
              x2 = make_float2(fast_exp2(x2.x), fast_exp2(x2.y));
              x3 = make_float2(fast_exp2(x3.x), fast_exp2(x3.y));
              acc0 = __fadd2_rn(acc0, x0);
              acc1 = __fadd2_rn(acc1, x1);
              acc2 = __fadd2_rn(acc2, x2);
              acc3 = __fadd2_rn(acc3, x3);
              const int w = e - 64 * h;
              if constexpr (FP8) {
                // e4m3, four keys per TMEM column, lowest key in the lowest byte
                pk[w / 4] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x0, __NV_SATFINITE, __NV_E4M3)) |
                            (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x1, __NV_SATFINITE, __NV_E4M3)) << 16);
                pk[w / 4 + 1] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x2, __NV_SATFINITE, __NV_E4M3)) |
                                (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x3, __NV_SATFINITE, __NV_E4M3)) << 16);
              } else {
                pk[w / 2] = pack_bf16(x0.x, x0.y);
                pk[w / 2 + 1] = pack_bf16(x1.x, x1.y);
                pk[w / 2 + 2] = pack_bf16(x2.x, x2.y);
                pk[w / 2 + 3] = pack_bf16(x3.x, x3.y);
              }
            }
            if constexpr (FP8)
              tmem_st16(tS + 16 * h, pk);
            else
              tmem_st32(tS + 32 * h, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(h ? &bars->p_hi[t] : &bars->p_full[t]);
          }
          const float2 accs = __fadd2_rn(__fadd2_rn(acc0, acc1), __fadd2_rn(acc2, acc3));
          l += accs.x + accs.y;
        } else {
          uint32_t pk[FP8 ? 32 : 64];
#pragma unroll
          for (int e = 0; e < 128; e += 8) {
            float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, nm2);
            float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), c2, nm2);
            float2 x2 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5])), c2, nm2);
            float2 x3 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7])), c2, nm2);
            x0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
            x1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
            x2 = make_float2(fast_exp2(x2.x), fast_exp2(x2.y));
            x3 = make_float2(fast_exp2(x3.x), fast_exp2(x3.y));
            acc0 = __fadd2_rn(acc0, x0);
            acc1 = __fadd2_rn(acc1, x1);
            acc2 = __fadd2_rn(acc2, x2);
            acc3 = __fadd2_rn(acc3, x3);
            if constexpr (FP8) {
              // e4m3, four keys per TMEM column, lowest key in the lowest byte
              pk[e / 4] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x0, __NV_SATFINITE, __NV_E4M3)) |
                          (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x1, __NV_SATFINITE, __NV_E4M3)) << 16);
              pk[e / 4 + 1] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x2, __NV_SATFINITE, __NV_E4M3)) |
                              (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x3, __NV_SATFINITE, __NV_E4M3)) << 16);
            } else {
              pk[e / 2] = pack_bf16(x0.x, x0.y);
              pk[e / 2 + 1] = pack_bf16(x1.x, x1.y);
              pk[e / 2 + 2] = pack_bf16(x2.x, x2.y);
              pk[e / 2 + 3] = pack_bf16(x3.x, x3.y);
            }
          }
          const float2 accs = __fadd2_rn(__fadd2_rn(acc0, acc1), __fadd2_rn(acc2, acc3));
          l += accs.x + accs.y;
          if constexpr (kSepP) {
            // P_t(j - 1) V has completed: P's columns are free and O holds the tiles before j
            if (j > 0) {
              if (!(ok = mbar_wait_warp(&bars->pv_done[t], ph_pv, p.status))) break;
              ph_pv ^= 1;
              tc_fence_after();
            }
            if constexpr (FP8)
              tmem_st32(tP, pk);
            else
              tmem_st64(tP, pk);
          } else {
            if constexpr (FP8)
              tmem_st32(tS, pk);
            else
              tmem_st64(tS, pk);
          }
          // O_t holds the tiles before j (their P V products completed before S_t(j) was
          // signalled, or, with separate P, before pv_done); rescale it, warp-uniformly, before
          // P is released
          if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ov[32];
              tmem_ld32(tO + c * 32, ov);
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
              tmem_st32(tO + c * 32, ov);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->p_full[t]);
        }
        }
        if constexpr (ROPE) {
          // (two-pass softmax) P is complete; rescale O, then release both halves at once
          if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ov[32];
              tmem_ld32(tO + c * 32, ov);
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
              tmem_st32(tO + c * 32, ov);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&bars->p_full[t]);
          if constexpr (kSplitP) mbar_arrive(&bars->p_hi[t]);
        }
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, LSE
      if (!(ok = mbar_wait(&bars->o_full[t], ph_o, p.status))) break;
      ph_o ^= 1;
      // separate P: the item's last P V completion is covered by o_full; step over its phase
      if constexpr (kSepP) ph_pv ^= 1;
      tc_fence_after();
      const float inv = p.v_scale / l;
      __nv_bfloat16* orow = p.o + ((static_cast<size_t>(b) * p.Hq + hq) * p.S + row) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + c * 32, ov);
        if (row < p.S) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(ov[q4 * 8 + 0]) * inv, __uint_as_float(ov[q4 * 8 + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(ov[q4 * 8 + 2]) * inv, __uint_as_float(ov[q4 * 8 + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(ov[q4 * 8 + 4]) * inv, __uint_as_float(ov[q4 * 8 + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(ov[q4 * 8 + 6]) * inv, __uint_as_float(ov[q4 * 8 + 7]) * inv);
            dst[q4] = w;
          }
        }
      }
      if (p.lse && row < p.S)
        p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.S + row] = (m_run + log2f(l)) * kLn2;
      tc_fence_before();
      mbar_arrive(&bars->o_empty[t]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------------------------------------
// One Q tile per item, S double-buffered in TMEM, K / V through a ring of 16 KB chunks: the head
// dim 256 kernel.  (The geometry below is written for any D whose rows are whole 128-byte
// boxes; at D = 128 the two-tile kernel above measured faster: fp8 causal S = 16384 3.96 ms
// against 5.84 ms with this one, so only D = 256 dispatches here.)
//
// At D = 256, 64 KB K and V tiles leave room for one stage each next to the 64 KB Q tile, so the
// next S could only start once the K stage had been refilled after the previous S: each KV step
// ran S, the softmax and P V one after the other.  Here the K / V stages form a ring of 16 KB
// chunks in the order the tensor core reads them: a K chunk is one 128-byte column box of a K
// tile (four K steps of S), a V chunk is kVKeys keys x all D dims, landed by one 4-D TMA copy as
// 128-byte-swizzled column groups.  TMEM holds S in two buffers (columns 0 and 128, S_j in
// buffer j & 1) and O in columns 256.., so S_{j+1} is computed while the softmax of step j runs,
// and the tensor core alternates S_{j+2}, P_{j+1} V, ...
//
//   warps 0-3   softmax (one TMEM lane quarter each; P released in two halves as above)
//   warp 4      TMA producer (Q tile, then the chunks in the MMA's order)
//   warp 5      MMA issuer
// ------------------------------------------------------------------------------------------------
constexpr int kT1Threads = 192;
constexpr int kT1Producer = 4;
constexpr int kT1Mma = 5;
constexpr int kT1MaxChunks = 12;
constexpr int kT1ChunkBytes = 16384;
constexpr int kT1QBoxBytes = BM * 128;  // one 128-byte column box of the Q tile

// Geometry by head dim and element size (2: bf16; 1: fp8 e5m2, P in e4m3).  Rows of D * ESZ
// bytes are kBoxes 128-byte column boxes.  A K chunk is one box of a K tile (four 32-byte K
// steps of S); a V chunk holds kVKeys keys of all D dims as kBoxes column groups, kSpc P V K
// steps (16 bf16 or 32 fp8 keys each).  P takes 8 TMEM columns per K step either way.  Each
// half of P (64 keys, released separately by the softmax) is whole V chunks, or (kSpc = all K
// steps of the tile: fp8 D = 128) half of the one V chunk.
template <int D, int ESZ>
struct T1Geo {
  static constexpr int kRowBytes = D * ESZ;
  static constexpr int kBoxElems = 128 / ESZ;
  static constexpr int kBoxes = kRowBytes / 128;
  static constexpr int kQBytes = BM * kRowBytes;
  static constexpr int kVKeys = kT1ChunkBytes / kRowBytes < BN ? kT1ChunkBytes / kRowBytes : BN;
  static constexpr int kVChunks = BN / kVKeys;
  static constexpr int kVGroupBytes = kVKeys * 128;
  static constexpr int kPVKeys = 32 / ESZ;
  static constexpr int kPVSteps = BN / kPVKeys;
  static constexpr int kSpc = kVKeys / kPVKeys;
  static constexpr int kChunks = D == 256 ? 8 : kT1MaxChunks;  // ring slots
  static constexpr int kRingOff = kQBytes;
  static constexpr int kBarOff = kRingOff + kChunks * kT1ChunkBytes;
  static constexpr int kSmemBytes = kBarOff + 1024 + 1024;
  static_assert(kRowBytes >= 128 && kRowBytes % 128 == 0, "rows of whole 128-byte boxes");
  static_assert(kSpc <= kPVSteps / 2 || kSpc == kPVSteps, "P halves and V chunks");
  static_assert(kChunks <= kT1MaxChunks, "barrier arrays");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

struct T1Bars {
  uint64_t full[kT1MaxChunks], empty[kT1MaxChunks];
  uint64_t q_full, q_empty;
  uint64_t s_full[2];  // S_j computed (buffer j & 1)
  uint64_t p_full, p_hi;  // P of keys 0..63 / 64..127 written
  uint64_t pv_done;       // the P V products of the step completed
  uint64_t o_full, o_empty;
  uint32_t tmem_slot;
};
static_assert(sizeof(T1Bars) <= 1024, "barrier block");

template <int D, int ESZ>
__global__ void __launch_bounds__(kT1Threads, 1)
    prefill_1tile_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params p) {
  using G = T1Geo<D, ESZ>;
  constexpr bool F8 = ESZ == 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  T1Bars* bars = reinterpret_cast<T1Bars*>(smem + G::kBarOff);
  uint8_t* ring = smem + G::kRingOff;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kChunks; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->p_hi, 128);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 128);
    fence_barrier_init();
  }
  if (warp == kT1Mma) tmem_alloc(&bars->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  const int rounds = (p.n_items + gridDim.x - 1) / gridDim.x;

  if (warp == kT1Producer) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t ph_qe = 0, ph = 0;
      int slot = 0;
      bool ok = true;
      auto next_slot = [&]() -> uint8_t* {
        if (!(ok = mbar_wait(&bars->empty[slot], ph ^ 1, p.status))) return nullptr;
        mbar_arrive_expect_tx(&bars->full[slot], kT1ChunkBytes);
        return ring + slot * kT1ChunkBytes;
      };
      auto advance = [&]() {
        if (++slot == G::kChunks) { slot = 0; ph ^= 1; }
      };
      for (int r = 0; r < rounds && ok; ++r) {
        const int it = item_for(r, blockIdx.x, gridDim.x);
        if (it >= p.n_items) continue;
        int m, b, hq;
        item_coords(p, it, m, b, hq);
        const int n = kv_tiles_for(p, m * BM);
        if (n == 0) continue;
        const int bhk = b * p.Hkv + hq / p.G;
        if (!(ok = mbar_wait(&bars->q_empty, ph_qe ^ 1, p.status))) break;
        ph_qe ^= 1;
        mbar_arrive_expect_tx(&bars->q_full, G::kQBytes);
#pragma unroll
        for (int bx = 0; bx < G::kBoxes; ++bx)
          tma_load_3d(smem + bx * kT1QBoxBytes, &tmQ, &bars->q_full, bx * G::kBoxElems,
                      m * BM, b * p.Hq + hq);
        // the chunks of K_j: its 128-byte column boxes
        auto load_k = [&](int j) {
          for (int bx = 0; bx < G::kBoxes && ok; ++bx) {
            uint8_t* dst = next_slot();
            if (!dst) return;
            tma_load_3d(dst, &tmK, &bars->full[slot], bx * G::kBoxElems, j * BN, bhk);
            advance();
          }
        };
        // the chunks of V_j: kVKeys keys each, all 256 dims in one 4-D copy
        auto load_v = [&](int j) {
          for (int c = 0; c < G::kVChunks && ok; ++c) {
            uint8_t* dst = next_slot();
            if (!dst) return;
            tma_load_4d(dst, &tmV, &bars->full[slot], 0, j * BN + c * G::kVKeys, 0, bhk);
            advance();
          }
        };
        load_k(0);
        if (n > 1) load_k(1);
        for (int j = 0; j < n && ok; ++j) {
          load_v(j);
          if (j + 2 < n) load_k(j + 2);
        }
      }
    }
  } else if (warp == kT1Mma) {
    // ------------------------------------------------------------------ MMA issuer
    // bf16 (format 1) x bf16, or e5m2 (1) x e5m2 for S and e4m3 (0) P x e5m2 V for P V
    const uint32_t idesc_s = make_idesc(1, 1, false, false, BN, BM);
    const uint32_t idesc_pv = make_idesc(F8 ? 0u : 1u, 1, false, true, D, BM);  // V MN-major
    const uint64_t q_desc0 = smem_desc(smem_u32(smem), 16, 1024, 2);
    const uint64_t r_desc0 = smem_desc(smem_u32(ring), 16, 1024, 2);  // K chunk (K-major)
    const uint64_t v_desc0 = smem_desc(smem_u32(ring), G::kVGroupBytes, 1024, 2);  // V chunk
    uint32_t ph = 0, ph_q = 0, ph_pf = 0, ph_oe = 0;
    int slot = 0;
    bool ok = true;
    auto wait_chunk = [&]() {
      ok = mbar_wait_warp(&bars->full[slot], ph, p.status);
      tc_fence_after();
      return ok;
    };
    auto release_chunk = [&]() {
      umma_commit_e(&bars->empty[slot]);
      if (++slot == G::kChunks) { slot = 0; ph ^= 1; }
    };
    // S_j = Q K_j^T into buffer `buf`: per K chunk (128 bytes of the rows), its four K steps
    auto issue_s = [&](int buf) {
      const uint32_t d = tmem + buf * 128;
      for (int bx = 0; bx < G::kBoxes && ok; ++bx) {
        if (!wait_chunk()) return;
        const uint64_t ad = q_desc0 + static_cast<uint64_t>((bx * kT1QBoxBytes) >> 4);
        const uint64_t bd = r_desc0 + static_cast<uint64_t>((slot * kT1ChunkBytes) >> 4);
        issue_batched<F8, false, 0, 4>(
            d, [&](int kk) { return ad + static_cast<uint64_t>((kk * 32) >> 4); },
            [&](int kk) { return bd + static_cast<uint64_t>((kk * 32) >> 4); }, idesc_s, bx > 0);
        release_chunk();
      }
    };
    // O += P_j V_j for half `h` of P_j (keys 64h..64h+63; P_j: TMEM columns of buffer `buf`,
    // 8 per K step): whole V chunks, or half of the tile's one V chunk
    constexpr int kH = G::kPVSteps / 2;  // K steps per half
    auto issue_pv = [&](int buf, auto hc, bool acc) {
      constexpr int h = decltype(hc)::value;
      const uint32_t pcol = tmem + buf * 128 + h * kH * 8;
      auto b_of = [&](int kin) {
        return v_desc0 + static_cast<uint64_t>((slot * kT1ChunkBytes + kin * G::kPVKeys * 128) >> 4);
      };
      if constexpr (G::kSpc <= kH) {
        for (int c = 0; c < kH / G::kSpc && ok; ++c) {
          if (!wait_chunk()) return;
          issue_batched<F8, true, 0, G::kSpc>(
              tmem + 256, [&](int kk) { return pcol + (c * G::kSpc + kk) * 8; },
              [&](int kk) { return b_of(kk); }, idesc_pv, acc || c > 0);
          release_chunk();
        }
      } else {
        if (h == 0 && !wait_chunk()) return;
        issue_batched<F8, true, h * kH, h * kH + kH>(
            tmem + 256, [&](int kk) { return pcol + (kk - h * kH) * 8; },
            [&](int kk) { return b_of(kk); }, idesc_pv, acc);
        if (h == 1) release_chunk();
      }
    };
    for (int r = 0; r < rounds && ok; ++r) {
      const int it = item_for(r, blockIdx.x, gridDim.x);
      if (it >= p.n_items) continue;
      int m, b, hq;
      item_coords(p, it, m, b, hq);
      const int n = kv_tiles_for(p, m * BM);
      if (n == 0) continue;
      if (!(ok = mbar_wait_warp(&bars->q_full, ph_q, p.status))) break;
      ph_q ^= 1;
      tc_fence_after();
      issue_s(0);
      umma_commit_e(&bars->s_full[0]);
      if (n > 1) {
        issue_s(1);
        umma_commit_e(&bars->s_full[1]);
      }
      if (n <= 2) umma_commit_e(&bars->q_empty);
      for (int j = 0; j < n && ok; ++j) {
        const int buf = j & 1;
        // P_j V_j in halves as the softmax releases them; O is free once the previous item's
        // epilogue has read it
        if (!(ok = mbar_wait_warp(&bars->p_full, ph_pf, p.status))) break;
        if (j == 0) {
          if (!(ok = mbar_wait_warp(&bars->o_empty, ph_oe ^ 1, p.status))) break;
          ph_oe ^= 1;
        }
        tc_fence_after();
        issue_pv(buf, std::integral_constant<int, 0>{}, j > 0);
        if (!ok) break;
        if (!(ok = mbar_wait_warp(&bars->p_hi, ph_pf, p.status))) break;
        ph_pf ^= 1;
        tc_fence_after();
        issue_pv(buf, std::integral_constant<int, 1>{}, true);
        if (!ok) break;
        umma_commit_e(&bars->pv_done);
        if (j == n - 1) umma_commit_e(&bars->o_full);
        // S_{j+2} into this buffer (after P_j V read P_j from it: the tensor core runs in order)
        if (j + 2 < n) {
          issue_s(buf);
          umma_commit_e(&bars->s_full[buf]);
          if (j + 2 == n - 1) umma_commit_e(&bars->q_empty);
        }
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------------ softmax warpgroup
    const int lrow = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + lane_off + 256;
    uint32_t ph_s[2] = {0, 0}, ph_o = 0, ph_pv = 0;
    bool ok = true;
    for (int r = 0; r < rounds && ok; ++r) {
      const int it = item_for(r, blockIdx.x, gridDim.x);
      if (it >= p.n_items) continue;
      int m, b, hq;
      item_coords(p, it, m, b, hq);
      const int r0 = m * BM;
      const int n = kv_tiles_for(p, r0);
      if (n == 0) continue;
      const int row = r0 + lrow;
      float m_run = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        const int buf = j & 1;
        const uint32_t tS = tmem + lane_off + buf * 128;
        if (!(ok = mbar_wait(&bars->s_full[buf], ph_s[buf], p.status))) break;
        ph_s[buf] ^= 1;
        tc_fence_after();
        const bool need_mask = (p.causal && j * BN + BN - 1 > r0 + p.off) || (j * BN + BN > p.Skv);
        const int lim = (p.causal ? min(row + p.off + 1, p.Skv) : p.Skv) - j * BN;
        uint32_t sr[128];
        tmem_ld128(tS, sr);
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 128; ++e)
            if (e >= lim) sr[e] = __float_as_uint(-INFINITY);
        }
        float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
        for (int e = 0; e < 128; e += 8) {
          a0 = fmax3(a0, __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
          a1 = fmax3(a1, __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
          a2 = fmax3(a2, __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
          a3 = fmax3(a3, __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
        }
        const float m_tile = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * p.c_log2;
        float f = 1.f;
        if (j == 0) {
          m_run = m_tile;
        } else if (m_tile > m_run + kRescaleThreshold) {
          f = fast_exp2(m_run - m_tile);
          l *= f;
          m_run = m_tile;
        }
        const float2 c2 = make_float2(p.c_log2, p.c_log2);
        const float2 nm2 = make_float2(-m_run, -m_run);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[F8 ? 16 : 32];  // 64 keys: packed bf16 pairs or e4m3 quads
#pragma unroll
          for (int e = 64 * h; e < 64 * h + 64; e += 8) {
            float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), c2, nm2);
            float2 x1 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), c2, nm2);
            float2 x2 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5])), c2, nm2);
            float2 x3 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7])), c2, nm2);
            x0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
            x1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
            x2 = make_float2(fast_exp2(x2.x), fast_exp2(x2.y));
            x3 = make_float2(fast_exp2(x3.x), fast_exp2(x3.y));
            acc0 = __fadd2_rn(acc0, x0);
            acc1 = __fadd2_rn(acc1, x1);
            acc2 = __fadd2_rn(acc2, x2);
            acc3 = __fadd2_rn(acc3, x3);
            const int w = e - 64 * h;
            if constexpr (F8) {
              // e4m3, four keys per TMEM column, lowest key in the lowest byte
              pk[w / 4] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x0, __NV_SATFINITE, __NV_E4M3)) |
                          (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x1, __NV_SATFINITE, __NV_E4M3)) << 16);
              pk[w / 4 + 1] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x2, __NV_SATFINITE, __NV_E4M3)) |
                              (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(x3, __NV_SATFINITE, __NV_E4M3)) << 16);
            } else {
              pk[w / 2] = pack_bf16(x0.x, x0.y);
              pk[w / 2 + 1] = pack_bf16(x1.x, x1.y);
              pk[w / 2 + 2] = pack_bf16(x2.x, x2.y);
              pk[w / 2 + 3] = pack_bf16(x3.x, x3.y);
            }
          }
          if (h == 0 && j > 0) {
            // P_{j-1} V has completed: O holds the tiles before j; rescale it (warp-uniformly,
            // eight columns at a time) before P_j V accumulates onto it
            if (!(ok = mbar_wait(&bars->pv_done, ph_pv, p.status))) break;
            ph_pv ^= 1;
            tc_fence_after();
            if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll 1
              for (int c = 0; c < D / 8; ++c) {
                uint32_t ov[8];
                tmem_ld8(tO + c * 8, ov);
#pragma unroll
                for (int e = 0; e < 8; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
                tmem_st8(tO + c * 8, ov);
              }
            }
          }
          if constexpr (F8)
            tmem_st16(tS + 16 * h, pk);
          else
            tmem_st32(tS + 32 * h, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(h ? &bars->p_hi : &bars->p_full);
        }
        if (!ok) break;
        const float2 accs = __fadd2_rn(__fadd2_rn(acc0, acc1), __fadd2_rn(acc2, acc3));
        l += accs.x + accs.y;
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, LSE.  The item's last pv_done completes with o_full: consume
      // it here, so that the phase the next item waits for is never two phases ahead
      if (!(ok = mbar_wait(&bars->o_full, ph_o, p.status))) break;
      ph_o ^= 1;
      if (!(ok = mbar_wait(&bars->pv_done, ph_pv, p.status))) break;
      ph_pv ^= 1;
      tc_fence_after();
      const float inv = p.v_scale / l;
      __nv_bfloat16* orow = p.o + ((static_cast<size_t>(b) * p.Hq + hq) * p.S + row) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + c * 32, ov);
        if (row < p.S) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(ov[q4 * 8 + 0]) * inv, __uint_as_float(ov[q4 * 8 + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(ov[q4 * 8 + 2]) * inv, __uint_as_float(ov[q4 * 8 + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(ov[q4 * 8 + 4]) * inv, __uint_as_float(ov[q4 * 8 + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(ov[q4 * 8 + 6]) * inv, __uint_as_float(ov[q4 * 8 + 7]) * inv);
            dst[q4] = w;
          }
        }
      }
      if (p.lse && row < p.S)
        p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.S + row] = (m_run + log2f(l)) * kLn2;
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kT1Mma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int RM, int ESZ, int NTT>
attn_status_t launch_typed(const void* q, const void* k, const void* v, void* o, float* lse,
                           float q_scale, float k_scale, float v_scale, int B, int Hq, int Hkv,
                           int S, int Skv, int kv_pitch, int causal, float scale,
                           const float2* table, int rope_k, int pos0, cudaStream_t st) {
  constexpr bool STAGED = ESZ == 1 && RM == 1;
  using C = Cfg<D, ESZ, STAGED, NTT>;
  // Q / K boxes: as the MMA reads them, or (STAGED) the fp8 staging tiles; V in its own geometry
  constexpr int kQKBoxElems = STAGED ? D : C::kBoxElems;
  constexpr int kQKSwz = STAGED ? 128 : C::kSwz;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_3d(&tq, q, ESZ, D, S, static_cast<uint64_t>(B) * Hq, kQKBoxElems, BM, kQKSwz) ||
      !make_tmap_3d(&tk, k, ESZ, D, Skv, static_cast<uint64_t>(B) * Hkv, kQKBoxElems, BN, kQKSwz,
                    kv_pitch) ||
      !make_tmap_3d(&tv, v, ESZ, D, Skv, static_cast<uint64_t>(B) * Hkv, C::kVBoxElems, BN,
                    C::kVSwz, kv_pitch))
    return ATTN_ERR_CUDA;
  Params p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.status = device_status_ptr();
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.S = S;
  p.Skv = Skv;
  p.off = Skv - S;
  p.rope_k = rope_k;
  p.causal = causal;
  constexpr int kRowsPerItem = NTT * BM;
  p.nM = (S + kRowsPerItem - 1) / kRowsPerItem;
  p.nKV = (Skv + BN - 1) / BN;
  p.n_items = p.nM * B * Hq;
  // causal, long prompts (more than 16 query-block levels, where the K/V streams outgrow L2):
  // blocks of levels give each stream at least 16 items per block while keeping the heaviest
  // levels first.  Shorter causal prompts keep one level per block, i.e. the plain
  // heaviest-first order the serpentine deal balances best (their K/V fit in L2 anyway).
  // Without the mask every item weighs the same: all levels of a stream run together.
  p.mblk = causal ? (p.nM > 16 ? std::max(1, 16 / p.G) : 1) : p.nM;
  p.c_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
  p.v_scale = v_scale;
  p.table = table;
  p.pos0 = pos0;
  auto kern = prefill_kernel<D, RM, ESZ, NTT>;
  if (!set_smem_attr(reinterpret_cast<const void*>(kern), C::kSmemBytes)) return ATTN_ERR_CUDA;
  const int grid = std::min(p.n_items, sm_count());
  kern<<<grid, threads_for(RM), C::kSmemBytes, st>>>(tq, tk, tv, p);
  return launch_status();
}

// one Q tile per item (bf16, or fp8 e5m2), no in-kernel RoPE (the rotation passes serve bf16)
template <int D, int ESZ>
attn_status_t launch_1tile(const void* q, const void* k, const void* v, void* o, float* lse,
                          float q_scale, float k_scale, float v_scale, int B, int Hq, int Hkv,
                          int S, int Skv, int kv_pitch, int causal, float scale, cudaStream_t st) {
  using G = T1Geo<D, ESZ>;
  const uint64_t pitch = kv_pitch ? static_cast<uint64_t>(kv_pitch) : static_cast<uint64_t>(Skv);
  CUtensorMap tq, tk, tv;
  // V as {128 bytes of a row, key, 128-byte column group, (batch, KV head)}: one box = a chunk
  const uint64_t vdims[4] = {static_cast<uint64_t>(G::kBoxElems), static_cast<uint64_t>(Skv),
                             static_cast<uint64_t>(G::kBoxes), static_cast<uint64_t>(B) * Hkv};
  const uint64_t vstrides[3] = {static_cast<uint64_t>(G::kRowBytes), 128,
                                pitch * G::kRowBytes};
  const uint32_t vbox[4] = {static_cast<uint32_t>(G::kBoxElems), static_cast<uint32_t>(G::kVKeys),
                            static_cast<uint32_t>(G::kBoxes), 1};
  if (!make_tmap_3d(&tq, q, ESZ, D, S, static_cast<uint64_t>(B) * Hq, G::kBoxElems, BM, 128) ||
      !make_tmap_3d(&tk, k, ESZ, D, Skv, static_cast<uint64_t>(B) * Hkv, G::kBoxElems, BN, 128,
                    kv_pitch) ||
      !make_tmap_4d(&tv, v, ESZ, vdims, vstrides, vbox))
    return ATTN_ERR_CUDA;
  Params p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.status = device_status_ptr();
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.S = S;
  p.Skv = Skv;
  p.off = Skv - S;
  p.rope_k = 0;
  p.causal = causal;
  p.nM = (S + BM - 1) / BM;
  p.nKV = (Skv + BN - 1) / BN;
  p.n_items = p.nM * B * Hq;
  p.mblk = causal ? (p.nM > 16 ? std::max(1, 16 / p.G) : 1) : p.nM;
  p.c_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
  p.v_scale = v_scale;
  p.table = nullptr;
  p.pos0 = 0;
  auto kern = prefill_1tile_kernel<D, ESZ>;
  if (!set_smem_attr(reinterpret_cast<const void*>(kern), G::kSmemBytes)) return ATTN_ERR_CUDA;
  const int grid = std::min(p.n_items, sm_count());
  kern<<<grid, kT1Threads, G::kSmemBytes, st>>>(tq, tk, tv, p);
  return launch_status();
}

std::atomic<int> g_forced_tiles{0};  // Q tiles per item for D <= 128 (0: the default, two)

}  // namespace

void force_prefill_tiles(int q_tiles) { g_forced_tiles.store(q_tiles); }

attn_status_t launch_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                             attn_dtype_t dt, float q_scale, float k_scale, float v_scale, int B,
                             int Hq, int Hkv, int S, int Skv, int kv_pitch, int D, int causal,
                             float scale, const float2* table, int rope_k, int pos0,
                             cudaStream_t st) {
  const int esz = dt == ATTN_BF16 ? 2 : 1;
  const int rm = table == nullptr ? 0 : 1;
  const int nt = D >= 256 ? 1 : (g_forced_tiles.load() == 1 ? 1 : 2);
#define ATTN_PREFILL_CASE(DD, RR, EE, NN)                                                    \
  if (D == DD && rm == RR && esz == EE && nt == NN)                                          \
    return launch_typed<DD, RR, EE, NN>(q, k, v, o, lse, q_scale, k_scale, v_scale, B, Hq,   \
                                        Hkv, S, Skv, kv_pitch, causal, scale, table, rope_k, \
                                        pos0, st);
  ATTN_PREFILL_CASE(128, 0, 2, 2)
  if (D == 256 && rm == 0)
    return esz == 2 ? launch_1tile<256, 2>(q, k, v, o, lse, q_scale, k_scale, v_scale, B, Hq, Hkv,
                                           S, Skv, kv_pitch, causal, scale, st)
                    : launch_1tile<256, 1>(q, k, v, o, lse, q_scale, k_scale, v_scale, B, Hq, Hkv,
                                           S, Skv, kv_pitch, causal, scale, st);
  ATTN_PREFILL_CASE(128, 1, 2, 2)
  ATTN_PREFILL_CASE(64, 0, 2, 2)
  ATTN_PREFILL_CASE(64, 1, 2, 2)
  ATTN_PREFILL_CASE(128, 0, 1, 2)
  ATTN_PREFILL_CASE(64, 0, 1, 2)
  ATTN_PREFILL_CASE(128, 1, 1, 2)
  // one Q tile per item (128-row items)
  ATTN_PREFILL_CASE(128, 0, 2, 1)
  ATTN_PREFILL_CASE(128, 1, 2, 1)
  ATTN_PREFILL_CASE(64, 0, 2, 1)
  ATTN_PREFILL_CASE(64, 1, 2, 1)
  ATTN_PREFILL_CASE(128, 0, 1, 1)
  ATTN_PREFILL_CASE(64, 0, 1, 1)
  ATTN_PREFILL_CASE(128, 1, 1, 1)
#undef ATTN_PREFILL_CASE
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
