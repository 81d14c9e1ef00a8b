// rope.cu — rope_apply: the unfused rotary position embedding pass over a [B,H,S,D] tensor.
//
// Row r = ((b*H + h)*S + s) is rotated at position pos0 + s: each pair (x_i, x_{i+D/2}) becomes
// (x_i c - x_{i+D/2} s, x_{i+D/2} c + x_i s) with (c, s) = table[pos][i].  The pass is HBM
// bound (every element read and written once); each thread moves 16-byte chunks of the first
// half of a row and the matching chunks of the second half, fully coalesced.  The interleaved
// convention pairs (x_{2i}, x_{2i+1}) with the same (c, s) = table[pos][i]; a 16-byte chunk then
// holds whole pairs.
#include "common.cuh"

namespace attn {
namespace {

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;  // elements per 16-byte chunk
  __device__ static void load(const void* p, float* f) {
    unpack(__ldg(reinterpret_cast<const uint4*>(p)), f);
  }
  __device__ static void unpack(const uint4& u, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 t = __bfloat1622float2(h[j]);
      f[2 * j] = t.x;
      f[2 * j + 1] = t.y;
    }
  }
  __device__ static void store(void* p, const float* f) {
    uint4 u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = pack_bf16(f[2 * j], f[2 * j + 1]);
    *reinterpret_cast<uint4*>(p) = u;
  }
  __device__ static float load1(const void* p, int i) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  }
  __device__ static void store1(void* p, int i, float f) {
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(f);
  }
};
template <>
struct Vec<__nv_fp8_e5m2> {
  static constexpr int N = 16;
  __device__ static void load(const void* p, float* f) {
    unpack(__ldg(reinterpret_cast<const uint4*>(p)), f);
  }
  __device__ static void unpack(const uint4& u, float* f) {
    const __nv_fp8x2_e5m2* h = reinterpret_cast<const __nv_fp8x2_e5m2*>(&u);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float2 t = static_cast<float2>(h[j]);
      f[2 * j] = t.x;
      f[2 * j + 1] = t.y;
    }
  }
  __device__ static void store(void* p, const float* f) {
    uint4 u;
    __nv_fp8x2_storage_t* w = reinterpret_cast<__nv_fp8x2_storage_t*>(&u);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      w[j] = __nv_cvt_float2_to_fp8x2(make_float2(f[2 * j], f[2 * j + 1]), __NV_SATFINITE,
                                      __NV_E5M2);
    *reinterpret_cast<uint4*>(p) = u;
  }
  __device__ static float load1(const void* p, int i) {
    return static_cast<float>(reinterpret_cast<const __nv_fp8_e5m2*>(p)[i]);
  }
  __device__ static void store1(void* p, int i, float f) {
    reinterpret_cast<__nv_fp8_e5m2*>(p)[i] = __nv_fp8_e5m2(f);
  }
};

// One thread per (row, 16-byte chunk of the first half).
template <typename T>
__global__ void __launch_bounds__(256) rope_vec_kernel(const T* __restrict__ x, T* y,
                                                       long long rows, int S, int D, int pos0,
                                                       const float2* __restrict__ table, float sgn) {
  constexpr int N = Vec<T>::N;
  const int half = D / 2;
  const int chunks = half / N;
  const long long total = rows * chunks;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long row = t / chunks;
    const int i0 = static_cast<int>(t - row * chunks) * N;
    const int pos = pos0 + static_cast<int>(row % S);
    const T* xr = x + row * D;
    T* yr = y + row * D;
    float a[N], b[N];
    Vec<T>::load(xr + i0, a);
    Vec<T>::load(xr + half + i0, b);
    const float2* cs = table + static_cast<long long>(pos) * half + i0;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      const float2 r = __ldg(cs + j);
      const float sn = r.y * sgn;
      const float a1 = a[j] * r.x - b[j] * sn;
      const float b1 = b[j] * r.x + a[j] * sn;
      a[j] = a1;
      b[j] = b1;
    }
    Vec<T>::store(yr + i0, a);
    Vec<T>::store(yr + half + i0, b);
  }
}

// One thread per (sequence b, position s, 16-byte chunk pair): its cos/sin are read once and
// applied to that chunk pair in all H heads, HU heads at a time so several loads are in flight.
// Consecutive threads take consecutive chunks of a row, then the next position, so every warp
// access covers whole rows of one head.
template <typename T, int HU>
__global__ void __launch_bounds__(256, 2) rope_pos_kernel(const T* __restrict__ x, T* y, int B,
                                                       int H, int S, int D, int pos0,
                                                       const float2* __restrict__ table, float sgn) {
  constexpr int N = Vec<T>::N;
  const int half = D / 2;
  const int chunks = half / N;
  const long long total = static_cast<long long>(B) * S * chunks;
  const size_t head_stride = static_cast<size_t>(S) * D;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long bs = t / chunks;
    const int i0 = static_cast<int>(t - bs * chunks) * N;
    const int s = static_cast<int>(bs % S);
    const long long b = bs / S;
    float2 r[N];
    const float2* cs = table + static_cast<long long>(pos0 + s) * half + i0;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      r[j] = __ldg(cs + j);
      r[j].y *= sgn;
    }
    const size_t row0 = (static_cast<size_t>(b) * H * S + s) * D + i0;
    for (int h = 0; h < H; h += HU) {
      uint4 ra[HU], rc[HU];  // raw chunks: all loads of the batch go out before any use
#pragma unroll
      for (int u = 0; u < HU; ++u)
        if (h + u < H) {
          const T* xr = x + row0 + static_cast<size_t>(h + u) * head_stride;
          ra[u] = __ldg(reinterpret_cast<const uint4*>(xr));
          rc[u] = __ldg(reinterpret_cast<const uint4*>(xr + half));
        }
#pragma unroll
      for (int u = 0; u < HU; ++u)
        if (h + u < H) {
          float a[N], c[N];
          Vec<T>::unpack(ra[u], a);
          Vec<T>::unpack(rc[u], c);
#pragma unroll
          for (int j = 0; j < N; ++j) {
            const float a1 = a[j] * r[j].x - c[j] * r[j].y;
            const float c1 = c[j] * r[j].x + a[j] * r[j].y;
            a[j] = a1;
            c[j] = c1;
          }
          T* yr = y + row0 + static_cast<size_t>(h + u) * head_stride;
          Vec<T>::store(yr, a);
          Vec<T>::store(yr + half, c);
        }
    }
  }
}

// Any even D: one thread per pair.
template <typename T>
__global__ void __launch_bounds__(256) rope_pair_kernel(const T* __restrict__ x, T* y,
                                                        long long rows, int S, int D, int pos0,
                                                        const float2* __restrict__ table, float sgn) {
  const int half = D / 2;
  const long long total = rows * half;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long row = t / half;
    const int i = static_cast<int>(t - row * half);
    const int pos = pos0 + static_cast<int>(row % S);
    const float2 r = table[static_cast<long long>(pos) * half + i];
    const float sn = r.y * sgn;
    const float a = Vec<T>::load1(x + row * D, i);
    const float b = Vec<T>::load1(x + row * D, i + half);
    Vec<T>::store1(y + row * D, i, a * r.x - b * sn);
    Vec<T>::store1(y + row * D, i + half, b * r.x + a * sn);
  }
}

// Interleaved pairs, one thread per (sequence b, position s, 16-byte chunk): the chunk's N/2
// pairs take table[pos][c*N/2 ..]; heads HU at a time as in rope_pos_kernel.
template <typename T, int HU>
__global__ void __launch_bounds__(256, 2) rope_il_pos_kernel(const T* __restrict__ x, T* y, int B,
                                                          int H, int S, int D, int pos0,
                                                          const float2* __restrict__ table,
                                                          float sgn) {
  constexpr int N = Vec<T>::N;
  const int chunks = D / N;
  const long long total = static_cast<long long>(B) * S * chunks;
  const size_t head_stride = static_cast<size_t>(S) * D;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long bs = t / chunks;
    const int c = static_cast<int>(t - bs * chunks);
    const int s = static_cast<int>(bs % S);
    const long long b = bs / S;
    float2 r[N / 2];
    const float2* cs = table + static_cast<long long>(pos0 + s) * (D / 2) + c * (N / 2);
#pragma unroll
    for (int j = 0; j < N / 2; ++j) {
      r[j] = __ldg(cs + j);
      r[j].y *= sgn;
    }
    const size_t row0 = (static_cast<size_t>(b) * H * S + s) * D + c * N;
    for (int h = 0; h < H; h += HU) {
      uint4 ra[HU];
#pragma unroll
      for (int u = 0; u < HU; ++u)
        if (h + u < H)
          ra[u] = __ldg(reinterpret_cast<const uint4*>(x + row0 + static_cast<size_t>(h + u) * head_stride));
#pragma unroll
      for (int u = 0; u < HU; ++u)
        if (h + u < H) {
          float a[N];
          Vec<T>::unpack(ra[u], a);
#pragma unroll
          for (int j = 0; j < N / 2; ++j) {
            const float e = a[2 * j], o = a[2 * j + 1];
            a[2 * j] = e * r[j].x - o * r[j].y;
            a[2 * j + 1] = o * r[j].x + e * r[j].y;
          }
          Vec<T>::store(y + row0 + static_cast<size_t>(h + u) * head_stride, a);
        }
    }
  }
}

// Interleaved pairs, any even D: one thread per pair.
template <typename T>
__global__ void __launch_bounds__(256) rope_il_pair_kernel(const T* __restrict__ x, T* y,
                                                           long long rows, int S, int D, int pos0,
                                                           const float2* __restrict__ table,
                                                           float sgn) {
  const int half = D / 2;
  const long long total = rows * half;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const long long row = t / half;
    const int i = static_cast<int>(t - row * half);
    const int pos = pos0 + static_cast<int>(row % S);
    const float2 r = table[static_cast<long long>(pos) * half + i];
    const float sn = r.y * sgn;
    const float e = Vec<T>::load1(x + row * D, 2 * i);
    const float o = Vec<T>::load1(x + row * D, 2 * i + 1);
    Vec<T>::store1(y + row * D, 2 * i, e * r.x - o * sn);
    Vec<T>::store1(y + row * D, 2 * i + 1, o * r.x + e * sn);
  }
}

template <typename T>
attn_status_t launch_typed_il(const void* x, void* y, int B, int H, int S, int D, int pos0,
                              const float2* table, float sgn, cudaStream_t st) {
  const int sms = sm_count();
  const int threads = 256;
  const long long cap = static_cast<long long>(sms) * 16;
  if (D % Vec<T>::N == 0) {
    const long long work = static_cast<long long>(B) * S * (D / Vec<T>::N);
    long long blocks = (work + threads - 1) / threads;
    if (blocks > cap) blocks = cap;
    // one 16-byte chunk per head (the half-split form moves two): twice the heads per batch
    // keep as many loads in flight
    constexpr int HU = Vec<T>::N == 8 ? 8 : 4;
    rope_il_pos_kernel<T, HU><<<static_cast<int>(blocks), threads, 0, st>>>(
        static_cast<const T*>(x), static_cast<T*>(y), B, H, S, D, pos0, table, sgn);
  } else {
    const long long rows = static_cast<long long>(B) * H * S;
    long long blocks = (rows * (D / 2) + threads - 1) / threads;
    if (blocks > cap) blocks = cap;
    rope_il_pair_kernel<T><<<static_cast<int>(blocks), threads, 0, st>>>(
        static_cast<const T*>(x), static_cast<T*>(y), rows, S, D, pos0, table, sgn);
  }
  return launch_status();
}

template <typename T>
attn_status_t launch_typed(const void* x, void* y, int B, int H, int S, int D, int pos0,
                           const float2* table, float sgn, cudaStream_t st) {
  const long long rows = static_cast<long long>(B) * H * S;
  const int sms = sm_count();
  const int threads = 256;
  if ((D / 2) % Vec<T>::N == 0 && H >= 4) {
    const long long work = static_cast<long long>(B) * S * ((D / 2) / Vec<T>::N);
    long long blocks = (work + threads - 1) / threads;
    const long long cap = static_cast<long long>(sms) * 16;
    if (blocks > cap) blocks = cap;
    constexpr int HU = Vec<T>::N == 8 ? 4 : 2;
    rope_pos_kernel<T, HU><<<static_cast<int>(blocks), threads, 0, st>>>(
        static_cast<const T*>(x), static_cast<T*>(y), B, H, S, D, pos0, table, sgn);
  } else if ((D / 2) % Vec<T>::N == 0) {
    const long long work = rows * ((D / 2) / Vec<T>::N);
    long long blocks = (work + threads - 1) / threads;
    const long long cap = static_cast<long long>(sms) * 16;
    if (blocks > cap) blocks = cap;
    rope_vec_kernel<T><<<static_cast<int>(blocks), threads, 0, st>>>(
        static_cast<const T*>(x), static_cast<T*>(y), rows, S, D, pos0, table, sgn);
  } else {
    const long long work = rows * (D / 2);
    long long blocks = (work + threads - 1) / threads;
    const long long cap = static_cast<long long>(sms) * 16;
    if (blocks > cap) blocks = cap;
    rope_pair_kernel<T><<<static_cast<int>(blocks), threads, 0, st>>>(
        static_cast<const T*>(x), static_cast<T*>(y), rows, S, D, pos0, table, sgn);
  }
  return launch_status();
}

}  // namespace

attn_status_t launch_rope(const void* x, void* y, attn_dtype_t dt, int B, int H, int S, int D,
                          int pos0, const float2* table, int interleaved, cudaStream_t st,
                          int inverse) {
  const float sgn = inverse ? -1.f : 1.f;  // the inverse rotation: sines negated
  if (interleaved) {
    if (dt == ATTN_BF16)
      return launch_typed_il<__nv_bfloat16>(x, y, B, H, S, D, pos0, table, sgn, st);
    return launch_typed_il<__nv_fp8_e5m2>(x, y, B, H, S, D, pos0, table, sgn, st);
  }
  if (dt == ATTN_BF16) return launch_typed<__nv_bfloat16>(x, y, B, H, S, D, pos0, table, sgn, st);
  return launch_typed<__nv_fp8_e5m2>(x, y, B, H, S, D, pos0, table, sgn, st);
}

}  // namespace attn
