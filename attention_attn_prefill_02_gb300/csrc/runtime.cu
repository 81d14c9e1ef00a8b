// runtime.cu — host-side runtime support: device status word, device checks, the cached RoPE
// cos/sin tables and TMA descriptor encoding through the driver entry point (so the library
// links only the static CUDA runtime and loads on machines without a GPU driver).
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "common.cuh"

namespace attn {

__device__ unsigned int g_status_word;

unsigned int* device_status_ptr() {
  static std::mutex mu;
  static std::map<int, unsigned int*> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  cache[dev] = static_cast<unsigned int*>(p);
  return static_cast<unsigned int*>(p);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

attn_status_t check_device() {
  int n = 0;
  cudaError_t e = cudaGetDeviceCount(&n);
  if (e != cudaSuccess || n == 0) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return ATTN_ERR_NO_DEVICE;
  return major == 10 ? ATTN_OK : ATTN_ERR_NO_DEVICE;
}

bool set_smem_attr(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int>, int> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_tuple(kernel, dev);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  done[key] = bytes;
  return true;
}

// ---------------------------------------------------------------------------------------------
// RoPE tables
// ---------------------------------------------------------------------------------------------

namespace {
struct RopeEntry {
  float2* ptr = nullptr;
  int npos = 0;
};
std::mutex g_rope_mu;
std::map<std::tuple<int, int, uint32_t>, RopeEntry> g_rope;
std::vector<float2*> g_rope_retired;  // grown-out tables stay alive: kernels may still read them
}  // namespace

const float2* rope_table_find(int D, float theta, int npos) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  uint32_t tbits;
  memcpy(&tbits, &theta, 4);
  std::lock_guard<std::mutex> lk(g_rope_mu);
  auto it = g_rope.find(std::make_tuple(dev, D, tbits));
  if (it == g_rope.end() || !it->second.ptr || it->second.npos < npos) return nullptr;
  return it->second.ptr;
}

const float2* rope_table(int D, float theta, int npos, attn_status_t* err) {
  *err = ATTN_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *err = ATTN_ERR_NO_DEVICE;
    return nullptr;
  }
  uint32_t tbits;
  memcpy(&tbits, &theta, 4);
  std::lock_guard<std::mutex> lk(g_rope_mu);
  RopeEntry& ent = g_rope[std::make_tuple(dev, D, tbits)];
  if (ent.ptr && ent.npos >= npos) return ent.ptr;
  int want = 4096;
  while (want < npos) want *= 2;
  const int half = D / 2;
  std::vector<float2> host(static_cast<size_t>(want) * half);
  std::vector<double> inv(half);
  for (int i = 0; i < half; ++i) inv[i] = std::pow(static_cast<double>(theta), -2.0 * i / D);
  for (int p = 0; p < want; ++p)
    for (int i = 0; i < half; ++i) {
      const double a = static_cast<double>(p) * inv[i];
      host[static_cast<size_t>(p) * half + i] =
          make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
    }
  float2* dptr = nullptr;
  if (cudaMalloc(&dptr, host.size() * sizeof(float2)) != cudaSuccess) {
    cudaGetLastError();
    *err = ATTN_ERR_CUDA;
    return nullptr;
  }
  if (cudaMemcpy(dptr, host.data(), host.size() * sizeof(float2), cudaMemcpyHostToDevice) !=
      cudaSuccess) {
    cudaFree(dptr);
    *err = ATTN_ERR_CUDA;
    return nullptr;
  }
  if (ent.ptr) g_rope_retired.push_back(ent.ptr);
  ent.ptr = dptr;
  ent.npos = want;
  return dptr;
}

// ---------------------------------------------------------------------------------------------
// TMA descriptors
// ---------------------------------------------------------------------------------------------

namespace {
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn encode_fn() {
  static EncodeFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeFn>(p);
  }();
  return fn;
}
}  // namespace

bool make_tmap_3d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner,
                  uint64_t mid, uint64_t outer, uint32_t box_inner, uint32_t box_mid,
                  int swizzle_bytes, uint64_t mid_pitch) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  if (mid_pitch == 0) mid_pitch = mid;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * elem_bytes, inner * mid_pitch * elem_bytes};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                          : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_4d(CUtensorMap* map, const void* base, int elem_bytes, const uint64_t dims[4],
                  const uint64_t strides[3], const uint32_t box[4]) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t s[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(map, dt, 4, const_cast<void*>(base), d, s, bx, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace attn
