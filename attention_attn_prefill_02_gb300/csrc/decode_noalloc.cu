// decode_noalloc.cu — attn_decode_noalloc: the split-KV decode with its scratch memory in a
// fixed, file-scope device array instead of a caller workspace, for callers that cannot
// allocate device memory when they call (see include/attn.h for who they are).
//
// The split partials live in g_decode_scratch (kNoAllocScratchBytes).  Host code cannot take
// that array's address directly (its name is a host-side stand-in), so the first call on each
// device looks the device address up with cudaGetSymbolAddress, with that device current, and
// caches it.  The kernels themselves are the same as attn_decode's.
#include <cmath>
#include <map>
#include <mutex>

#include "common.cuh"

namespace attn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch on the current device; resolved once per device.
void* scratch_address(attn_status_t* err) {
  static std::mutex mu;
  static std::map<int, void*> addr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    *err = ATTN_ERR_NO_DEVICE;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  auto it = addr.find(dev);
  if (it != addr.end()) return it->second;
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    *err = ATTN_ERR_CUDA;
    return nullptr;
  }
  addr[dev] = p;
  return p;
}

bool finite_pos(float x) { return std::isfinite(x) && x > 0.f; }

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" ATTN_API attn_status_t attn_decode_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cache_len, int Lmax,
    void* o, float* lse, attn_dtype_t dtype, int B, int Hq, int Hkv, int D, float softmax_scale,
    int rope, float rope_theta, attn_stream_t stream) {
  if (!q || !k_cache || !v_cache || !cache_len || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cache_len) & 3u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP8_E5M2) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  int il = 0;
  if (!split_rope_arg(rope, 1, &rope, &il)) return ATTN_ERR_INVALID_ARG;
  if (rope && !finite_pos(rope_theta)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16 || dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(Lmax) > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  const DecodePlan plan = plan_decode(B, Hq, Hkv, D, Lmax);
  if (plan.ws_bytes > kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
  const float2* tab = nullptr;
  if (rope) {
    tab = rope_table_find(D, rope_theta, Lmax + 1);  // never builds a table here
    if (!tab) return ATTN_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if (plan.ws_bytes > 0) {
    scratch = scratch_address(&st);
    if (!scratch) return st;
  }
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  return launch_decode(q, k_cache, v_cache, cache_len, Lmax, o, lse, B, Hq, Hkv, D, scale, tab,
                       il, scratch, plan, reinterpret_cast<cudaStream_t>(stream));
}
