// static_scratch.cu -- fixed device scratch for callers that cannot allocate.
//
// fp8rl_gemm_blockscaled_ws needs a workspace from its caller.  Some callers
// have no device allocator of their own (plain C code linked against this
// library without a framework that manages device memory), or must not
// allocate on their path (an allocation can synchronise the device, or fail
// under memory pressure in a long-running serving loop).  For them,
// fp8rl_gemm_blockscaled_static uses this array instead: a file-scope device
// variable, created when this module is loaded, never allocated or freed by a
// call.  It lives in a translation unit of its own.  With lazy module loading
// (CUDA_MODULE_LOADING=LAZY, the CUDA 12 default) a process that never calls
// that entry point does not load it; with CUDA_MODULE_LOADING=EAGER every
// device the process uses holds the 24 MiB from the time the library loads.
#include <mutex>

#include "common.cuh"

namespace fp8rl {

// Capacity: the stream-K layout for one 128 x 256 fp32 partial tile per SM
// plus header and flags is 19.9 MB on a 152-SM GB300; 24 MiB leaves room for
// that and nothing more is needed.
constexpr size_t kStaticScratchBytes = size_t(24) << 20;

static __device__ __align__(256) uint8_t g_gemm_scratch[kStaticScratchBytes];

// Device address of the scratch in the current context, or null (*status
// says why).  The first call on each device (and again after the device's
// context was replaced, e.g. by cudaDeviceReset), with that device current,
// looks the array up and zeroes its first `clear_bytes` (the stream-K header
// and flags, which must start at zero); later calls return the cached address.
// need_bytes above the capacity is rejected with FP8RL_ERR_UNSUPPORTED.
void* static_gemm_scratch(size_t need_bytes, size_t clear_bytes, fp8rl_status* status) {
  static std::mutex mu;
  static void* cache[64] = {};
  static uint64_t cache_ctx[64] = {};
  *status = FP8RL_OK;
  if (need_bytes > kStaticScratchBytes || clear_bytes > need_bytes) {
    *status = FP8RL_ERR_UNSUPPORTED;
    return nullptr;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *status = FP8RL_ERR_CUDA;
    return nullptr;
  }
  const uint64_t ctx = current_context_id();
  if (!ctx) {
    *status = FP8RL_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev] || cache_ctx[dev] != ctx) {
    cache[dev] = nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gemm_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      *status = FP8RL_ERR_CUDA;
      return nullptr;
    }
    if (cudaMemset(p, 0, clear_bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      *status = FP8RL_ERR_CUDA;
      return nullptr;
    }
    cache[dev] = p;
    cache_ctx[dev] = ctx;
  }
  return cache[dev];
}

}  // namespace fp8rl
