// api.cu -- status reporting of the C ABI and the device error word.
//
// Kernels that wait on mbarriers bound every wait; when one runs out they set
// a bit in this word and leave through their normal teardown (no trap), so
// the CUDA context stays usable.  fp8rl_sync_status() reads and clears it.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace fp8rl {

// one word per device that loads the library (a module-scope variable: no
// allocation is ever made for it)
static __device__ uint32_t g_error_word;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

uint64_t current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return 0;
  if (!ctx) {
    // no context on this thread yet: cudaSetDevice makes the current device's
    // primary context current (CUDA 12 and later)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return static_cast<uint64_t>(id) + 1;
}

// device address of the error word in the current context (cached per device
// together with the context it was looked up in)
uint32_t* device_error_word() {
  static std::mutex mu;
  static uint32_t* cache[64] = {};
  static uint64_t cache_ctx[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  const uint64_t ctx = current_context_id();
  if (!ctx) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev] || cache_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    cache[dev] = static_cast<uint32_t*>(p);
    cache_ctx[dev] = ctx;
  }
  return cache[dev];
}

}  // namespace fp8rl

using namespace fp8rl;

extern "C" FP8RL_API fp8rl_status fp8rl_sync_status(void* stream) {
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(cs) != cudaSuccess) return FP8RL_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return FP8RL_ERR_CUDA;
  uint32_t* word = device_error_word();
  if (!word) return FP8RL_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_error_word, sizeof v, 0, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
    return FP8RL_ERR_CUDA;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbolAsync(g_error_word, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, cs) != cudaSuccess)
    return FP8RL_ERR_CUDA;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return FP8RL_ERR_CUDA;
  if (v & kErrDeviceCheck) return FP8RL_ERR_DEVICE_CHECK;
  if (v & kErrTimeout) return FP8RL_ERR_TIMEOUT;
  return FP8RL_OK;
}

extern "C" FP8RL_API const char* fp8rl_status_string(fp8rl_status s) {
  switch (s) {
    case FP8RL_OK: return "FP8RL_OK";
    case FP8RL_ERR_INVALID_ARG: return "FP8RL_ERR_INVALID_ARG";
    case FP8RL_ERR_SHAPE: return "FP8RL_ERR_SHAPE";
    case FP8RL_ERR_ALIGNMENT: return "FP8RL_ERR_ALIGNMENT";
    case FP8RL_ERR_UNSUPPORTED: return "FP8RL_ERR_UNSUPPORTED";
    case FP8RL_ERR_CUDA: return "FP8RL_ERR_CUDA";
    case FP8RL_ERR_TIMEOUT: return "FP8RL_ERR_TIMEOUT";
    case FP8RL_ERR_DEVICE_CHECK: return "FP8RL_ERR_DEVICE_CHECK";
  }
  return "FP8RL_ERR_UNKNOWN";
}

extern "C" FP8RL_API int32_t fp8rl_version(void) { return 100; }
