// api.cu -- status reporting of the C ABI and the device error word.
//
// Kernels that wait on mbarriers bound every wait; when one runs out they set
// a bit in this word and leave through their normal teardown (no trap), so
// the CUDA context stays usable.  fp8rl_sync_status() reads and clears it.
#include <mutex>

#include "common.cuh"

namespace fp8rl {

// one word per device that loads the library (a module-scope variable: no
// allocation is ever made for it)
static __device__ uint32_t g_error_word;

// device address of the error word on the current device (cached per device)
uint32_t* device_error_word() {
  static std::mutex mu;
  static uint32_t* cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<uint32_t*>(p);
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
  }
  return "FP8RL_ERR_UNKNOWN";
}

extern "C" FP8RL_API int32_t fp8rl_version(void) { return 100; }
