// gemm.cu -- block-scaled W8A8 GEMMs (host validation; the tcgen05 kernels follow).
#include "common.cuh"

namespace fp8rl {
namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

fp8rl_status check_gemm(const void* xq, const void* x_scale, const void* wq, const void* w_scale,
                        const void* y, int64_t m, int64_t n, int64_t k, fp8rl_scale_fmt fmt) {
  if (fmt != FP8RL_SCALE_FP32 && fmt != FP8RL_SCALE_UE8M0) return FP8RL_ERR_INVALID_ARG;
  if (m < 0 || n < 0 || k < 0) return FP8RL_ERR_INVALID_ARG;
  if (n % 128 || k % 128) return FP8RL_ERR_SHAPE;
  if (m == 0 || n == 0) return FP8RL_OK;
  if (!xq || !x_scale || !wq || !w_scale || !y) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(y, 16)) return FP8RL_ERR_ALIGNMENT;
  if (fmt == FP8RL_SCALE_FP32 && (!aligned(x_scale, 4) || !aligned(w_scale, 4))) return FP8RL_ERR_ALIGNMENT;
  return FP8RL_OK;
}
}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" FP8RL_API fp8rl_status fp8rl_gemm_blockscaled(const void* xq, const void* x_scale,
                                                         const void* wq, const void* w_scale, void* y,
                                                         int64_t m, int64_t n, int64_t k,
                                                         fp8rl_scale_fmt fmt, void* stream) {
  fp8rl_status st = check_gemm(xq, x_scale, wq, w_scale, y, m, n, k, fmt);
  if (st != FP8RL_OK || m == 0 || n == 0) return st;
  (void)stream;
  return FP8RL_ERR_UNSUPPORTED;
}

extern "C" FP8RL_API fp8rl_status fp8rl_grouped_gemm_blockscaled(const void* xq, const void* x_scale,
                                                                 const void* wq, const void* w_scale,
                                                                 const int32_t* d_offsets,
                                                                 int64_t num_experts, int64_t rows,
                                                                 int64_t n, int64_t k, void* y,
                                                                 fp8rl_scale_fmt fmt, void* stream) {
  if (num_experts < 1 || !d_offsets) return FP8RL_ERR_INVALID_ARG;
  fp8rl_status st = check_gemm(xq, x_scale, wq, w_scale, y, rows, n, k, fmt);
  if (st != FP8RL_OK || rows == 0 || n == 0) return st;
  (void)stream;
  return FP8RL_ERR_UNSUPPORTED;
}
