// kv.cu -- FP8 KV cache: per-step per-tensor scale calibration and the
// quantised append of K and V rows.
//
// FP8-RL page, "Method steps", step 3: the KV cache is stored in FP8, and its
// quantisation scales are recomputed before every RL step's rollout from the
// first forward pass of the freshly synced policy, so that they follow the
// updated weights.  One fp32 scale per tensor (the pages leave the
// granularity open; per tensor is the plainest reading), scale = amax / 448
// of the calibration pass, all-zero tensors get 1.0.  Rows appended later are
// quantised with those fixed scales: the IEEE fp32 quotient x / scale rounded
// to nearest-even E4M3, saturating at +-448 when a later token exceeds the
// calibrated range.
//
// Both kernels are HBM-bound streams: a warp takes a token row, its lanes
// 16-byte pieces (8 bf16) of it.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8rl {
namespace {

constexpr int kKvThreads = 256;  // 8 warps
constexpr int kKvCtasPerSm = 8;

__device__ __forceinline__ uint4 ld_nc_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

struct KvTensors {
  const uint16_t* x[3];
  int64_t cols[3], ld[3];
  int32_t vec[3];
};

// The amax words start at zero (an empty tensor keeps 0: scale 1.0).  This
// kernel is launched in stream order (it begins once everything before it on
// the stream has completed) and lets the amax kernel start at once.
__global__ void kv_zero_kernel(uint32_t* amax_bits, int n) {
  ptx::grid_dep_launch_dependents();
  if ((int)threadIdx.x < n) amax_bits[threadIdx.x] = 0u;
}

// amax of tensor blockIdx.y (rows x cols bf16) into amax_bits[blockIdx.y]:
// the fp32 bit pattern of the magnitude (non-negative floats order like
// unsigned integers, so atomicMax is exact and the result is independent of
// the order of the updates).  Launched behind kv_zero_kernel with
// programmatic stream serialisation: that kernel began only after every
// earlier kernel of the stream had completed, so K, V and Q are read at once;
// the wait for its completion (the zeroed words) comes before the atomicMax.
__global__ void __launch_bounds__(kKvThreads) kv_amax_kernel(KvTensors ts, int64_t rows, uint32_t* amax_bits) {
  ptx::grid_dep_launch_dependents();
  const int ti = blockIdx.y;
  // selected, not indexed: an indexed parameter struct is copied to local memory
  const uint16_t* x = ti == 0 ? ts.x[0] : ti == 1 ? ts.x[1] : ts.x[2];
  const int64_t cols = ti == 0 ? ts.cols[0] : ti == 1 ? ts.cols[1] : ts.cols[2];
  const int64_t ld = ti == 0 ? ts.ld[0] : ti == 1 ? ts.ld[1] : ts.ld[2];
  const bool vec = ti == 0 ? ts.vec[0] : ti == 1 ? ts.vec[1] : ts.vec[2];
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kKvThreads / 32);
  uint32_t acc = 0;  // packed |bf16| maxima
  for (int64_t r = (int64_t)blockIdx.x * (kKvThreads / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
    const uint16_t* row = x + r * ld;
    if (vec) {
      // four 16-byte pieces per lane per trip, all loads issued before use
      for (int64_t c0 = (int64_t)lane * 8; c0 < cols; c0 += 4 * 256) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t c = c0 + j * 256;
          v[j] = c + 8 <= cols ? ld_nc_u4(row + c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) acc = absmax_u4(acc, v[j]);
        for (int j = 0; j < 4; ++j) {  // a ragged last piece (cols % 8 != 0)
          const int64_t c = c0 + j * 256;
          if (c < cols && c + 8 > cols)
            for (int e = 0; c + e < cols; ++e) acc = absmax_bf16x2(acc, (uint32_t)row[c + e]);
        }
      }
    } else {
      for (int64_t c = (int64_t)lane * 8; c < cols; c += 256)
        for (int e = 0; e < 8 && c + e < cols; ++e) acc = absmax_bf16x2(acc, (uint32_t)row[c + e]);
    }
  }
  uint32_t m = max(acc & 0xFFFFu, acc >> 16) << 16;
  m = __reduce_max_sync(0xffffffffu, m);
  __shared__ uint32_t red[kKvThreads / 32];
  if (lane == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < kKvThreads / 32 ? red[threadIdx.x] : 0u;
    m = __reduce_max_sync(0xffffffffu, m);
    if (threadIdx.x == 0) {
      ptx::grid_dep_wait();
      if (m != 0) atomicMax(amax_bits + ti, m);
    }
  }
}

// amax bits -> fp32 scale, in place (after the amax kernel has completed)
__global__ void kv_scale_kernel(float* scales, int n) {
  ptx::grid_dep_wait();
  const int i = threadIdx.x;
  if (i < n) scales[i] = scale_fp32(scales[i]);  // the word holds the amax's bits
}

// Row t of K and V to cache row slots[t]; rows whose slot is outside
// [0, num_slots) are skipped (padding).
__global__ void __launch_bounds__(kKvThreads) kv_append_kernel(const uint16_t* __restrict__ k,
                                                               const uint16_t* __restrict__ v, int64_t tokens,
                                                               int64_t dim, int64_t ldk, int64_t ldv,
                                                               const int32_t* __restrict__ slots,
                                                               uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                                                               int64_t ldc, int64_t num_slots,
                                                               const float* __restrict__ scales, int vec) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kKvThreads / 32);
  const float sk = scales[0], sv = scales[1];
  const float rk = __frcp_rn(sk), rv = __frcp_rn(sv);
  for (int64_t t = (int64_t)blockIdx.x * (kKvThreads / 32) + (threadIdx.x >> 5); t < tokens; t += warps) {
    const int64_t slot = slots[t];
    if (slot < 0 || slot >= num_slots) continue;  // warp-uniform
    const uint16_t* kr = k + t * ldk;
    const uint16_t* vr = v + t * ldv;
    uint8_t* kd = kc + slot * ldc;
    uint8_t* vd = vc + slot * ldc;
    for (int64_t c = (int64_t)lane * 8; c < dim; c += 256) {
      if (vec && c + 8 <= dim) {
        const uint4 xk = ld_nc_u4(kr + c), xv = ld_nc_u4(vr + c);
        const uint2 qk = quant8_div(xk, sk, rk), qv = quant8_div(xv, sv, rv);
        *reinterpret_cast<uint2*>(kd + c) = qk;
        *reinterpret_cast<uint2*>(vd + c) = qv;
      } else {
        for (int e = 0; e < 8 && c + e < dim; ++e) {
          const float xk = bf16_lo((uint32_t)kr[c + e]), xv = bf16_lo((uint32_t)vr[c + e]);
          kd[c + e] = (uint8_t)(e4m3x2(__fdiv_rn(xk, sk), 0.0f) & 0xFFu);
          vd[c + e] = (uint8_t)(e4m3x2(__fdiv_rn(xv, sv), 0.0f) & 0xFFu);
        }
      }
    }
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t kv_grid(int64_t rows) {
  const int64_t ctas = (rows + kKvThreads / 32 - 1) / (kKvThreads / 32);
  return std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)sm_count() * kKvCtasPerSm));
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" FP8RL_API fp8rl_status fp8rl_kv_calibrate(const void* k_bf16, const void* v_bf16, const void* q_bf16,
                                                     int64_t tokens, int64_t kv_dim, int64_t ldk, int64_t ldv,
                                                     int64_t q_dim, int64_t ldq, float* d_scales, void* stream) {
  if (tokens < 0 || kv_dim < 0 || ldk < kv_dim || ldv < kv_dim) return FP8RL_ERR_INVALID_ARG;
  if (q_bf16 && (q_dim < 0 || ldq < q_dim)) return FP8RL_ERR_INVALID_ARG;
  if (!d_scales || (tokens > 0 && kv_dim > 0 && (!k_bf16 || !v_bf16))) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(d_scales, 4) || !aligned(k_bf16, 2) || !aligned(v_bf16, 2) || !aligned(q_bf16, 2))
    return FP8RL_ERR_ALIGNMENT;
  const int n = q_bf16 ? 3 : 2;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint32_t* words = reinterpret_cast<uint32_t*>(d_scales);
  // zero the amax words, reduce, convert: each kernel after the first starts
  // while the one before it runs, and waits for it before it touches d_scales
  kv_zero_kernel<<<1, 32, 0, cs>>>(words, n);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = cs;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  if (tokens > 0) {
    KvTensors ts{};
    const void* xs[3] = {k_bf16, v_bf16, q_bf16};
    const int64_t cols[3] = {kv_dim, kv_dim, q_dim}, lds[3] = {ldk, ldv, ldq};
    for (int i = 0; i < n; ++i) {
      ts.x[i] = static_cast<const uint16_t*>(xs[i]);
      ts.cols[i] = cols[i];
      ts.ld[i] = lds[i];
      ts.vec[i] = aligned(xs[i], 16) && (lds[i] * 2) % 16 == 0;
    }
    // one grid slice per tensor, each warp a row at a time (a flat stream of
    // 16-byte pieces over all three tensors, one resident wave, measured
    // 30-50 % slower on GB300 after an L2 flush at 8192 and 32768 tokens)
    cfg.gridDim = dim3((unsigned)kv_grid(tokens), (unsigned)n);
    cfg.blockDim = dim3(kKvThreads);
    if (cudaLaunchKernelEx(&cfg, kv_amax_kernel, ts, tokens, words) != cudaSuccess) {
      cudaGetLastError();
      return FP8RL_ERR_CUDA;
    }
  }
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  if (cudaLaunchKernelEx(&cfg, kv_scale_kernel, d_scales, n) != cudaSuccess) {
    cudaGetLastError();
    return FP8RL_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}

extern "C" FP8RL_API fp8rl_status fp8rl_kv_append(const void* k_bf16, const void* v_bf16, int64_t tokens,
                                                  int64_t kv_dim, int64_t ldk, int64_t ldv,
                                                  const int32_t* d_slot_mapping, void* k_cache, void* v_cache,
                                                  int64_t ld_cache, int64_t num_slots, const float* d_scales,
                                                  void* stream) {
  if (tokens < 0 || kv_dim < 0 || num_slots < 0 || ldk < kv_dim || ldv < kv_dim || ld_cache < kv_dim)
    return FP8RL_ERR_INVALID_ARG;
  if (tokens == 0 || kv_dim == 0) return FP8RL_OK;
  if (!k_bf16 || !v_bf16 || !d_slot_mapping || !k_cache || !v_cache || !d_scales) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(k_bf16, 2) || !aligned(v_bf16, 2) || !aligned(d_slot_mapping, 4) || !aligned(d_scales, 4))
    return FP8RL_ERR_ALIGNMENT;
  const int vec = aligned(k_bf16, 16) && aligned(v_bf16, 16) && (ldk * 2) % 16 == 0 && (ldv * 2) % 16 == 0 &&
                  aligned(k_cache, 8) && aligned(v_cache, 8) && ld_cache % 8 == 0;
  kv_append_kernel<<<(unsigned)kv_grid(tokens), kKvThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(k_bf16), static_cast<const uint16_t*>(v_bf16), tokens, kv_dim, ldk, ldv,
      d_slot_mapping, static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), ld_cache, num_slots,
      d_scales, vec);
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}
