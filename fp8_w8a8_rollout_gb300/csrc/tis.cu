// tis.cu -- token-level truncated importance sampling weights and the
// train-inference mismatch KL estimate.
//
// FP8-RL page, "Method steps", step 4: each token sampled by the FP8 rollout
// policy is re-scored by the training policy; the weight is the probability
// ratio pi_theta / pi_fp8 = exp(lp_train - lp_rollout), truncated at C (2 in
// the pages; the pages' clip to [-C, C] is min(w, C) as w > 0).
// Precision-alignment page, "how the gap is measured": the mismatch is the
// mean over generated tokens of lp_rollout - lp_train.
//
// A token mask marks the generated tokens; others get weight 0 and stay out
// of the mean.  The weight: the fp32 difference, CUDA's expf, fminf with C.
// The mean: each difference lp_rollout - lp_train is made exact in fp32 by
// Knuth's TwoSum (the rounded sum plus its error term), the pairs are summed
// in an fp32 (hi, lo) accumulator (hi by TwoSum again, lo plainly: its own
// rounding is 2^-24 of terms already 2^-24 below hi), and every 64 tokens the
// pair is folded into the thread's fp64 sum.  GB300's fp64 pipe is narrow:
// fp64 conversions and adds per token made the kernel fp64-bound.  Thread
// sums then meet in a fixed tree per CTA and the CTA partials in a fixed tree
// in one CTA -- the same bits on every run of the same size on a given GPU
// (the grid is one wave of resident CTAs).  HBM-bound: 13
// bytes per token (two fp32 reads, the mask, the fp32 weight).
#include <algorithm>

#include "common.cuh"

namespace fp8rl {
namespace {

constexpr int kTisThreads = 256;
constexpr int kTisMaxCtas = 4096;       // workspace bound; the grid is one wave of resident CTAs
constexpr int kTisTokensPerCta = 8192;  // below this many per CTA the grid shrinks
constexpr int kTisFinalThreads = 1024;
constexpr int kTrips = 4;  // float4 loads of each input in flight per thread

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

__device__ __forceinline__ float tis_weight(float lt, float lr, float clip) {
  return fminf(expf(lt - lr), clip);
}

// Knuth's TwoSum: s + e == a + b exactly (round-to-nearest fp32, no
// reassociation: plain adds, which nvcc does not contract or reorder)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  const float av = __fsub_rn(s, bv);
  e = __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv));
}

// lp_rollout - lp_train added exactly (up to the lo word's rounding) to (hi, lo)
__device__ __forceinline__ void acc_diff(float lr, float lt, float& hi, float& lo) {
  float d, de, s, se;
  two_sum(lr, -lt, d, de);
  two_sum(hi, d, s, se);
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(se, de));
}

__global__ void __launch_bounds__(kTisThreads, 3) tis_partial_kernel(const float* __restrict__ lp_train,
                                                                 const float* __restrict__ lp_rollout,
                                                                 const uint8_t* __restrict__ mask, int64_t n,
                                                                 float clip, float* __restrict__ w,
                                                                 double* __restrict__ part_sum,
                                                                 unsigned long long* __restrict__ part_cnt,
                                                                 int vec) {
  double sum = 0.0;
  float hi = 0.0f, lo = 0.0f;  // fp32 pair, folded into sum every 64 tokens
  uint32_t cnt = 0, trips = 0;
  const int64_t stride = (int64_t)gridDim.x * kTisThreads;
  const int64_t tid = (int64_t)blockIdx.x * kTisThreads + threadIdx.x;
  if (vec) {
    const int64_t n4 = n / 4;
    // kTrips float4 trips per loop: all their loads are in flight together
    for (int64_t i0 = tid; i0 < n4; i0 += kTrips * stride) {
      float4 a[kTrips], b[kTrips];
      uint32_t mk[kTrips];
#pragma unroll
      for (int u = 0; u < kTrips; ++u) {
        const int64_t i = i0 + u * stride;
        const bool in = i < n4;
        a[u] = in ? __ldcs(reinterpret_cast<const float4*>(lp_train) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        b[u] = in ? __ldcs(reinterpret_cast<const float4*>(lp_rollout) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        mk[u] = !in ? 0u : mask ? __ldcs(reinterpret_cast<const unsigned int*>(mask) + i) : 0x01010101u;
      }
#pragma unroll
      for (int u = 0; u < kTrips; ++u) {
        const int64_t i = i0 + u * stride;
        if (i >= n4) break;
        const float lt[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, lr[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
        float o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool on = (mk[u] >> (8 * j)) & 0xFFu;
          o[j] = on ? tis_weight(lt[j], lr[j], clip) : 0.0f;
          if (on) {
            acc_diff(lr[j], lt[j], hi, lo);
            ++cnt;
          }
        }
        __stcs(reinterpret_cast<float4*>(w) + i, make_float4(o[0], o[1], o[2], o[3]));
      }
      if ((++trips & (16 / kTrips - 1)) == 0) {  // every 64 tokens
        sum += (double)hi + (double)lo;
        hi = lo = 0.0f;
      }
    }
    for (int64_t i = n4 * 4 + tid; i < n; i += stride) {
      const bool on = mask ? mask[i] != 0 : true;
      w[i] = on ? tis_weight(lp_train[i], lp_rollout[i], clip) : 0.0f;
      if (on) {
        acc_diff(lp_rollout[i], lp_train[i], hi, lo);
        ++cnt;
      }
    }
  } else {
    for (int64_t i = tid; i < n; i += stride) {
      const bool on = mask ? mask[i] != 0 : true;
      w[i] = on ? tis_weight(lp_train[i], lp_rollout[i], clip) : 0.0f;
      if (on) {
        acc_diff(lp_rollout[i], lp_train[i], hi, lo);
        ++cnt;
      }
      if ((++trips & 63) == 0) {
        sum += (double)hi + (double)lo;
        hi = lo = 0.0f;
      }
    }
  }
  sum += (double)hi + (double)lo;
  // fixed-shape tree: lanes, then the CTA's warps in order
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    sum += __shfl_xor_sync(0xffffffffu, sum, d);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, d);
  }
  __shared__ double ws[kTisThreads / 32];
  __shared__ uint32_t wc[kTisThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    ws[warp] = sum;
    wc[warp] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    unsigned long long c = 0;
    for (int i = 0; i < kTisThreads / 32; ++i) {
      s += ws[i];
      c += wc[i];
    }
    part_sum[blockIdx.x] = s;
    part_cnt[blockIdx.x] = c;
  }
}

// out: [0] mean (0 when no token is selected), [1] sum, [2] token count.
// Thread i adds partials i, i + 1024, ... in order; then a fixed tree.
__global__ void __launch_bounds__(kTisFinalThreads) tis_final_kernel(const double* __restrict__ part_sum,
                                                                    const unsigned long long* __restrict__ part_cnt,
                                                                    int parts, double* __restrict__ out) {
  double s = 0.0;
  unsigned long long c = 0;
  for (int i = threadIdx.x; i < parts; i += kTisFinalThreads) {
    s += part_sum[i];
    c += part_cnt[i];
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, d);
    c += __shfl_xor_sync(0xffffffffu, c, d);
  }
  __shared__ double ws[kTisFinalThreads / 32];
  __shared__ unsigned long long wc[kTisFinalThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    ws[warp] = s;
    wc[warp] = c;
  }
  __syncthreads();
  if (warp == 0) {
    s = ws[lane];
    c = wc[lane];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, d);
      c += __shfl_xor_sync(0xffffffffu, c, d);
    }
    if (lane == 0) {
      out[0] = c ? s / (double)c : 0.0;
      out[1] = s;
      out[2] = (double)c;
    }
  }
}

int64_t tis_grid(int64_t n) {
  static int resident = 0;  // CTAs of the partial kernel resident per SM, asked once
  static int sms = 0;
  if (resident == 0) {
    int dev = 0, r = 0, m = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&m, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || m <= 0)
      m = 152;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, tis_partial_kernel, kTisThreads, 0) != cudaSuccess || r < 1)
      r = 1;
    resident = r;
    sms = m;
  }
  const int64_t wave = std::min<int64_t>(kTisMaxCtas, (int64_t)sms * resident);
  return std::max<int64_t>(1, std::min<int64_t>(wave, (n + kTisTokensPerCta - 1) / kTisTokensPerCta));
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" FP8RL_API size_t fp8rl_tis_workspace_size(int64_t n) {
  if (n < 0) return 0;
  return (size_t)std::max<int64_t>(1, std::min<int64_t>(kTisMaxCtas, (n + kTisTokensPerCta - 1) / kTisTokensPerCta)) *
         16;
}

extern "C" FP8RL_API fp8rl_status fp8rl_tis_weights(const float* d_lp_train, const float* d_lp_rollout,
                                                    const uint8_t* d_mask, int64_t n, float clip, float* d_w,
                                                    double* d_kl, void* d_workspace, size_t workspace_bytes,
                                                    void* stream) {
  if (n < 0 || !(clip > 0.0f) || !d_kl || !d_workspace) return FP8RL_ERR_INVALID_ARG;
  if (n > 0 && (!d_lp_train || !d_lp_rollout || !d_w)) return FP8RL_ERR_INVALID_ARG;
  if (workspace_bytes < fp8rl_tis_workspace_size(n)) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(d_lp_train, 4) || !aligned(d_lp_rollout, 4) || !aligned(d_w, 4) || !aligned(d_kl, 8) ||
      !aligned(d_workspace, 8))
    return FP8RL_ERR_ALIGNMENT;
  const int64_t grid = tis_grid(n);
  double* part_sum = static_cast<double*>(d_workspace);
  unsigned long long* part_cnt = reinterpret_cast<unsigned long long*>(part_sum + grid);
  const int vec = aligned(d_lp_train, 16) && aligned(d_lp_rollout, 16) && aligned(d_w, 16) && aligned(d_mask, 4);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  tis_partial_kernel<<<(unsigned)grid, kTisThreads, 0, cs>>>(d_lp_train, d_lp_rollout, d_mask, n, clip, d_w,
                                                              part_sum, part_cnt, vec);
  tis_final_kernel<<<1, kTisFinalThreads, 0, cs>>>(part_sum, part_cnt, (int)grid, d_kl);
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}
