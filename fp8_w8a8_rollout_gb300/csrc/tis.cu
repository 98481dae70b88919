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
// Knuth's TwoSum (the rounded sum plus its error term) and accumulated in an
// fp32 (hi, lo) pair -- hi by TwoSum again, lo plainly, whose own rounding is
// 2^-24 of terms already 2^-24 below hi.  GB300's fp64 pipe is narrow: fp64
// conversions and adds per token made the kernel fp64-bound.  Each CTA takes
// fixed 4096-token chunks; its threads' pairs meet in a fixed tree and the
// CTA's pair is its partial; the last CTA to finish (an atomic ticket in the
// workspace header, reset by that CTA) adds the partials the same way, in an
// order fixed by their index, and converts to fp64 once.  The grid depends on n alone, so the result has the same bits on
// every run and device.  HBM-bound: 13 bytes per token (two fp32 reads, the
// mask, the fp32 weight).
#include <algorithm>

#include "common.cuh"

namespace fp8rl {
namespace {

constexpr int kTisThreads = 256;
constexpr int kTrips = 4;                                     // float4 loads of each input per thread
constexpr int64_t kTisChunk = (int64_t)kTisThreads * 4 * kTrips;  // 4096 tokens per CTA and chunk
constexpr int64_t kTisMaxCtas = 65536;                        // more tokens: CTAs take several chunks

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// the grid, and the number of partials, are a function of n alone: the
// summation order (and so the result's bits) does not depend on the device
int64_t tis_grid(int64_t n) {
  return std::max<int64_t>(1, std::min<int64_t>(kTisMaxCtas, (n + kTisChunk - 1) / kTisChunk));
}

__device__ __forceinline__ float tis_weight(float lt, float lr, float clip) {
  return fminf(expf(lt - lr), clip);
}

// Knuth's TwoSum: s + e == a + b exactly (round-to-nearest fp32; explicit
// _rn adds, which the compiler neither contracts nor reorders)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  const float av = __fsub_rn(s, bv);
  e = __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv));
}

// (hi, lo) += (bhi, blo): hi by TwoSum, the error terms into lo
__device__ __forceinline__ void pair_add(float& hi, float& lo, float bhi, float blo) {
  float s, e;
  two_sum(hi, bhi, s, e);
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(e, blo));
}

// lp_rollout - lp_train, made exact by TwoSum, added to (hi, lo)
__device__ __forceinline__ void acc_diff(float lr, float lt, float& hi, float& lo) {
  float d, de;
  two_sum(lr, -lt, d, de);
  pair_add(hi, lo, d, de);
}

__device__ __forceinline__ void tis_token(float lt, float lr, bool on, float clip, float& w, float& hi, float& lo,
                                          uint32_t& cnt) {
  w = on ? tis_weight(lt, lr, clip) : 0.0f;
  if (on) {
    acc_diff(lr, lt, hi, lo);
    ++cnt;
  }
}

// One 4096-token chunk per CTA and trip of the outer loop: thread i takes
// float4 i, i + 256, i + 512, i + 768 of the chunk (coalesced), all loads
// first.  The per-thread (hi, lo) pairs meet in the CTA by pair additions
// in a fixed tree; the CTA's partial is the pair's fp64 value.
__global__ void __launch_bounds__(kTisThreads) tis_partial_kernel(const float* __restrict__ lp_train,
                                                                 const float* __restrict__ lp_rollout,
                                                                 const uint8_t* __restrict__ mask, int64_t n,
                                                                 float clip, float* __restrict__ w,
                                                                 uint4* __restrict__ part,
                                                                 uint32_t* __restrict__ ticket,
                                                                 double* __restrict__ out, int vec) {
  float hi = 0.0f, lo = 0.0f;
  uint32_t cnt = 0;
  for (int64_t c0 = (int64_t)blockIdx.x * kTisChunk; c0 < n; c0 += (int64_t)gridDim.x * kTisChunk) {
    if (vec && c0 + kTisChunk <= n) {
      const int64_t q0 = c0 / 4 + threadIdx.x;
      float4 a[kTrips], b[kTrips];
      uint32_t mk[kTrips];
#pragma unroll
      for (int u = 0; u < kTrips; ++u) {
        a[u] = __ldcs(reinterpret_cast<const float4*>(lp_train) + q0 + u * kTisThreads);
        b[u] = __ldcs(reinterpret_cast<const float4*>(lp_rollout) + q0 + u * kTisThreads);
        mk[u] = mask ? __ldcs(reinterpret_cast<const unsigned int*>(mask) + q0 + u * kTisThreads) : 0x01010101u;
      }
#pragma unroll
      for (int u = 0; u < kTrips; ++u) {
        float4 o;
        tis_token(a[u].x, b[u].x, mk[u] & 0xFFu, clip, o.x, hi, lo, cnt);
        tis_token(a[u].y, b[u].y, (mk[u] >> 8) & 0xFFu, clip, o.y, hi, lo, cnt);
        tis_token(a[u].z, b[u].z, (mk[u] >> 16) & 0xFFu, clip, o.z, hi, lo, cnt);
        tis_token(a[u].w, b[u].w, mk[u] >> 24, clip, o.w, hi, lo, cnt);
        __stcs(reinterpret_cast<float4*>(w) + q0 + u * kTisThreads, o);
      }
    } else {
      // a ragged last chunk, or unaligned arrays: token by token
      const int64_t c1 = min(n, c0 + kTisChunk);
      for (int64_t i = c0 + threadIdx.x; i < c1; i += kTisThreads) {
        float wi;
        tis_token(lp_train[i], lp_rollout[i], mask ? mask[i] != 0 : true, clip, wi, hi, lo, cnt);
        w[i] = wi;
      }
    }
  }
  // fixed-shape tree: lanes, then the CTA's warps in order
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const float ohi = __shfl_xor_sync(0xffffffffu, hi, d);
    const float olo = __shfl_xor_sync(0xffffffffu, lo, d);
    pair_add(hi, lo, ohi, olo);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, d);
  }
  __shared__ float whi[kTisThreads / 32], wlo[kTisThreads / 32];
  __shared__ uint32_t wc[kTisThreads / 32];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    whi[warp] = hi;
    wlo[warp] = lo;
    wc[warp] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float h = whi[0], l = wlo[0];
    uint32_t c = wc[0];
    for (int i = 1; i < kTisThreads / 32; ++i) {
      pair_add(h, l, whi[i], wlo[i]);
      c += wc[i];
    }
    part[blockIdx.x] = make_uint4(__float_as_uint(h), __float_as_uint(l), c, 0u);
    __threadfence();  // the partial is visible before the ticket is taken
    last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  // The last CTA to finish adds every partial, in an order fixed by the
  // partial's index (not by which CTA came last): thread i takes partials
  // i, i + 256, ... (loads issued in batches of 8), then a fixed tree.
  __threadfence();
  hi = lo = 0.0f;
  unsigned long long c = 0;
  const int parts = gridDim.x;
  for (int i0 = threadIdx.x; i0 < parts; i0 += 8 * kTisThreads) {
    uint4 p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * kTisThreads;
      p[j] = i < parts ? __ldcg(part + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      pair_add(hi, lo, __uint_as_float(p[j].x), __uint_as_float(p[j].y));
      c += p[j].z;
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const float ohi = __shfl_xor_sync(0xffffffffu, hi, d);
    const float olo = __shfl_xor_sync(0xffffffffu, lo, d);
    pair_add(hi, lo, ohi, olo);
    c += __shfl_xor_sync(0xffffffffu, c, d);
  }
  __shared__ unsigned long long wc64[kTisThreads / 32];
  __syncthreads();  // the first tree's shared values are no longer read
  if (lane == 0) {
    whi[warp] = hi;
    wlo[warp] = lo;
    wc64[warp] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float h = whi[0], l = wlo[0];
    unsigned long long cc = wc64[0];
    for (int i = 1; i < kTisThreads / 32; ++i) {
      pair_add(h, l, whi[i], wlo[i]);
      cc += wc64[i];
    }
    const double sum = (double)h + (double)l;
    out[0] = cc ? sum / (double)cc : 0.0;
    out[1] = sum;
    out[2] = (double)cc;
    *ticket = 0u;  // ready for the next call on this workspace
  }
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

// workspace: a 16-byte header (the CTA ticket), then one 16-byte partial per CTA
extern "C" FP8RL_API size_t fp8rl_tis_workspace_size(int64_t n) {
  if (n < 0) return 0;
  return 16 + (size_t)tis_grid(n) * 16;
}

extern "C" FP8RL_API fp8rl_status fp8rl_tis_weights(const float* d_lp_train, const float* d_lp_rollout,
                                                    const uint8_t* d_mask, int64_t n, float clip, float* d_w,
                                                    double* d_kl, void* d_workspace, size_t workspace_bytes,
                                                    void* stream) {
  if (n < 0 || !(clip > 0.0f) || !d_kl || !d_workspace) return FP8RL_ERR_INVALID_ARG;
  if (n > 0 && (!d_lp_train || !d_lp_rollout || !d_w)) return FP8RL_ERR_INVALID_ARG;
  if (workspace_bytes < fp8rl_tis_workspace_size(n)) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(d_lp_train, 4) || !aligned(d_lp_rollout, 4) || !aligned(d_w, 4) || !aligned(d_kl, 8) ||
      !aligned(d_workspace, 16))
    return FP8RL_ERR_ALIGNMENT;
  const int64_t grid = tis_grid(n);
  uint32_t* ticket = static_cast<uint32_t*>(d_workspace);
  uint4* part = static_cast<uint4*>(d_workspace) + 1;
  const int vec = aligned(d_lp_train, 16) && aligned(d_lp_rollout, 16) && aligned(d_w, 16) && aligned(d_mask, 4);
  tis_partial_kernel<<<(unsigned)grid, kTisThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      d_lp_train, d_lp_rollout, d_mask, n, clip, d_w, part, ticket, d_kl, vec);
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}
