// quant.cu -- weight-sync (128x128 block) and activation (1x128 group) E4M3
// quantisers for sm_103a.
//
// FP8-RL page, "Prerequisites / FP8 quantisation format": one scale per
// 128x128 weight block, W_hat = round(W / scale) in E4M3; "Method steps",
// step 1: weights quantised once per sync, activations in every forward pass.
//
// Both kernels are HBM-bound streams (2 bytes in, 1 byte + a scale out per
// element).  Each thread issues several independent 16-byte non-allocating
// loads before it touches any of them, so that enough bytes are in flight per
// SM; the block maximum is reduced in registers, across the warp with one
// redux and across warps through shared memory; the codes leave as 16-byte
// stores.  Grids are persistent: a multiple of the SM count, striding over the
// blocks or groups.
#include <algorithm>
#include <atomic>
#include <vector>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8rl {

// ============================================================================
// weight blocks
// ============================================================================

struct WDesc {
  const uint16_t* w;
  uint8_t* q;
  void* scale;
  int64_t n, k, ldw, ldq;
  int64_t kbs;          // blocks along K
  int64_t block_begin;  // first global block index of this matrix
  int32_t vec;          // rows are 16-byte aligned: vector path allowed
  int32_t pad;
};

template <int MAXD>
struct WBatch {
  int32_t count;
  int32_t pad;
  int64_t total_blocks;
  uint32_t* err;  // device error word (debug builds' store checks)
  WDesc d[MAXD];
};

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// a hint: fetch the line holding p into L2 (p must point into the tensor)
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

template <int MAXD>
__device__ __forceinline__ int find_desc(const WBatch<MAXD>& b, int64_t blk) {
  if (MAXD == 1) return 0;
  int lo = 0, hi = b.count - 1;  // largest d with block_begin <= blk
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (b.d[mid].block_begin <= blk) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// One CTA of 256 threads quantises one 128x128 block per loop iteration.
// Full, aligned blocks: thread t owns rows (t/8) + 32 i, i = 0..3, and the 16
// columns starting at 16 (t%8): four rows x 32 bytes in, four 16-byte stores out.
template <int MAXD, bool UE8M0>
__global__ void __launch_bounds__(256) quant_weight_kernel(const __grid_constant__ WBatch<MAXD> batch) {
  __shared__ uint32_t red[2][8];
  const int t = threadIdx.x, warp = t >> 5;
  int parity = 0;
  for (int64_t blk = blockIdx.x; blk < batch.total_blocks; blk += gridDim.x, parity ^= 1) {
    const WDesc& D = batch.d[find_desc<MAXD>(batch, blk)];
    const int64_t local = blk - D.block_begin;
    const int64_t nb = local / D.kbs, kb = local - nb * D.kbs;
    const int64_t r0 = nb * kBlock, c0 = kb * kBlock;
    const bool full = D.vec && r0 + kBlock <= D.n && c0 + kBlock <= D.k;
    if (full) {
      const int rs = t >> 3, cc = (t & 7) * 16;
      uint4 v[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint16_t* p = D.w + (r0 + rs + 32 * i) * D.ldw + c0 + cc;
        v[i][0] = ld_stream(p);
        v[i][1] = ld_stream(p + 8);
      }
      uint32_t acc = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc = absmax_u4(absmax_u4(acc, v[i][0]), v[i][1]);
      uint32_t am = __reduce_max_sync(0xffffffffu, (acc & 0xFFFFu) > (acc >> 16) ? (acc & 0xFFFFu) : (acc >> 16));
      if ((t & 31) == 0) red[parity][warp] = am;
      __syncthreads();
      uint32_t m8 = red[parity][0];
#pragma unroll
      for (int w = 1; w < 8; ++w) m8 = max(m8, red[parity][w]);
      const float amax = __uint_as_float(m8 << 16);
      const bool scale_in = dcheck(local < (D.n + kBlock - 1) / kBlock * D.kbs, batch.err);
      if (UE8M0) {
        const int e = scale_ue8m0_exponent(amax);
        const float f = exp2_neg(e);
        if (t == 0 && scale_in) static_cast<uint8_t*>(D.scale)[local] = (uint8_t)(e + 127);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint2 a = quant8_mul(v[i][0], f), b = quant8_mul(v[i][1], f);
          if (dcheck(r0 + rs + 32 * i < D.n && c0 + cc + 16 <= D.k, batch.err))
            st_stream(D.q + (r0 + rs + 32 * i) * D.ldq + c0 + cc, make_uint4(a.x, a.y, b.x, b.y));
        }
      } else {
        const float s = scale_fp32(amax);
        const float rcp = __frcp_rn(s);
        if (t == 0 && scale_in) static_cast<float*>(D.scale)[local] = s;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint2 a = quant8_div(v[i][0], s, rcp), b = quant8_div(v[i][1], s, rcp);
          if (dcheck(r0 + rs + 32 * i < D.n && c0 + cc + 16 <= D.k, batch.err))
            st_stream(D.q + (r0 + rs + 32 * i) * D.ldq + c0 + cc, make_uint4(a.x, a.y, b.x, b.y));
        }
      }
    } else {
      // ragged or unaligned block: scalar loads with bounds, two passes
      const int64_t rows = min((int64_t)kBlock, D.n - r0), cols = min((int64_t)kBlock, D.k - c0);
      uint32_t acc = 0;
      for (int idx = t; idx < kBlock * kBlock; idx += 256) {
        const int r = idx >> 7, c = idx & 127;
        if (r < rows && c < cols) acc = max(acc, (uint32_t)(D.w[(r0 + r) * D.ldw + c0 + c] & 0x7FFFu));
      }
      uint32_t am = __reduce_max_sync(0xffffffffu, acc);
      if ((t & 31) == 0) red[parity][warp] = am;
      __syncthreads();
      uint32_t m8 = red[parity][0];
      for (int w = 1; w < 8; ++w) m8 = max(m8, red[parity][w]);
      const float amax = __uint_as_float(m8 << 16);
      int e = 0;
      float s = 1.0f, f = 1.0f;
      const bool scale_in = dcheck(local < (D.n + kBlock - 1) / kBlock * D.kbs, batch.err);
      if (UE8M0) {
        e = scale_ue8m0_exponent(amax);
        f = exp2_neg(e);
        if (t == 0 && scale_in) static_cast<uint8_t*>(D.scale)[local] = (uint8_t)(e + 127);
      } else {
        s = scale_fp32(amax);
        if (t == 0 && scale_in) static_cast<float*>(D.scale)[local] = s;
      }
      for (int idx = t; idx < kBlock * kBlock; idx += 256) {
        const int r = idx >> 7, c = idx & 127;
        if (r < rows && c < cols && dcheck(r0 + r < D.n && c0 + c < D.k, batch.err)) {
          const float x = __uint_as_float((uint32_t)D.w[(r0 + r) * D.ldw + c0 + c] << 16);
          const float y = UE8M0 ? x * f : __fdiv_rn(x, s);
          D.q[(r0 + r) * D.ldq + c0 + c] = (uint8_t)(e4m3x2(y, 0.0f) & 0xFFu);
        }
      }
    }
  }
}

// ============================================================================
// activation groups
// ============================================================================

// Four lanes quantise one 1x128 group (32 elements each, as four 16-byte
// pieces interleaved so that the four lanes of a group read 64 contiguous
// bytes per load).  A warp task is one K group g of kActRows = 8 consecutive
// rows, so the per-group work (max over 4 lanes, the scale, its reciprocal)
// is shared by 8 groups per warp instruction, and the 8 scales land in one
// 32-byte run of the [K/128][m] scale array.  Tasks are numbered g-major and
// taken with a warp-uniform stride; each warp loads its next task before it
// quantises the current one, so its loads stay in flight while it computes.
constexpr int kActRows = 8;

struct ActTask {
  int32_t row;  // this lane's row
  int64_t c0;   // first column of the group
  bool live, full;
};

__device__ __forceinline__ ActTask act_task(int32_t t, int32_t rblocks, int32_t m, int64_t k, int vec, int sub) {
  ActTask a;
  const int32_t g = t / rblocks;
  a.row = (t - g * rblocks) * kActRows + sub;
  a.c0 = (int64_t)g * kBlock;
  a.live = a.row < m;
  a.full = vec && a.c0 + kBlock <= k;
  return a;
}

__device__ __forceinline__ void act_load(const uint16_t* __restrict__ x, int64_t ldx, int64_t k, const ActTask& a,
                                         int part, uint4 (&v)[4]) {
  const uint16_t* src = x + (int64_t)a.row * ldx + a.c0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int piece = part + 4 * j;  // 8 elements each
    if (a.live && a.full) {
      v[j] = ld_stream(src + piece * 8);
    } else if (a.live) {
      uint32_t h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int64_t c = a.c0 + piece * 8 + e;
        h[e] = c < k ? (uint32_t)src[piece * 8 + e] : 0u;
      }
      v[j] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
    } else {
      v[j] = make_uint4(0, 0, 0, 0);
    }
  }
}

template <bool UE8M0>
__device__ __forceinline__ void act_quant_store(const uint4 (&v)[4], const ActTask& a, int32_t m, int64_t k,
                                                uint8_t* __restrict__ q, int64_t ldq, void* __restrict__ scale,
                                                int part, uint32_t* err) {
  uint32_t acc = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) acc = absmax_u4(acc, v[j]);
  uint32_t am = max(acc & 0xFFFFu, acc >> 16);
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
  if (!a.live) return;
  if (!dcheck(a.row < m && a.c0 < k, err)) return;
  const float amax = __uint_as_float(am << 16);
  const int64_t sidx = (a.c0 / kBlock) * m + a.row;
  uint2 codes[4];
  if (UE8M0) {
    const int e = scale_ue8m0_exponent(amax);
    const float f = exp2_neg(e);
#pragma unroll
    for (int j = 0; j < 4; ++j) codes[j] = quant8_mul(v[j], f);
    if (part == 0) static_cast<uint8_t*>(scale)[sidx] = (uint8_t)(e + 127);
  } else {
    const float s = scale_fp32(amax);
    const float rcp = __frcp_rn(s);
#pragma unroll
    for (int j = 0; j < 4; ++j) codes[j] = quant8_div(v[j], s, rcp);
    if (part == 0) static_cast<float*>(scale)[sidx] = s;
  }
  uint8_t* dst = q + (int64_t)a.row * ldq + a.c0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int piece = part + 4 * j;
    if (a.full) {
      if (dcheck(a.c0 + piece * 8 + 8 <= k, err))
        asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(dst + piece * 8), "r"(codes[j].x), "r"(codes[j].y)
                     : "memory");
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (a.c0 + piece * 8 + e < k)
          dst[piece * 8 + e] = (uint8_t)(((e < 4 ? codes[j].x : codes[j].y) >> (8 * (e & 3))) & 0xFFu);
    }
  }
}

template <bool UE8M0>
__global__ void __launch_bounds__(256, 3) quant_act_kernel(const uint16_t* __restrict__ x, int32_t m,
                                                        int64_t k, int64_t ldx, uint8_t* __restrict__ q,
                                                        int64_t ldq, void* __restrict__ scale,
                                                        int32_t groups, int vec, uint32_t* err) {
  const int lane = threadIdx.x & 31, sub = lane >> 2, part = lane & 3;
  const int32_t warp = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int32_t warp_count = gridDim.x * 8;
  const int32_t rblocks = (m + kActRows - 1) / kActRows;
  const int32_t tasks = rblocks * groups;  // the host keeps m * groups below 2^31
  // the next kernel of the stream may start (it waits for this grid before
  // reading the codes); this grid's input comes from the earlier ones
  ptx::grid_dep_launch_dependents();
  ptx::grid_dep_wait();
  if (warp >= tasks) return;
  uint4 va[4], vb[4];
  ActTask ta = act_task(warp, rblocks, m, k, vec, sub);
  act_load(x, ldx, k, ta, part, va);
  // two tasks per trip, so that the two register sets keep fixed names
  for (int32_t t = warp; t < tasks; t += 2 * warp_count) {
    const int32_t t1 = t + warp_count, t2 = t + 2 * warp_count;
    ActTask tb;
    if (t1 < tasks) {
      tb = act_task(t1, rblocks, m, k, vec, sub);
      act_load(x, ldx, k, tb, part, vb);
    }
    act_quant_store<UE8M0>(va, ta, m, k, q, ldq, scale, part, err);
    if (t2 < tasks) {
      ta = act_task(t2, rblocks, m, k, vec, sub);
      act_load(x, ldx, k, ta, part, va);
    }
    if (t1 < tasks) act_quant_store<UE8M0>(vb, tb, m, k, q, ldq, scale, part, err);
  }
}

// ============================================================================
// the device codec alone (fp32 -> E4M3), for whole-format checks
// ============================================================================

__global__ void __launch_bounds__(256) e4m3_encode_kernel(const float* __restrict__ in, int64_t n,
                                                          uint8_t* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 2;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2; i < n; i += stride) {
    const float a = in[i], b = (i + 1 < n) ? in[i + 1] : 0.0f;
    const uint32_t c = e4m3x2(a, b);
    out[i] = (uint8_t)(c & 0xFFu);
    if (i + 1 < n) out[i + 1] = (uint8_t)(c >> 8);
  }
}

// ============================================================================
// host side
// ============================================================================

namespace {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// resident CTAs per SM of a 256-thread kernel (at least 1), asked once per
// kernel; concurrent first calls store the same value
template <typename K>
int ctas_per_sm(K kernel) {
  static std::atomic<int> cached{0};
  int c = cached.load(std::memory_order_relaxed);
  if (c == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, kernel, 256, 0) != cudaSuccess || c < 1) c = 1;
    cached.store(c, std::memory_order_relaxed);
  }
  return c;
}

fp8rl_status check_weight(const fp8rl_weight_desc& d, fp8rl_scale_fmt fmt) {
  if (d.n < 0 || d.k < 0 || d.ldw < d.k || d.ldq < d.k) return FP8RL_ERR_INVALID_ARG;
  if (d.n == 0 || d.k == 0) return FP8RL_OK;
  if (!d.w_bf16 || !d.q_e4m3 || !d.w_scale) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(d.w_bf16, 16) || !aligned(d.q_e4m3, 16)) return FP8RL_ERR_ALIGNMENT;
  if (fmt == FP8RL_SCALE_FP32 && !aligned(d.w_scale, 4)) return FP8RL_ERR_ALIGNMENT;
  return FP8RL_OK;
}

constexpr int kMaxBatch = 256;
constexpr int kWeightCtasPerSm = 4;  // 256 threads each, about 64 registers

template <int MAXD>
fp8rl_status launch_weight(const WBatch<MAXD>& b, fp8rl_scale_fmt fmt, cudaStream_t stream) {
  if (b.total_blocks == 0) return FP8RL_OK;
  // the same whole number of blocks for every CTA (no partly idle last round)
  const int64_t resident = (int64_t)sm_count() * kWeightCtasPerSm;
  const int64_t per_cta = (b.total_blocks + resident - 1) / resident;
  const int64_t grid = (b.total_blocks + per_cta - 1) / per_cta;
  if (fmt == FP8RL_SCALE_UE8M0)
    quant_weight_kernel<MAXD, true><<<(unsigned)grid, 256, 0, stream>>>(b);
  else
    quant_weight_kernel<MAXD, false><<<(unsigned)grid, 256, 0, stream>>>(b);
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}

WDesc make_desc(const fp8rl_weight_desc& s, int64_t begin) {
  WDesc d{};
  d.w = static_cast<const uint16_t*>(s.w_bf16);
  d.q = static_cast<uint8_t*>(s.q_e4m3);
  d.scale = s.w_scale;
  d.n = s.n;
  d.k = s.k;
  d.ldw = s.ldw;
  d.ldq = s.ldq;
  d.kbs = (s.k + kBlock - 1) / kBlock;
  d.block_begin = begin;
  d.vec = (s.ldw * 2) % 16 == 0 && s.ldq % 16 == 0;
  return d;
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" FP8RL_API fp8rl_status fp8rl_quant_weight_blockwise(const void* w_bf16, int64_t n,
                                                               int64_t k, int64_t ldw, void* q_e4m3,
                                                               int64_t ldq, void* w_scale,
                                                               fp8rl_scale_fmt fmt, void* stream) {
  if (fmt != FP8RL_SCALE_FP32 && fmt != FP8RL_SCALE_UE8M0) return FP8RL_ERR_INVALID_ARG;
  fp8rl_weight_desc s{w_bf16, q_e4m3, w_scale, n, k, ldw, ldq};
  fp8rl_status st = check_weight(s, fmt);
  if (st != FP8RL_OK || n == 0 || k == 0) return st;
  WBatch<1> b{};
  b.err = device_error_word();
  if (!b.err) return FP8RL_ERR_CUDA;
  b.count = 1;
  b.d[0] = make_desc(s, 0);
  b.total_blocks = ((n + kBlock - 1) / kBlock) * b.d[0].kbs;
  return launch_weight(b, fmt, static_cast<cudaStream_t>(stream));
}

extern "C" FP8RL_API fp8rl_status fp8rl_quant_weight_blockwise_batched(const fp8rl_weight_desc* descs,
                                                                       int32_t count,
                                                                       fp8rl_scale_fmt fmt,
                                                                       void* stream) {
  if (fmt != FP8RL_SCALE_FP32 && fmt != FP8RL_SCALE_UE8M0) return FP8RL_ERR_INVALID_ARG;
  if (count < 0 || (count > 0 && !descs)) return FP8RL_ERR_INVALID_ARG;
  for (int32_t i = 0; i < count; ++i) {
    fp8rl_status st = check_weight(descs[i], fmt);
    if (st != FP8RL_OK) return st;
  }
  // heap-allocated host staging: the parameter block is ~18 KB
  std::vector<WBatch<kMaxBatch>> staged(1);
  WBatch<kMaxBatch>& b = staged[0];
  b.err = nullptr;  // looked up before the first launch (a batch of empty matrices touches no device)
  int32_t i = 0;
  while (i < count) {
    b.count = 0;
    b.total_blocks = 0;
    for (; i < count && b.count < kMaxBatch; ++i) {
      const fp8rl_weight_desc& s = descs[i];
      if (s.n == 0 || s.k == 0) continue;
      b.d[b.count] = make_desc(s, b.total_blocks);
      b.total_blocks += ((s.n + kBlock - 1) / kBlock) * b.d[b.count].kbs;
      ++b.count;
    }
    if (b.count == 0) continue;
    if (!b.err && !(b.err = device_error_word())) return FP8RL_ERR_CUDA;
    fp8rl_status st = launch_weight(b, fmt, static_cast<cudaStream_t>(stream));
    if (st != FP8RL_OK) return st;
  }
  return FP8RL_OK;
}

extern "C" FP8RL_API fp8rl_status fp8rl_quant_act_group(const void* x_bf16, int64_t m, int64_t k,
                                                        int64_t ldx, void* q_e4m3, int64_t ldq,
                                                        void* x_scale, fp8rl_scale_fmt fmt,
                                                        void* stream) {
  if (fmt != FP8RL_SCALE_FP32 && fmt != FP8RL_SCALE_UE8M0) return FP8RL_ERR_INVALID_ARG;
  fp8rl_weight_desc s{x_bf16, q_e4m3, x_scale, m, k, ldx, ldq};
  fp8rl_status st = check_weight(s, fmt);
  if (st != FP8RL_OK || m == 0 || k == 0) return st;
  const int64_t groups = (k + kBlock - 1) / kBlock;
  const int64_t tasks = m * groups;
  if (tasks > (int64_t)INT32_MAX - (1 << 20)) return FP8RL_ERR_SHAPE;  // 32-bit task numbering
  const int64_t warp_tasks = ((m + kActRows - 1) / kActRows) * groups;
  const int occ = fmt == FP8RL_SCALE_UE8M0 ? ctas_per_sm(quant_act_kernel<true>) : ctas_per_sm(quant_act_kernel<false>);
  // Every warp gets the same whole number of tasks (the last round of a
  // striding loop is otherwise partly idle: 3.37 tasks per resident warp at
  // 8192 x 4096 left a third of the warps working in the fourth round).
  const int64_t resident_warps = (int64_t)sm_count() * occ * 8;
  const int64_t per_warp = (warp_tasks + resident_warps - 1) / resident_warps;
  const int64_t grid = std::max<int64_t>(1, (warp_tasks + 8 * per_warp - 1) / (8 * per_warp));
  const int vec = (ldx * 2) % 16 == 0 && ldq % 8 == 0;
  uint32_t* err = device_error_word();
  if (!err) return FP8RL_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(256);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  // start while the previous kernel of the stream finishes (the kernel waits
  // for it before reading X): at decode sizes the launch is most of the cost
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  const uint16_t* xp = static_cast<const uint16_t*>(x_bf16);
  uint8_t* qp = static_cast<uint8_t*>(q_e4m3);
  const int32_t m32 = (int32_t)m, g32 = (int32_t)groups;
  const cudaError_t e =
      fmt == FP8RL_SCALE_UE8M0
          ? cudaLaunchKernelEx(&cfg, quant_act_kernel<true>, xp, m32, k, ldx, qp, ldq, x_scale, g32, vec, err)
          : cudaLaunchKernelEx(&cfg, quant_act_kernel<false>, xp, m32, k, ldx, qp, ldq, x_scale, g32, vec, err);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FP8RL_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}

extern "C" FP8RL_API fp8rl_status fp8rl_e4m3_encode(const float* d_in, int64_t n, uint8_t* d_out,
                                                   void* stream) {
  if (n < 0 || (n > 0 && (!d_in || !d_out))) return FP8RL_ERR_INVALID_ARG;
  if (n == 0) return FP8RL_OK;
  if (!aligned(d_in, 4)) return FP8RL_ERR_ALIGNMENT;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((n + 511) / 512, (int64_t)sm_count() * 8));
  e4m3_encode_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(d_in, n, d_out);
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}
