// moe.cu -- MoE expert dispatch plan and the weighted combine around the
// grouped GEMM, driven by replayed routing indices.
//
// Routing-replay page, "R3: Rollout Routing Replay": the rollout records each
// token's top-k expert indices per MoE layer as integers, and experts are fed
// from those indices.  The plan turns a [T][k] index array into the grouped
// layout the grouped GEMM reads:
//   offsets[e]      first row of expert e's segment (exclusive prefix sum of
//                   the per-expert pair counts), offsets[E] = routed pairs
//   row_of_pair[p]  the row pair p = t * k + j occupies, -1 if dropped
//   token_of_row[r] the token row r came from, -1 for the unused tail
// Rows inside a segment follow increasing pair order (the stable order);
// an index outside [0, E) drops its pair.
//
// Up to 8192 pairs and 256 experts, one CTA does the whole plan (below);
// larger plans take three small kernels, deterministic and independent of
// timing:
//   count  one CTA per tile of pairs: per-expert histogram in shared memory
//   scan   one CTA: the exclusive scan over experts of their totals, then
//          per expert the running count over tiles: each tile's first row
//   rank   one warp per tile: walks its pairs 32 at a time in order; lanes
//          with the same expert find each other (one ballot per bit of the
//          expert id) and take consecutive rows from the tile's running row
//          counter
//
// Dispatch: each token row quantised once in 1x128 groups and written to all
// rows its pairs occupy (below, with the kernel).
//
// Combine: out[t] = sum_j gate[t][j] * y[row_of_pair[t * k + j]], fp32
// fused multiply-adds in slot order, one bf16 rounding.  A thread per 16-byte
// piece of an output row, with the k source pieces loaded before any is used.
// HBM-bound: k rows read, one written per token.
#include <algorithm>
#include <atomic>

#include "common.cuh"

namespace fp8rl {
namespace {

constexpr int kPlanMinTile = 1024;  // pairs per tile (at least)
constexpr int kPlanMaxTiles = 32;   // tiles are widened beyond this many
constexpr int kPlanMaxExperts = 8192;
constexpr int kMaxTopk = 32;
constexpr int kScanThreads = 1024;
constexpr int kCombineThreads = 256;

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct PlanShape {
  int64_t pairs, tile, tiles;
};

PlanShape plan_shape(int64_t tokens, int64_t topk) {
  PlanShape s;
  s.pairs = tokens * topk;
  s.tile = kPlanMinTile;
  while ((s.pairs + s.tile - 1) / s.tile > kPlanMaxTiles) s.tile *= 2;
  s.tiles = (s.pairs + s.tile - 1) / s.tile;
  return s;
}

// Lanes holding the same key as this lane, for keys below 2^bits: one ballot
// per key bit (match.any does the same in one instruction, but takes about a
// thousand cycles when most of the 32 keys differ, as expert ids do).
__device__ __forceinline__ uint32_t match_key(uint32_t key, int bits) {
  uint32_t m = 0xffffffffu;
  for (int b = 0; b < bits; ++b) {
    const bool on = (key >> b) & 1u;
    const uint32_t bb = __ballot_sync(0xffffffffu, on);
    m &= on ? bb : ~bb;
  }
  return m;
}

// bits needed for the keys 0 .. experts (experts itself marks a dropped pair)
int key_bits(int64_t experts) {
  int b = 1;
  while ((int64_t{1} << b) <= experts) ++b;
  return b;
}

__global__ void __launch_bounds__(256) moe_count_kernel(const int32_t* __restrict__ idx, int32_t pairs,
                                                       int32_t tile, int32_t experts, int32_t* __restrict__ counts) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < experts; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int32_t p0 = blockIdx.x * tile;
  const int32_t p1 = min(pairs, p0 + tile);
#pragma unroll 4
  for (int32_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int32_t e = idx[p];
    if (e >= 0 && e < experts) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < experts; e += blockDim.x) counts[(int64_t)blockIdx.x * experts + e] = hist[e];
}

// counts[tiles][E] in, each tile's first row per expert out (in place);
// offsets[E + 1].  Thread e holds its expert's (at most kPlanMaxTiles)
// counts in registers, so all loads are in flight at once; experts beyond
// kScanThreads take a second and later round of the same.
__global__ void __launch_bounds__(kScanThreads) moe_scan_kernel(int32_t* __restrict__ base, int32_t tiles,
                                                               int32_t experts, int32_t* __restrict__ offsets) {
  __shared__ int32_t warp_sum[kScanThreads / 32];
  __shared__ int32_t carry;  // rows of the experts of earlier rounds
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  for (int e0 = 0; e0 < experts; e0 += kScanThreads) {
    const int e = e0 + threadIdx.x;
    int32_t c[kPlanMaxTiles];
    int32_t mine = 0;
#pragma unroll
    for (int b = 0; b < kPlanMaxTiles; ++b) {
      c[b] = (e < experts && b < tiles) ? base[(int64_t)b * experts + e] : 0;
      mine += c[b];
    }
    int32_t incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    __syncthreads();  // carry is set; warp_sum is free
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int32_t w = warp_sum[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int32_t v = __shfl_up_sync(0xffffffffu, w, d);
        if (lane >= d) w += v;
      }
      warp_sum[lane] = w;
    }
    __syncthreads();
    int32_t run = carry + incl - mine + (warp > 0 ? warp_sum[warp - 1] : 0);
    if (e < experts) {
      offsets[e] = run;
#pragma unroll
      for (int b = 0; b < kPlanMaxTiles; ++b) {
        if (b < tiles) base[(int64_t)b * experts + e] = run;
        run += c[b];
      }
    }
    __syncthreads();  // everyone has read carry
    if (threadIdx.x == 0) carry += warp_sum[kScanThreads / 32 - 1];
  }
  __syncthreads();
  if (threadIdx.x == 0) offsets[experts] = carry;
}

__global__ void __launch_bounds__(32) moe_rank_kernel(const int32_t* __restrict__ idx, int32_t pairs, int32_t tile,
                                                     int32_t topk, int32_t experts, int32_t bits,
                                                     const int32_t* __restrict__ base,
                                                     const int32_t* __restrict__ offsets,
                                                     int32_t* __restrict__ row_of_pair,
                                                     int32_t* __restrict__ token_of_row) {
  extern __shared__ int32_t next_row[];  // [experts]
  const int lane = threadIdx.x;
  for (int e = lane; e < experts; e += 32) next_row[e] = base[(int64_t)blockIdx.x * experts + e];
  __syncwarp();
  const int32_t p0 = blockIdx.x * tile;
  const int32_t p1 = min(pairs, p0 + tile);
  const uint32_t lt_mask = (1u << lane) - 1u;
  // 1024 pairs per round: all 32 loads of a lane in flight at once, then
  // 32 steps of 32 consecutive pairs
  for (int32_t q0 = p0; q0 < p1; q0 += 1024) {
    int32_t ev[32];
#pragma unroll
    for (int s = 0; s < 32; ++s) {
      const int32_t p = q0 + s * 32 + lane;
      ev[s] = p < p1 ? idx[p] : -1;
    }
#pragma unroll
    for (int s = 0; s < 32; ++s) {
      const int32_t p = q0 + s * 32 + lane;
      const int32_t e = ev[s];
      const bool live = e >= 0 && e < experts;
      const uint32_t same = match_key(live ? (uint32_t)e : (uint32_t)experts, bits);
      int32_t row = -1;
      if (live) row = next_row[e] + __popc(same & lt_mask);
      __syncwarp();  // every lane has read its counter before the leaders move them
      if (live && (same & lt_mask) == 0) next_row[e] += __popc(same);
      __syncwarp();
      if (p < p1) {
        row_of_pair[p] = row;
        if (live) token_of_row[row] = p / topk;
      }
    }
  }
  // the rows past the routed pairs carry no token
  for (int64_t r = (int64_t)offsets[experts] + (int64_t)blockIdx.x * 32 + lane; r < pairs;
       r += (int64_t)gridDim.x * 32)
    token_of_row[r] = -1;
}

// The whole plan in one CTA, for up to kSmallPlanPairs pairs and
// kSmallPlanExperts experts (decode-size batches): each of the 32 warps
// takes a contiguous chunk of at most 256 pairs and keeps its
// indices in registers; pass 1 counts them into the warp's own histogram row
// (shared-memory atomics), a block scan turns the rows into
// each warp's first row per expert and the offsets, pass 2 ranks as above.
constexpr int kSmallPlanPairs = 8 * 1024;
constexpr int kSmallPlanExperts = 256;

__global__ void __launch_bounds__(1024) moe_plan_small_kernel(const int32_t* __restrict__ idx, int32_t pairs,
                                                             int32_t topk, int32_t experts, int32_t bits,
                                                             int32_t* __restrict__ offsets,
                                                             int32_t* __restrict__ row_of_pair,
                                                             int32_t* __restrict__ token_of_row) {
  extern __shared__ int32_t hist[];  // [32][experts], then total[experts]
  int32_t* total = hist + 32 * experts;
  __shared__ int32_t warp_sum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32 * experts; i += 1024) hist[i] = 0;
  const int32_t chunk = (pairs + 32 * 32 - 1) / (32 * 32) * 32;  // <= 1024, a multiple of 32
  const int32_t p0 = min(pairs, warp * chunk), p1 = min(pairs, p0 + chunk);
  int32_t ev[32];
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    const int32_t p = p0 + s * 32 + lane;
    ev[s] = p < p1 ? idx[p] : -1;
  }
  __syncthreads();
  int32_t* h = hist + warp * experts;
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    if (p0 + s * 32 >= p1) break;  // warp-uniform
    const int32_t e = ev[s];
    if (e >= 0 && e < experts) atomicAdd(&h[e], 1);  // counts only: the order does not matter
  }
  __syncthreads();
  // per expert: the running count over warps, then the scan over experts
  int32_t mine = 0;
  if (threadIdx.x < experts) {
    const int e = threadIdx.x;
    int32_t run = 0;
    for (int w = 0; w < 32; ++w) {
      const int32_t c = hist[w * experts + e];
      hist[w * experts + e] = run;
      run += c;
    }
    mine = run;
  }
  int32_t incl = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = warp_sum[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += v;
    }
    warp_sum[lane] = w;
  }
  __syncthreads();
  const int32_t start = incl - mine + (warp > 0 ? warp_sum[warp - 1] : 0);
  if (threadIdx.x < experts) {
    total[threadIdx.x] = start;
    offsets[threadIdx.x] = start;
  }
  if (threadIdx.x == 0) offsets[experts] = warp_sum[31];
  __syncthreads();
  for (int i = threadIdx.x; i < 32 * experts; i += 1024) hist[i] += total[i % experts];
  __syncthreads();
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    const int32_t p = p0 + s * 32 + lane;
    if (p0 + s * 32 >= p1) break;  // warp-uniform
    const int32_t e = ev[s];
    const bool live = e >= 0 && e < experts;
    const uint32_t same = match_key(live ? (uint32_t)e : (uint32_t)experts, bits);
    int32_t row = -1;
    if (live) row = h[e] + __popc(same & lt_mask);
    __syncwarp();
    if (live && (same & lt_mask) == 0) h[e] += __popc(same);
    __syncwarp();
    if (p < p1) {
      row_of_pair[p] = row;
      if (live) token_of_row[row] = p / topk;
    }
  }
  for (int32_t r = warp_sum[31] + threadIdx.x; r < pairs; r += 1024) token_of_row[r] = -1;
}

__device__ __forceinline__ uint4 ld_nc_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void fma_piece(float (&acc)[8], float w, uint4 v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = fmaf(w, bf16_lo(u[i]), acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, bf16_hi(u[i]), acc[2 * i + 1]);
  }
}

// Dispatch with 1x128 quantisation.  A warp task is 1024 columns of one
// token (two 512-column rounds); lane l takes columns [16 l, 16 l + 16) of a
// round, so a group of 128 columns is 8 consecutive lanes and its amax meets
// in 3 shuffles.  Each group's codes and scale are written to every row the
// token's pairs occupy: a warp store covers 512 contiguous bytes of a
// destination row.  Tasks are taken with a warp-uniform stride, and each
// warp loads its next task (row chunk and row map) before it quantises and
// stores the current one.  The quotient and its rounding are the activation
// quantiser's (IEEE fp32 x / s, nearest-even E4M3, saturating), so the bytes
// equal those of quantising gathered rows.
constexpr int kDispatchThreads = 256;
constexpr int kDispatchTaskCols = 1024;

__device__ __forceinline__ uint4 load16_bf16(const uint16_t* src, int64_t c, int64_t k, bool vec) {
  if (vec && c + 8 <= k) return ld_nc_u4(src + c);
  uint32_t h[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) h[e] = c + e < k ? (uint32_t)src[c + e] : 0u;
  return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
}

__device__ __forceinline__ void store_codes(uint8_t* dst, uint2 code, int64_t c, int64_t k) {
  for (int e = 0; e < 8 && c + e < k; ++e) dst[e] = (uint8_t)(((e < 4 ? code.x : code.y) >> (8 * (e & 3))) & 0xFFu);
}

struct DispatchTask {
  uint4 v[2][2];   // this lane's 16 columns of each round
  int32_t row;     // lane j < topk: the row of the token's pair j
  int64_t c0;      // first column of the task
  int64_t token;
};

__device__ __forceinline__ void dispatch_load(DispatchTask& d, int64_t task, int64_t chunks,
                                              const uint16_t* __restrict__ x, int64_t k, int64_t ldx,
                                              const int32_t* __restrict__ row_of_pair, int32_t topk, int64_t rows,
                                              bool vec, int lane) {
  d.token = task / chunks;
  d.c0 = (task - d.token * chunks) * kDispatchTaskCols;
  d.row = lane < topk ? row_of_pair[d.token * topk + lane] : -1;
  if (d.row >= rows) d.row = -1;
  const uint16_t* src = x + d.token * ldx;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int64_t cr = d.c0 + 512 * i;
    const int64_t c = cr + 16 * lane;
    if (vec && cr + 512 <= k) {
      d.v[i][0] = ld_nc_u4(src + c);
      d.v[i][1] = ld_nc_u4(src + c + 8);
    } else if (cr < k) {
      d.v[i][0] = load16_bf16(src, c, k, vec);
      d.v[i][1] = load16_bf16(src, c + 8, k, vec);
    }
  }
}

template <bool UE8M0>
__device__ __forceinline__ void dispatch_store(const DispatchTask& d, int64_t k, int32_t topk, int64_t rows,
                                               uint8_t* __restrict__ q, int64_t ldq, void* __restrict__ scale,
                                               bool vec, int lane) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int64_t cr = d.c0 + 512 * i;
    if (cr >= k) break;  // warp-uniform: past the row
    const bool full = vec && cr + 512 <= k && ldq % 16 == 0;
    const int64_t c = cr + 16 * lane;
    uint32_t am = absmax_u4(absmax_u4(0u, d.v[i][0]), d.v[i][1]);
    am = max(am & 0xFFFFu, am >> 16);
#pragma unroll
    for (int s = 1; s < 8; s <<= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, s));
    const float amax = __uint_as_float(am << 16);
    uint2 c_lo, c_hi;
    uint32_t sbits;
    if (UE8M0) {
      const int e = scale_ue8m0_exponent(amax);
      const float f = exp2_neg(e);
      c_lo = quant8_mul(d.v[i][0], f);
      c_hi = quant8_mul(d.v[i][1], f);
      sbits = (uint32_t)(e + 127);
    } else {
      const float sc = scale_fp32(amax);
      const float r = __frcp_rn(sc);
      c_lo = quant8_div(d.v[i][0], sc, r);
      c_hi = quant8_div(d.v[i][1], sc, r);
      sbits = __float_as_uint(sc);
    }
    const uint4 code = make_uint4(c_lo.x, c_lo.y, c_hi.x, c_hi.y);
    const bool lead = (lane & 7) == 0 && c < k;  // the group's first lane writes its scale
    const int64_t sidx = (c / kBlock) * rows;
    for (int j = 0; j < topk; ++j) {
      const int32_t row = __shfl_sync(0xffffffffu, d.row, j);
      if (row < 0) continue;  // warp-uniform
      uint8_t* dst = q + (int64_t)row * ldq + c;
      if (full) {
        *reinterpret_cast<uint4*>(dst) = code;
      } else if (c < k) {
        if (vec && c + 16 <= k) {
          *reinterpret_cast<uint2*>(dst) = c_lo;
          *reinterpret_cast<uint2*>(dst + 8) = c_hi;
        } else {
          store_codes(dst, c_lo, c, k);
          if (c + 8 < k) store_codes(dst + 8, c_hi, c + 8, k);
        }
      }
      if (lead) {
        if (UE8M0)
          static_cast<uint8_t*>(scale)[sidx + row] = (uint8_t)sbits;
        else
          static_cast<float*>(scale)[sidx + row] = __uint_as_float(sbits);
      }
    }
  }
}

template <bool UE8M0>
__global__ void __launch_bounds__(kDispatchThreads) moe_dispatch_kernel(
    const uint16_t* __restrict__ x, int64_t tokens, int64_t k, int64_t ldx, const int32_t* __restrict__ row_of_pair,
    int32_t topk, int64_t rows, uint8_t* __restrict__ q, int64_t ldq, void* __restrict__ scale, int vec) {
  const int lane = threadIdx.x & 31;
  const int64_t chunks = (k + kDispatchTaskCols - 1) / kDispatchTaskCols;
  const int64_t tasks = tokens * chunks;
  const int64_t wc = (int64_t)gridDim.x * (kDispatchThreads / 32);
  const int64_t warp = (int64_t)blockIdx.x * (kDispatchThreads / 32) + (threadIdx.x >> 5);
  if (warp >= tasks) return;
  DispatchTask da, db;
  dispatch_load(da, warp, chunks, x, k, ldx, row_of_pair, topk, rows, vec, lane);
  // two tasks per trip, so that the two register sets keep fixed names
  for (int64_t t = warp; t < tasks; t += 2 * wc) {
    const int64_t t1 = t + wc, t2 = t + 2 * wc;
    if (t1 < tasks) dispatch_load(db, t1, chunks, x, k, ldx, row_of_pair, topk, rows, vec, lane);
    dispatch_store<UE8M0>(da, k, topk, rows, q, ldq, scale, vec, lane);
    if (t2 < tasks) dispatch_load(da, t2, chunks, x, k, ldx, row_of_pair, topk, rows, vec, lane);
    if (t1 < tasks) dispatch_store<UE8M0>(db, k, topk, rows, q, ldq, scale, vec, lane);
  }
}

template <typename K>
int ctas_per_sm(K kernel, int threads) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) n = 1;
  return n;
}

// One thread per (token, 16-byte piece of the output row), grid-strided.
// The token's slot rows and gates are read through L1 (all pieces of a token
// share them); the 8 source loads of a slot group are issued before their
// multiply-adds.
__global__ void __launch_bounds__(kCombineThreads) moe_combine_kernel(
    const uint16_t* __restrict__ y, int32_t y_rows, int64_t n, int64_t ldy, const int32_t* __restrict__ row_of_pair,
    const float* __restrict__ gate, int32_t tokens, int32_t topk, uint16_t* __restrict__ out, int64_t ldo,
    int32_t pieces, int vec) {
  const int32_t total = tokens * pieces;  // the host keeps this below 2^31
  for (int32_t i = blockIdx.x * kCombineThreads + threadIdx.x; i < total; i += gridDim.x * kCombineThreads) {
    const int32_t t = i / pieces;
    const int64_t c = (int64_t)(i - t * pieces) * 8;
    const bool full = vec && c + 8 <= n;
    const int32_t* rp = row_of_pair + (int64_t)t * topk;
    const float* gp = gate + (int64_t)t * topk;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    for (int j0 = 0; j0 < topk; j0 += 8) {
      int32_t rows[8];
      float ws[8];
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rows[j] = j0 + j < topk ? __ldg(rp + j0 + j) : -1;
        if (rows[j] >= y_rows) rows[j] = -1;  // a row y does not have adds nothing
        ws[j] = j0 + j < topk ? __ldg(gp + j0 + j) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[j] = (full && rows[j] >= 0) ? ld_nc_u4(y + (int64_t)rows[j] * ldy + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (rows[j] < 0) continue;
        if (full) {
          fma_piece(acc, ws[j], v[j]);
        } else {
          const uint16_t* src = y + (int64_t)rows[j] * ldy + c;
          for (int e = 0; e < 8 && c + e < n; ++e) acc[e] = fmaf(ws[j], bf16_lo((uint32_t)src[e]), acc[e]);
        }
      }
    }
    uint16_t* dst = out + (int64_t)t * ldo + c;
    if (full) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(bf16x2_rn(acc[0], acc[1]), bf16x2_rn(acc[2], acc[3]),
                                                  bf16x2_rn(acc[4], acc[5]), bf16x2_rn(acc[6], acc[7]));
    } else {
      for (int e = 0; e < 8 && c + e < n; ++e) dst[e] = (uint16_t)(bf16x2_rn(acc[e], 0.0f) & 0xFFFFu);
    }
  }
}

// asked once; concurrent first calls store the same value
int combine_ctas_per_sm() {
  static std::atomic<int> cached{0};
  int c = cached.load(std::memory_order_relaxed);
  if (c == 0) {
    c = ctas_per_sm(moe_combine_kernel, kCombineThreads);
    cached.store(c, std::memory_order_relaxed);
  }
  return c;
}

}  // namespace
}  // namespace fp8rl

using namespace fp8rl;

extern "C" FP8RL_API size_t fp8rl_moe_plan_workspace_size(int64_t tokens, int64_t topk, int64_t experts) {
  if (tokens < 0 || topk < 1 || topk > kMaxTopk || experts < 1 || experts > kPlanMaxExperts) return 0;
  const PlanShape s = plan_shape(tokens, topk);
  return (size_t)(std::max<int64_t>(s.tiles, 1) * experts * 4 + 255) / 256 * 256;
}

extern "C" FP8RL_API fp8rl_status fp8rl_moe_plan(const int32_t* d_topk, int64_t tokens, int64_t topk,
                                                 int64_t experts, int32_t* d_offsets, int32_t* d_row_of_pair,
                                                 int32_t* d_token_of_row, void* d_workspace,
                                                 size_t workspace_bytes, void* stream) {
  if (tokens < 0 || topk < 1 || topk > kMaxTopk || experts < 1) return FP8RL_ERR_INVALID_ARG;
  if (experts > kPlanMaxExperts || tokens * topk > (int64_t)INT32_MAX - 4096) return FP8RL_ERR_SHAPE;
  if (!d_offsets || !d_workspace || (tokens > 0 && (!d_topk || !d_row_of_pair || !d_token_of_row)))
    return FP8RL_ERR_INVALID_ARG;
  if (workspace_bytes < fp8rl_moe_plan_workspace_size(tokens, topk, experts)) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(d_topk, 4) || !aligned(d_offsets, 4) || !aligned(d_row_of_pair, 4) || !aligned(d_token_of_row, 4) ||
      !aligned(d_workspace, 4))
    return FP8RL_ERR_ALIGNMENT;
  const PlanShape s = plan_shape(tokens, topk);
  int32_t* base = static_cast<int32_t*>(d_workspace);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (s.pairs <= kSmallPlanPairs && experts <= kSmallPlanExperts) {
    moe_plan_small_kernel<<<1, 1024, (size_t)33 * experts * 4, cs>>>(d_topk, (int32_t)s.pairs, (int32_t)topk,
                                                                     (int32_t)experts, key_bits(experts), d_offsets,
                                                                     d_row_of_pair, d_token_of_row);
    return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
  }
  const size_t hist_bytes = (size_t)experts * 4;
  // shared memory: one int per expert, at most 32 KB (below the 48 KB default)
  if (s.tiles > 0)
    moe_count_kernel<<<(unsigned)s.tiles, 256, hist_bytes, cs>>>(d_topk, (int32_t)s.pairs, (int32_t)s.tile,
                                                                 (int32_t)experts, base);
  moe_scan_kernel<<<1, kScanThreads, hist_bytes, cs>>>(base, (int32_t)s.tiles, (int32_t)experts, d_offsets);
  if (s.tiles > 0)
    moe_rank_kernel<<<(unsigned)s.tiles, 32, hist_bytes, cs>>>(d_topk, (int32_t)s.pairs, (int32_t)s.tile,
                                                               (int32_t)topk, (int32_t)experts, key_bits(experts),
                                                               base, d_offsets,
                                                               d_row_of_pair, d_token_of_row);
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}

extern "C" FP8RL_API fp8rl_status fp8rl_moe_dispatch_quant(const void* x_bf16, int64_t tokens, int64_t k,
                                                           int64_t ldx, const int32_t* d_row_of_pair,
                                                           int64_t topk, int64_t rows, void* q_e4m3,
                                                           int64_t ldq, void* x_scale, fp8rl_scale_fmt fmt,
                                                           void* stream) {
  if (fmt != FP8RL_SCALE_FP32 && fmt != FP8RL_SCALE_UE8M0) return FP8RL_ERR_INVALID_ARG;
  if (tokens < 0 || rows < 0 || k < 0 || topk < 1 || topk > kMaxTopk || ldx < k || ldq < k)
    return FP8RL_ERR_INVALID_ARG;
  if (tokens == 0 || rows == 0 || k == 0) return FP8RL_OK;
  if (!x_bf16 || !q_e4m3 || !x_scale || !d_row_of_pair) return FP8RL_ERR_INVALID_ARG;
  if (rows > INT32_MAX) return FP8RL_ERR_SHAPE;
  if (!aligned(x_bf16, 16) || !aligned(q_e4m3, 16) || !aligned(d_row_of_pair, 4)) return FP8RL_ERR_ALIGNMENT;
  if (fmt == FP8RL_SCALE_FP32 && !aligned(x_scale, 4)) return FP8RL_ERR_ALIGNMENT;
  const int vec = (ldx * 2) % 16 == 0 && ldq % 8 == 0;
  static std::atomic<int> occ[2];  // asked once per format (zero until then)
  const int u = fmt == FP8RL_SCALE_UE8M0;
  int resident = occ[u].load(std::memory_order_relaxed);
  if (resident == 0) {
    resident = u ? ctas_per_sm(moe_dispatch_kernel<true>, kDispatchThreads)
                 : ctas_per_sm(moe_dispatch_kernel<false>, kDispatchThreads);
    occ[u].store(resident, std::memory_order_relaxed);
  }
  // one wave of resident CTAs (the SMs share the tasks evenly; a warp's
  // tasks overlap its neighbours' on the same SM)
  const int64_t tasks = tokens * ((k + kDispatchTaskCols - 1) / kDispatchTaskCols);
  const int64_t ctas = (tasks + kDispatchThreads / 32 - 1) / (kDispatchThreads / 32);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)sm_count() * resident));
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  uint8_t* q = static_cast<uint8_t*>(q_e4m3);
  if (u)
    moe_dispatch_kernel<true><<<(unsigned)grid, kDispatchThreads, 0, cs>>>(x, tokens, k, ldx, d_row_of_pair,
                                                                          (int32_t)topk, rows, q, ldq, x_scale, vec);
  else
    moe_dispatch_kernel<false><<<(unsigned)grid, kDispatchThreads, 0, cs>>>(x, tokens, k, ldx, d_row_of_pair,
                                                                           (int32_t)topk, rows, q, ldq, x_scale, vec);
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}

extern "C" FP8RL_API fp8rl_status fp8rl_moe_combine(const void* y_bf16, int64_t rows, int64_t n, int64_t ldy,
                                                    const int32_t* d_row_of_pair, const float* d_gate,
                                                    int64_t tokens, int64_t topk, void* out_bf16, int64_t ldo,
                                                    void* stream) {
  if (rows < 0 || n < 0 || tokens < 0 || topk < 1 || topk > kMaxTopk || ldy < n || ldo < n)
    return FP8RL_ERR_INVALID_ARG;
  if (tokens == 0 || n == 0) return FP8RL_OK;
  if ((rows > 0 && !y_bf16) || !d_row_of_pair || !d_gate || !out_bf16) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(y_bf16, 2) || !aligned(out_bf16, 2) || !aligned(d_row_of_pair, 4) || !aligned(d_gate, 4))
    return FP8RL_ERR_ALIGNMENT;
  const int64_t pieces = (n + 7) / 8;
  if (rows > INT32_MAX || tokens * pieces > (int64_t)INT32_MAX - (1 << 20)) return FP8RL_ERR_SHAPE;
  const int vec = aligned(y_bf16, 16) && aligned(out_bf16, 16) && (ldy * 2) % 16 == 0 && (ldo * 2) % 16 == 0;
  const int64_t ctas = (tokens * pieces + kCombineThreads - 1) / kCombineThreads;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)sm_count() * combine_ctas_per_sm()));
  moe_combine_kernel<<<(unsigned)grid, kCombineThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(y_bf16), (int32_t)rows, n, ldy, d_row_of_pair, d_gate, (int32_t)tokens, (int32_t)topk,
      static_cast<uint16_t*>(out_bf16), ldo, (int32_t)pieces, vec);
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}
