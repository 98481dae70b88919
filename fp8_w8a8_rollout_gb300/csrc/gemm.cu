// gemm.cu -- block-scaled W8A8 GEMMs on sm_103a tensor cores (tcgen05 + TMEM).
//
//   Y[m][n] = bf16_rne( sum_kb sx[kb][m] * sw[n/128][kb] * P_kb[m][n] )
//
// P_kb is the product of the E4M3 tiles over one 128-wide K chunk, accumulated
// in fp32 by the tensor cores; the two chunk scales are applied in fp32 on the
// way out of TMEM and Y is rounded to bf16 once ("FP8-RL", "Core method":
// compute-level W8A8 linears with 128x128 weight blocks; "Where Rounding
// Happens Matters": keep fp32 inside the fused region, round once).
//
// One CTA computes a 128 x BN output tile (BN = 128 or 256):
//   warp 0, one lane   TMA producer: per K chunk, a 128x128 E4M3 tile of X and a
//                      BN x 128 tile of W (128-byte swizzle) into a ring of
//                      shared-memory stages;
//   warp 1, one lane   MMA issuer: four tcgen05.mma (M=128, N=BN, K=32) per chunk
//                      into one of two TMEM accumulators, then commits;
//   warps 2, 3         idle (they complete warpgroup 0);
//   warps 4..          epilogue, 64 accumulator columns per warp (four warps per
//                      column slice cover the 128 TMEM lanes): per chunk,
//                      tcgen05.ld the partial product, fold
//                      it into fp32 registers with sx * sw, release the TMEM
//                      buffer (so the tensor cores fill the other one meanwhile);
//                      finally round to bf16 and store.
// Every mbarrier wait is bounded; a wait that runs out raises a CTA abort flag
// and the device error word, and all roles leave through the common teardown,
// which releases TMEM.
//
// The MoE grouped variant is the same kernel over row segments: CTA x-index ->
// (expert, 128-row tile of that expert's segment) from the device offsets;
// rows past the segment end are computed and not stored.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8rl {

void* static_gemm_scratch(size_t need_bytes, size_t clear_bytes, fp8rl_status* status);  // static_scratch.cu
// decode.cu: dense products with at most 128 rows, operands swapped (UNSUPPORTED: use this file's kernel)
fp8rl_status decode_gemm(const void* xq, const void* x_scale, const void* wq, const void* w_scale, void* y,
                         int64_t rows, int64_t n, int64_t k, bool ue8m0, uint32_t* err, uint64_t timeout_ns,
                         int fault_skip_kb, int force_splits, cudaStream_t stream);
// decode.cu: the same with the 1x128 activation quantisation inside (at most 16 rows)
fp8rl_status decode_gemm_qx(const void* x_bf16, int64_t ldx, const void* wq, const void* w_scale, void* y,
                            int64_t rows, int64_t n, int64_t k, bool ue8m0, void* xq_out, void* sx_out,
                            uint32_t* err, uint64_t timeout_ns, int fault_skip_kb, int force_splits,
                            cudaStream_t stream);

namespace {

using namespace ptx;

constexpr int kBM = 128;     // tile rows (tcgen05 M)
constexpr int kBK = 128;     // K chunk: one scale block, one 128-byte swizzle row
constexpr int kUmmaK = 32;   // K of one E4M3 tcgen05.mma

// EPI 0: bf16 Y.  EPI 1: the fused gate-up epilogue (SiLU(gate) * up kept in
// fp32, quantised to E4M3 in 1x128 groups); needs 256-wide tiles.
// OUT: finished tiles leave through shared memory and TMA stores (one
// 32-row x 64-column bf16 box per epilogue warp, in a slot of its own), which
// takes the operand ring down to what fits beside the slots.
// MX: UE8M0 scales applied by the tensor cores (tcgen05.mma kind::mxf8f6f4
// with scale factors in TMEM): one accumulator per tile instead of one per K
// chunk, so the epilogue reads TMEM once per tile.
template <int BN, int AROWS = kBM, int EPI = 0, bool OUT = false, bool MX = false>
struct Cfg {
  static constexpr int kStageBytesRaw = AROWS * kBK + BN * kBK;
  static constexpr int kCols = 64;                      // accumulator columns per epilogue thread
  static constexpr int kEpiWarps = 4 * (BN / kCols);    // 4 TMEM lane quadrants x column slices
  static constexpr int kOutSlotBytes = 32 * kCols * 2;  // one warp's 32 x 64 bf16 box
  static constexpr int kOutBytes = OUT ? kEpiWarps * kOutSlotBytes : 0;
  // chunk-scale ring filled by the scale-loader warp: per K chunk the tile's
  // 128 activation scales and its BN/128 weight scales, as fp32.  MX needs no
  // ring in shared memory: the epilogue warps write the scale factors of each
  // group of four consecutive K chunks into one of kScaleSlots TMEM slots
  static constexpr int kScaleSlots = 16;
  static constexpr int kScaleSlotFloats = kBM + 4;
  static constexpr int kScaleRingBytes = MX ? 0 : kScaleSlots * kScaleSlotFloats * 4;
  // TMEM columns: MX keeps its accumulators in [0, 256) and the scale factors
  // of each slot in 16 columns from 256 on: row r of A's factor in lane r,
  // column r / 32; column n of B's in lane n mod 32 of every lane quadrant,
  // column 4 + n / 32.  The MMA picks a byte of each 32-bit cell (one per
  // 32-wide K block); our scales are per 128-wide chunk, so all four K blocks
  // of a chunk use the same byte and the cell's four bytes hold four
  // consecutive chunks: chunk c reads byte c mod 4 of slot (c / 4) mod slots
  static constexpr int kMxSfCol0 = 256;
  static constexpr int kMxSfColsPerSlot = 16;
  static_assert(!MX || kMxSfCol0 + kScaleSlots * kMxSfColsPerSlot <= 512, "MX scale factors fit in TMEM");
  static_assert(!MX || 4 + 4 * (BN / 128) <= kMxSfColsPerSlot, "MX scale factors of one chunk");
  // operand stages: as many as fit in about 200 KB of shared memory, or, with
  // the output slots, in the 227 KB a CTA may use
  static constexpr int kStagesFit =
      OUT ? (227 * 1024 - 3 * 1024 - 1024 - kOutBytes - kScaleRingBytes - (EPI ? 2 * 4 * 128 * 4 : 0) -
             3 * 256 * 4) /
                kStageBytesRaw
          : (200 * 1024) / kStageBytesRaw;
  static constexpr int kStages = kStagesFit > 12 ? 12 : kStagesFit;
  static constexpr int kThreads = 128 + kEpiWarps * 32; // warpgroup 0: producer, MMA, two idle warps
  // K chunks handed from the MMA issuer to the epilogue per synchronisation:
  // a 128-wide tile's TMEM buffer holds two chunk partials side by side
  static constexpr int kGroup = (BN == 128 && !MX) ? 2 : 1;
  // TMEM accumulator buffers (all 512 columns; MX: the 256 below its scale factors)
  static constexpr int kAccBufs = MX ? 256 / BN : 512 / (BN * kGroup);
  static constexpr int kTmemCols = 512;
  static constexpr int kABytes = AROWS * kBK;  // activation rows loaded per stage
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBookBytes = 1024;  // barriers and small shared state
  // fused epilogue: per-row maxima of the four column slices, two tiles deep
  static constexpr int kRedBytes = EPI ? 2 * 4 * kBM * 4 : 0;
  static constexpr int kTileCacheBytes = 3 * 256 * 4;  // grouped: the experts' segments (TileMap)
  static constexpr int kSharedEnd = kStages * kStageBytes + kBookBytes + kScaleRingBytes + kRedBytes + kTileCacheBytes;
  static constexpr int kOutOffset = (kSharedEnd + 1023) / 1024 * 1024;  // 1024-aligned for the 128-byte swizzle
  static constexpr int kSmemBytes = 1024 + (OUT ? kOutOffset + kOutBytes : kSharedEnd);
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(EPI == 0 || BN == 256, "the fused epilogue pairs 128 gate with 128 up columns");
  static_assert(!MX || (EPI == 0 && AROWS == kBM), "MX: plain bf16 epilogue, 128-row activation stages");
  static constexpr int kPartPitch = BN + 4;  // floats per row of a split-K partial tile
  static_assert(kBM * kPartPitch * 4 <= kStages * kStageBytes, "partial tile must fit over the stages");
  static_assert((2 * kStages + 2 * kAccBufs + 2 * kScaleSlots + 2) * 8 + 16 <= kBookBytes, "bookkeeping");
  // register split for BN = 256 (640 threads launch with <= 96 each): the role
  // warpgroup gives registers back, the four epilogue warpgroups take them.
  // 128 * kRoleRegs + 512 * kEpiRegs must not exceed 640 * (registers at
  // launch); the host checks that before launching.
  static constexpr bool kSplitRegs = BN == 256;
  static constexpr int kRoleRegs = 56;
  static constexpr int kRoleRegsStreamK = 64;  // its schedule state needs a little more
  static constexpr int kEpiRegs = 104;
  // MX: the epilogue keeps no running sums; the role warps get more
  // (measured: below 80 they spill a little, 72 with 96 epilogue registers
  // still fits the launch's allocation)
  static constexpr int kRoleRegsMx = 80;
  static constexpr int kEpiRegsMx = 96;
  static constexpr int kMinLaunchRegs =
      (128 * (kRoleRegsStreamK > kRoleRegs ? kRoleRegsStreamK : kRoleRegs) + kEpiWarps * 32 * kEpiRegs + kThreads - 1) /
      kThreads;
};

struct GemmArgs {
  const void* sx;            // [K/128][rows], fp32 or UE8M0 bytes
  const void* sw;            // [experts][N/128][K/128]
  __nv_bfloat16* y;          // [rows][N]
  const int32_t* offsets;    // device [experts + 1], or null: one segment [0, rows)
  int32_t rows, n, k, experts;
  uint32_t* err;
  uint64_t timeout_ns;
  int32_t fault_skip_kb;     // test hook: the producer never fills this K chunk (-1: off)
  int32_t wait_mode;         // bit 0: producer and MMA threads poll; bit 1: epilogue polls
  int32_t l2_prefetch;       // K chunks ahead of the shared-memory loads that are prefetched into L2
  int32_t splits;            // K splits; > 1 only for a launch in clusters of `splits` CTAs along z
  // stream-K (cooperative launch): partial tiles meet in a caller-provided workspace
  // fused gate-up epilogue: h = SiLU(gate) * up, [rows][n / 2] E4M3 codes and
  // [n / 256][rows] scales (the weight's 128-row blocks alternate gate, up)
  uint8_t* hq;
  void* h_scale;
  uint32_t* ws_head;         // [0] epoch of the last completed launch, [1] CTAs finished in this launch
  uint32_t* ws_flag;         // [gridDim.x] slot of CTA b holds this launch's partial: == epoch + 1
  // [gridDim.x][BN / 4][32] float4: one 128 x BN fp32 partial tile per CTA,
  // stored as each epilogue thread holds it (warp, 4-column step, lane), so
  // that every warp-wide access is 512 contiguous bytes
  float* ws_part;
};

// The (tile, first K chunk, end K chunk) segments one CTA works through, in
// order.  Data-parallel: whole tiles blockIdx.x, +gridDim.x, ...  Stream-K: the
// CTA's share of all tiles' K iterations, which may begin inside one tile and
// end inside another.  Split-K cluster: one segment of the CTA's own tile.
// kernel schedules
constexpr int kDataParallel = 0;  // persistent CTAs stride over whole tiles
constexpr int kSplitK = 1;        // one tile per cluster, its K chunks split over the cluster's CTAs
constexpr int kStreamK = 2;       // the K iterations of all tiles divided evenly over the CTAs

template <int MODE>
struct Schedule {
  // data-parallel (and the first part of stream-K): u = next whole tile, below
  // dp_tiles.  Stream-K: then the CTA's share [v, v_end) of the K iterations of
  // the remaining tiles.  Split-K cluster: the CTA's K chunks [u, v_end), once.
  // (The host keeps gridDim.x x the stream-K iteration count below 2^31.)
  int u, dp_tiles, num_kb;
  int v, v_end;
  __device__ __forceinline__ bool next(int& t, int& lo, int& hi) {
    if (MODE == kSplitK) {
      if (u > (int)v_end) return false;
      t = 0;
      lo = u;
      hi = (int)v_end;
      u = (int)v_end + 1;
      return true;
    }
    if (u < dp_tiles) {
      t = u;
      u += gridDim.x;
      lo = 0;
      hi = num_kb;
      return true;
    }
    if (MODE != kStreamK || v >= v_end) return false;
    const int r = v / num_kb;
    t = dp_tiles + r;
    lo = v - r * num_kb;
    hi = min(num_kb, lo + (v_end - v));
    v += hi - lo;
    return true;
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Stream-K tile owner, for one thread's n4 x 4 columns: `srow` (shared
// memory) holds this CTA's partial; the same values of the partial tile of
// every CTA after this one whose K range starts inside the tile (the tile's
// iterations end at tile_end) are added in CTA order, each once its flag shows
// this launch's epoch.  part0: the thread's first float4 in slot 0; the next
// steps follow 32 float4 apart.  Warp-collective.  Kept out of line so that
// its registers are not added to the epilogue's.
__device__ __noinline__ bool streamk_fold(float4* srow, const float* part0, int64_t slot_floats,
                                          const uint32_t* flags, uint32_t epoch, uint32_t tile_end, uint32_t iters,
                                          int n4, bool row_ok, volatile int* abortv, uint32_t* err,
                                          uint64_t timeout_ns) {
  for (uint32_t q = blockIdx.x + 1; q < gridDim.x && q * iters / gridDim.x < tile_end; ++q) {
    bool ok = flag_wait_bounded(flags + q, epoch, abortv, err, timeout_ns);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    if (!row_ok) continue;
    const float* part = part0 + (int64_t)q * slot_floats;
#pragma unroll 8
    for (int j = 0; j < n4; ++j) {
      const float4 v = ld_cg_f32x4(part + 128 * j);
      float4 w = srow[j];
      w.x += v.x;
      w.y += v.y;
      w.z += v.z;
      w.w += v.w;
      srow[j] = w;
    }
  }
  return true;
}

// Calls fn(t, lo, nseg) for the segments of this CTA in order, while fn
// returns true.  The data-parallel and split-K kernels keep a plain loop over
// whole tiles (the role warps' loops are latency-critical: measured on GB300,
// driving them through the general schedule cost the data-parallel kernel
// ~4%); only the stream-K kernel walks the general schedule.
template <int MODE, typename F>
__device__ __forceinline__ void for_each_segment(const Schedule<MODE>& s0, int total_tiles, F&& fn) {
  if constexpr (MODE == kStreamK) {
    Schedule<MODE> s = s0;
    int t, lo, hi;
    while (s.next(t, lo, hi))
      if (!fn(t, lo, hi - lo)) return;
  } else if constexpr (MODE == kSplitK) {
    fn(0, s0.u, s0.v_end - s0.u);
  } else {
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x)
      if (!fn(t, 0, s0.num_kb)) return;
  }
}

// Scales are fetched as the aligned 32-bit word that holds them (a UE8M0 byte
// sits inside its word; the word never crosses the end of the allocation's
// last 4-byte unit, so it cannot leave mapped memory).
template <bool UE8M0>
__device__ __forceinline__ const void* scale_word(const void* p, int64_t idx) {
  if (UE8M0) return static_cast<const uint8_t*>(p) + (idx & ~(int64_t)3);
  return static_cast<const float*>(p) + idx;
}

// idx: the scale's element index, or only its low 32 bits (the byte position
// within the word is idx mod 4)
template <bool UE8M0>
__device__ __forceinline__ float scale_value(uint32_t word, uint32_t idx) {
  if (UE8M0) {
    const uint32_t b = (word >> (8 * (idx & 3))) & 0xFFu;
    return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
  }
  return __uint_as_float(word);
}


// Rows of the m-tile with index m_idx: (expert, first row, end of the expert's
// segment).  Dense: one segment [0, rows).  Grouped: a running prefix over the
// experts of their 128-row tile counts, 32 experts per step.  Warp-collective.
struct TileRows {
  int expert, row0, seg_end;
};

__device__ __forceinline__ TileRows tile_rows(const GemmArgs& a, int m_idx, int lane) {
  if (a.offsets == nullptr) return TileRows{0, m_idx * kBM, a.rows};
  TileRows tr{-1, 0, 0};
  int done = 0;
  for (int e0 = 0; e0 < a.experts && tr.expert < 0; e0 += 32) {
    const int ex = e0 + lane;
    int start = 0, end = 0;
    if (ex < a.experts) {
      start = min(max(a.offsets[ex], 0), a.rows);
      end = min(max(a.offsets[ex + 1], 0), a.rows);
      end = max(end, start);
    }
    const int tiles = (end - start + kBM - 1) / kBM;
    int incl = tiles;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const int excl = incl - tiles;
    const bool hit = tiles > 0 && m_idx >= done + excl && m_idx < done + incl;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      const int src = __ffs(m) - 1;
      tr.expert = __shfl_sync(0xffffffffu, ex, src);
      tr.row0 = __shfl_sync(0xffffffffu, start, src) + (m_idx - done - __shfl_sync(0xffffffffu, excl, src)) * kBM;
      tr.seg_end = __shfl_sync(0xffffffffu, end, src);
    }
    done += __shfl_sync(0xffffffffu, incl, 31);
  }
  return tr;
}

// number of 128-row tiles over all segments (warp-collective)
__device__ __forceinline__ int count_m_tiles(const GemmArgs& a, int lane) {
  if (a.offsets == nullptr) return (a.rows + kBM - 1) / kBM;
  int total = 0;
  for (int e0 = 0; e0 < a.experts; e0 += 32) {
    const int ex = e0 + lane;
    int tiles = 0;
    if (ex < a.experts) {
      const int start = min(max(a.offsets[ex], 0), a.rows);
      const int end = max(min(max(a.offsets[ex + 1], 0), a.rows), start);
      tiles = (end - start + kBM - 1) / kBM;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) tiles += __shfl_xor_sync(0xffffffffu, tiles, off);
    total += tiles;
  }
  return total;
}

// Grouped products with at most kTileCacheExperts experts keep each expert's
// segment (start, end) and the running count of m-tiles in shared memory,
// built once per CTA, so that every role finds a tile's rows with a binary
// search there instead of a scan over the offsets in global memory per tile
// (measured on GB300: the scan's round trips stalled the producer at every
// tile boundary of the MoE expert GEMMs).
constexpr int kTileCacheExperts = 256;
struct TileMap {
  // shared-memory address of [0, E) segment starts (clamped as in
  // tile_rows), [E, 2E) segment ends, [2E, 3E) m-tiles of experts 0..e,
  // E = kTileCacheExperts
  uint32_t t;
  bool cached;
  __device__ __forceinline__ int get(int i) const {
    int v;
    asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(t + 4u * (uint32_t)i));
    return v;
  }
  __device__ __forceinline__ void put(int i, int v) const {
    asm volatile("st.shared.s32 [%0], %1;" ::"r"(t + 4u * (uint32_t)i), "r"(v) : "memory");
  }
  __device__ __forceinline__ int start(int e) const { return get(e); }
  __device__ __forceinline__ int end(int e) const { return get(kTileCacheExperts + e); }
  __device__ __forceinline__ int incl(int e) const { return get(2 * kTileCacheExperts + e); }
};

// fills the map (warp-collective; one warp) and returns the m-tile count
__device__ __forceinline__ int build_tile_map(const GemmArgs& a, const TileMap& tm, int lane) {
  int carry = 0;
  for (int e0 = 0; e0 < a.experts; e0 += 32) {
    const int ex = e0 + lane;
    int start = 0, end = 0;
    if (ex < a.experts) {
      start = min(max(a.offsets[ex], 0), a.rows);
      end = min(max(a.offsets[ex + 1], 0), a.rows);
      end = max(end, start);
    }
    const int tiles = (end - start + kBM - 1) / kBM;
    int incl = tiles;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (ex < a.experts) {
      tm.put(ex, start);
      tm.put(kTileCacheExperts + ex, end);
      tm.put(2 * kTileCacheExperts + ex, carry + incl);
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  return carry;
}

// tile_rows from the map: the expert is the first whose running tile count
// exceeds m_idx (experts without tiles never are); not warp-collective
__device__ __forceinline__ TileRows tile_rows_cached(const GemmArgs& a, const TileMap& tm, int m_idx) {
  int lo = 0, hi = a.experts - 1;
  if (hi < 0 || tm.incl(hi) <= m_idx) return TileRows{-1, 0, 0};
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (tm.incl(mid) > m_idx) hi = mid; else lo = mid + 1;
  }
  const int start = tm.start(lo), end = tm.end(lo);
  const int tiles = (end - start + kBM - 1) / kBM;
  return TileRows{lo, start + (m_idx - (tm.incl(lo) - tiles)) * kBM, end};
}

// AROWS < 128 (decode-sized M, at most AROWS rows in the only m-tile): each
// stage holds just AROWS activation rows; the M = 128 MMA reads the rest of
// its A rows from whatever shared memory follows, which only feeds accumulator
// rows >= AROWS that are never stored.
// OUT: finished tiles leave through shared memory and TMA stores (data-
// parallel kernels with 128-row tiles; the host chooses it per launch).
// MX: UE8M0 scales applied by the tensor cores (data-parallel tiles, bf16 out).
template <int BN, int AROWS, bool UE8M0, int MODE, int EPI = 0, bool OUT = false, bool MX = false>
__global__ void __launch_bounds__(Cfg<BN, AROWS, EPI>::kThreads, 1)
    gemm_blockscaled_kernel(const __grid_constant__ CUtensorMap tmap_x,
                            const __grid_constant__ CUtensorMap tmap_w,
                            const __grid_constant__ CUtensorMap tmap_y, const GemmArgs a) {
  static_assert(!OUT || (MODE == kDataParallel && EPI == 0 && AROWS == kBM), "staged output: data-parallel tiles");
  static_assert(!MX || (UE8M0 && MODE == kDataParallel), "MX: UE8M0 scales, data-parallel tiles");
  using C = Cfg<BN, AROWS, EPI, OUT, MX>;
  static_assert(EPI == 0 || MODE == kDataParallel, "the fused epilogue needs whole tiles");
  constexpr bool SPLITK = MODE == kSplitK;
  constexpr bool STREAMK = MODE == kStreamK;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + C::kStages * C::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(base_ptr + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + C::kAccBufs;
  uint64_t* drain = tempty + C::kAccBufs;
  uint64_t* sfull = drain + 1;                // scale slot filled (1 arrival: the loader)
  uint64_t* sempty = sfull + C::kScaleSlots;  // scale slot read (one arrival per epilogue warp; MX: the MMA
                                              // thread's commit once the copy into TMEM has read it)
  uint64_t* published = sempty + C::kScaleSlots;  // stream-K partial stored (one arrival per epilogue warp)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(published + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* shared_m_tiles = abort_flag + 1;
  uint32_t* shared_epoch = reinterpret_cast<uint32_t*>(shared_m_tiles + 1);
  float* scale_ring = reinterpret_cast<float*>(base_ptr + C::kStages * C::kStageBytes + C::kBookBytes);
  float* row_max = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(scale_ring) + C::kScaleRingBytes);  // EPI 1
  // (the map is rebuilt from base_ptr and the parameters at each use, so it
  // holds no registers across the role loops)
#define FP8RL_TMAP                                                                                    \
  TileMap {                                                                                           \
    base + (uint32_t)(C::kStages * C::kStageBytes + C::kBookBytes + C::kScaleRingBytes + C::kRedBytes), \
        a.offsets != nullptr && a.experts <= kTileCacheExperts                                        \
  }
  uint8_t* out_slots = base_ptr + C::kOutOffset;                         // OUT only

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_kb = a.k / kBK;
  const int n_tiles = a.n / BN;
  // split-K: one tile per CTA (m-tile blockIdx.x, n-tile blockIdx.y), this
  // CTA's K chunks [kb_lo, kb_lo + nloc); the partial tiles of a cluster are
  // summed through distributed shared memory at the end.  Otherwise the CTA is
  // persistent: tiles blockIdx.x, blockIdx.x + gridDim.x, ...
  const int splits = SPLITK ? a.splits : 1;
  const int split = SPLITK ? (int)cluster_ctarank() : 0;
  const int kb_lo = (int)((int64_t)num_kb * split / splits);
  const int nloc = (int)((int64_t)num_kb * (split + 1) / splits) - kb_lo;

  if (warp == 0) {
    const int mt = SPLITK ? 0 : (FP8RL_TMAP.cached ? build_tile_map(a, FP8RL_TMAP, lane) : count_m_tiles(a, lane));
    if (lane == 0) *shared_m_tiles = mt;
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), C::kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(published), C::kEpiWarps);
    for (int q = 0; q < C::kScaleSlots; ++q) {
      mbar_init(smem_u32(&sfull[q]), MX ? 4 : 1);  // MX: one epilogue warp per lane quadrant
      mbar_init(smem_u32(&sempty[q]), MX ? 1 : C::kEpiWarps);
    }
    *abort_flag = 0;
    // stream-K flags of this launch carry the value epoch + 1; the epoch in the
    // workspace header advances only after every CTA has read it (below)
    if (STREAMK) *shared_epoch = ld_acquire_gpu(a.ws_head) + 1;
    fence_barrier_init();
  }
  __syncthreads();
  const int m_tiles = *shared_m_tiles;
  const int total_tiles = SPLITK ? 1 : m_tiles * n_tiles;
  Schedule<MODE> sched0;
  sched0.num_kb = num_kb;
  // stream-K: whole waves of tiles first (data-parallel, in the same order as
  // the data-parallel kernel); the last partial wave plus one full wave are
  // divided by K iterations
  int sk_tiles = 0;
  if (STREAMK) {
    const int rem = total_tiles % (int)gridDim.x;
    sk_tiles = rem == 0 ? 0 : rem + (total_tiles >= (int)gridDim.x ? (int)gridDim.x : 0);
  }
  const int sk_iters = sk_tiles * num_kb;
  if (SPLITK) {
    sched0.u = kb_lo;
    sched0.dp_tiles = 0;
    sched0.v = kb_lo + nloc;
    sched0.v_end = kb_lo + nloc;
  } else {
    sched0.u = blockIdx.x;
    sched0.dp_tiles = total_tiles - sk_tiles;
    sched0.v = STREAMK ? (int)(blockIdx.x * (uint32_t)sk_iters / gridDim.x) : 0;
    sched0.v_end = STREAMK ? (int)((blockIdx.x + 1) * (uint32_t)sk_iters / gridDim.x) : 0;
  }
  // The last stream-K CTA to finish advances the workspace epoch: every CTA
  // read the old one before it counted itself as finished.
  auto streamk_finish = [&]() {
    if (STREAMK && threadIdx.x == 0) {
      const uint32_t before = atom_add_acq_rel_gpu(a.ws_head + 1, 1u);
      if (before == gridDim.x - 1) {
        a.ws_head[1] = 0;
        st_release_gpu(a.ws_head, *shared_epoch);
      }
    }
  };
  // CTA-uniform: nothing to do (more CTAs than tiles or iterations)
  if (!SPLITK && sched0.u >= sched0.dp_tiles && sched0.v >= sched0.v_end) {
    streamk_finish();
    return;
  }
  auto tile_coords = [&](int t, int& m_idx, int& n_tile) {
    if (SPLITK) {
      m_idx = blockIdx.x;
      n_tile = blockIdx.y;
    } else if (a.offsets == nullptr) {
      // dense: m-tile fastest, so that the tiles in flight share a few weight
      // n-tiles and the whole (smaller) activation matrix stays in L2
      m_idx = t % m_tiles;
      n_tile = t / m_tiles;
    } else {
      // grouped: n-tile fastest, so that each activation tile is read once for
      // all n-tiles of its expert and each expert's weights serve its few
      // m-tiles back to back
      m_idx = t / n_tiles;
      n_tile = t % n_tiles;
    }
  };

  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abortv = abort_flag;

  if (warp < 4) {
    // the UE8M0 scale loader (byte decode) with staged tile stores runs
    // better with the stream-K budget (measured on GB300: 8192 x 24576 x 4096
    // 788 -> 756 us); with register stores the extra registers cost 4-7%
    if (C::kSplitRegs)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(MX ? C::kRoleRegsMx
                                                             : (STREAMK || (UE8M0 && OUT)) ? C::kRoleRegsStreamK
                                                                                           : C::kRoleRegs));
    if constexpr (!STREAMK) {
      // Data-parallel and split-K: plain loops over whole tiles (or the
      // cluster's one tile).  These loops are latency-critical; measured on
      // GB300, driving them through the general segment schedule (below)
      // cost the data-parallel kernel ~4% (fp32 scales) to ~9% (UE8M0).
      const int first_tile = SPLITK ? 0 : (int)blockIdx.x;
      const int tile_stride = SPLITK ? 1 : (int)gridDim.x;
        if (warp == 0) {
          // ---------------------------------------------------------- TMA producer
          if (lane == 0) {
            prefetch_tensormap(&tmap_x);
            prefetch_tensormap(&tmap_w);
          }
          uint32_t g = 0;  // chunks issued by this CTA so far (position in the stage ring)
          bool alive = true;
          for (int t = first_tile; t < total_tiles && alive; t += tile_stride) {
            int m_idx, n_tile;
            tile_coords(t, m_idx, n_tile);
            const TileRows tr = (FP8RL_TMAP.cached ? tile_rows_cached(a, FP8RL_TMAP, m_idx) : tile_rows(a, m_idx, lane));
            if (lane == 0) {
              const int wrow0 = tr.expert * a.n + n_tile * BN;
              for (int it = 0; it < nloc; ++it, ++g) {
                const int kb = kb_lo + it;
                const int s = g % C::kStages;
                const uint32_t ph = (g / C::kStages) & 1;
                if (!mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1, abortv, a.err, a.timeout_ns, !(a.wait_mode & 1))) {
                  alive = false;
                  break;
                }
                if ((int)g == a.fault_skip_kb) continue;
                if (a.l2_prefetch > 0 && it + a.l2_prefetch < nloc) {
                  tma_prefetch_l2_2d(&tmap_x, (kb + a.l2_prefetch) * kBK, tr.row0);
                  tma_prefetch_l2_2d(&tmap_w, (kb + a.l2_prefetch) * kBK, wrow0);
                }
                const uint32_t fb = smem_u32(&full[s]);
                mbar_arrive_expect_tx(fb, C::kStageBytes);
                tma_load_2d(sA + s * C::kABytes, &tmap_x, kb * kBK, tr.row0, fb);
                tma_load_2d(sB + s * C::kBBytes, &tmap_w, kb * kBK, wrow0, fb);
              }
            }
            alive = __shfl_sync(0xffffffffu, alive, 0);
          }
          if (lane == 0 && *abortv) {
            // let the copies still in flight land before shared memory is released
            for (uint32_t j = g > (uint32_t)C::kStages ? g - C::kStages : 0; j < g; ++j) {
              if ((int)j == a.fault_skip_kb) continue;
              mbar_wait_bounded(smem_u32(&full[j % C::kStages]), (j / C::kStages) & 1, nullptr, nullptr, 10000000ull);
            }
          }
          __syncwarp();
        } else if (warp == 1) {
          // ---------------------------------------------------------- MMA issuer
          if (lane == 0 && MX) {
            // One accumulator per tile: per K chunk, four block-scaled MMAs
            // (32-wide K blocks) accumulate into it, all reading the chunk's
            // scale-factor byte c mod 4 of its group's TMEM slot.  The MMA
            // thread waits for a slot once per group of four chunks (once the
            // epilogue warps have written it) and releases it after the
            // group's last chunk; a slot is rewritten only after that commit.
            const int my_tiles = (total_tiles - first_tile + tile_stride - 1) / tile_stride;
            const uint32_t total_chunks = (uint32_t)my_tiles * (uint32_t)nloc;
            uint32_t g = 0;   // chunks consumed (stage ring position)
            uint32_t gs = 0;  // chunks consumed (scale-factor position)
            bool alive = true;
            for (int tt = 0; tt < my_tiles && alive; ++tt) {
              const int buf = tt % C::kAccBufs;
              const uint32_t bph = (tt / C::kAccBufs) & 1;
              if (!mbar_wait_bounded(smem_u32(&tempty[buf]), bph ^ 1, abortv, a.err, a.timeout_ns,
                                     !(a.wait_mode & 1))) {
                alive = false;
                break;
              }
              const uint32_t d = tmem + buf * BN;
              for (int it = 0; it < nloc; ++it, ++g, ++gs) {
                const int s = g % C::kStages;
                const uint32_t grp = gs >> 2, j = gs & 3u;
                const int q = grp % C::kScaleSlots;
                if (!mbar_wait_bounded(smem_u32(&full[s]), (g / C::kStages) & 1, abortv, a.err, a.timeout_ns,
                                       !(a.wait_mode & 1)) ||
                    (j == 0 && !mbar_wait_bounded(smem_u32(&sfull[q]), (grp / C::kScaleSlots) & 1, abortv, a.err,
                                                  a.timeout_ns, !(a.wait_mode & 1)))) {
                  alive = false;
                  break;
                }
                tc_fence_after();
                const uint32_t sf_t = tmem + C::kMxSfCol0 + q * C::kMxSfColsPerSlot;
                const uint32_t a0 = sA + s * C::kABytes, b0 = sB + s * C::kBBytes;
                const uint32_t idesc = idesc_mx_e4m3_ue8m0(kBM, BN, 0, 0) | (j << 4) | (j << 29);
#pragma unroll
                for (int k = 0; k < kBK / kUmmaK; ++k)
                  mma_mx_e4m3(d, sw128_kmajor_desc(a0 + k * kUmmaK), sw128_kmajor_desc(b0 + k * kUmmaK), idesc,
                              sf_t, sf_t + 4, (it > 0 || k > 0) ? 1u : 0u);
                mma_commit(smem_u32(&empty[s]));
                if (j == 3 || gs + 1 == total_chunks) mma_commit(smem_u32(&sempty[q]));
              }
              if (alive) mma_commit(smem_u32(&tfull[buf]));
            }
            if (*abortv) {
              // no MMA or copy may still be using TMEM when it is released
              mma_commit(smem_u32(drain));
              mbar_wait_bounded(smem_u32(drain), 0, nullptr, nullptr, 10000000ull);
            }
          } else if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
            const int my_tiles = (total_tiles - first_tile + tile_stride - 1) / tile_stride;
            uint32_t g = 0;  // chunks consumed (stage ring position)
            uint32_t c = 0;  // chunk groups handed to the epilogue (TMEM ring position)
            bool alive = true;
            for (int tt = 0; tt < my_tiles && alive; ++tt) {
              for (int it = 0; it < nloc && alive; it += C::kGroup, ++c) {
                const int gsz = min(C::kGroup, nloc - it);
                const int buf = c % C::kAccBufs;
                const uint32_t bph = (c / C::kAccBufs) & 1;
                if (!mbar_wait_bounded(smem_u32(&tempty[buf]), bph ^ 1, abortv, a.err, a.timeout_ns,
                                       !(a.wait_mode & 1))) {
                  alive = false;
                  break;
                }
                for (int j = 0; j < gsz; ++j, ++g) {
                  const int s = g % C::kStages;
                  const uint32_t ph = (g / C::kStages) & 1;
                  if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abortv, a.err, a.timeout_ns, !(a.wait_mode & 1))) {
                    alive = false;
                    break;
                  }
                  tc_fence_after();
                  const uint32_t d = tmem + (buf * C::kGroup + j) * BN;
                  const uint32_t a0 = sA + s * C::kABytes, b0 = sB + s * C::kBBytes;
                  #pragma unroll
                  for (int k = 0; k < kBK / kUmmaK; ++k)
                    mma_e4m3(d, sw128_kmajor_desc(a0 + k * kUmmaK), sw128_kmajor_desc(b0 + k * kUmmaK), idesc,
                             k > 0 ? 1u : 0u);
                  mma_commit(smem_u32(&empty[s]));
                }
                if (alive) mma_commit(smem_u32(&tfull[buf]));
              }
            }
            if (*abortv) {
              // no MMA may still be writing TMEM when it is released
              mma_commit(smem_u32(drain));
              mbar_wait_bounded(smem_u32(drain), 0, nullptr, nullptr, 10000000ull);
            }
          }
          __syncwarp();
        } else if (warp == 2 && !MX) {
          // ---------------------------------------------------------- scale loader
          // Runs up to kScaleSlots K chunks ahead of the epilogue, so the latency
          // of these small loads never paces the pipeline.  Lane l loads the
          // activation scales of rows l, l+32, l+64, l+96 of the tile.
          uint32_t gs = 0;
          bool alive = true;
          for (int t = first_tile; t < total_tiles && alive; t += tile_stride) {
            int m_idx, n_tile;
            tile_coords(t, m_idx, n_tile);
            // (the scan: the map's lookup would not fit the role warps'
            // registers here, and this warp runs kScaleSlots chunks ahead)
            const TileRows tr = tile_rows(a, m_idx, lane);
            const int64_t sw_row = ((int64_t)tr.expert * (a.n / 128) + (n_tile * BN >> 7)) * num_kb;
            // batches of kLoadBatch chunks: all their loads first, then the stores
            constexpr int kLoadBatch = 4;
            for (int it0 = 0; it0 < nloc && alive; it0 += kLoadBatch) {
              // raw words first (all loads of the batch in flight), decoded at the store
              uint32_t v[kLoadBatch][4];
              uint32_t w[kLoadBatch];
              int64_t vi[kLoadBatch][4], wi[kLoadBatch];
              #pragma unroll
              for (int b = 0; b < kLoadBatch; ++b) {
                const int kb = kb_lo + it0 + b;
                const bool live = it0 + b < nloc;
                #pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int grow = tr.row0 + lane + 32 * j;
                  vi[b][j] = (int64_t)kb * a.rows + grow;
                  v[b][j] = (live && grow < tr.seg_end)
                                ? __ldg(static_cast<const uint32_t*>(scale_word<UE8M0>(a.sx, vi[b][j])))
                                : 0u;
                }
                wi[b] = sw_row + (int64_t)(lane < BN / 128 ? lane : 0) * num_kb + kb;
                w[b] = (live && lane < BN / 128) ? __ldg(static_cast<const uint32_t*>(scale_word<UE8M0>(a.sw, wi[b])))
                                                   : 0u;
              }
              #pragma unroll
              for (int b = 0; b < kLoadBatch; ++b) {
                if (it0 + b >= nloc) break;
                const int q = gs % C::kScaleSlots;
                const uint32_t ph = (gs / C::kScaleSlots) & 1;
                const bool got = mbar_wait_bounded(smem_u32(&sempty[q]), ph ^ 1, abortv, a.err, a.timeout_ns,
                                                   !(a.wait_mode & 1));
                alive = __all_sync(0xffffffffu, got);
                if (!alive) break;
                float* slot = scale_ring + q * C::kScaleSlotFloats;
                #pragma unroll
                for (int j = 0; j < 4; ++j)
                  slot[lane + 32 * j] = tr.row0 + lane + 32 * j < tr.seg_end ? scale_value<UE8M0>(v[b][j], vi[b][j]) : 0.0f;
                if (lane < BN / 128) slot[kBM + lane] = scale_value<UE8M0>(w[b], wi[b]);
                __syncwarp();  // orders the lanes' stores before lane 0's release
                if (lane == 0) mbar_arrive(smem_u32(&sfull[q]));
                ++gs;
              }
            }
          }
        }
    } else {
      // stream-K: the CTA's segments, possibly starting and ending inside tiles
      if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
          prefetch_tensormap(&tmap_x);
          prefetch_tensormap(&tmap_w);
        }
        uint32_t g = 0;  // chunks issued by this CTA so far (position in the stage ring)
        bool alive = true;
        for_each_segment<MODE>(sched0, total_tiles, [&](int t, int lo, int nseg) {
          int m_idx, n_tile;
          tile_coords(t, m_idx, n_tile);
          const TileRows tr = (FP8RL_TMAP.cached ? tile_rows_cached(a, FP8RL_TMAP, m_idx) : tile_rows(a, m_idx, lane));
          if (lane == 0) {
            const int wrow0 = tr.expert * a.n + n_tile * BN;
            for (int it = 0; it < nseg; ++it, ++g) {
              const int kb = lo + it;
              const int s = g % C::kStages;
              const uint32_t ph = (g / C::kStages) & 1;
              if (!mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1, abortv, a.err, a.timeout_ns, !(a.wait_mode & 1))) {
                alive = false;
                break;
              }
              if ((int)g == a.fault_skip_kb) continue;
              if (a.l2_prefetch > 0 && it + a.l2_prefetch < nseg) {
                tma_prefetch_l2_2d(&tmap_x, (kb + a.l2_prefetch) * kBK, tr.row0);
                tma_prefetch_l2_2d(&tmap_w, (kb + a.l2_prefetch) * kBK, wrow0);
              }
              const uint32_t fb = smem_u32(&full[s]);
              mbar_arrive_expect_tx(fb, C::kStageBytes);
              tma_load_2d(sA + s * C::kABytes, &tmap_x, kb * kBK, tr.row0, fb);
              tma_load_2d(sB + s * C::kBBytes, &tmap_w, kb * kBK, wrow0, fb);
            }
          }
          alive = __shfl_sync(0xffffffffu, alive, 0);
          return alive;
        });
        if (lane == 0 && *abortv) {
          // let the copies still in flight land before shared memory is released
          for (uint32_t j = g > (uint32_t)C::kStages ? g - C::kStages : 0; j < g; ++j) {
            if ((int)j == a.fault_skip_kb) continue;
            mbar_wait_bounded(smem_u32(&full[j % C::kStages]), (j / C::kStages) & 1, nullptr, nullptr, 10000000ull);
          }
        }
        __syncwarp();
      } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
          constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
          uint32_t g = 0;  // chunks consumed (stage ring position)
          uint32_t c = 0;  // chunk groups handed to the epilogue (TMEM ring position)
          bool alive = true;
          for_each_segment<MODE>(sched0, total_tiles, [&](int, int, int nseg) {
            for (int it = 0; it < nseg && alive; it += C::kGroup, ++c) {
              const int gsz = min(C::kGroup, nseg - it);
              const int buf = c % C::kAccBufs;
              const uint32_t bph = (c / C::kAccBufs) & 1;
              if (!mbar_wait_bounded(smem_u32(&tempty[buf]), bph ^ 1, abortv, a.err, a.timeout_ns,
                                     !(a.wait_mode & 1))) {
                alive = false;
                break;
              }
              for (int j = 0; j < gsz; ++j, ++g) {
                const int s = g % C::kStages;
                const uint32_t ph = (g / C::kStages) & 1;
                if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abortv, a.err, a.timeout_ns, !(a.wait_mode & 1))) {
                  alive = false;
                  break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (buf * C::kGroup + j) * BN;
                const uint32_t a0 = sA + s * C::kABytes, b0 = sB + s * C::kBBytes;
  #pragma unroll
                for (int k = 0; k < kBK / kUmmaK; ++k)
                  mma_e4m3(d, sw128_kmajor_desc(a0 + k * kUmmaK), sw128_kmajor_desc(b0 + k * kUmmaK), idesc,
                           k > 0 ? 1u : 0u);
                mma_commit(smem_u32(&empty[s]));
              }
              if (alive) mma_commit(smem_u32(&tfull[buf]));
            }
            return alive;
          });
          if (*abortv) {
            // no MMA may still be writing TMEM when it is released
            mma_commit(smem_u32(drain));
            mbar_wait_bounded(smem_u32(drain), 0, nullptr, nullptr, 10000000ull);
          }
        }
        __syncwarp();
      } else if (warp == 2) {
        // ---------------------------------------------------------- scale loader
        // Runs up to kScaleSlots K chunks ahead of the epilogue, so the latency
        // of these small loads never paces the pipeline.  Lane l loads the
        // activation scales of rows l, l+32, l+64, l+96 of the tile.
        uint32_t gs = 0;
        bool alive = true;
        for_each_segment<MODE>(sched0, total_tiles, [&](int t, int lo, int nseg) {
          int m_idx, n_tile;
          tile_coords(t, m_idx, n_tile);
          const TileRows tr = (FP8RL_TMAP.cached ? tile_rows_cached(a, FP8RL_TMAP, m_idx) : tile_rows(a, m_idx, lane));
          const int64_t sw_row = ((int64_t)tr.expert * (a.n / 128) + (n_tile * BN >> 7)) * num_kb;
          // batches of kLoadBatch chunks: all their loads first, then the stores
          constexpr int kLoadBatch = 4;
          // low bits of the scales' element indices (a UE8M0 scale's byte
          // position within its word) are recomputed at the store: this kernel
          // has fewer registers to spare
          const int64_t wbase = sw_row + (int64_t)(lane < BN / 128 ? lane : 0) * num_kb;
          for (int it0 = 0; it0 < nseg && alive; it0 += kLoadBatch) {
            // raw words first (all loads of the batch in flight), decoded at the store
            uint32_t v[kLoadBatch][4];
            uint32_t w[kLoadBatch];
#pragma unroll
            for (int b = 0; b < kLoadBatch; ++b) {
              const int kb = lo + it0 + b;
              const bool live = it0 + b < nseg;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int grow = tr.row0 + lane + 32 * j;
                v[b][j] = (live && grow < tr.seg_end)
                              ? __ldg(static_cast<const uint32_t*>(scale_word<UE8M0>(a.sx, (int64_t)kb * a.rows + grow)))
                              : 0u;
              }
              w[b] = (live && lane < BN / 128)
                         ? __ldg(static_cast<const uint32_t*>(scale_word<UE8M0>(a.sw, wbase + kb)))
                         : 0u;
            }
#pragma unroll
            for (int b = 0; b < kLoadBatch; ++b) {
              if (it0 + b >= nseg) break;
              const int q = gs % C::kScaleSlots;
              const uint32_t ph = (gs / C::kScaleSlots) & 1;
              const bool got = mbar_wait_bounded(smem_u32(&sempty[q]), ph ^ 1, abortv, a.err, a.timeout_ns,
                                                 !(a.wait_mode & 1));
              alive = __all_sync(0xffffffffu, got);
              if (!alive) break;
              float* slot = scale_ring + q * C::kScaleSlotFloats;
              const uint32_t kb = (uint32_t)(lo + it0 + b);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int grow = tr.row0 + lane + 32 * j;
                slot[lane + 32 * j] =
                    grow < tr.seg_end ? scale_value<UE8M0>(v[b][j], kb * (uint32_t)a.rows + (uint32_t)grow) : 0.0f;
              }
              if (lane < BN / 128) slot[kBM + lane] = scale_value<UE8M0>(w[b], (uint32_t)wbase + kb);
              __syncwarp();  // orders the lanes' stores before lane 0's release
              if (lane == 0) mbar_arrive(smem_u32(&sfull[q]));
              ++gs;
            }
          }
          return alive;
        });
      } else if (STREAMK && lane == 0) {
        // ---------------------------------------------------------- publisher
        // A CTA whose stream-K share starts inside a tile computes that tile's
        // later K chunks first and publishes the partial: once every epilogue
        // warp has stored its part, the flag of this CTA's slot is raised.  A
        // warp that gave up never arrives; then nothing is published, and the
        // tile's owner gives up as well.
        if (sched0.v < sched0.v_end && sched0.v % num_kb != 0 &&
            mbar_wait_bounded(smem_u32(published), 0, abortv, a.err, a.timeout_ns, !(a.wait_mode & 2)) && !*abortv)
          st_release_gpu(a.ws_flag + blockIdx.x, *shared_epoch);
      }
    }
  } else {
    if (C::kSplitRegs) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(MX ? C::kEpiRegsMx : C::kEpiRegs));
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 4;
    const int quad = warp & 3;   // TMEM lanes this warp may read: 32*quad .. +31
    const int slice = ew >> 2;   // which kCols columns of the tile
    const int r = quad * 32 + lane;
    // EPI 0: columns [kCols * slice, +kCols).  EPI 1: gate columns
    // [32 * slice, +32) and the matching up columns 128 further on.
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16) + (EPI ? 32 * slice : slice * C::kCols);
    uint32_t tiles_done = 0;  // fused epilogue: which half of row_max
    uint32_t g = 0;   // chunk groups folded so far (TMEM ring position)
    uint32_t gs = 0;  // chunks whose scales were taken (scale ring position)
    bool ok = true;
    // MX: the epilogue warps write the scale factors of this CTA's K chunks
    // (numbered across its tiles) into TMEM, four consecutive chunks per slot
    // (one per byte of each cell); group G is written by the four warps of
    // slice G mod (kEpiWarps / 4), one per lane quadrant, up to kMxLead
    // chunks ahead of the tile being accumulated.  A warp writes every
    // kEpiWarps / 4-th group, so its scale loads have that many groups of
    // MMAs to arrive in.
    constexpr int kMxStep = C::kEpiWarps / 4;
    constexpr uint32_t kMxLead = 4 * (C::kScaleSlots / 2);  // chunks of lead into the next tile
    // (the count for every kernel: the block-scaled ones alone use it)
    const uint32_t mx_total =
        (uint32_t)((total_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x) * (uint32_t)num_kb;
    uint32_t mx_next = (uint32_t)slice;  // this warp's next group to write
    uint32_t mx_tile = 0;                // tiles of this CTA drained so far
    // write group mx_next's scale factors into its TMEM slot once the MMAs
    // that last read the slot have completed; false when a wait ran out
    auto mx_write = [&]() -> bool {
      const uint32_t grp = mx_next;
      mx_next += kMxStep;
      uint32_t xw = 0u, b0 = 0u, b1 = 0u;  // cell bytes: byte j for chunk 4 grp + j
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t c = 4u * grp + (uint32_t)j;
        uint32_t xb = 127u, wb0 = 127u, wb1 = 127u;
        if (c < mx_total) {
          const int tseq = (int)(c / (uint32_t)num_kb), kbc = (int)(c - (uint32_t)tseq * (uint32_t)num_kb);
          int mi, nt;
          tile_coords((int)blockIdx.x + tseq * (int)gridDim.x, mi, nt);
          const TileRows st = (FP8RL_TMAP.cached ? tile_rows_cached(a, FP8RL_TMAP, mi) : tile_rows(a, mi, lane));  // warp-collective
          const int srow = st.row0 + quad * 32 + lane;
          if (srow < st.seg_end) {
            const int64_t xi = (int64_t)kbc * a.rows + srow;
            xb = (__ldg(static_cast<const uint32_t*>(scale_word<true>(a.sx, xi))) >> (8 * ((uint32_t)xi & 3u))) &
                 0xFFu;
          }
          const int64_t wi = ((int64_t)st.expert * (a.n / 128) + (nt * BN >> 7)) * num_kb + kbc;
          wb0 = (__ldg(static_cast<const uint32_t*>(scale_word<true>(a.sw, wi))) >> (8 * ((uint32_t)wi & 3u))) &
                0xFFu;
          wb1 = wb0;
          if (BN == 256)
            wb1 = (__ldg(static_cast<const uint32_t*>(scale_word<true>(a.sw, wi + num_kb))) >>
                   (8 * ((uint32_t)(wi + num_kb) & 3u))) &
                  0xFFu;
        }
        xw |= xb << (8 * j);
        b0 |= wb0 << (8 * j);
        b1 |= wb1 << (8 * j);
      }
      const int q = grp % C::kScaleSlots;
      bool got = mbar_wait_bounded(smem_u32(&sempty[q]), ((grp / C::kScaleSlots) & 1) ^ 1, abortv, a.err,
                                   a.timeout_ns, !(a.wait_mode & 2));
      got = __all_sync(0xffffffffu, got);
      if (!got) return false;
      tc_fence_after();
      const uint32_t sf = tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::kMxSfCol0 + q * C::kMxSfColsPerSlot;
      tmem_st_32x32b_x1(sf + quad, xw);
      const uint32_t bw[8] = {b0, b0, b0, b0, b1, b1, b1, b1};
      tmem_st_32x32b_x8(sf + 4, bw);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sfull[q]));
      return true;
    };
    Schedule<MODE> sch = sched0;
    int t, lo, hi;
    while (ok && sch.next(t, lo, hi)) {
      const int nseg = hi - lo;
      int m_idx, n_tile;
      tile_coords(t, m_idx, n_tile);
      // (the fused epilogue keeps the scan: the map's lookup would not leave
      // it the registers it holds)
      const TileRows tr =
          (EPI == 0 && FP8RL_TMAP.cached) ? tile_rows_cached(a, FP8RL_TMAP, m_idx) : tile_rows(a, m_idx, lane);
      const int n0 = n_tile * BN;
      const int grow = tr.row0 + r;
      const bool row_ok = grow < tr.seg_end;
      const bool warp_idle = AROWS < kBM && tr.row0 + quad * 32 >= tr.seg_end;  // warp-uniform
      const int nb = (n0 + slice * C::kCols) >> 7;
      // fp32 accumulators as packed pairs (fma.rn.f32x2: two round-to-nearest
      // FMAs per instruction, the same results as scalar FMAs)
      uint64_t acc[C::kCols / 2];
#pragma unroll
      for (int j = 0; j < C::kCols / 2; ++j) acc[j] = 0ull;
      const int sw_lane = nb - (n0 >> 7);  // which of the tile's weight scales
      if constexpr (MX) {
        // scale factors up to kMxLead chunks into the next tile, so the
        // MMA thread can start it while this tile drains and stores
        const uint32_t lim = min(mx_total, (mx_tile + 1) * (uint32_t)num_kb + kMxLead);
        while (ok && 4u * mx_next < lim) ok = mx_write();
        ++mx_tile;
        // the whole tile's scaled sum is in one accumulator: read this
        // thread's 64 columns and hand the buffer back to the MMA thread
        const int buf = g % C::kAccBufs;
        const uint32_t bph = (g / C::kAccBufs) & 1;
        ++g;
        ok = mbar_wait_bounded(smem_u32(&tfull[buf]), bph, abortv, a.err, a.timeout_ns, !(a.wait_mode & 2));
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < C::kCols / 32; ++cc) {
            uint64_t v[16];
            tmem_ld_32x32b_x32_pairs(t_lane + buf * BN + cc * 32, v);
#pragma unroll
            for (int q = 0; q < 16; ++q) acc[cc * 16 + q] = v[q];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
        }
      }
      for (int it = 0; !MX && it < nseg; it += C::kGroup, ++g) {
        const int gsz = min(C::kGroup, nseg - it);
        const int buf = g % C::kAccBufs;
        const uint32_t bph = (g / C::kAccBufs) & 1;
        ok = mbar_wait_bounded(smem_u32(&tfull[buf]), bph, abortv, a.err, a.timeout_ns, !(a.wait_mode & 2));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; j < gsz; ++j, ++gs) {
          const int q = gs % C::kScaleSlots;
          ok = mbar_wait_bounded(smem_u32(&sfull[q]), (gs / C::kScaleSlots) & 1, abortv, a.err, a.timeout_ns,
                                 !(a.wait_mode & 2));
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          const float* slot = scale_ring + q * C::kScaleSlotFloats;
          const float f = slot[r] * slot[kBM + (EPI ? 0 : sw_lane)];
          const float f_up = EPI ? slot[r] * slot[kBM + 1] : f;  // the up half's weight block
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sempty[q]));  // the values are in registers
          if (warp_idle) continue;  // every row of this warp is past the segment
          const uint32_t taddr = t_lane + (buf * C::kGroup + j) * BN;
          if constexpr (!C::kSplitRegs && EPI == 0 && C::kCols == 64) {
            // registers to spare (no split): the chunk's 64 columns in one
            // TMEM round trip instead of two
            const uint64_t f2 = f32x2(f, f);
            uint64_t v[32];
            tmem_ld_32x32b_x64_pairs(taddr, v);
#pragma unroll
            for (int q = 0; q < 32; ++q) acc[q] = fma_f32x2(v[q], f2, acc[q]);
          } else {
#pragma unroll
            for (int cc = 0; cc < C::kCols / 32; ++cc) {
              const float fc = cc == 0 ? f : f_up;
              const uint64_t f2 = f32x2(fc, fc);
              uint64_t v[16];
              tmem_ld_32x32b_x32_pairs(taddr + cc * (EPI ? 128 : 32), v);
#pragma unroll
              for (int q = 0; q < 16; ++q) acc[cc * 16 + q] = fma_f32x2(v[q], f2, acc[cc * 16 + q]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));  // one arrival per warp
      }
      if constexpr (EPI == 1) {
        // h = SiLU(gate) * up for this thread's 32 columns, kept in fp32 (the
        // single rounding of the fused region is the E4M3 one below); SiLU
        // with the fast exponential and division intrinsics (a few ulp)
        float hmax = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float g0, g1, u0, u1;
          f32x2_unpack(acc[j], g0, g1);
          f32x2_unpack(acc[16 + j], u0, u1);
          const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
          const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
          acc[j] = f32x2(h0, h1);
          hmax = fmaxf(hmax, fmaxf(fabsf(h0), fabsf(h1)));
        }
        // the group is the row's 128 h columns, held by the four warps of this
        // TMEM lane quadrant: their maxima meet in shared memory (two buffers:
        // a warp may start the next tile's exchange while another still reads
        // this one) behind the quadrant's own barrier
        float* red = row_max + (tiles_done++ & 1) * 4 * kBM;
        red[slice * kBM + r] = hmax;
        asm volatile("bar.sync %0, 128;" ::"r"(1 + quad) : "memory");
        // every warp reaches its quadrant's barrier for every tile (a warp whose
        // wait ran out still finishes the tile), and all of them leave here
        // once any wait has run out
        if (*abortv) break;
        const float amax = fmaxf(fmaxf(red[r], red[kBM + r]), fmaxf(red[2 * kBM + r], red[3 * kBM + r]));
        if (ok && row_ok &&
            dcheck(grow < a.rows && n_tile * 128 + slice * 32 + 32 <= a.n / 2 && n_tile < a.n / 256, a.err)) {
          uint32_t w[8];
          if (UE8M0) {
            const int e = scale_ue8m0_exponent(amax);
            const float fs = exp2_neg(e);
            const uint64_t f2 = f32x2(fs, fs);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float h0, h1, h2, h3;
              f32x2_unpack(mul_f32x2(acc[2 * j], f2), h0, h1);
              f32x2_unpack(mul_f32x2(acc[2 * j + 1], f2), h2, h3);
              w[j] = e4m3x2(h0, h1) | (e4m3x2(h2, h3) << 16);
            }
            if (slice == 0) static_cast<uint8_t*>(a.h_scale)[(int64_t)n_tile * a.rows + grow] = (uint8_t)(e + 127);
          } else {
            const float sc = scale_fp32(amax);
            const float rc = __frcp_rn(sc);
            if (sc >= kFastDivMinScale) {
              // the correctly rounded quotient h / sc, on pairs (formed from
              // -h so that every rounding, signed zeros included, matches the
              // scalar sequence q0 = h r, e = q0 sc - h, q = q0 - e r)
              const uint64_t s2 = f32x2(sc, sc), nr2 = f32x2(-rc, -rc);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                uint32_t half[2];
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                  const uint64_t nx = acc[2 * j + p] ^ 0x8000000080000000ull;
                  const uint64_t q0 = mul_f32x2(nx, nr2);
                  const uint64_t e = fma_f32x2(q0, s2, nx);
                  float q_lo, q_hi;
                  f32x2_unpack(fma_f32x2(e, nr2, q0), q_lo, q_hi);
                  half[p] = e4m3x2(q_lo, q_hi);
                }
                w[j] = half[0] | (half[1] << 16);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                float h[4];
                f32x2_unpack(acc[2 * j], h[0], h[1]);
                f32x2_unpack(acc[2 * j + 1], h[2], h[3]);
                w[j] = e4m3x2(__fdiv_rn(h[0], sc), __fdiv_rn(h[1], sc)) |
                       (e4m3x2(__fdiv_rn(h[2], sc), __fdiv_rn(h[3], sc)) << 16);
              }
            }
            if (slice == 0) static_cast<float*>(a.h_scale)[(int64_t)n_tile * a.rows + grow] = sc;
          }
          uint4* dst = reinterpret_cast<uint4*>(a.hq + (int64_t)grow * (a.n / 2) + n_tile * 128 + slice * 32);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        continue;
      }
      bool store_y = !SPLITK;
      if (STREAMK && !(lo == 0 && hi == num_kb)) {
        if (lo > 0) {
          // a later part of tile t (a CTA has at most one, in its first
          // stream-K segment): publish the partial in this CTA's slot
          store_y = false;
          if (ok && row_ok) {
            float4* slot = reinterpret_cast<float4*>(a.ws_part + (int64_t)blockIdx.x * kBM * BN) +
                           ew * (C::kCols / 4) * 32 + lane;
#pragma unroll
            for (int j = 0; j < C::kCols / 4; ++j) {
              float4 v;
              f32x2_unpack(acc[2 * j], v.x, v.y);
              f32x2_unpack(acc[2 * j + 1], v.z, v.w);
              slot[32 * j] = v;
            }
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(published));  // warp 3 raises the flag
        } else {
          // the head of tile t, which is this CTA's last segment: every MMA has
          // completed, so the operand stages are idle.  The accumulators wait
          // there (padded rows, as for split-K) while the parts that the
          // following CTAs published are added in CTA order; the sums leave
          // from there.
          store_y = false;
          float4* srow = reinterpret_cast<float4*>(reinterpret_cast<float*>(base_ptr) + r * C::kPartPitch +
                                                   slice * C::kCols);
#pragma unroll
          for (int j = 0; j < C::kCols / 4; ++j) {
            float4 v;
            f32x2_unpack(acc[2 * j], v.x, v.y);
            f32x2_unpack(acc[2 * j + 1], v.z, v.w);
            srow[j] = v;
          }
          const bool folded =
              streamk_fold(srow, a.ws_part + (int64_t)(ew * (C::kCols / 4) * 32 + lane) * 4, (int64_t)kBM * BN, a.ws_flag,
                           *shared_epoch, (uint32_t)((t - sch.dp_tiles + 1) * num_kb), (uint32_t)sk_iters,
                           C::kCols / 4, ok && row_ok, abortv, a.err, a.timeout_ns);
          if (folded && ok && row_ok && !*abortv &&
              dcheck(grow < a.rows && n0 + slice * C::kCols + C::kCols <= a.n, a.err)) {
            uint4* dst = reinterpret_cast<uint4*>(a.y + (int64_t)grow * a.n + n0 + slice * C::kCols);
            const bool wide = (reinterpret_cast<uintptr_t>(a.y) & 31) == 0;
#pragma unroll 1
            for (int j = 0; j < C::kCols / 16; ++j) {
              const float4 s0 = srow[4 * j], s1 = srow[4 * j + 1], s2 = srow[4 * j + 2], s3 = srow[4 * j + 3];
              const uint4 h0 = make_uint4(pack_bf16x2(s0.x, s0.y), pack_bf16x2(s0.z, s0.w),
                                          pack_bf16x2(s1.x, s1.y), pack_bf16x2(s1.z, s1.w));
              const uint4 h1 = make_uint4(pack_bf16x2(s2.x, s2.y), pack_bf16x2(s2.z, s2.w),
                                          pack_bf16x2(s3.x, s3.y), pack_bf16x2(s3.z, s3.w));
              if (wide) {
                st_global_v8(dst + 2 * j, h0, h1);
              } else {
                dst[2 * j] = h0;
                dst[2 * j + 1] = h1;
              }
            }
          }
        }
      }
      if (store_y) {
        bool staged = false;
        if constexpr (OUT) {
          // The warp's 32-row x 64-column box goes to its shared slot in the
          // 128-byte swizzled layout (16-byte chunk c of row r at position
          // c ^ (r mod 8): 8 lanes cover all banks) and leaves in one TMA
          // store, so the warp moves on without waiting for global memory.
          // Dense boxes may run past the last row (the store clips them);
          // grouped boxes must lie inside the expert's segment, else the rows
          // go out one by one below.
          const int box_row0 = tr.row0 + quad * 32;
          const bool box_ok = a.offsets == nullptr ? box_row0 < a.rows : box_row0 + 32 <= tr.seg_end;
          if (__all_sync(0xffffffffu, ok && box_ok && !*abortv &&
                                     dcheck(box_row0 < a.rows && n0 + slice * C::kCols + C::kCols <= a.n, a.err))) {
            uint8_t* slot = out_slots + ew * C::kOutSlotBytes;
            if (lane == 0) bulk_wait_group_read0();  // this slot's previous box has been read
            __syncwarp();
#pragma unroll
            for (int c = 0; c < C::kCols / 8; ++c) {
              float x[8];
#pragma unroll
              for (int q = 0; q < 4; ++q) f32x2_unpack(acc[4 * c + q], x[2 * q], x[2 * q + 1]);
              *reinterpret_cast<uint4*>(slot + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                  make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                             pack_bf16x2(x[6], x[7]));
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmap_y, smem_u32(slot), n0 + slice * C::kCols, box_row0);
              bulk_commit_group();
            }
            staged = true;
          }
        }
        if (!staged && ok && row_ok && !*abortv &&
            dcheck(grow < a.rows && n0 + slice * C::kCols + C::kCols <= a.n, a.err)) {
          // the row segment leaves as full 32-byte sectors (one 256-bit store
          // per 16 columns) when the output allows it
          uint4* dst = reinterpret_cast<uint4*>(a.y + (int64_t)grow * a.n + n0 + slice * C::kCols);
          const bool wide = (reinterpret_cast<uintptr_t>(a.y) & 31) == 0;
#pragma unroll
          for (int j = 0; j < C::kCols / 16; ++j) {
            uint4 h[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float x[8];
#pragma unroll
              for (int q = 0; q < 4; ++q) f32x2_unpack(acc[8 * j + 4 * e + q], x[2 * q], x[2 * q + 1]);
              h[e] = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                                pack_bf16x2(x[6], x[7]));
            }
            if (wide) {
              st_global_v8(dst + 2 * j, h[0], h[1]);
            } else {
              dst[2 * j] = h[0];
              dst[2 * j + 1] = h[1];
            }
          }
        }
      } else if (SPLITK && row_ok) {
        // this split's fp32 partial tile, row-major with a 4-float pad per row,
        // over the operand stages (every MMA that read them has completed)
        float4* prow = reinterpret_cast<float4*>(reinterpret_cast<float*>(base_ptr) + r * C::kPartPitch +
                                                 slice * C::kCols);
#pragma unroll
        for (int j = 0; j < C::kCols / 4; ++j) {
          float4 v;
          f32x2_unpack(acc[2 * j], v.x, v.y);
          f32x2_unpack(acc[2 * j + 1], v.z, v.w);
          prow[j] = v;
        }
      }
    }
    if constexpr (OUT) {
      // every TMA store of this warp has completed before shared memory is
      // released and the kernel ends
      if (lane == 0) bulk_wait_group0();
      __syncwarp();
    }
  }
  if (SPLITK) {
    // sum the cluster's partial tiles: rank `split` owns a run of 8-column
    // chunks of every valid row; the (row, chunk) items are spread over all
    // epilogue threads (neighbouring threads take neighbouring chunks), each
    // issues every rank's loads before adding them in rank order, then rounds
    // to bf16 once
    cluster_sync();
    if (warp >= 4) {
      const TileRows tr = tile_rows(a, blockIdx.x, lane);
      const int rows = min(kBM, tr.seg_end - tr.row0);
      const int n0 = blockIdx.y * BN;
      constexpr int kChunks = BN / 8;
      const int ch_lo = kChunks * split / splits, ch_hi = kChunks * (split + 1) / splits;
      const int nch = ch_hi - ch_lo;
      const uint32_t part0 = smem_u32(base_ptr);
      if (!*abortv && nch > 0) {
        for (int item = threadIdx.x - 128; item < rows * nch; item += C::kEpiWarps * 32) {
          const int r = item / nch, ch = ch_lo + (item - r * nch);
          const uint32_t src = part0 + (uint32_t)(r * C::kPartPitch + ch * 8) * 4u;
          float4 u[8], w[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q < splits) {
              const uint32_t ra = mapa_shared(src, (uint32_t)q);
              u[q] = ld_dsmem_f32x4(ra);
              w[q] = ld_dsmem_f32x4(ra + 16);
            }
          float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q < splits) {
              x[0] += u[q].x; x[1] += u[q].y; x[2] += u[q].z; x[3] += u[q].w;
              x[4] += w[q].x; x[5] += w[q].y; x[6] += w[q].z; x[7] += w[q].w;
            }
          if (dcheck(tr.row0 + r < a.rows && n0 + ch * 8 + 8 <= a.n, a.err))
          *reinterpret_cast<uint4*>(a.y + (int64_t)(tr.row0 + r) * a.n + n0 + ch * 8) =
              make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                         pack_bf16x2(x[6], x[7]));
        }
      }
    }
    cluster_sync();  // no CTA leaves while its partial may still be read
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  streamk_finish();
}

#undef FP8RL_TMAP

// ---------------------------------------------------------------- tensor-core pairs
//
// UE8M0 products on tensor-core pairs: a cluster of two CTAs on neighbouring
// SMs computes a 256 x 256 output tile with tcgen05 cta_group::2.  Per K chunk
// each CTA loads its own 128 activation rows and its half (128 rows) of the
// tile's 256 weight rows, 32 KB instead of the 48 KB that a 128 x 256 tile of
// one CTA needs for the same work per SM (measured on GB300, operand delivery
// is what bounds the one-CTA tile).  The even CTA's MMA thread issues
// block-scaled M = 256 MMAs that read both CTAs' shared memory and accumulate
// the whole tile in both CTAs' TMEM (rows 0..127 in the even CTA, 128..255 in
// the odd one); each CTA's epilogue warps write that CTA's scale factors (its
// rows' activation scales and the tile's two weight scales) into its own
// TMEM a few chunks ahead, as in the one-CTA block-scaled kernel, and read
// and store its own 128 rows once per tile.
//   Both producers' copies complete on the even CTA's stage barrier, whose
// arrival the even producer makes with both CTAs' byte count; both CTAs'
// scale-factor writers arrive on the even CTA's scale barrier; the MMA
// thread's commits arrive in both CTAs; both epilogues hand the accumulator
// back on the even CTA's barrier.  (With fp32 scales the chunk accumulators would have to cross the
// pair every K chunk: measured at half the one-CTA kernel's speed on GB300,
// so fp32 keeps one CTA per tile.)
struct PairCfg {
  static constexpr int kBN = 256;                // tile columns
  static constexpr int kABytes = kBM * kBK;      // this CTA's 128 activation rows
  static constexpr int kBBytes = 128 * kBK;      // this CTA's 128 of the 256 weight rows
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kCols = 64;               // accumulator columns per epilogue thread
  static constexpr int kEpiWarps = 16;
  static constexpr int kThreads = 128 + kEpiWarps * 32;
  // scale-factor slots in TMEM, four K chunks each (the one-CTA block-scaled
  // kernel's layout); no ring in shared memory
  static constexpr int kScaleSlots = 16;
  static constexpr int kScaleRingBytes = 0;
  static constexpr int kSfCol0 = 256;            // TMEM: the accumulator in [0, 256)
  static constexpr int kSfColsPerSlot = 16;
  static_assert(kSfCol0 + kScaleSlots * kSfColsPerSlot <= 512, "scale factors fit in TMEM");
  static constexpr int kBookBytes = 1024;
  static constexpr int kStagesFit = (200 * 1024) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr int kTmemCols = 512;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBookBytes + kScaleRingBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert((2 * kStages + 2 * kScaleSlots + 4) * 8 + 32 <= kBookBytes, "bookkeeping");
  // the roles (the MMA thread's copies, cluster waits and descriptors) need
  // more than the one-CTA kernel's (measured: spills below 80); the epilogue
  // holds no running sums
  static constexpr int kRoleRegs = 80;
  static constexpr int kEpiRegs = 96;
  static constexpr int kMinLaunchRegs = (128 * kRoleRegs + kEpiWarps * 32 * kEpiRegs + kThreads - 1) / kThreads;
};

__global__ void __launch_bounds__(PairCfg::kThreads, 1)
    gemm_pair_mx_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                        const GemmArgs a) {
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + C::kStages * C::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(base_ptr + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* sfull = drain + 1;
  uint64_t* sempty = sfull + C::kScaleSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sempty + C::kScaleSlots);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  uint32_t* issued = reinterpret_cast<uint32_t*>(abort_flag + 1);  // chunks this CTA's producer issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the CTA that issues the pair's MMAs
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  const int num_kb = a.k / kBK;
  const int m_pairs = (a.rows + 2 * kBM - 1) / (2 * kBM);
  const int n_tiles = a.n / C::kBN;
  const int total = m_pairs * n_tiles;

  if (threadIdx.x == 32) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);   // the even producer's arrival with both CTAs' bytes
      mbar_init(smem_u32(&empty[s]), 1);  // the MMA thread's commit
    }
    mbar_init(smem_u32(tfull), 1);
    mbar_init(smem_u32(tempty), 2 * C::kEpiWarps);  // both CTAs' epilogue warps
    mbar_init(smem_u32(drain), 1);
    for (int q = 0; q < C::kScaleSlots; ++q) {
      mbar_init(smem_u32(&sfull[q]), 8);   // both CTAs' writers, one warp per lane quadrant
      mbar_init(smem_u32(&sempty[q]), 1);  // the MMA thread's commit after the chunk's MMAs
    }
    *abort_flag = 0;
    *issued = 0;
    fence_barrier_init();
  }
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any copy or arrival targets them
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abortv = abort_flag;
  auto coords = [&](int pt, int& mp, int& n_tile) {
    mp = pt % m_pairs;  // m-pairs fastest: the pairs in flight share a few weight tiles
    n_tile = pt / m_pairs;
  };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRoleRegs));
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      uint32_t g = 0;
      if (lane == 0) {
        prefetch_tensormap(&tmap_x);
        prefetch_tensormap(&tmap_w);
        const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);
        bool alive = true;
        for (int pt = pair; pt < total && alive; pt += npairs) {
          int mp, n_tile;
          coords(pt, mp, n_tile);
          const int row0 = mp * 2 * kBM + (int)rank * kBM;
          const int wrow0 = n_tile * C::kBN + (int)rank * 128;
          for (int kb = 0; kb < num_kb; ++kb, ++g) {
            const int s = g % C::kStages;
            if (!mbar_wait_bounded(smem_u32(&empty[s]), ((g / C::kStages) & 1) ^ 1, abortv, a.err, a.timeout_ns,
                                   !(a.wait_mode & 1))) {
              alive = false;
              break;
            }
            if ((int)g == a.fault_skip_kb) continue;
            if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * C::kStageBytes);
            const uint32_t fb = full0 + 8u * (uint32_t)s;
            tma_load_2d_pair(sA + s * C::kABytes, &tmap_x, kb * kBK, row0, fb);
            tma_load_2d_pair(sB + s * C::kBBytes, &tmap_w, kb * kBK, wrow0, fb);
          }
        }
        *issued = g;
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer (even CTA)
      if (lane == 0 && rank == 0) {
        const uint32_t total_chunks = (uint32_t)((total - pair + npairs - 1) / npairs) * (uint32_t)num_kb;
        uint32_t g = 0, gs = 0, tt = 0;
        bool alive = true;
        for (int pt = pair; pt < total && alive; pt += npairs, ++tt) {
          if (!mbar_wait_bounded_cluster(smem_u32(tempty), (tt & 1) ^ 1, abortv, a.err, a.timeout_ns)) {
            alive = false;
            break;
          }
          for (int kb = 0; kb < num_kb; ++kb, ++g, ++gs) {
            const int s = g % C::kStages;
            const uint32_t grp = gs >> 2, j = gs & 3u;
            const int q = grp % C::kScaleSlots;
            if (!mbar_wait_bounded(smem_u32(&full[s]), (g / C::kStages) & 1, abortv, a.err, a.timeout_ns,
                                   !(a.wait_mode & 1)) ||
                (j == 0 && !mbar_wait_bounded_cluster(smem_u32(&sfull[q]), (grp / C::kScaleSlots) & 1, abortv,
                                                      a.err, a.timeout_ns))) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t sf_t = tmem + C::kSfCol0 + q * C::kSfColsPerSlot;
            const uint32_t a0 = sA + s * C::kABytes, b0 = sB + s * C::kBBytes;
            const uint32_t idesc = idesc_mx_e4m3_ue8m0(2 * kBM, C::kBN, 0, 0) | (j << 4) | (j << 29);
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k)
              mma_mx_e4m3_pair(tmem, sw128_kmajor_desc(a0 + k * kUmmaK), sw128_kmajor_desc(b0 + k * kUmmaK), idesc,
                               sf_t, sf_t + 4, (kb > 0 || k > 0) ? 1u : 0u);
            mma_commit_pair(smem_u32(&empty[s]));
            if (j == 3 || gs + 1 == total_chunks) mma_commit_pair(smem_u32(&sempty[q]));
          }
          if (alive) mma_commit_pair(smem_u32(tfull));
        }
        if (*abortv) {
          // no MMA or copy may still be using either CTA's TMEM when it is released
          mma_commit_pair(smem_u32(drain));
          mbar_wait_bounded(smem_u32(drain), 0, nullptr, nullptr, 10000000ull);
        }
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kEpiRegs));
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 4;
    const int quad = warp & 3;
    const int slice = ew >> 2;
    const int r = quad * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16) + slice * C::kCols;
    // the accumulator is handed back, and the scale factors announced, on the
    // even CTA's barriers (its own shared::cluster addresses for the even CTA)
    const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
    const uint32_t sfull_leader = mapa_shared(smem_u32(&sfull[0]), 0);
    // Scale factors of the pair's K chunks (numbered across its tiles), four
    // consecutive chunks per TMEM slot (one per byte of each cell): group G
    // is written into this CTA's TMEM by the four warps of slice G mod 4, one
    // per lane quadrant, up to 32 chunks ahead of the tile being accumulated.
    const uint32_t sf_total = (uint32_t)((total - pair + npairs - 1) / npairs) * (uint32_t)num_kb;
    uint32_t sf_next = (uint32_t)slice;  // this warp's next group
    auto sf_write = [&]() -> bool {
      const uint32_t grp = sf_next;
      sf_next += 4;
      uint32_t xw = 0u, b0 = 0u, b1 = 0u;  // cell bytes: byte j for chunk 4 grp + j
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t c = 4u * grp + (uint32_t)j;
        uint32_t xb = 127u, wb0 = 127u, wb1 = 127u;
        if (c < sf_total) {
          const int tseq = (int)(c / (uint32_t)num_kb), kbc = (int)(c - (uint32_t)tseq * (uint32_t)num_kb);
          int mp, nt;
          coords(pair + tseq * npairs, mp, nt);
          const int srow = mp * 2 * kBM + (int)rank * kBM + quad * 32 + lane;
          if (srow < a.rows) {
            const int64_t xi = (int64_t)kbc * a.rows + srow;
            xb = (__ldg(static_cast<const uint32_t*>(scale_word<true>(a.sx, xi))) >> (8 * ((uint32_t)xi & 3u))) &
                 0xFFu;
          }
          const int64_t wi = (int64_t)(nt * C::kBN >> 7) * num_kb + kbc;
          wb0 = (__ldg(static_cast<const uint32_t*>(scale_word<true>(a.sw, wi))) >> (8 * ((uint32_t)wi & 3u))) &
                0xFFu;
          wb1 = (__ldg(static_cast<const uint32_t*>(scale_word<true>(a.sw, wi + num_kb))) >>
                 (8 * ((uint32_t)(wi + num_kb) & 3u))) &
                0xFFu;
        }
        xw |= xb << (8 * j);
        b0 |= wb0 << (8 * j);
        b1 |= wb1 << (8 * j);
      }
      const int q = grp % C::kScaleSlots;
      bool got = mbar_wait_bounded(smem_u32(&sempty[q]), ((grp / C::kScaleSlots) & 1) ^ 1, abortv, a.err,
                                   a.timeout_ns, !(a.wait_mode & 2));
      got = __all_sync(0xffffffffu, got);
      if (!got) return false;
      tc_fence_after();
      const uint32_t sf = tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::kSfCol0 + q * C::kSfColsPerSlot;
      tmem_st_32x32b_x1(sf + quad, xw);
      const uint32_t bw[8] = {b0, b0, b0, b0, b1, b1, b1, b1};
      tmem_st_32x32b_x8(sf + 4, bw);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(sfull_leader + 8u * (uint32_t)q);
      return true;
    };
    uint32_t tt = 0;
    bool ok = true;
    for (int pt = pair; ok && pt < total; pt += npairs, ++tt) {
      const uint32_t lim = min(sf_total, (tt + 1) * (uint32_t)num_kb + 4u * (C::kScaleSlots / 2));
      while (ok && 4u * sf_next < lim) ok = sf_write();
      if (!ok) break;
      int mp, n_tile;
      coords(pt, mp, n_tile);
      const int row0 = mp * 2 * kBM + (int)rank * kBM;
      const int n0 = n_tile * C::kBN;
      const int grow = row0 + r;
      const bool row_ok = grow < a.rows;
      uint64_t acc[C::kCols / 2];
      ok = mbar_wait_bounded(smem_u32(tfull), tt & 1, abortv, a.err, a.timeout_ns, !(a.wait_mode & 2));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // straight into the accumulator registers, 32 columns per round trip
      tmem_ld_32x32b_x32_pairs(t_lane, *reinterpret_cast<uint64_t(*)[16]>(&acc[0]));
      tmem_ld_32x32b_x32_pairs(t_lane + 32, *reinterpret_cast<uint64_t(*)[16]>(&acc[16]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader);
      if (row_ok && !*abortv && dcheck(grow < a.rows && n0 + slice * C::kCols + C::kCols <= a.n, a.err)) {
        uint4* dst = reinterpret_cast<uint4*>(a.y + (int64_t)grow * a.n + n0 + slice * C::kCols);
        const bool wide = (reinterpret_cast<uintptr_t>(a.y) & 31) == 0;
#pragma unroll
        for (int j = 0; j < C::kCols / 16; ++j) {
          uint4 h[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float x[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) f32x2_unpack(acc[8 * j + 4 * e + q], x[2 * q], x[2 * q + 1]);
            h[e] = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                              pack_bf16x2(x[6], x[7]));
          }
          if (wide) {
            st_global_v8(dst + 2 * j, h[0], h[1]);
          } else {
            dst[2 * j] = h[0];
            dst[2 * j + 1] = h[1];
          }
        }
      }
    }
  }
  // Teardown.  Every copy either CTA issued completes on the even CTA's stage
  // barriers: after a wait ran out anywhere, the even CTA's producer lets the
  // last stages' copies of both CTAs land before shared memory is released.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (rank == 0 && threadIdx.x == 0) {
    const uint32_t peer_abort = ld_dsmem_u32(mapa_shared(smem_u32(abort_flag), 1));
    if (*abortv || peer_abort) {
      const uint32_t peer_issued = ld_dsmem_u32(mapa_shared(smem_u32(issued), 1));
      const uint32_t gmax = *issued > peer_issued ? *issued : peer_issued;
      for (uint32_t j = gmax > (uint32_t)C::kStages ? gmax - C::kStages : 0; j < gmax; ++j) {
        if ((int)j == a.fault_skip_kb) continue;
        mbar_wait_bounded(smem_u32(&full[j % C::kStages]), (j / C::kStages) & 1, nullptr, nullptr, 10000000ull);
      }
    }
  }
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

fp8rl_status check_gemm(const void* xq, const void* x_scale, const void* wq, const void* w_scale,
                        const void* y, int64_t m, int64_t n, int64_t k, fp8rl_scale_fmt fmt) {
  if (fmt != FP8RL_SCALE_FP32 && fmt != FP8RL_SCALE_UE8M0) return FP8RL_ERR_INVALID_ARG;
  if (m < 0 || n < 0 || k < 0) return FP8RL_ERR_INVALID_ARG;
  if (n % 128 || k % 128) return FP8RL_ERR_SHAPE;
  if (m == 0 || n == 0) return FP8RL_OK;
  if (m > INT32_MAX || n > INT32_MAX || k > INT32_MAX) return FP8RL_ERR_SHAPE;
  if (!xq || !x_scale || !wq || !w_scale || !y) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(y, 16)) return FP8RL_ERR_ALIGNMENT;
  if (fmt == FP8RL_SCALE_FP32 && (!aligned(x_scale, 4) || !aligned(w_scale, 4))) return FP8RL_ERR_ALIGNMENT;
  return FP8RL_OK;
}

// test hooks (set through fp8rl_debug_set)
struct Debug {
  int bn = 0;                     // 0: choose; 128 or 256: force the tile width
  int fault_skip_kb = -1;         // the producer skips this K chunk (forces a timeout)
  int wait_mode = 0;              // which roles poll instead of suspending (bits: 1 producer/MMA, 2 epilogue)
  int l2_prefetch = 0;            // K chunks of L2 prefetch beyond the shared-memory ring
  int splits = 0;                 // 0: choose; 1..8: force the split-K cluster size
  int streamk = 0;                // with a workspace: 0 choose, 1 never, 2 always (dense, M > 32)
  int streamk_grid = 0;           // 0: one CTA per SM (at most one per K iteration); else this many
  int out_stage = 0;              // data-parallel tile stores: 0 choose, 1 through shared memory + TMA, 2 from registers
  int decode = 0;                 // dense rows <= 128: 0 choose, 1 the swapped-operand decode kernel, 2 the 128-row-tile one
  int mx = 0;                     // UE8M0 data-parallel tiles: 0 choose, 1 the per-chunk promotion, 2 the block-scaled MMA
  int pair = 0;                   // dense data-parallel tiles on tensor-core pairs: 0 choose, 1 always, 2 never
  uint64_t timeout_ns = 2000000000ull;
};
Debug g_debug;
std::mutex g_mu;
std::atomic<int> g_pdl_off{0};    // test hook 13: launch without programmatic stream serialisation

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// row-major E4M3 matrix [outer][inner] (inner contiguous), boxes of box_outer rows x 128 bytes
// bf16 output [rows][n] for the epilogue's TMA stores: boxes of 32 rows x 64
// columns (128 bytes), 128-byte swizzle
bool make_out_map(CUtensorMap* map, void* base, uint64_t n, uint64_t rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {n, rows};
  cuuint64_t strides[1] = {n * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
  bool ok = false;
  int sms = 0;
};

DeviceInfo device_info() {
  static DeviceInfo cache[64];
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return {};
  std::lock_guard<std::mutex> lock(g_mu);
  if (!done[dev]) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cache[dev].ok = major == 10 && minor == 3;
    cache[dev].sms = sms;
    done[dev] = true;
  }
  return cache[dev];
}

// clusters of `splits` CTAs along z that can be resident at once (0: none)
template <typename K>
int max_active_clusters(K kernel, dim3 grid, int threads, int smem, int splits) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = splits;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Per device and kernel instantiation, what does not depend on the call's
// pointers is established once: the shared-memory opt-in, the register check
// of the setmaxnreg split, and for each split count whether its clusters fit.
struct KernelState {
  uint64_t ctx = 0;  // the context the attributes were set in (redone when it changes)
  bool ready = false;
  bool regs_ok = false;
  bool attr_ok = false;
  int cluster_capacity[9] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};  // clusters resident at once
};

template <int BN, int AROWS, bool UE8M0, int MODE, int EPI, bool OUT, bool MX>
KernelState& kernel_state(int dev) {
  static KernelState st[64];
  return st[dev];
}

// Stream-K workspace: a 256-byte header (epoch, finished-CTA count), one flag
// word per CTA, then one 128 x 256 fp32 partial tile per CTA.
struct StreamKLayout {
  size_t flag_off, part_off, bytes;
};

StreamKLayout streamk_layout(int max_ctas) {
  StreamKLayout l;
  l.flag_off = 256;
  l.part_off = l.flag_off + (((size_t)max_ctas * 4 + 255) / 256) * 256;
  l.bytes = l.part_off + (size_t)max_ctas * kBM * 256 * 4;
  return l;
}

template <int BN, int AROWS, bool UE8M0, int MODE, int EPI = 0, bool OUT = false, bool MX = false>
fp8rl_status launch(const void* xq, const void* wq, int64_t experts, int64_t m_tiles_bound, int sms,
                    GemmArgs args, int splits, cudaStream_t stream, int streamk_grid = 0) {
  using C = Cfg<BN, AROWS, EPI, OUT, MX>;
  constexpr bool SPLITK = MODE == kSplitK;
  auto kernel = gemm_blockscaled_kernel<BN, AROWS, UE8M0, MODE, EPI, OUT, MX>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8RL_ERR_CUDA;
  KernelState& ks = kernel_state<BN, AROWS, UE8M0, MODE, EPI, OUT, MX>(dev);
  const uint64_t ctx = current_context_id();
  if (!ctx) return FP8RL_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!ks.ready || ks.ctx != ctx) {
      ks = KernelState{};
      ks.ctx = ctx;
      cudaFuncAttributes fa;
      ks.regs_ok = cudaFuncGetAttributes(&fa, kernel) == cudaSuccess &&
                   // setmaxnreg.inc waits until the block has the registers it asks
                   // for: the launch allocation must cover the split or it waits forever
                   (!C::kSplitRegs || fa.numRegs >= C::kMinLaunchRegs);
      ks.attr_ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) ==
                   cudaSuccess;
      ks.ready = true;
    }
    if (!ks.attr_ok) return FP8RL_ERR_CUDA;
    if (!ks.regs_ok) return FP8RL_ERR_UNSUPPORTED;  // the caller retries with 128-wide tiles
    // the largest split count not above the request whose clusters (one per
    // tile) are all resident at once: measured on GB300, clusters of 3 fit 46
    // at a time, so 48 tiles split three ways ran as two waves
    const int64_t cluster_count = m_tiles_bound * (args.n / BN);
    while (SPLITK && splits > 1) {
      if (ks.cluster_capacity[splits] < 0)
        ks.cluster_capacity[splits] =
            max_active_clusters(kernel, dim3(1, 1, (unsigned)splits), C::kThreads, C::kSmemBytes, splits);
      if (ks.cluster_capacity[splits] >= cluster_count) break;
      --splits;
    }
  }
  if (SPLITK && splits == 1) return FP8RL_ERR_UNSUPPORTED;  // the caller launches the plain kernel
  CUtensorMap mx, mw, my;
  if (!make_map(&mx, xq, args.k, args.rows, AROWS)) return FP8RL_ERR_CUDA;
  if (!make_map(&mw, wq, args.k, (uint64_t)experts * args.n, BN)) return FP8RL_ERR_CUDA;
  if (OUT) {
    if (!make_out_map(&my, args.y, args.n, args.rows)) return FP8RL_ERR_CUDA;
  } else {
    my = mx;  // unused by this kernel
  }
  args.splits = splits;
  // split-K: one CTA per (m-tile, n-tile, split); otherwise persistent CTAs,
  // at most one per SM, striding over the tiles
  const int64_t tiles_bound = m_tiles_bound * (args.n / BN);
  dim3 grid = SPLITK ? dim3((unsigned)m_tiles_bound, (unsigned)(args.n / BN), (unsigned)splits)
                     : dim3((unsigned)std::min<int64_t>(tiles_bound, sms), 1, 1);
  if (MODE == kStreamK) {
    // stream-K: every CTA gets at least one K iteration (dense: the tile count
    // is exact); the launch is cooperative because tile owners wait for the
    // CTAs that hold the rest of their tiles
    const int64_t iters = tiles_bound * (args.k / kBK);
    const int want = streamk_grid > 0 ? streamk_grid : sms;
    grid = dim3((unsigned)std::min<int64_t>(iters, std::min(want, sms)), 1, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, mx, mw, my, args) != cudaSuccess) {
      cudaGetLastError();
      return FP8RL_ERR_CUDA;
    }
  } else if (!SPLITK) {
    kernel<<<grid, C::kThreads, C::kSmemBytes, stream>>>(mx, mw, my, args);
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = splits;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, mx, mw, my, args) != cudaSuccess) return FP8RL_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}

// A dense data-parallel UE8M0 product on tensor-core pairs (clusters of two CTAs).
fp8rl_status launch_pair(const void* xq, const void* wq, GemmArgs args, cudaStream_t stream) {
  using C = PairCfg;
  auto kernel = gemm_pair_mx_kernel;
  static KernelState st[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8RL_ERR_CUDA;
  KernelState& ks = st[dev];
  const uint64_t ctx = current_context_id();
  if (!ctx) return FP8RL_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!ks.ready || ks.ctx != ctx) {
      ks = KernelState{};
      ks.ctx = ctx;
      cudaFuncAttributes fa;
      // setmaxnreg.inc waits until the block has the registers it asks for
      ks.regs_ok = cudaFuncGetAttributes(&fa, kernel) == cudaSuccess && fa.numRegs >= C::kMinLaunchRegs;
      ks.attr_ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) ==
                   cudaSuccess;
      if (ks.attr_ok) {
        // pairs resident at once (a persistent grid needs no more)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(C::kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
          cudaGetLastError();
          n = 0;
        }
        ks.cluster_capacity[2] = n;
      }
      ks.ready = true;
    }
    if (!ks.attr_ok) return FP8RL_ERR_CUDA;
    if (!ks.regs_ok || ks.cluster_capacity[2] < 1) return FP8RL_ERR_UNSUPPORTED;
  }
  CUtensorMap mx, mw;
  if (!make_map(&mx, xq, args.k, args.rows, kBM)) return FP8RL_ERR_CUDA;
  if (!make_map(&mw, wq, args.k, args.n, 128)) return FP8RL_ERR_CUDA;
  const int64_t pairs_total = ((int64_t)args.rows + 2 * kBM - 1) / (2 * kBM) * (args.n / C::kBN);
  const int64_t clusters = std::min<int64_t>(pairs_total, ks.cluster_capacity[2]);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, mx, mw, args) != cudaSuccess) {
    cudaGetLastError();
    return FP8RL_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? FP8RL_OK : FP8RL_ERR_CUDA;
}

fp8rl_status run(const void* xq, const void* x_scale, const void* wq, const void* w_scale,
                 const int32_t* d_offsets, int64_t experts, int64_t rows, int64_t n, int64_t k, void* y,
                 fp8rl_scale_fmt fmt, void* stream, void* workspace = nullptr) {
  const DeviceInfo di = device_info();
  if (!di.ok) return FP8RL_ERR_UNSUPPORTED;
  uint32_t* err = device_error_word();
  if (!err) return FP8RL_ERR_CUDA;
  Debug dbg;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    dbg = g_debug;
  }
  GemmArgs args{};
  args.sx = x_scale;
  args.sw = w_scale;
  args.y = static_cast<__nv_bfloat16*>(y);
  args.offsets = d_offsets;
  args.rows = (int32_t)rows;
  args.n = (int32_t)n;
  args.k = (int32_t)k;
  args.experts = (int32_t)experts;
  args.err = err;
  args.timeout_ns = dbg.timeout_ns;
  args.fault_skip_kb = dbg.fault_skip_kb;
  args.wait_mode = dbg.wait_mode;
  args.l2_prefetch = dbg.l2_prefetch;
  // decode sizes (dense, at most 64 rows): the swapped-operand kernel of
  // decode.cu (measured on GB300, Qwen3-8B projections with weights from
  // HBM: 30-50% faster than the 128-row-tile kernel at 17 and 32 rows, 5-30%
  // at 64).  Its 128-column form (one CTA per SM) beats the tile kernel at
  // 65..128 rows only where the weight's 128-row blocks leave room for four
  // K splits in one wave (fp32 scales, 128 rows: 4096 x 4096 10.6 against
  // 14.0 us, 4096 x 12288 even; 6144 x 4096 even with two splits, 24576 x
  // 4096 1.8x slower), so only those shapes take it.  The test hook forces
  // either kernel.
  const bool narrow = fmt == FP8RL_SCALE_FP32 && n / 128 * 4 <= di.sms && k >= 4096;
  const bool decode_shape = !d_offsets && (rows <= 64 || (rows <= 128 && (dbg.decode == 1 || narrow)));
  if (decode_shape && dbg.decode != 2 && dbg.streamk != 2) {
    const fp8rl_status st = decode_gemm(xq, x_scale, wq, w_scale, y, rows, n, k, fmt == FP8RL_SCALE_UE8M0, err,
                                        dbg.timeout_ns, dbg.fault_skip_kb, dbg.splits,
                                        static_cast<cudaStream_t>(stream));
    if (st != FP8RL_ERR_UNSUPPORTED) return st;
  }
  const int64_t m_tiles = (rows + kBM - 1) / kBM;
  // Tile width by estimated time: whole waves of tiles x the time of one tile.
  // Measured on GB300 (K = 4096): a 128 x 256 tile takes ~1.35x as long as a
  // 128 x 128 one (half the operand traffic per flop).
  const int64_t sms64 = di.sms;
  const int64_t cost128 = (m_tiles * (n / 128) + sms64 - 1) / sms64 * 100;
  const int64_t cost256 = n % 256 ? INT64_MAX : (m_tiles * (n / 256) + sms64 - 1) / sms64 * 135;
  int bn = dbg.bn;
  if (bn != 128 && bn != 256) bn = (d_offsets ? m_tiles * (n / 256) >= 2 * sms64 : cost256 <= cost128) ? 256 : 128;
  if (bn == 256 && n % 256) bn = 128;
  // split K across a cluster when the tiles alone leave SMs idle (dense only):
  // decode-sized M streams the weights through every SM
  const int64_t num_kb = k / kBK;
  int splits = 1;
  if (!d_offsets) {
    const int64_t tiles = m_tiles * (n / 128);
    if (dbg.splits > 0)
      splits = dbg.splits;
    else if (m_tiles * (n / bn) < di.sms && tiles < di.sms)
      splits = (int)std::min<int64_t>(std::min<int64_t>(8, di.sms / tiles), num_kb / 2);
    splits = (int)std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(splits, 8), num_kb));
  }
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool ue = fmt == FP8RL_SCALE_UE8M0;
  // an upper bound on the 128-row tiles (grouped: every expert may end in a partial tile)
  const int64_t mt_bound = d_offsets ? m_tiles + experts : m_tiles;
  const int sms = di.sms;
  // decode-sized M: load only 32 activation rows per stage (deeper weight pipeline)
  const bool short_a = !d_offsets && rows <= 32;
  // dense UE8M0 products with more than one m-tile and 256-wide weight
  // blocks: tiles of 256 x 256 on tensor-core pairs (clusters of two CTAs)
  // UE8M0 on the block-scaled MMA (one accumulator per tile) unless K is
  // short: measured on GB300, the MoE expert pair (T = 4096) gate-up at
  // K = 2048 126 vs 142 us, but down at K = 768 112 vs 94 us (six chunks a
  // tile leave the scale-factor writes and the register stores exposed)
  const bool mx = ue && (dbg.mx == 2 || (dbg.mx == 0 && num_kb >= 16));
  const bool pair_ok = mx && !d_offsets && n % 256 == 0 && rows > kBM && !short_a;
  if (pair_ok && dbg.pair == 1) {
    const fp8rl_status st = launch_pair(xq, wq, args, cs);
    if (st != FP8RL_ERR_UNSUPPORTED) return st;
  }
  if (workspace && !d_offsets && !short_a && dbg.streamk != 1) {
    // stream-K when whole tiles would leave the last wave of SMs mostly idle
    // (measured on GB300: it pays when that wave is at most ~30% full, between
    // one and eight waves; with less than one wave, whole tiles are faster)
    const int sbn = (dbg.bn == 128 || n % 256) ? 128 : 256;
    const int64_t tiles = m_tiles * (n / sbn);
    const bool uneven = splits == 1 && tiles > sms64 && tiles < 8 * sms64 && (tiles % sms64) * 10 <= 3 * sms64;
    // the kernel counts stream-K iterations (at most two waves of tiles) times
    // the grid in 32 bits
    const bool fits = 2 * (int64_t)sms * num_kb * sms < ((int64_t)1 << 31);
    if (fits && (dbg.streamk == 2 || uneven)) {
      const StreamKLayout l = streamk_layout(sms);
      char* ws = static_cast<char*>(workspace);
      args.ws_head = reinterpret_cast<uint32_t*>(ws);
      args.ws_flag = reinterpret_cast<uint32_t*>(ws + l.flag_off);
      args.ws_part = reinterpret_cast<float*>(ws + l.part_off);
      fp8rl_status st;
      if (sbn == 256) {
        st = ue ? launch<256, kBM, true, kStreamK>(xq, wq, experts, mt_bound, sms, args, 1, cs, dbg.streamk_grid)
                : launch<256, kBM, false, kStreamK>(xq, wq, experts, mt_bound, sms, args, 1, cs, dbg.streamk_grid);
        if (st != FP8RL_ERR_UNSUPPORTED) return st;
      }
      return ue ? launch<128, kBM, true, kStreamK>(xq, wq, experts, mt_bound, sms, args, 1, cs, dbg.streamk_grid)
                : launch<128, kBM, false, kStreamK>(xq, wq, experts, mt_bound, sms, args, 1, cs, dbg.streamk_grid);
    }
  }
  if (splits > 1) {
    // split-K clusters use 128-wide tiles
    fp8rl_status st;
    if (short_a)
      st = ue ? launch<128, 32, true, kSplitK>(xq, wq, experts, mt_bound, sms, args, splits, cs)
              : launch<128, 32, false, kSplitK>(xq, wq, experts, mt_bound, sms, args, splits, cs);
    else
      st = ue ? launch<128, kBM, true, kSplitK>(xq, wq, experts, mt_bound, sms, args, splits, cs)
              : launch<128, kBM, false, kSplitK>(xq, wq, experts, mt_bound, sms, args, splits, cs);
    if (st != FP8RL_ERR_UNSUPPORTED) return st;
  }
  if (short_a)
    return ue ? launch<128, 32, true, kDataParallel>(xq, wq, experts, mt_bound, sms, args, 1, cs)
              : launch<128, 32, false, kDataParallel>(xq, wq, experts, mt_bound, sms, args, 1, cs);
  // Tiles leave through shared memory and TMA stores unless K is deep: the
  // slots cost the operand ring a stage, which only deep-K tiles feel more
  // than the store they save (measured on GB300: 8192 x 24576 x 4096 +6%,
  // 1024 x 6144 x 4096 +5%, grouped MoE +5..14%; 8192 x 4096 x 12288 -3%).
  const bool staged = dbg.out_stage == 1 || (dbg.out_stage != 2 && k <= 4096);
  if (mx) {
    // UE8M0: the tensor cores apply the power-of-two scales themselves
    // (block-scaled MMA), one accumulator per tile; the tile stores stay in
    // the epilogue's registers (measured on GB300: 8192 x 24576 x 4096 0.559
    // vs 0.604 ms through shared memory, every shape faster), since the
    // store does not hold up the next tile's MMAs
    if (bn == 256) {
      const fp8rl_status st =
          launch<256, kBM, true, kDataParallel, 0, false, true>(xq, wq, experts, mt_bound, sms, args, 1, cs);
      if (st != FP8RL_ERR_UNSUPPORTED) return st;
    }
    return launch<128, kBM, true, kDataParallel, 0, false, true>(xq, wq, experts, mt_bound, sms, args, 1, cs);
  }
  if (bn == 256) {
    const fp8rl_status st =
        staged ? (ue ? launch<256, kBM, true, kDataParallel, 0, true>(xq, wq, experts, mt_bound, sms, args, 1, cs)
                     : launch<256, kBM, false, kDataParallel, 0, true>(xq, wq, experts, mt_bound, sms, args, 1, cs))
               : (ue ? launch<256, kBM, true, kDataParallel>(xq, wq, experts, mt_bound, sms, args, 1, cs)
                     : launch<256, kBM, false, kDataParallel>(xq, wq, experts, mt_bound, sms, args, 1, cs));
    if (st != FP8RL_ERR_UNSUPPORTED) return st;
  }
  if (staged)
    return ue ? launch<128, kBM, true, kDataParallel, 0, true>(xq, wq, experts, mt_bound, sms, args, 1, cs)
              : launch<128, kBM, false, kDataParallel, 0, true>(xq, wq, experts, mt_bound, sms, args, 1, cs);
  return ue ? launch<128, kBM, true, kDataParallel>(xq, wq, experts, mt_bound, sms, args, 1, cs)
            : launch<128, kBM, false, kDataParallel>(xq, wq, experts, mt_bound, sms, args, 1, cs);
}

// The fused gate-up GEMM: the same kernel with the SwiGLU-quantise epilogue,
// 256-wide tiles (128 gate + the matching 128 up columns), whole tiles.
fp8rl_status run_swiglu(const void* xq, const void* x_scale, const void* wq, const void* w_scale,
                        const int32_t* d_offsets, int64_t experts, int64_t rows, int64_t inter, int64_t k,
                        void* hq, void* h_scale, fp8rl_scale_fmt fmt, void* stream) {
  const DeviceInfo di = device_info();
  if (!di.ok) return FP8RL_ERR_UNSUPPORTED;
  uint32_t* err = device_error_word();
  if (!err) return FP8RL_ERR_CUDA;
  Debug dbg;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    dbg = g_debug;
  }
  GemmArgs args{};
  args.sx = x_scale;
  args.sw = w_scale;
  args.offsets = d_offsets;
  args.rows = (int32_t)rows;
  args.n = (int32_t)(2 * inter);
  args.k = (int32_t)k;
  args.experts = (int32_t)experts;
  args.err = err;
  args.timeout_ns = dbg.timeout_ns;
  args.fault_skip_kb = dbg.fault_skip_kb;
  args.wait_mode = dbg.wait_mode;
  args.l2_prefetch = dbg.l2_prefetch;
  args.hq = static_cast<uint8_t*>(hq);
  args.h_scale = h_scale;
  const int64_t m_tiles = (rows + kBM - 1) / kBM;
  const int64_t mt_bound = d_offsets ? m_tiles + experts : m_tiles;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return fmt == FP8RL_SCALE_UE8M0
             ? launch<256, kBM, true, kDataParallel, 1>(xq, wq, experts, mt_bound, di.sms, args, 1, cs)
             : launch<256, kBM, false, kDataParallel, 1>(xq, wq, experts, mt_bound, di.sms, args, 1, cs);
}

}  // namespace

bool pdl_enabled() { return g_pdl_off.load() == 0; }

namespace {

// fp8rl_gemm_act_quant at decode sizes: one kernel that quantises X and
// multiplies; UNSUPPORTED when the shape or layout needs the two-call path
fp8rl_status run_act_quant_fused(const void* x_bf16, int64_t ldx, const void* wq, const void* w_scale, void* y,
                                 int64_t m, int64_t n, int64_t k, fp8rl_scale_fmt fmt, void* xq, void* x_scale,
                                 void* stream) {
  const DeviceInfo di = device_info();
  if (!di.ok) return FP8RL_ERR_UNSUPPORTED;
  Debug dbg;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    dbg = g_debug;
  }
  if (m > 16 || dbg.decode == 2 || dbg.streamk == 2) return FP8RL_ERR_UNSUPPORTED;
  uint32_t* err = device_error_word();
  if (!err) return FP8RL_ERR_CUDA;
  return decode_gemm_qx(x_bf16, ldx, wq, w_scale, y, m, n, k, fmt == FP8RL_SCALE_UE8M0, xq, x_scale, err,
                        dbg.timeout_ns, dbg.fault_skip_kb, dbg.splits, static_cast<cudaStream_t>(stream));
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
  return run(xq, x_scale, wq, w_scale, nullptr, 1, m, n, k, y, fmt, stream);
}

extern "C" FP8RL_API fp8rl_status fp8rl_gemm_act_quant(const void* x_bf16, int64_t ldx, const void* wq,
                                                       const void* w_scale, void* y, int64_t m, int64_t n,
                                                       int64_t k, fp8rl_scale_fmt fmt, void* xq, void* x_scale,
                                                       void* stream) {
  fp8rl_status st = check_gemm(xq, x_scale, wq, w_scale, y, m, n, k, fmt);
  if (st != FP8RL_OK || m == 0) return st;
  if (!x_bf16 || ldx < k) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 2)) return FP8RL_ERR_ALIGNMENT;
  if (n > 0) {
    st = run_act_quant_fused(x_bf16, ldx, wq, w_scale, y, m, n, k, fmt, xq, x_scale, stream);
    if (st != FP8RL_ERR_UNSUPPORTED) return st;
  }
  st = fp8rl_quant_act_group(x_bf16, m, k, ldx, xq, k, x_scale, fmt, stream);
  if (st != FP8RL_OK || n == 0) return st;
  return run(xq, x_scale, wq, w_scale, nullptr, 1, m, n, k, y, fmt, stream);
}

extern "C" FP8RL_API fp8rl_status fp8rl_gemm_workspace_size(size_t* bytes) {
  if (!bytes) return FP8RL_ERR_INVALID_ARG;
  *bytes = 0;
  const DeviceInfo di = device_info();
  if (!di.ok) return FP8RL_ERR_UNSUPPORTED;
  *bytes = streamk_layout(di.sms).bytes;
  return FP8RL_OK;
}

extern "C" FP8RL_API fp8rl_status fp8rl_gemm_blockscaled_ws(const void* xq, const void* x_scale,
                                                            const void* wq, const void* w_scale, void* y,
                                                            int64_t m, int64_t n, int64_t k,
                                                            fp8rl_scale_fmt fmt, void* workspace,
                                                            size_t workspace_bytes, void* stream) {
  fp8rl_status st = check_gemm(xq, x_scale, wq, w_scale, y, m, n, k, fmt);
  if (st != FP8RL_OK) return st;
  if (!workspace) return FP8RL_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return FP8RL_ERR_ALIGNMENT;
  if (m == 0 || n == 0) return FP8RL_OK;
  const DeviceInfo di = device_info();
  if (!di.ok) return FP8RL_ERR_UNSUPPORTED;
  if (workspace_bytes < streamk_layout(di.sms).bytes) return FP8RL_ERR_INVALID_ARG;
  return run(xq, x_scale, wq, w_scale, nullptr, 1, m, n, k, y, fmt, stream, workspace);
}

extern "C" FP8RL_API fp8rl_status fp8rl_gemm_blockscaled_static(const void* xq, const void* x_scale,
                                                                const void* wq, const void* w_scale, void* y,
                                                                int64_t m, int64_t n, int64_t k,
                                                                fp8rl_scale_fmt fmt, void* stream) {
  fp8rl_status st = check_gemm(xq, x_scale, wq, w_scale, y, m, n, k, fmt);
  if (st != FP8RL_OK || m == 0 || n == 0) return st;
  const DeviceInfo di = device_info();
  if (!di.ok) return FP8RL_ERR_UNSUPPORTED;
  const StreamKLayout l = streamk_layout(di.sms);
  void* scratch = static_gemm_scratch(l.bytes, l.part_off, &st);
  if (!scratch) return st;
  return run(xq, x_scale, wq, w_scale, nullptr, 1, m, n, k, y, fmt, stream, scratch);
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
  if (num_experts > INT32_MAX / 2 || num_experts * n > INT32_MAX) return FP8RL_ERR_SHAPE;
  return run(xq, x_scale, wq, w_scale, d_offsets, num_experts, rows, n, k, y, fmt, stream);
}

extern "C" FP8RL_API fp8rl_status fp8rl_gemm_swiglu_quant(const void* xq, const void* x_scale,
                                                          const void* wq_gate_up, const void* w_scale_gate_up,
                                                          int64_t m, int64_t inter, int64_t k, void* hq,
                                                          void* h_scale, fp8rl_scale_fmt fmt, void* stream) {
  if (inter < 0) return FP8RL_ERR_INVALID_ARG;
  fp8rl_status st = check_gemm(xq, x_scale, wq_gate_up, w_scale_gate_up, hq, m, 2 * inter, k, fmt);
  if (st != FP8RL_OK || m == 0 || inter == 0) return st;
  if (!h_scale) return FP8RL_ERR_INVALID_ARG;
  if (fmt == FP8RL_SCALE_FP32 && !aligned(h_scale, 4)) return FP8RL_ERR_ALIGNMENT;
  if (2 * inter > INT32_MAX) return FP8RL_ERR_SHAPE;
  return run_swiglu(xq, x_scale, wq_gate_up, w_scale_gate_up, nullptr, 1, m, inter, k, hq, h_scale, fmt, stream);
}

extern "C" FP8RL_API fp8rl_status fp8rl_grouped_gemm_swiglu_quant(
    const void* xq, const void* x_scale, const void* wq_gate_up, const void* w_scale_gate_up,
    const int32_t* d_offsets, int64_t num_experts, int64_t rows, int64_t inter, int64_t k, void* hq,
    void* h_scale, fp8rl_scale_fmt fmt, void* stream) {
  if (num_experts < 1 || !d_offsets || inter < 0) return FP8RL_ERR_INVALID_ARG;
  fp8rl_status st = check_gemm(xq, x_scale, wq_gate_up, w_scale_gate_up, hq, rows, 2 * inter, k, fmt);
  if (st != FP8RL_OK || rows == 0 || inter == 0) return st;
  if (!h_scale) return FP8RL_ERR_INVALID_ARG;
  if (fmt == FP8RL_SCALE_FP32 && !aligned(h_scale, 4)) return FP8RL_ERR_ALIGNMENT;
  if (num_experts > INT32_MAX / 2 || num_experts * 2 * inter > INT32_MAX) return FP8RL_ERR_SHAPE;
  return run_swiglu(xq, x_scale, wq_gate_up, w_scale_gate_up, d_offsets, num_experts, rows, inter, k, hq, h_scale,
                    fmt, stream);
}

extern "C" FP8RL_API fp8rl_status fp8rl_debug_set(int32_t key, int64_t value) {
  // the hooks change every later call of the process: only a process that
  // asked for them (tests, profiling) may set one; restoring the defaults is
  // always allowed
  if (key != 0) {
    const char* on = std::getenv("FP8RL_TEST_HOOKS");
    if (!on || std::strcmp(on, "1") != 0) return FP8RL_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  switch (key) {
    case 1:
      if (value != 0 && value != 128 && value != 256) return FP8RL_ERR_INVALID_ARG;
      g_debug.bn = (int)value;
      return FP8RL_OK;
    case 2:
      g_debug.fault_skip_kb = value < 0 ? -1 : (int)value;
      return FP8RL_OK;
    case 3:
      if (value <= 0) return FP8RL_ERR_INVALID_ARG;
      g_debug.timeout_ns = (uint64_t)value;
      return FP8RL_OK;
    case 4:
      if (value < 0 || value > 3) return FP8RL_ERR_INVALID_ARG;
      g_debug.wait_mode = (int)value;
      return FP8RL_OK;
    case 5:
      if (value < 0 || value > 64) return FP8RL_ERR_INVALID_ARG;
      g_debug.l2_prefetch = (int)value;
      return FP8RL_OK;
    case 6:
      if (value < 0 || value > 8) return FP8RL_ERR_INVALID_ARG;
      g_debug.splits = (int)value;
      return FP8RL_OK;
    case 7:
      if (value < 0 || value > 2) return FP8RL_ERR_INVALID_ARG;
      g_debug.streamk = (int)value;
      return FP8RL_OK;
    case 8:
      if (value < 0 || value > 1024) return FP8RL_ERR_INVALID_ARG;
      g_debug.streamk_grid = (int)value;
      return FP8RL_OK;
    case 9:
      if (value < 0 || value > 2) return FP8RL_ERR_INVALID_ARG;
      g_debug.out_stage = (int)value;
      return FP8RL_OK;
    case 10:
      if (value < 0 || value > 2) return FP8RL_ERR_INVALID_ARG;
      g_debug.decode = (int)value;
      return FP8RL_OK;
    case 11:
      if (value < 0 || value > 2) return FP8RL_ERR_INVALID_ARG;
      g_debug.mx = (int)value;
      return FP8RL_OK;
    case 12:
      if (value < 0 || value > 2) return FP8RL_ERR_INVALID_ARG;
      g_debug.pair = (int)value;
      return FP8RL_OK;
    case 13:
      if (value < 0 || value > 1) return FP8RL_ERR_INVALID_ARG;
      g_pdl_off.store((int)value);
      return FP8RL_OK;
    case 0:
      g_debug = Debug{};
      g_pdl_off.store(0);
      return FP8RL_OK;
  }
  return FP8RL_ERR_INVALID_ARG;
}
