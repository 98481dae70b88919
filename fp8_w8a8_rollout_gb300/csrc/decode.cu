// decode.cu -- the block-scaled W8A8 GEMM for decode-sized M (up to 128
// tokens; by default the GEMMs route at most 64 here), with the operands
// swapped.
//
// Same product as gemm.cu (FP8-RL page, "Method steps": E4M3 operands, one
// scale per 128x128 weight block and per 1x128 activation group, fp32
// accumulation, one bf16 rounding): Y[m][n] = bf16(sum over 128-wide K chunks
// kb of sx[kb][m] * sw[n/128][kb] * P_kb[m][n]).  At decode sizes the weights
// are the whole cost (HBM-bound), so the tensor-core tile is turned around:
// the MMA's 128 rows are 128 weight rows and its N is the token count padded
// to NT = 16, 32, 64 or 128.  A CTA's accumulator is then 128 x NT fp32 (four
// buffers, two at 128 columns, so the MMA runs ahead of the epilogue), four
// epilogue warps per 32 token columns promote each chunk with up to 32
// multiply-adds per thread (instead of a 128 x 128 tile of which only the
// first rows are real), and every operand stage carries 16 KB of weights and
// only NT rows of activations.  Up to 32 columns the chunk scales reach the
// epilogue 32 chunks at a time (one lane per chunk, shared by shuffles); with
// more columns (more warps, fewer registers each) every warp keeps a ring of
// eight chunks' scales in shared memory, filled ahead by asynchronous copies.
//
// Split K: a cluster of `splits` CTAs (grid y) shares one 128-row weight
// block, each a contiguous K range; their fp32 partials meet through
// distributed shared memory, summed in rank order, every rank's 16-byte
// pieces requested before the first is added.
//
// Launch (measured on GB300, 16 tokens, weights streamed from HBM): a power
// of two of splits that keeps about two CTAs per SM, as many stages as let
// two CTAs share an SM; the first stages' weight tiles are requested by the
// thread that initialises the barriers, before the block's setup completes.
// With overlapped launches (programmatic stream serialisation) the kernel
// lets the next one start at once and waits for the previous one only
// before it loads activations and scales of X or writes Y.  Qwen3-8B
// projections at 16 tokens, back to back: 6144 x 4096 11.0 -> 7.8 us,
// 4096 x 4096 7.4 -> 6.7, 4096 x 12288 14.4 -> 11.7, 24576 x 4096 20.8 -> 19.5.
//
// Roles (192 threads): warp 0 lane 0 the TMA producer, warp 1 the TMEM
// allocator and (lane 0) the MMA issuer, warps 2-5 the epilogue (TMEM lane
// quadrant = warp mod 4, thread = weight row).  Every wait is bounded, as in
// gemm.cu: on expiry the CTA raises its abort flag and the device error word,
// all roles leave their loops, and every thread still reaches the cluster
// barriers and the common teardown.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8rl {
namespace {

using namespace ptx;

constexpr int kDecMaxStages = 12; // operand stages at most (one CTA per SM)
constexpr int kDecMaxAccBufs = 4; // accumulator buffers at most
constexpr int kDecMaxSplits = 8;  // K splits per weight block (cluster size)
constexpr int kDecRing = 8;       // chunks of scales in flight per epilogue warp (64 tokens and more)
constexpr int kDecRingSlot = 40;  // words per ring slot: 32 token scales, the weight scale, padding
constexpr int kDecQRing = 16;     // chunks of in-kernel activation scales kept (fused quantisation)
constexpr int kDecRows = 128;   // weight rows per tile (the MMA's M)
constexpr int kDecWBytes = kDecRows * 128;  // one 128-wide K chunk of the weight block

struct DecArgs {
  const void* sx;  // [K/128][rows] fp32 or UE8M0 bytes
  const void* sw;  // [N/128][K/128]
  __nv_bfloat16* y;
  int32_t rows, n, k, splits;
  int32_t stages;  // operand stages in shared memory (at most kDecMaxStages)
  uint32_t* err;
  uint64_t timeout_ns;
  int32_t fault_skip_kb;  // test hook: the producer never fills this K chunk (-1: off)
  // fused activation quantisation: the E4M3 codes [rows][k] and scales
  // [k/128][rows] written out as fp8rl_quant_act_group writes them (by the
  // CTAs of the first weight block; null: not written)
  uint8_t* xq_out;
  void* sx_out;
};

// NT token columns (16, 32, 64 or 128): up to 32 per epilogue thread, so 4
// epilogue warps (one per TMEM lane quadrant) for every 32 columns.  QX: the
// kernel quantises the bf16 activations itself (more warps; NT <= 32).
template <int NT, bool QX = false>
struct DecCfg {
  static_assert(!QX || NT <= 32, "fused quantisation up to 32 token columns");
  static constexpr int kSlice = NT < 32 ? NT : 32;   // token columns per epilogue thread
  static constexpr int kEpiWarps = 4 * (NT / kSlice);
  // activation quantiser warps (four tokens each per pass; two at 32
  // columns, where four would not leave the registers for two CTAs per SM)
  static constexpr int kQWarps = QX ? (NT <= 16 ? 4 : 2) : 0;
  static constexpr int kThreads = 64 + 32 * (kEpiWarps + kQWarps);
  static constexpr int kAccBufs = NT <= 64 ? 4 : 2;   // 256 TMEM columns at most, two CTAs per SM
  static constexpr int kTmemCols = kAccBufs * NT < 32 ? 32 : kAccBufs * NT;  // a power of two
  static constexpr int kXBytes = NT * 128;            // E4M3 activation codes of a chunk
  // Fused quantisation: the activations travel through their own ring of
  // kXRing slots (the chunk's codes, then their bf16 source), so that their
  // quantisation runs ahead of the MMA without holding a weight stage.
  static constexpr int kXRing = QX ? 4 : 0;
  static constexpr int kXRingDiv = QX ? kXRing : 1;  // the ring as a divisor (reached only when QX)
  static constexpr int kXRawBytes = NT * 256;
  static constexpr int kXSlotBytes = kXBytes + kXRawBytes;
  static constexpr int kStageBytes = kDecWBytes + (QX ? 0 : kXBytes);  // a weight stage (+ the codes unfused)
  static constexpr int kTmaBytes = kStageBytes;                         // what a stage's copies bring
  static constexpr int kBookBytes = 512;
  // the activation ring, the epilogue warps' scale rings (64 token columns
  // and more) and the in-kernel activation scales (fused quantisation)
  static constexpr int kFixedBytes = kXRing * kXSlotBytes + kBookBytes +
                                     (NT > 32 ? kEpiWarps * kDecRing * kDecRingSlot * 4 : 0) +
                                     (QX ? kDecQRing * NT * 4 : 0);
  static constexpr int smem_bytes(int stages) { return 1024 + stages * kStageBytes + kFixedBytes; }
  // the most stages one CTA can hold (227 KB of shared memory per block)
  static constexpr int kStagesFit = (227 * 1024 - 1024 - kFixedBytes) / kStageBytes;
  static constexpr int kMaxStages = kStagesFit < kDecMaxStages ? kStagesFit : kDecMaxStages;
  // the most stages that let two CTAs share an SM (228 KB of shared memory,
  // 1 KB of it reserved per CTA); below three, one CTA per SM with more
  static constexpr int kPairStages = (114 * 1024 - 1024 - 1024 - kFixedBytes) / kStageBytes;
  static constexpr bool kPairs = kPairStages >= 3;
  static constexpr int kStages = kPairs ? kPairStages : kMaxStages;
  static constexpr int kMinBlocks = kPairs ? 2 : 1;
  static_assert(kStages >= 2 && kStages <= kDecMaxStages, "stages");
  static_assert(kDecRows * NT * 4 <= kStages * kStageBytes, "the split partial fits over the operand stages");
  static_assert(kAccBufs <= kDecMaxAccBufs, "accumulators");
  static_assert((3 * kDecMaxStages + 2 * kDecMaxAccBufs + 1 + kDecQRing) * 8 + 8 <= kBookBytes, "bookkeeping");
  static_assert(3 * kXRing <= kDecMaxStages, "activation ring barriers");
  // the quantiser runs at most kXRing chunks ahead of the MMA, the MMA the
  // accumulators ahead of the epilogue
  static_assert(kXRing + kDecMaxAccBufs < kDecQRing, "the activation-scale ring outlives its readers");
};

// a scale as fp32: the word holding it (a UE8M0 byte sits in an aligned
// 32-bit word), decoded as gemm.cu does: byte b -> 2^(b - 127)
template <bool UE8M0>
__device__ __forceinline__ float dec_scale(const void* p, int64_t idx) {
  if (UE8M0) {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(p) + (idx & ~(int64_t)3)));
    const uint32_t b = (w >> (8 * (idx & 3))) & 0xFFu;
    return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
  }
  return __ldg(static_cast<const float*>(p) + idx);
}

// 16 bytes of another CTA's shared memory (a cluster address from mapa);
// volatile keeps it after the cluster barrier that makes the data valid
__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// two fp32 values rounded to nearest-even bf16, the first in the low half
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// the scale 2^(b - 127) of UE8M0 byte `which` of a 32-bit word (byte 0: 2^-127)
__device__ __forceinline__ float ue8m0_word_to_f32(uint32_t word, uint32_t which) {
  const uint32_t b = (word >> (8u * which)) & 0xFFu;
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// TMEM allocation with the column count as an immediate operand
template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_alloc_n(uint32_t slot_smem) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "n"(NCOLS)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[W]) {
  if constexpr (W == 32) {
    tmem_ld_32x32b_x32(taddr, v);
  } else {
    tmem_ld_32x32b_x16(taddr, v);
  }
}

template <int NT, bool UE8M0, bool QX>
__global__ void __launch_bounds__(DecCfg<NT, QX>::kThreads, DecCfg<NT, QX>::kMinBlocks)
    gemm_decode_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                       const DecArgs a) {
  using C = DecCfg<NT, QX>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const int stages = a.stages;
  const uint32_t sW = base;                                 // stages x 16 KB
  const uint32_t sX = base + stages * kDecWBytes;           // stages x NT x 128 B (unfused)
  const uint32_t xring = base + stages * C::kStageBytes;    // kXRing x (codes | bf16) (fused quantisation)
  uint8_t* book = base_ptr + stages * C::kStageBytes + C::kXRing * C::kXSlotBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(book);
  uint64_t* empty = full + kDecMaxStages;
  uint64_t* xfull = empty + kDecMaxStages;  // [kXRing] an activation slot's bf16 chunk has landed
  uint64_t* xready = xfull + 4;             // [kXRing] ... its codes are written (quantiser warps)
  uint64_t* xempty = xready + 4;            // [kXRing] ... the MMAs that read them have completed
  uint64_t* tfull = xfull + kDecMaxStages;
  uint64_t* tempty = tfull + kDecMaxAccBufs;
  uint64_t* drain = tempty + kDecMaxAccBufs;
  uint64_t* qready = drain + 1;  // [kDecQRing]: a chunk's activation scales are in the ring (fused quantisation)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qready + kDecQRing);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  volatile int* abortv = abort_flag;
  const uint32_t ring = smem_u32(book + C::kBookBytes);  // epilogue scale rings
  float* qring = reinterpret_cast<float*>(book + C::kBookBytes);  // [kDecQRing][NT] (fused quantisation)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = blockIdx.x;
  const int splits = a.splits;
  const int split = splits > 1 ? (int)cluster_ctarank() : 0;
  const int num_kb = a.k / 128;
  const int kb_lo = (int)((int64_t)num_kb * split / splits);
  const int nloc = (int)((int64_t)num_kb * (split + 1) / splits) - kb_lo;
  const int pre = nloc < stages ? nloc : stages;  // stages filled before the loop

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int r = 0; r < C::kXRing; ++r) {
      mbar_init(smem_u32(&xfull[r]), 1);
      mbar_init(smem_u32(&xready[r]), C::kQWarps);
      mbar_init(smem_u32(&xempty[r]), 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(smem_u32(&tfull[b]), 1);
      mbar_init(smem_u32(&tempty[b]), C::kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(smem_u32(drain), 1);
    if (QX)
      for (int r = 0; r < kDecQRing; ++r) mbar_init(smem_u32(&qready[r]), C::kQWarps);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_shared();  // the barriers are seen by this thread's copies below
    // No kernel of this library that lets a dependent start early writes
    // weights (the weight quantiser does not), so the first stages' weight
    // tiles are requested at once, before the block's setup completes and
    // before the wait for the earlier kernels of the stream; the
    // activations, their outputs, are loaded after that wait.
    prefetch_tensormap(&tmap_w);
    for (int j = 0; j < pre; ++j) {
      if (kb_lo + j == a.fault_skip_kb) continue;
      const uint32_t fb = smem_u32(&full[j]);
      mbar_arrive_expect_tx(fb, C::kTmaBytes);
      tma_load_2d(sW + j * kDecWBytes, &tmap_w, (kb_lo + j) * 128, nblk * kDecRows, fb);
    }
  }
  if (warp == 1) tmem_alloc_n<C::kTmemCols>(smem_u32(tmem_slot));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The next kernel of the stream may start now (when launched with
  // programmatic stream serialisation: it waits for this grid's completion
  // before it reads anything this grid writes).
  grid_dep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_x);
      grid_dep_wait();
      // fused quantisation: activation chunk c into slot c mod kXRing once the
      // MMAs of chunk c - kXRing have completed; false when a wait ran out
      int xissued = 0;
      auto issue_x = [&](int c) {
        const int xs = c % C::kXRingDiv;
        if (c >= C::kXRing &&
            !mbar_wait_bounded(smem_u32(&xempty[xs]), ((c / C::kXRingDiv) - 1) & 1, abortv, a.err, a.timeout_ns))
          return false;
        mbar_arrive_expect_tx(smem_u32(&xfull[xs]), C::kXRawBytes);
        tma_load_2d(xring + xs * C::kXSlotBytes + C::kXBytes, &tmap_x, (kb_lo + c) * 128, 0, smem_u32(&xfull[xs]));
        xissued = c + 1;
        return true;
      };
      if (QX) {
        for (int c = 0; c < nloc && c < C::kXRing; ++c) issue_x(c);
      } else {
        for (int j = 0; j < pre; ++j)
          if (kb_lo + j != a.fault_skip_kb)
            tma_load_2d(sX + j * C::kXBytes, &tmap_x, (kb_lo + j) * 128, 0, smem_u32(&full[j]));
      }
      int it = pre;
      bool alive = true;
      for (; it < nloc; ++it) {
        const int s = it % stages;
        const uint32_t ph = (it / stages) & 1;
        if (!mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1, abortv, a.err, a.timeout_ns)) {
          alive = false;
          break;
        }
        // (the MMAs of chunk it - stages have completed: so have those that
        // free the activation slot of chunk it - stages + kXRing)
        const int c = it - stages + C::kXRing;
        if (QX && c >= xissued && c < nloc && !issue_x(c)) {
          alive = false;
          break;
        }
        const int kb = kb_lo + it;
        if (kb == a.fault_skip_kb) continue;  // the MMA's wait on this stage runs out
        const uint32_t fb = smem_u32(&full[s]);
        mbar_arrive_expect_tx(fb, C::kTmaBytes);
        tma_load_2d(sW + s * kDecWBytes, &tmap_w, kb * 128, nblk * kDecRows, fb);
        if (!QX) tma_load_2d(sX + s * C::kXBytes, &tmap_x, kb * 128, 0, fb);
      }
      if (QX)
        while (alive && xissued < nloc && issue_x(xissued)) {
        }
      if (*abortv) {
        // let the copies still in flight land before shared memory is released
        for (int j = it > stages ? it - stages : 0; j < it; ++j)
          if (kb_lo + j != a.fault_skip_kb)
            mbar_wait_bounded(smem_u32(&full[j % stages]), (j / stages) & 1, nullptr, nullptr, 10000000ull);
        for (int c = xissued > C::kXRing ? xissued - C::kXRing : 0; c < xissued; ++c)
          mbar_wait_bounded(smem_u32(&xfull[c % C::kXRingDiv]), (c / C::kXRingDiv) & 1, nullptr, nullptr, 10000000ull);
      }
    } else {
      grid_dep_wait();
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    grid_dep_wait();
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kDecRows, NT);
      for (int it = 0; it < nloc; ++it) {
        const int buf = it % C::kAccBufs;
        const uint32_t bph = (it / C::kAccBufs) & 1;
        if (!mbar_wait_bounded(smem_u32(&tempty[buf]), bph ^ 1, abortv, a.err, a.timeout_ns)) break;
        const int s = it % stages;
        const uint32_t ph = (it / stages) & 1;
        if (!mbar_wait_bounded(smem_u32(&full[s]), ph, abortv, a.err, a.timeout_ns)) break;
        const int xs = QX ? it % C::kXRingDiv : 0;
        if (QX && !mbar_wait_bounded(smem_u32(&xready[xs]), (it / C::kXRingDiv) & 1, abortv, a.err, a.timeout_ns)) break;
        tc_fence_after();
        const uint32_t a0 = sW + s * kDecWBytes;
        const uint32_t b0 = QX ? xring + xs * C::kXSlotBytes : sX + s * C::kXBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_e4m3(tmem + buf * NT, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32), idesc,
                   kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&empty[s]));
        if (QX) mma_commit(smem_u32(&xempty[xs]));
        mma_commit(smem_u32(&tfull[buf]));
      }
      if (*abortv) {
        // no MMA may still be writing TMEM when it is released
        mma_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, nullptr, nullptr, 10000000ull);
      }
    }
    __syncwarp();
  }

  if (QX && warp >= 2 + C::kEpiWarps) {
    // ------------------------------------------------------------ activation quantiser
    // Chunk c's bf16 activations [NT][128] land in activation slot c mod
    // kXRing (requested by the producer; a slot is refilled once the MMAs that
    // read its codes have completed).  Each warp quantises 4 tokens per pass (eight lanes per
    // token, 16 values each) with the arithmetic of the activation quantiser,
    // so the codes and scales are those fp8rl_quant_act_group writes: E4M3
    // codes into the slot in the 128-byte-swizzled layout the MMA reads, the
    // scale into the chunk's ring slot for the epilogue.  The first weight
    // block's CTAs also write both out.
    grid_dep_wait();  // the activations come from earlier kernels; nothing is written before they end
    const int qw = warp - (2 + C::kEpiWarps);
    const int part = lane & 7;
    const bool out = a.xq_out != nullptr && nblk == 0;
    for (int it = 0; it < nloc; ++it) {
      const int xs = it % C::kXRingDiv;
      bool got = mbar_wait_bounded(smem_u32(&xfull[xs]), (it / C::kXRingDiv) & 1, abortv, a.err, a.timeout_ns);
      got = __all_sync(0xffffffffu, got);
      if (!got) break;
      const int kb = kb_lo + it;
      const uint8_t* slot = base_ptr + (xring - base) + xs * C::kXSlotBytes;
      constexpr int kPasses = NT / (4 * (C::kQWarps > 0 ? C::kQWarps : 1));
      uint2 keep[kPasses][2];  // the codes and scales, written out after the release
      float keep_s[kPasses];
      uint32_t keep_b[kPasses];
#pragma unroll
      for (int pass = 0; pass < kPasses; ++pass) {
        const int t = (pass * C::kQWarps + qw) * 4 + (lane >> 3);  // this lane's token
        const uint8_t* src = slot + C::kXBytes + t * 256;
        uint4 v[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) v[j] = *reinterpret_cast<const uint4*>(src + (part + 8 * j) * 16);
        uint32_t acc = 0;
#pragma unroll
        for (int j = 0; j < 2; ++j) acc = absmax_u4(acc, v[j]);
        uint32_t am = max(acc & 0xFFFFu, acc >> 16);
        am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
        am = max(am, __shfl_xor_sync(0xffffffffu, am, 4));
        const float amax = __uint_as_float(am << 16);
        uint2 codes[2];
        float sf;
        uint32_t sbyte = 0;
        if (UE8M0) {
          const int e = scale_ue8m0_exponent(amax);
          const float f = exp2_neg(e);
#pragma unroll
          for (int j = 0; j < 2; ++j) codes[j] = quant8_mul(v[j], f);
          sbyte = (uint32_t)(e + 127);
          sf = sbyte == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(sbyte << 23);
        } else {
          sf = scale_fp32(amax);
          const float rcp = __frcp_rn(sf);
#pragma unroll
          for (int j = 0; j < 2; ++j) codes[j] = quant8_div(v[j], sf, rcp);
        }
        uint8_t* dst = const_cast<uint8_t*>(slot) + t * 128;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int piece = part + 8 * j;  // 8 codes: half of 16-byte chunk piece / 2
          *reinterpret_cast<uint2*>(dst + (((piece >> 1) ^ (t & 7)) << 4) + (piece & 1) * 8) = codes[j];
        }
        if (part == 0) qring[(it % kDecQRing) * NT + t] = sf;
        keep[pass][0] = codes[0];
        keep[pass][1] = codes[1];
        keep_s[pass] = sf;
        keep_b[pass] = sbyte;
      }
      fence_proxy_async_shared();  // the codes are read by the tensor cores
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&xready[xs]));
        mbar_arrive(smem_u32(&qready[it % kDecQRing]));
      }
      if (out) {
#pragma unroll
        for (int pass = 0; pass < kPasses; ++pass) {
          const int t = (pass * C::kQWarps + qw) * 4 + (lane >> 3);
          if (t < a.rows) {
            uint8_t* q = a.xq_out + (int64_t)t * a.k + (int64_t)kb * 128;
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (dcheck(kb * 128 + (part + 8 * j) * 8 + 8 <= a.k, a.err))
                *reinterpret_cast<uint2*>(q + (part + 8 * j) * 8) = keep[pass][j];
            if (part == 0) {
              const int64_t si = (int64_t)kb * a.rows + t;
              if (UE8M0)
                static_cast<uint8_t*>(a.sx_out)[si] = (uint8_t)keep_b[pass];
              else
                static_cast<float*>(a.sx_out)[si] = keep_s[pass];
            }
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- epilogue
  // thread = one weight row (TMEM lane) x kSlice token columns
  const bool epi = warp >= 2 && warp < 2 + C::kEpiWarps;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;  // weight row within the block
  const int slice = epi ? (warp - 2) >> 2 : 0;
  const int tok0 = slice * C::kSlice;  // this thread's first token column
  constexpr int S = C::kSlice;
  float acc[S];
#pragma unroll
  for (int m = 0; m < S; ++m) acc[m] = 0.0f;
  bool ok = true;
  if (epi) {
    grid_dep_wait();  // the activation scales come from earlier kernels
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16) + tok0;
    if constexpr (NT <= 32) {
      // The chunks' scales, 32 chunks at a time: lane j loads chunk w0 + j's
      // weight scale and its NT activation scales (one round trip to memory
      // per 32 chunks instead of one per chunk), and each chunk's values
      // reach the whole warp by shuffles.
      float wsw = 0.0f, wsx[S];
      for (int it = 0; it < nloc; ++it) {
        const int j = it & 31;
        if (j == 0) {
          const int c = it + lane;
          const int kb = kb_lo + (c < nloc ? c : it);
          wsw = dec_scale<UE8M0>(a.sw, (int64_t)nblk * num_kb + kb);
          if (!QX) {
#pragma unroll
            for (int m = 0; m < S; ++m) wsx[m] = m < a.rows ? dec_scale<UE8M0>(a.sx, (int64_t)kb * a.rows + m) : 0.0f;
          }
        }
        const int buf = it % C::kAccBufs;
        const uint32_t bph = (it / C::kAccBufs) & 1;
        ok = mbar_wait_bounded(smem_u32(&tfull[buf]), bph, abortv, a.err, a.timeout_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float fx[S];  // fused quantisation: this chunk's activation scales, read before the release
        if (QX) {
          // (the slot is refilled only after this chunk's release: the
          // quantiser runs at most the stages plus the accumulators ahead)
          ok = mbar_wait_bounded(smem_u32(&qready[it % kDecQRing]), (it / kDecQRing) & 1, abortv, a.err,
                                 a.timeout_ns);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
#pragma unroll
          for (int m = 0; m < S; ++m) fx[m] = qring[(it % kDecQRing) * NT + m];
        }
        uint32_t v[S];
        tmem_ld_cols<S>(t_lane + buf * NT, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
        // the activation scale times the weight scale, then one fused
        // multiply-add per token: the 128-row-tile kernel's arithmetic
        const float swv = __shfl_sync(0xffffffffu, wsw, j);
#pragma unroll
        for (int m = 0; m < S; ++m)
          acc[m] = fmaf(__uint_as_float(v[m]), (QX ? fx[m] : __shfl_sync(0xffffffffu, wsx[m], j)) * swv, acc[m]);
      }
    } else {
      // The chunks' scales through a ring of kDecRing slots per warp, filled
      // kDecRing chunks ahead by asynchronous 4-byte copies: lane t copies
      // the word holding token tok0 + t's scale (zeros past the last token),
      // lane 0 also the weight scale's word; every lane then reads the whole
      // slot (broadcast).  One round trip per chunk, kDecRing chunks ahead.
      const uint32_t my_ring = ring + (uint32_t)((warp - 2) * kDecRing * kDecRingSlot * 4);
      const int tok = tok0 + lane;
      auto issue = [&](int c) {  // chunk c of this CTA's range into its slot
        const uint32_t slot = my_ring + (uint32_t)((c % kDecRing) * kDecRingSlot * 4);
        if (c < nloc) {
          const int64_t kb = kb_lo + c;
          const int64_t xi = kb * a.rows + (tok < a.rows ? tok : 0);
          const int64_t wi = (int64_t)nblk * num_kb + kb;
          const uint8_t* xs = static_cast<const uint8_t*>(a.sx);
          const uint8_t* ws = static_cast<const uint8_t*>(a.sw);
          cp_async_4(slot + 4u * (uint32_t)lane, UE8M0 ? xs + (xi & ~(int64_t)3) : xs + 4 * xi, tok < a.rows ? 4u : 0u);
          if (lane == 0) cp_async_4(slot + 4u * 32u, UE8M0 ? ws + (wi & ~(int64_t)3) : ws + 4 * wi, 4u);
        }
        cp_async_commit();  // empty past the range: the group count stays uniform
      };
      for (int c = 0; c < kDecRing; ++c) issue(c);
      for (int it = 0; it < nloc; ++it) {
        const int buf = it % C::kAccBufs;
        const uint32_t bph = (it / C::kAccBufs) & 1;
        ok = mbar_wait_bounded(smem_u32(&tfull[buf]), bph, abortv, a.err, a.timeout_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t v[S];
        tmem_ld_cols<S>(t_lane + buf * NT, v);
        cp_async_wait<kDecRing - 1>();  // this chunk's scales have landed (this lane's copies)
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();  // ... and every lane's
        if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
        const int64_t kb = kb_lo + it;
        const uint32_t slot = my_ring + (uint32_t)((it % kDecRing) * kDecRingSlot * 4);
        const uint32_t* sp = reinterpret_cast<const uint32_t*>(base_ptr) + (slot - base) / 4;
        uint32_t wword = sp[32];
        const int64_t wi = (int64_t)nblk * num_kb + kb;
        const float swv = UE8M0 ? ue8m0_word_to_f32(wword, (uint32_t)(wi & 3)) : __uint_as_float(wword);
#pragma unroll
        for (int m4 = 0; m4 < S; m4 += 4) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(sp + m4);
          const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int m = m4 + q;
            const float f = UE8M0 ? ue8m0_word_to_f32(ww[q], (uint32_t)((kb * a.rows + tok0 + m) & 3)) : __uint_as_float(ww[q]);
            acc[m] = fmaf(__uint_as_float(v[m]), f * swv, acc[m]);
          }
        }
        __syncwarp();  // every lane has read the slot before it is refilled
        issue(it + kDecRing);
      }
      cp_async_wait<0>();  // no copy into the ring outlives the loop
    }
  }
  __syncthreads();  // every MMA has been consumed: the operand stages are free
  const bool write = !*abortv;
  float* part = reinterpret_cast<float*>(base_ptr);  // [NT][128] fp32 over the first weight stage
  if (splits == 1) {
    if (epi && write) {
      __nv_bfloat16* dst = a.y + (int64_t)tok0 * a.n + (int64_t)nblk * kDecRows + row;
#pragma unroll
      for (int m = 0; m < S; ++m)  // a constant bound keeps acc in registers
        if (tok0 + m < a.rows && dcheck(nblk * kDecRows + row < a.n, a.err))
          dst[(int64_t)m * a.n] = __float2bfloat16_rn(acc[m]);
    }
  } else {
    if (epi) {
#pragma unroll
      for (int m = 0; m < S; ++m) part[(tok0 + m) * kDecRows + row] = acc[m];
    }
    cluster_sync();  // every CTA's partial is in its shared memory
    if (write) {
      // This CTA's share of the outputs, four weight rows of one token at a
      // time, each the sum of the cluster's partials in rank order: all
      // ranks' 16-byte pieces are requested before the first is added.
      const int quads = a.rows * (kDecRows / 4);
      const int q0 = (int)((int64_t)quads * split / splits), q1 = (int)((int64_t)quads * (split + 1) / splits);
      const uint32_t pbase = smem_u32(part);
      for (int q = q0 + (int)threadIdx.x; q < q1; q += C::kThreads) {
        float4 p[kDecMaxSplits];
#pragma unroll
        for (int r = 0; r < kDecMaxSplits; ++r)
          if (r < splits) p[r] = ld_dsmem_f32x4(mapa_shared(pbase + 16u * (uint32_t)q, r));
        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll
        for (int r = 0; r < kDecMaxSplits; ++r)
          if (r < splits) {
            s0 += p[r].x;
            s1 += p[r].y;
            s2 += p[r].z;
            s3 += p[r].w;
          }
        const int m = q / (kDecRows / 4), nr = (q - m * (kDecRows / 4)) * 4;
        if (dcheck(m < a.rows && nblk * kDecRows + nr + 4 <= a.n, a.err)) {
          const uint32_t lo = pack_bf16x2_rn(s0, s1), hi = pack_bf16x2_rn(s2, s3);
          asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(a.y + (int64_t)m * a.n + (int64_t)nblk * kDecRows + nr),
                       "r"(lo), "r"(hi)
                       : "memory");
        }
      }
    }
    // No CTA leaves while its partial may still be read.  The values this
    // CTA loaded were consumed before the arrival, and nothing written here
    // is read through the cluster afterwards, so the arrival need not
    // release (a release would also wait for the Y stores to complete).
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

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

// E4M3 [outer][inner] row-major, boxes of box_outer rows x 128 bytes, 128-byte
// swizzle (rows past `outer` read as zeros)
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

struct DecState {
  uint64_t ctx = 0;  // the context the attributes were set in (redone when it changes)
  bool ready = false, ok = false;
  int sms = 0;
};

// bf16 [outer][inner] with row stride ld elements, boxes of box_outer rows x
// 128 elements, no swizzle (the fused quantisation's source; rows past
// `outer` read as zeros)
bool make_map_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                   uint32_t box_outer) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {128, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT, bool UE8M0, bool QX>
DecState& dec_state(int dev) {
  static DecState st[64];
  return st[dev];
}

std::mutex g_dec_mu;

// x: the E4M3 codes, or (QX) the bf16 activations with row stride ldx
template <int NT, bool UE8M0, bool QX = false>
fp8rl_status launch_decode(const void* x, const void* wq, const DecArgs& args0, int force_splits,
                           cudaStream_t stream, int64_t ldx = 0) {
  using C = DecCfg<NT, QX>;
  auto kernel = gemm_decode_kernel<NT, UE8M0, QX>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8RL_ERR_CUDA;
  DecState& st = dec_state<NT, UE8M0, QX>(dev);
  DecArgs args = args0;
  const int nblocks = args.n / kDecRows;
  const int num_kb = args.k / 128;
  const uint64_t ctx = current_context_id();
  if (!ctx) return FP8RL_ERR_CUDA;
  int splits = 1;
  const int stages = C::kStages;
  {
    std::lock_guard<std::mutex> lock(g_dec_mu);
    if (!st.ready || st.ctx != ctx) {
      st = DecState{};
      st.ctx = ctx;
      int sms = 0;
      st.ok = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0 &&
              cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   C::smem_bytes(C::kMaxStages)) == cudaSuccess &&
              cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) == cudaSuccess &&
              // the whole unified L1 as shared memory, so that two CTAs fit on an SM
              cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared) == cudaSuccess;
      st.sms = sms;
      st.ready = true;
    }
    if (!st.ok) return FP8RL_ERR_UNSUPPORTED;
    // K splits (measured on GB300 at 16 tokens, weights streamed from HBM):
    // about two CTAs per SM with few stages each beat one deep CTA per SM
    // (more CTAs keep more weight rows in flight at once), and a split count
    // that divides the K chunks evenly (a power of two) beats an uneven one.
    // Clusters that cannot all be resident at once simply run later; the
    // occupancy query reports one CTA per SM for clustered launches of this
    // kernel, but two run (measured: 6144 x 4096 weights in 4 splits, 192
    // CTAs, 7.9 us against 9.4 us for the 2 splits that query allows).
    // (64 and 128 token columns: C::kMinBlocks CTAs per SM, by shared memory.)
    if (force_splits > 0) {
      splits = std::min(std::min(force_splits, kDecMaxSplits), num_kb);
    } else {
      const int64_t slots = (int64_t)C::kMinBlocks * st.sms;
      while (splits * 2 <= kDecMaxSplits && (int64_t)nblocks * splits * 2 <= slots && num_kb / (splits * 2) >= 2)
        splits *= 2;
    }
  }
  args.splits = splits;
  args.stages = stages;
  CUtensorMap mw, mx;
  if (!make_map(&mw, wq, args.k, args.n, kDecRows)) return FP8RL_ERR_CUDA;
  if (QX ? !make_map_bf16(&mx, x, args.k, args.rows, (uint64_t)ldx, NT) : !make_map(&mx, x, args.k, args.rows, NT))
    return FP8RL_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nblocks, (unsigned)splits, 1);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::smem_bytes(stages);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (splits > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = splits;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl_enabled()) {
    // start while the previous kernel of the stream finishes: the prologue
    // and the first weight stages overlap its tail (the kernel waits for it
    // before loading activations or writing Y)
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kernel, mw, mx, args) != cudaSuccess) {
    cudaGetLastError();
    return FP8RL_ERR_CUDA;
  }
  return FP8RL_OK;
}

}  // namespace

// Called by the GEMM entry points for dense products with rows <= 128 (the
// arguments already validated); UNSUPPORTED lets the caller fall back to the
// 128-row-tile kernel.
fp8rl_status decode_gemm(const void* xq, const void* x_scale, const void* wq, const void* w_scale, void* y,
                         int64_t rows, int64_t n, int64_t k, bool ue8m0, uint32_t* err, uint64_t timeout_ns,
                         int fault_skip_kb, int force_splits, cudaStream_t stream) {
  if (rows < 1 || rows > 128 || n % kDecRows || k % 128) return FP8RL_ERR_UNSUPPORTED;
  DecArgs a{};
  a.sx = x_scale;
  a.sw = w_scale;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.rows = (int32_t)rows;
  a.n = (int32_t)n;
  a.k = (int32_t)k;
  a.err = err;
  a.timeout_ns = timeout_ns;
  a.fault_skip_kb = fault_skip_kb;
  a.xq_out = nullptr;
  a.sx_out = nullptr;
  if (rows <= 16)
    return ue8m0 ? launch_decode<16, true>(xq, wq, a, force_splits, stream)
                 : launch_decode<16, false>(xq, wq, a, force_splits, stream);
  if (rows <= 32)
    return ue8m0 ? launch_decode<32, true>(xq, wq, a, force_splits, stream)
                 : launch_decode<32, false>(xq, wq, a, force_splits, stream);
  if (rows <= 64)
    return ue8m0 ? launch_decode<64, true>(xq, wq, a, force_splits, stream)
                 : launch_decode<64, false>(xq, wq, a, force_splits, stream);
  return ue8m0 ? launch_decode<128, true>(xq, wq, a, force_splits, stream)
               : launch_decode<128, false>(xq, wq, a, force_splits, stream);
}

// The decode GEMM with the activation quantisation inside (at most 16 rows):
// bf16 X [rows][k] (row stride ldx elements, 16-byte aligned rows) is
// quantised in 1x128 groups exactly as fp8rl_quant_act_group does; the codes
// and scales are also written to xq_out ([rows][k]) and sx_out ([k/128][rows])
// when those are given.  UNSUPPORTED for shapes it does not take.
fp8rl_status decode_gemm_qx(const void* x_bf16, int64_t ldx, const void* wq, const void* w_scale, void* y,
                            int64_t rows, int64_t n, int64_t k, bool ue8m0, void* xq_out, void* sx_out,
                            uint32_t* err, uint64_t timeout_ns, int fault_skip_kb, int force_splits,
                            cudaStream_t stream) {
  // (up to 16 rows: with 32 token columns the in-kernel quantisation is
  // slower than the separate quantiser, measured on GB300)
  if (rows < 1 || rows > 16 || n % kDecRows || k % 128 || (ldx * 2) % 16 ||
      (reinterpret_cast<uintptr_t>(x_bf16) & 15))
    return FP8RL_ERR_UNSUPPORTED;
  DecArgs a{};
  a.sx = nullptr;
  a.sw = w_scale;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.rows = (int32_t)rows;
  a.n = (int32_t)n;
  a.k = (int32_t)k;
  a.err = err;
  a.timeout_ns = timeout_ns;
  a.fault_skip_kb = fault_skip_kb;
  a.xq_out = static_cast<uint8_t*>(xq_out);
  a.sx_out = sx_out;
  return ue8m0 ? launch_decode<16, true, true>(x_bf16, wq, a, force_splits, stream, ldx)
               : launch_decode<16, false, true>(x_bf16, wq, a, force_splits, stream, ldx);
}

}  // namespace fp8rl
