// common.cuh -- device-side numerics shared by the quantiser and GEMM kernels.
//
// E4M3 conversion uses the hardware convert (cvt.rn.satfinite.e4m3x2.f32:
// round-to-nearest-even, saturating to +-448); the scale is the IEEE fp32
// quotient amax / 448 and each element is rounded from the IEEE fp32 quotient
// x / scale (FP8-RL page, "Prerequisites / FP8 quantisation format", read as
// scale = amax / 448).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8rl.h"

namespace fp8rl {

constexpr int kBlock = 128;         // weight block edge and activation group width
constexpr float kE4M3Max = 448.0f;  // largest finite E4M3 magnitude

// ------------------------------------------------------------------ bf16 pairs

// the two bf16 values packed in a 32-bit word, low half first
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// |a| and |b| of two packed bf16 values, then the per-half unsigned max; the
// magnitude bit patterns of non-negative floats order like unsigned integers.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t u) {
  return __vmaxu2(acc, u & 0x7FFF7FFFu);
}
__device__ __forceinline__ float absmax_bf16x2_to_f32(uint32_t acc) {
  uint32_t lo = acc & 0xFFFFu, hi = acc >> 16;
  return __uint_as_float((lo > hi ? lo : hi) << 16);
}

// ------------------------------------------------------------------ E4M3

// two fp32 values -> two E4M3 codes (a in the low byte, b in the high byte)
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// ------------------------------------------------------------------ scales

// fp32 scale of a block with absolute maximum amax (zeros: 1.0)
__device__ __forceinline__ float scale_fp32(float amax) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, kE4M3Max);
}

// Correctly rounded x / s from r = RN(1/s), in three fp32 operations
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990: with r the correctly
// rounded reciprocal and q0 = RN(x r) within one ulp of x / s, the remainder
// x - q0 s is exact under an FMA and one more FMA gives RN(x / s)).  The
// remainder is formed as q0 s - x and subtracted, so that x = -0 gives -0.
// Valid while s, x / s and the remainder stay in the normal range; callers use
// it only for scales s >= kFastDivMinScale, where every quotient that can round
// to a non-zero E4M3 code is a normal number.  Checked bit for bit against IEEE
// division by the GPU tests: every bf16 x against every amax mantissa at
// exponents across the whole range, both sides of the threshold included (the
// quotient is unchanged when x and amax share a power-of-two shift away from
// the ends of the range).
constexpr float kFastDivMinScale = 0x1p-80f;

__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(q0, s, -x);
  return __fmaf_rn(-e, r, q0);
}

// ------------------------------------------------------------------ fp32 pairs
// Two IEEE fp32 operations per instruction (mul/fma.rn.f32x2, no flush of
// subnormals): the same results as the scalar operations on each half.

__device__ __forceinline__ uint64_t pair_of(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}

__device__ __forceinline__ uint64_t pair_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint64_t pair_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// two E4M3 codes (low byte from the low half) of an fp32 pair
__device__ __forceinline__ uint32_t e4m3x2_pair(uint64_t p) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
  return e4m3x2(lo, hi);
}

// div_by_scale on the two bf16 values of word w, as pairs.  Written from -x
// (one XOR of the packed sign bits): q0 = (-x)(-r) = RN(x r), the remainder
// q0 s + (-x) and q = q0 + e (-r) round exactly as the scalar form, signed
// zeros included.
__device__ __forceinline__ uint64_t div_by_scale_pair(uint32_t w, uint64_t s2, uint64_t nr2) {
  const uint32_t nw = w ^ 0x80008000u;
  const uint64_t nx = pair_of(bf16_lo(nw), bf16_hi(nw));
  const uint64_t q0 = pair_mul(nx, nr2);
  const uint64_t e = pair_fma(q0, s2, nx);
  return pair_fma(e, nr2, q0);
}

// UE8M0 exponent: smallest e with 448 * 2^e >= amax, in [-127, 127]; zeros: 0.
// Exact integer form: for a normal amax = (1 + m / 2^23) 2^(E - 127) and
// 448 = 1.75 * 2^8, e = E - 135 when 1 + m / 2^23 <= 1.75 (m <= 0x600000),
// else E - 134.  A subnormal amax is below 448 * 2^-127 and clamps to -127.
__device__ __forceinline__ int scale_ue8m0_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (b == 0) return 0;
  const int E = (int)(b >> 23);
  if (E == 0) return -127;
  const int e = E - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as an fp32 (e in [-126, 127] gives a normal number; -127 -> 2^127)
__device__ __forceinline__ float exp2_neg(int e) { return __int_as_float((127 - e) << 23); }

// ------------------------------------------------------------------ eight values

// 8 bf16 (one uint4) -> 8 E4M3 codes (two 32-bit words), fp32-scale variant:
// IEEE division for tiny scales, else the three-operation division by the
// block's correctly rounded reciprocal rcp (same result, see div_by_scale).
__device__ __forceinline__ uint2 quant8_div(uint4 v, float s, float rcp) {
  uint2 r;
  if (s >= kFastDivMinScale) {
    const uint64_t s2 = pair_of(s, s), nr2 = pair_of(-rcp, -rcp);
    r.x = e4m3x2_pair(div_by_scale_pair(v.x, s2, nr2)) | (e4m3x2_pair(div_by_scale_pair(v.y, s2, nr2)) << 16);
    r.y = e4m3x2_pair(div_by_scale_pair(v.z, s2, nr2)) | (e4m3x2_pair(div_by_scale_pair(v.w, s2, nr2)) << 16);
  } else {
    r.x = e4m3x2(__fdiv_rn(bf16_lo(v.x), s), __fdiv_rn(bf16_hi(v.x), s)) |
          (e4m3x2(__fdiv_rn(bf16_lo(v.y), s), __fdiv_rn(bf16_hi(v.y), s)) << 16);
    r.y = e4m3x2(__fdiv_rn(bf16_lo(v.z), s), __fdiv_rn(bf16_hi(v.z), s)) |
          (e4m3x2(__fdiv_rn(bf16_lo(v.w), s), __fdiv_rn(bf16_hi(v.w), s)) << 16);
  }
  return r;
}

// the same with an exact power-of-two multiplier (UE8M0 variant)
__device__ __forceinline__ uint2 quant8_mul(uint4 v, float f) {
  const uint64_t f2 = pair_of(f, f);
  auto one = [&](uint32_t w) { return e4m3x2_pair(pair_mul(pair_of(bf16_lo(w), bf16_hi(w)), f2)); };
  uint2 r;
  r.x = one(v.x) | (one(v.y) << 16);
  r.y = one(v.z) | (one(v.w) << 16);
  return r;
}

__device__ __forceinline__ uint32_t absmax_u4(uint32_t acc, uint4 v) {
  acc = absmax_bf16x2(acc, v.x);
  acc = absmax_bf16x2(acc, v.y);
  acc = absmax_bf16x2(acc, v.z);
  return absmax_bf16x2(acc, v.w);
}

// ------------------------------------------------------------------ errors

// bits recorded in a device error word
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrDeviceCheck = 2u;

// Debug builds (compiled with FP8RL_DEBUG): the kernels check the index of
// each global store against its buffer before storing; a failed check sets
// kErrDeviceCheck in the device error word and the store is skipped (no
// trap).  Release builds compile the checks away.
__device__ __forceinline__ bool dcheck(bool ok, uint32_t* err) {
#ifdef FP8RL_DEBUG
  if (!ok && err) atomicOr(err, kErrDeviceCheck);
  return ok;
#else
  (void)err;
  return true;
#endif
}

// the device error word of the current device and context (api.cu)
uint32_t* device_error_word();

// A process-unique id of the CUDA context current on this thread, making the
// runtime's primary context of the current device current first if there is
// none yet; 0 if it cannot be found.  Per-device host caches of device
// addresses and function attributes keep the id they were made under and are
// rebuilt when it changes (a cudaDeviceReset destroys the context: addresses
// cached from the old one would point nowhere).  api.cu.
uint64_t current_context_id();

// Whether the activation quantiser and the decode GEMM are launched with
// programmatic stream serialisation (on unless test hook 13 turns it off;
// gemm.cu)
bool pdl_enabled();

}  // namespace fp8rl
