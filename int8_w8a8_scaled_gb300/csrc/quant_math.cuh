// quant_math.cuh -- the quantiser's element arithmetic, shared by the
// stand-alone quantiser kernels (quant.cu) and the matmul that quantises its
// own activations (gemm.cu), so that both produce the same codes and scales.
//
// "[Kernel] Support Fp8 Checkpoints (Dynamic + Static)", review thread: the
// dynamic scale is absmax / 448 (e4m3) or absmax / 127 (int8), the code is
// the input divided by the scale, clamped to the finite range and rounded;
// "Enable scaled FP8 (e4m3fn) KV cache on ROCm (AMD GPU)", "Scaling
// semantics": a tensor with no scale (all zeros here) has the factor 1.0.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace w8a8 {
namespace {  // each translation unit keeps its own copy

template <int KIND>
__device__ __forceinline__ float cvt_in(uint16_t b) {
  if (KIND == 0) return __bfloat162float(__ushort_as_bfloat16(b));
  return __half2float(__ushort_as_half(b));
}

// 8 consecutive 16-bit inputs from a 128-bit word.
template <int KIND>
__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = cvt_in<KIND>(static_cast<uint16_t>(u[j] & 0xFFFFu));
    f[2 * j + 1] = cvt_in<KIND>(static_cast<uint16_t>(u[j] >> 16));
  }
}

// Two fp32 -> two e4m3 codes (low byte = first), RNE, saturating; NaN -> 0x7F.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  uint32_t out = r;
  if (a != a) out = (out & 0xFF00u) | 0x7Fu;
  if (b != b) out = (out & 0x00FFu) | 0x7F00u;
  return out;
}

// Four fp32 -> four e4m3 codes in one word (low byte = first).  The
// satfinite conversion never gives 0x7F / 0xFF for a number (its largest
// magnitude is 0x7E), so the NaN codes are exactly the bytes whose low seven
// bits are all ones; their sign bit is cleared once for the whole word
// (0x7F + 1 carries into the byte's top bit and no further).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  const uint32_t w = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  const uint32_t nan_top = ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
  return w & ~nan_top;
}

__device__ __forceinline__ uint32_t int8x1(float a) {
  int i;
  asm("cvt.rni.s32.f32 %0, %1;" : "=r"(i) : "f"(a));  // RNE; NaN -> 0; saturates to int32
  i = max(-128, min(127, i));
  return static_cast<uint32_t>(i) & 0xFFu;
}

template <int QK>
__device__ __forceinline__ uint32_t enc4(float a, float b, float c, float d) {
  if (QK == 0) return e4m3x4(a, b, c, d);
  return int8x1(a) | (int8x1(b) << 8) | (int8x1(c) << 16) | (int8x1(d) << 24);
}

template <int QK>
__device__ __forceinline__ uint8_t enc1(float a) {
  if (QK == 0) return static_cast<uint8_t>(e4m3x2(a, 0.f) & 0xFFu);
  return static_cast<uint8_t>(int8x1(a));
}

// Correctly rounded x / s without a per-element division.
//
// With y = RN(1/s) (one IEEE division per thread), q0 = RN(x*y) lies within
// one ulp of x/s, so the (negated) remainder q0*s - x is exact in one FMA
// and RN(q0 - (q0*s - x)*y) is the correctly rounded quotient RN(x/s)
// (Markstein's correction step for IEEE division with a correctly rounded
// reciprocal).  Taking the remainder negated also gets the sign of a zero
// quotient right: for x = -0 both addends of the correction are -0.
// Preconditions: s and y are normal finite floats (checked per thread;
// otherwise the plain IEEE division is used) and no intermediate overflows.
// kBounded: the quotient is known to stay near the code range (dynamic
// scales: s is absmax / 448 or absmax / 127, so |x / s| cannot exceed the
// largest code by more than a rounding); otherwise quotients beyond
// kSatQuot, far past the largest code, are taken as q0 uncorrected -- they
// saturate whatever their last bits, and this covers q0 = +-inf (x*y
// overflowed, or x is infinite), where the correction would make a NaN.
// A NaN x gives a NaN quotient either way.  Quotients in the fp32 subnormal
// range all encode to a signed zero, whatever their last bits.
__device__ __forceinline__ bool recip_ok(float s, float* y) {
  const float r = __fdiv_rn(1.0f, s);
  *y = r;
  const uint32_t es = (__float_as_uint(s) >> 23) & 0xFFu, er = (__float_as_uint(r) >> 23) & 0xFFu;
  return es != 0u && es != 0xFFu && er != 0u && er != 0xFFu;
}

constexpr float kSatQuot = 1024.f;

template <bool kBounded>
__device__ __forceinline__ float div_by(float x, float s, float y, bool ok) {
  if (!ok) return __fdiv_rn(x, s);
  const float q0 = __fmul_rn(x, y);
  const float nrem = __fmaf_rn(q0, s, -x);
  const float q1 = __fmaf_rn(-nrem, y, q0);
  if (kBounded) return q1;
  return fabsf(q0) < kSatQuot ? q1 : q0;
}

// Codes of 4 / 8 / 16 consecutive values and of one value; `bounded` picks
// the division without the saturation guard (dynamic scales).
template <int QK, bool kB>
__device__ __forceinline__ uint32_t quant4(const float* f, float s, float y, bool ok) {
  return enc4<QK>(div_by<kB>(f[0], s, y, ok), div_by<kB>(f[1], s, y, ok), div_by<kB>(f[2], s, y, ok),
                  div_by<kB>(f[3], s, y, ok));
}

template <int QK>
__device__ __forceinline__ uint2 quant8(const float* f, float s, float y, bool ok, bool bounded) {
  uint2 o;
  if (bounded) {
    o.x = quant4<QK, true>(f, s, y, ok);
    o.y = quant4<QK, true>(f + 4, s, y, ok);
  } else {
    o.x = quant4<QK, false>(f, s, y, ok);
    o.y = quant4<QK, false>(f + 4, s, y, ok);
  }
  return o;
}

template <int QK>
__device__ __forceinline__ uint4 quant16(const float* f, float s, float y, bool ok, bool bounded) {
  const uint2 a = quant8<QK>(f, s, y, ok, bounded), b = quant8<QK>(f + 8, s, y, ok, bounded);
  return make_uint4(a.x, a.y, b.x, b.y);
}

template <int QK>
__device__ __forceinline__ uint8_t quant1(float x, float s, float y, bool ok, bool bounded) {
  return enc1<QK>(bounded ? div_by<true>(x, s, y, ok) : div_by<false>(x, s, y, ok));
}

template <int QK>
__device__ __forceinline__ float scale_from_amax(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, QK == 0 ? 448.f : 127.f) : 1.f;
}

}  // namespace
}  // namespace w8a8
