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

__device__ __forceinline__ uint32_t int8x1(float a) {
  int i;
  asm("cvt.rni.s32.f32 %0, %1;" : "=r"(i) : "f"(a));  // RNE; NaN -> 0; saturates to int32
  i = max(-128, min(127, i));
  return static_cast<uint32_t>(i) & 0xFFu;
}

template <int QK>
__device__ __forceinline__ uint32_t enc4(float a, float b, float c, float d) {
  if (QK == 0) return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
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
// one ulp of x/s, so the remainder x - s*q0 is exact in one FMA and
// RN(q0 + remainder*y) is the correctly rounded quotient RN(x/s)
// (Markstein's correction step for IEEE division with a correctly rounded
// reciprocal).  Preconditions: s and y are normal finite floats (checked per
// thread; otherwise the plain IEEE division is used) and no intermediate
// overflows -- when x*y overflows, q0 = +-inf already gives the code of the
// exact quotient (saturation), and the NaN the correction step would make is
// replaced by q0.  A zero remainder means q0 is exact; it is returned as is
// (q0 + 0 would turn -0 into +0).  Quotients in the fp32 subnormal range all
// encode to a signed zero, whatever their last bits.
__device__ __forceinline__ bool recip_ok(float s, float* y) {
  const float r = __fdiv_rn(1.0f, s);
  *y = r;
  const uint32_t es = (__float_as_uint(s) >> 23) & 0xFFu, er = (__float_as_uint(r) >> 23) & 0xFFu;
  return es != 0u && es != 0xFFu && er != 0u && er != 0xFFu;
}

__device__ __forceinline__ float div_by(float x, float s, float y, bool ok) {
  if (!ok) return __fdiv_rn(x, s);
  const float q0 = __fmul_rn(x, y);
  const float rem = __fmaf_rn(-q0, s, x);
  const float q1 = __fmaf_rn(rem, y, q0);
  // rem == 0: q0 is the exact quotient (and keeps the sign of a zero, which
  // q0 + 0 would lose for x = -0)
  return (rem == 0.0f || q1 != q1) ? q0 : q1;
}

template <int QK>
__device__ __forceinline__ float scale_from_amax(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, QK == 0 ? 448.f : 127.f) : 1.f;
}

}  // namespace
}  // namespace w8a8
