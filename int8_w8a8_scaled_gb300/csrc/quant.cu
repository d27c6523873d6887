// quant.cu -- the scaled quantiser and dequantiser kernels (sm_103a).
//
// Semantics ("Enable scaled FP8 (e4m3fn) KV cache on ROCm (AMD GPU)", section
// "Scaling semantics"; "[Kernel] Support Fp8 Checkpoints (Dynamic + Static)",
// PR description): scale = absmax / 448 for e4m3 (absmax / 127 for int8),
// computed at run time (dynamic) or given (static), per tensor or per row
// (token); q = sat_round(x / scale); dequant = decode(q) * scale.
//
// Exactness rules (the codes must match a correctly rounded reference bit
// for bit): x / scale is the correctly rounded fp32 quotient -- computed with
// a reciprocal and an exact-remainder correction step (div_by), or __fdiv_rn
// where its preconditions fail; never a bare reciprocal multiply; e4m3 uses the hardware round-to-nearest-even satfinite
// conversion with NaN canonicalised to 0x7F; int8 rounds half to even and
// saturates; absmax uses fmaxf from 0 so NaN never wins.
//
// Kernels:
//  - quant_rows: one 256-thread CTA per row; the row is read once into
//    registers with 128-bit loads (up to 8 * 256 * VPT elements), reduced
//    to absmax with warp shuffles (dynamic per-row), then converted from the
//    registers and written with 64-bit stores.  Rows longer than the
//    register budget are re-read (they are still in L2).
//  - absmax_flat + quant_flat: dynamic per-tensor needs the absmax of the
//    whole tensor before any code is written, so it is two grid-stride
//    passes over a contiguous tensor (the absmax word is reduced with
//    atomicMax on the float's bit pattern, valid for non-negative floats).
//  - quant_flat alone: static per-tensor on a contiguous tensor.
//  - dequant_flat / dequant_rows: decode(q) * scale rounded to bf16/fp16.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "quant_math.cuh"
#include "sm103_ptx.cuh"

namespace w8a8 {

namespace {

constexpr int kRowThreads = 256;
constexpr long long kBulkRowMaxCols = 65536;  // 128 KB of 16-bit row in shared memory

// Programmatic dependent launch.  Every kernel here is launched with the
// programmatic-serialisation attribute.  It first lets the next kernel in
// the stream be scheduled (that kernel's own wait still holds it back until
// this one has finished and its memory is visible), then waits for the
// preceding kernel and its memory before touching global memory.  Letting
// the successor in early lets a matmul stream its weights while this kernel
// and the one before it finish.  A kernel is launched only after every CTA of
// its predecessor has been scheduled, and every wait is on an earlier kernel,
// so the chain cannot deadlock.  Both instructions are no-ops without the
// attribute.
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl_smem(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, cudaStream_t st, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

__device__ __forceinline__ float load_f(const uint16_t* p, int kind) {
  const uint16_t b = *p;
  return kind == 0 ? __bfloat162float(__ushort_as_bfloat16(b)) : __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide max over kRowThreads threads; result broadcast to all.
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = (l < kRowThreads / 32) ? red[l] : 0.f;
  r = warp_max(r);
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------- per-row quantiser

// Per-row quantiser for rows whose start and length are 16-byte multiples:
// one thread pulls the whole row into shared memory with a single bulk async
// copy (no chain of dependent loads, which matters when a decode step has one
// row per kernel), then all threads reduce absmax and convert from shared
// memory in short loops (small code: the kernel runs cold on few SMs).  One
// CTA per row: with several CTAs per SM at different phases, one CTA's copy
// is in flight while another converts.  (A persistent two-row ring per CTA
// measured 6 % slower at the prefill sizes.)
template <int XK, int QK>
__global__ void __launch_bounds__(kRowThreads)
    quant_row_bulk_kernel(const uint16_t* __restrict__ x, long long ld_x, long long cols,
                          uint8_t* __restrict__ q, long long ld_q, float* __restrict__ scale, int per_row,
                          int dynamic) {
  extern __shared__ __align__(16) uint4 row_s[];
  __shared__ uint64_t bar;
  __shared__ float red[kRowThreads / 32];
  const long long row = blockIdx.x;
  const uint32_t bytes = static_cast<uint32_t>(cols * 2);
  // Start the row's trip into L2 before waiting on the preceding kernel (a
  // prefetch only reads: whatever that kernel writes, the copy below reads
  // after the wait), then trigger / wait as every kernel here does.
  if (threadIdx.x == 0) bulk_prefetch_l2(x + row * ld_x, bytes);
  allow_dependents();
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(smem_addr(&bar), bytes);
    bulk_load(smem_addr(row_s), x + row * ld_x, bytes, smem_addr(&bar));
  }
  __syncthreads();
  // on a timeout (flagged in the device status) every thread leaves together,
  // before the block-wide reductions below, once the copy in flight has had a
  // second bounded wait to land
  if (!__syncthreads_and(mbar_wait(smem_addr(&bar), 0))) {
    if (threadIdx.x == 0) mbar_wait(smem_addr(&bar), 0);
    return;
  }
  const int nvec = static_cast<int>(cols / 8);
  float s;
  if (dynamic) {
    float amax = 0.f;
#pragma unroll 4
    for (int v = threadIdx.x; v < nvec; v += kRowThreads) {
      float f[8];
      unpack8<XK>(row_s[v], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
    amax = block_max(amax, red);
    s = scale_from_amax<QK>(amax);
    if (threadIdx.x == 0) scale[row] = s;
  } else {
    s = scale[per_row ? row : 0];
  }
  float y;
  const bool ok = recip_ok(s, &y);
  uint2* qr = reinterpret_cast<uint2*>(q + row * ld_q);
#pragma unroll 2
  for (int v = threadIdx.x; v < nvec; v += kRowThreads) {
    float f[8];
    unpack8<XK>(row_s[v], f);
    qr[v] = quant8<QK>(f, s, y, ok, dynamic);
  }
}

// VPT = 128-bit vectors cached per thread (0: vector path disabled, scalar).
template <int XK, int QK, int VPT>
__global__ void __launch_bounds__(kRowThreads)
    quant_rows_kernel(const uint16_t* __restrict__ x, long long ld_x, long long cols,
                      uint8_t* __restrict__ q, long long ld_q, float* __restrict__ scale,
                      int per_row, int dynamic) {
  allow_dependents();
  __shared__ float red[kRowThreads / 32];
  const long long row = blockIdx.x;
  const uint16_t* xr = x + row * ld_x;
  uint8_t* qr = q + row * ld_q;

  if (VPT > 0) {
    const long long nvec = cols / 8;
    uint4 cache[VPT > 0 ? VPT : 1];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const long long v = threadIdx.x + static_cast<long long>(i) * kRowThreads;
      if (v < nvec) {
        cache[i] = __ldcs(reinterpret_cast<const uint4*>(xr) + v);
        if (dynamic) {
          float f[8];
          unpack8<XK>(cache[i], f);
#pragma unroll
          for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
        }
      }
    }
    // vectors beyond the register cache, and the scalar tail
    for (long long v = threadIdx.x + static_cast<long long>(VPT) * kRowThreads; dynamic && v < nvec;
         v += kRowThreads) {
      float f[8];
      unpack8<XK>(__ldg(reinterpret_cast<const uint4*>(xr) + v), f);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
    for (long long j = nvec * 8 + threadIdx.x; dynamic && j < cols; j += kRowThreads)
      amax = fmaxf(amax, fabsf(cvt_in<XK>(xr[j])));

    float s;
    if (dynamic) {
      amax = block_max(amax, red);
      s = scale_from_amax<QK>(amax);
      if (threadIdx.x == 0) scale[row] = s;
    } else {
      s = scale[per_row ? row : 0];
    }
    float y;
    const bool ok = recip_ok(s, &y);

#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const long long v = threadIdx.x + static_cast<long long>(i) * kRowThreads;
      if (v < nvec) {
        float f[8];
        unpack8<XK>(cache[i], f);
        uint2 o;
        o = quant8<QK>(f, s, y, ok, dynamic);
        reinterpret_cast<uint2*>(qr)[v] = o;
      }
    }
    for (long long v = threadIdx.x + static_cast<long long>(VPT) * kRowThreads; v < nvec;
         v += kRowThreads) {
      float f[8];
      unpack8<XK>(__ldg(reinterpret_cast<const uint4*>(xr) + v), f);
      uint2 o;
      o = quant8<QK>(f, s, y, ok, dynamic);
      reinterpret_cast<uint2*>(qr)[v] = o;
    }
    for (long long j = nvec * 8 + threadIdx.x; j < cols; j += kRowThreads)
      qr[j] = quant1<QK>(cvt_in<XK>(xr[j]), s, y, ok, dynamic);
  } else {
    // scalar path for unaligned layouts
    float s;
    if (dynamic) {
      float amax = 0.f;
      for (long long j = threadIdx.x; j < cols; j += kRowThreads)
        amax = fmaxf(amax, fabsf(cvt_in<XK>(xr[j])));
      amax = block_max(amax, red);
      s = scale_from_amax<QK>(amax);
      if (threadIdx.x == 0) scale[row] = s;
    } else {
      s = scale[per_row ? row : 0];
    }
    float y;
    const bool ok = recip_ok(s, &y);
    for (long long j = threadIdx.x; j < cols; j += kRowThreads)
      qr[j] = quant1<QK>(cvt_in<XK>(xr[j]), s, y, ok, dynamic);
  }
}

// ---------------------------------------------------------------- per-tensor (flat)

template <int XK>
__global__ void __launch_bounds__(256)
    absmax_flat_kernel(const uint16_t* __restrict__ x, long long n, unsigned* __restrict__ word) {
  allow_dependents();
  __shared__ float red[8];
  float amax = 0.f;
  const long long nvec = n / 8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  // 4 independent 128-bit loads in flight per thread
  for (; v + 3 * stride < nvec; v += 4 * stride) {
    uint4 w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) w[u] = __ldg(reinterpret_cast<const uint4*>(x) + v + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float f[8];
      unpack8<XK>(w[u], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
  }
  for (; v < nvec; v += stride) {
    float f[8];
    unpack8<XK>(__ldg(reinterpret_cast<const uint4*>(x) + v), f);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
  }
  for (long long j = nvec * 8 + blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; j < n;
       j += stride)
    amax = fmaxf(amax, fabsf(cvt_in<XK>(x[j])));
  amax = warp_max(amax);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) red[w] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float r = (l < 8) ? red[l] : 0.f;
    r = warp_max(r);
    // non-negative, non-NaN floats order like their bit patterns
    if (l == 0 && r > 0.f) atomicMax(word, __float_as_uint(r));
  }
}

// Per-row absmax of a strided tensor, reduced into one word (per-tensor
// dynamic on a non-contiguous view).
template <int XK>
__global__ void __launch_bounds__(kRowThreads)
    absmax_rows_kernel(const uint16_t* __restrict__ x, long long ld_x, long long cols,
                       unsigned* __restrict__ word) {
  allow_dependents();
  __shared__ float red[kRowThreads / 32];
  const uint16_t* xr = x + static_cast<long long>(blockIdx.x) * ld_x;
  float amax = 0.f;
  for (long long j = threadIdx.x; j < cols; j += kRowThreads) amax = fmaxf(amax, fabsf(cvt_in<XK>(xr[j])));
  amax = block_max(amax, red);
  if (threadIdx.x == 0 && amax > 0.f) atomicMax(word, __float_as_uint(amax));
}

// q = enc(x / s) over a contiguous tensor, s from the absmax word (dynamic)
// or from scale[0] (static).  16 elements per thread per step.
template <int XK, int QK>
__global__ void __launch_bounds__(256, 4)
    quant_flat_kernel(const uint16_t* __restrict__ x, long long n, uint8_t* __restrict__ q,
                      float* __restrict__ scale, const unsigned* __restrict__ word, int dynamic) {
  allow_dependents();
  float s;
  if (dynamic) {
    s = scale_from_amax<QK>(__uint_as_float(*word));
    if (blockIdx.x == 0 && threadIdx.x == 0) scale[0] = s;
  } else {
    s = __ldg(scale);
  }
  float y;
  const bool ok = recip_ok(s, &y);
  const long long n16 = n / 16;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // The grid walks the tensor back to front: after the absmax pass (front to
  // back) the tail it read last is still in L2, so a tensor up to about the
  // L2 size is read from DRAM once.  rv(v) is the 16-element group visited
  // at virtual position v.
  auto rv = [n16](long long v) { return n16 - 1 - v; };
  long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  for (; v + stride < n16; v += 2 * stride) {
    uint4 w[4];
    w[0] = __ldcs(reinterpret_cast<const uint4*>(x) + 2 * rv(v));
    w[1] = __ldcs(reinterpret_cast<const uint4*>(x) + 2 * rv(v) + 1);
    w[2] = __ldcs(reinterpret_cast<const uint4*>(x) + 2 * rv(v + stride));
    w[3] = __ldcs(reinterpret_cast<const uint4*>(x) + 2 * rv(v + stride) + 1);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float f[16];
      unpack8<XK>(w[2 * u], *reinterpret_cast<float(*)[8]>(f));
      unpack8<XK>(w[2 * u + 1], *reinterpret_cast<float(*)[8]>(f + 8));
      uint4 o;
      o = quant16<QK>(f, s, y, ok, dynamic);
      __stcs(reinterpret_cast<uint4*>(q) + rv(u == 0 ? v : v + stride), o);
    }
  }
  for (; v < n16; v += stride) {
    float f[16];
    unpack8<XK>(__ldcs(reinterpret_cast<const uint4*>(x) + 2 * rv(v)), *reinterpret_cast<float(*)[8]>(f));
    unpack8<XK>(__ldcs(reinterpret_cast<const uint4*>(x) + 2 * rv(v) + 1), *reinterpret_cast<float(*)[8]>(f + 8));
    uint4 o;
    o = quant16<QK>(f, s, y, ok, dynamic);
    __stcs(reinterpret_cast<uint4*>(q) + rv(v), o);
  }
  for (long long j = n16 * 16 + blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; j < n;
       j += stride)
    q[j] = quant1<QK>(cvt_in<XK>(x[j]), s, y, ok, dynamic);
}

// Per-row quantiser driven by a per-tensor scale from the absmax word (the
// second pass of dynamic per-tensor on a strided view).
template <int XK, int QK>
__global__ void __launch_bounds__(kRowThreads)
    quant_rows_from_word_kernel(const uint16_t* __restrict__ x, long long ld_x, long long cols,
                                uint8_t* __restrict__ q, long long ld_q, float* __restrict__ scale,
                                const unsigned* __restrict__ word) {
  allow_dependents();
  const float s = scale_from_amax<QK>(__uint_as_float(*word));
  if (blockIdx.x == 0 && threadIdx.x == 0) scale[0] = s;
  float y;
  const bool ok = recip_ok(s, &y);
  const uint16_t* xr = x + static_cast<long long>(blockIdx.x) * ld_x;
  uint8_t* qr = q + static_cast<long long>(blockIdx.x) * ld_q;
  for (long long j = threadIdx.x; j < cols; j += kRowThreads) qr[j] = quant1<QK>(cvt_in<XK>(xr[j]), s, y, ok, true);
}

// ---------------------------------------------------------------- dequantiser

template <int QK>
__device__ __forceinline__ float dec1(uint8_t c) {
  if (QK == 0) {
    __nv_fp8_e4m3 v;
    v.__x = c;
    return static_cast<float>(v);  // exact
  }
  return static_cast<float>(static_cast<int8_t>(c));
}

template <int YK>
__device__ __forceinline__ uint16_t out16(float y) {
  if (YK == 0) return __bfloat16_as_ushort(__float2bfloat16_rn(y));
  return __half_as_ushort(__float2half_rn(y));
}

// two outputs RN(a), RN(b) in one 32-bit word, a in the low half
template <int YK>
__device__ __forceinline__ uint32_t out16x2(float a, float b) {
  if (YK == 0) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 codes (one 16-byte word, first code in the low byte) -> decode(q) * s
// rounded to 16 bits, two per output word.  e4m3 decodes four codes per
// conversion (exactly, through f16); the products and roundings are those
// of dec1 and out16 one by one.
template <int QK, int YK>
__device__ __forceinline__ void dequant16(const uint4& w, float s, uint32_t (&o)[8]) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
  if (QK == 0) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t h01, h23;
      e4m3x4_to_f16x2x2(words[j], h01, h23);
      const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
      const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
      o[2 * j] = out16x2<YK>(f01.x * s, f01.y * s);
      o[2 * j + 1] = out16x2<YK>(f23.x * s, f23.y * s);
    }
  } else {
    const uint8_t* bb = reinterpret_cast<const uint8_t*>(&w);
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = out16x2<YK>(dec1<QK>(bb[2 * j]) * s, dec1<QK>(bb[2 * j + 1]) * s);
  }
}

template <int QK, int YK>
__global__ void __launch_bounds__(256)
    dequant_flat_kernel(const uint8_t* __restrict__ q, long long n, const float* __restrict__ scale,
                        uint16_t* __restrict__ y) {
  allow_dependents();
  const float s = __ldg(scale);
  const long long n16 = n / 16;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; v < n16; v += stride) {
    const uint4 w = __ldcs(reinterpret_cast<const uint4*>(q) + v);
    uint32_t o[8];
    dequant16<QK, YK>(w, s, o);
    uint4* d = reinterpret_cast<uint4*>(y) + 2 * v;
    __stcs(d, make_uint4(o[0], o[1], o[2], o[3]));
    __stcs(d + 1, make_uint4(o[4], o[5], o[6], o[7]));
  }
  for (long long j = n16 * 16 + blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; j < n;
       j += stride)
    y[j] = out16<YK>(dec1<QK>(q[j]) * s);
}

// Streaming per-tensor quantiser passes for a contiguous tensor (n % 16 == 0,
// 16-byte aligned): chunks of kQzChunk elements pulled into shared memory by
// bulk copies, one thread issuing, kQzStages chunks in flight per CTA (a ring
// of that depth), all threads working from shared memory.  With several
// CTAs per SM that keeps ~100 KB per SM on its way from HBM.
constexpr int kQzChunk = 4096;  // elements per chunk: 8 KB of bf16 / fp16
#ifndef W8A8_QZ_ABS_STAGES
#define W8A8_QZ_ABS_STAGES 4
#endif
#ifndef W8A8_QZ_CVT_STAGES
#define W8A8_QZ_CVT_STAGES 2
#endif
// ring depths: the absmax pass only streams, so it keeps more chunks in
// flight; the convert pass is bound by its per-element arithmetic and keeps
// a shallow ring so that more CTAs (warps) fit an SM
constexpr int kQzAbsStages = W8A8_QZ_ABS_STAGES;
constexpr int kQzCvtStages = W8A8_QZ_CVT_STAGES;

// Chunk ring shared by the two passes: chunk c of this CTA (its i-th) goes
// to slot i % kQzStages; the loads run kQzStages - 1 chunks ahead.
template <int kQzStages>
struct QzRing {
  long long n, nchunks, step;
  bool reverse;  // visit the chunks back to front
  __device__ long long phys(long long c) const { return reverse ? nchunks - 1 - c : c; }
  __device__ uint32_t elems(long long c) const {
    const long long rem = n - phys(c) * kQzChunk;
    return static_cast<uint32_t>(rem < kQzChunk ? rem : kQzChunk);
  }
  // thread 0: issue the load of this CTA's i-th chunk, if it exists
  __device__ bool issue(int i, const uint16_t* x, uint16_t (*buf)[kQzChunk], uint64_t* bar) const {
    const long long c = blockIdx.x + static_cast<long long>(i) * step;
    if (c >= nchunks) return false;
    const int slot = i % kQzStages;
    mbar_arrive_expect_tx(smem_addr(&bar[slot]), elems(c) * 2);
    // the absmax pass keeps what it reads in L2 for the convert pass, which
    // walks the tensor back to front and reads it for the last time
    bulk_load_hint(smem_addr(buf[slot]), x + phys(c) * kQzChunk, elems(c) * 2, smem_addr(&bar[slot]),
                   reverse ? policy_evict_first() : policy_evict_last());
    return true;
  }
  // thread 0, after a failed wait at chunk i: let the loads still in flight
  // (chunks i .. i + kQzStages - 2 that were issued) land, bounded, before
  // the CTA exits and its shared memory is released
  __device__ void drain(int i, uint64_t* bar) const {
    for (int j = i; j < i + kQzStages - 1; ++j) {
      if (blockIdx.x + static_cast<long long>(j) * step >= nchunks) break;
      mbar_wait(smem_addr(&bar[j % kQzStages]), (j / kQzStages) & 1);
    }
  }
};

// Pass 1: absmax of the whole tensor (front to back) into the word.
template <int XK>
__global__ void __launch_bounds__(256)
    absmax_bulk_kernel(const uint16_t* __restrict__ x, long long n, unsigned* __restrict__ word) {
  __shared__ __align__(128) uint16_t in_buf[kQzAbsStages][kQzChunk];
  __shared__ uint64_t bar[kQzAbsStages];
  __shared__ float red[8];
  allow_dependents();
  QzRing<kQzAbsStages> ring{n, (n + kQzChunk - 1) / kQzChunk, gridDim.x, false};
  if (threadIdx.x == 0) {
    for (int j = 0; j < kQzAbsStages; ++j) mbar_init(smem_addr(&bar[j]), 1);
    fence_barrier_init();
    for (int j = 0; j < kQzAbsStages - 1; ++j) ring.issue(j, x, in_buf, bar);
  }
  __syncthreads();
  float amax = 0.f;
  int i = 0;
  bool failed = false;
  for (long long c = blockIdx.x; c < ring.nchunks; c += ring.step, ++i) {
    // the slot of chunk i + S - 1 was released by the barrier ending chunk i - 1
    if (threadIdx.x == 0) ring.issue(i + kQzAbsStages - 1, x, in_buf, bar);
    const int slot = i % kQzAbsStages;
    const bool got = mbar_wait(smem_addr(&bar[slot]), (i / kQzAbsStages) & 1);
    if (!__syncthreads_and(got)) {
      failed = true;
      break;
    }
    const int e0 = threadIdx.x * 16;
    if (e0 < static_cast<int>(ring.elems(c))) {
      const uint4* p = reinterpret_cast<const uint4*>(in_buf[slot] + e0);
      float f[8];
      unpack8<XK>(p[0], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
      unpack8<XK>(p[1], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
    __syncthreads();  // the slot is refilled S - 1 chunks on
  }
  if (threadIdx.x == 0 && failed) ring.drain(i, bar);
  amax = warp_max(amax);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) red[w] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float r = (l < 8) ? red[l] : 0.f;
    r = warp_max(r);
    // non-negative, non-NaN floats order like their bit patterns
    if (l == 0 && r > 0.f) atomicMax(word, __float_as_uint(r));
  }
}

// Pass 2: codes of the whole tensor with the scale from the word (dynamic)
// or scale[0] (static).  The chunks are visited back to front, so a tensor
// about the size of L2 finds the tail pass 1 read last still there.  Codes
// leave through two output buffers, each written back by one bulk store.
template <int XK, int QK>
__global__ void __launch_bounds__(256)
    quant_bulk_kernel(const uint16_t* __restrict__ x, long long n, uint8_t* __restrict__ q,
                      float* __restrict__ scale, const unsigned* __restrict__ word, int dynamic) {
  __shared__ __align__(128) uint16_t in_buf[kQzCvtStages][kQzChunk];
  __shared__ __align__(128) uint8_t out_buf[2][kQzChunk];
  __shared__ uint64_t bar[kQzCvtStages];
  allow_dependents();
  float s;
  if (dynamic) {
    s = scale_from_amax<QK>(__uint_as_float(*word));
    if (blockIdx.x == 0 && threadIdx.x == 0) scale[0] = s;
  } else {
    s = __ldg(scale);
  }
  float y;
  const bool ok = recip_ok(s, &y);
  QzRing<kQzCvtStages> ring{n, (n + kQzChunk - 1) / kQzChunk, gridDim.x, true};
  if (threadIdx.x == 0) {
    for (int j = 0; j < kQzCvtStages; ++j) mbar_init(smem_addr(&bar[j]), 1);
    fence_barrier_init();
    for (int j = 0; j < kQzCvtStages - 1; ++j) ring.issue(j, x, in_buf, bar);
  }
  __syncthreads();
  int i = 0;
  bool failed = false;
  for (long long c = blockIdx.x; c < ring.nchunks; c += ring.step, ++i) {
    const int ob = i & 1;
    if (threadIdx.x == 0) {
      ring.issue(i + kQzCvtStages - 1, x, in_buf, bar);
      bulk_wait_read<1>();  // the store two chunks back has read out_buf[ob]
    }
    const int slot = i % kQzCvtStages;
    const bool got = mbar_wait(smem_addr(&bar[slot]), (i / kQzCvtStages) & 1);
    if (!__syncthreads_and(got)) {
      failed = true;
      break;
    }
    const uint4* p = reinterpret_cast<const uint4*>(in_buf[slot] + threadIdx.x * 16);
    float f[16];
    unpack8<XK>(p[0], *reinterpret_cast<float(*)[8]>(f));
    unpack8<XK>(p[1], *reinterpret_cast<float(*)[8]>(f + 8));
    uint4 o;
    o = quant16<QK>(f, s, y, ok, dynamic);
    reinterpret_cast<uint4*>(out_buf[ob])[threadIdx.x] = o;
    fence_proxy_async_shared();
    __syncthreads();
    if (threadIdx.x == 0) {
      bulk_store(q + ring.phys(c) * kQzChunk, smem_addr(out_buf[ob]), ring.elems(c));
      bulk_commit();
    }
  }
  if (threadIdx.x == 0) {
    if (failed) ring.drain(i, bar);
    bulk_wait_all();
  }
}

// Streaming dequantiser for a contiguous tensor (n % 16 == 0, 16-byte
// aligned): each CTA walks chunks of kDqChunk codes with a two-deep ring.
// One thread pulls the next chunk into shared memory with a bulk copy while
// all threads convert the current one into a shared output buffer, which one
// bulk store writes back.  No per-thread global loads or stores: the bulk
// engine keeps whole chunks in flight in both directions.
constexpr int kDqChunk = 4096;  // codes per chunk: 4 KB in, 8 KB out

template <int QK, int YK>
__global__ void __launch_bounds__(256)
    dequant_bulk_kernel(const uint8_t* __restrict__ q, long long n, const float* __restrict__ scale,
                        uint16_t* __restrict__ y) {
  __shared__ __align__(128) uint8_t in_buf[2][kDqChunk];
  __shared__ __align__(128) uint16_t out_buf[2][kDqChunk];
  __shared__ uint64_t bar[2];
  allow_dependents();
  const float s = __ldg(scale);
  const long long nchunks = (n + kDqChunk - 1) / kDqChunk;
  const long long step = gridDim.x;
  auto chunk_bytes = [&](long long c) {
    const long long rem = n - c * kDqChunk;
    return static_cast<uint32_t>(rem < kDqChunk ? rem : kDqChunk);
  };
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar[0]), 1);
    mbar_init(smem_addr(&bar[1]), 1);
    fence_barrier_init();
    const long long c0 = blockIdx.x;
    if (c0 < nchunks) {
      mbar_arrive_expect_tx(smem_addr(&bar[0]), chunk_bytes(c0));
      // codes are read once: behind everything else in L2
      bulk_load_hint(smem_addr(in_buf[0]), q + c0 * kDqChunk, chunk_bytes(c0), smem_addr(&bar[0]),
                     policy_evict_first());
    }
  }
  __syncthreads();
  int i = 0;
  bool failed = false, next_issued = false;
  for (long long c = blockIdx.x; c < nchunks; c += step, ++i) {
    const int b = i & 1;
    next_issued = false;
    if (threadIdx.x == 0) {
      const long long next = c + step;
      next_issued = next < nchunks;
      if (next_issued) {  // in_buf[b ^ 1] was consumed last iteration
        mbar_arrive_expect_tx(smem_addr(&bar[b ^ 1]), chunk_bytes(next));
        bulk_load_hint(smem_addr(in_buf[b ^ 1]), q + next * kDqChunk, chunk_bytes(next), smem_addr(&bar[b ^ 1]),
                       policy_evict_first());
      }
      bulk_wait_read<1>();  // the store two chunks back has read out_buf[b]
    }
    // every thread waits for the chunk; on a timeout (flagged in the device
    // status) all of them leave together
    const bool got = mbar_wait(smem_addr(&bar[b]), (i >> 1) & 1);
    if (!__syncthreads_and(got)) {
      failed = true;
      break;
    }
    const uint4 w = reinterpret_cast<const uint4*>(in_buf[b])[threadIdx.x];
    uint32_t o[8];
    dequant16<QK, YK>(w, s, o);
    uint4* d = reinterpret_cast<uint4*>(out_buf[b]) + 2 * threadIdx.x;
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
    fence_proxy_async_shared();
    __syncthreads();
    if (threadIdx.x == 0) {
      bulk_store(y + c * kDqChunk, smem_addr(out_buf[b]), chunk_bytes(c) * 2);
      bulk_commit();
    }
  }
  if (threadIdx.x == 0) {
    if (failed) {
      // let this CTA's copies in flight land (bounded) before it exits
      mbar_wait(smem_addr(&bar[i & 1]), (i >> 1) & 1);
      if (next_issued) mbar_wait(smem_addr(&bar[(i & 1) ^ 1]), ((i + 1) >> 1) & 1);
    }
    bulk_wait_all();
  }
}

template <int QK, int YK>
__global__ void __launch_bounds__(kRowThreads)
    dequant_rows_kernel(const uint8_t* __restrict__ q, long long ld_q, long long cols,
                        const float* __restrict__ scale, int per_row, uint16_t* __restrict__ y,
                        long long ld_y) {
  allow_dependents();
  const long long row = blockIdx.x;
  const float s = __ldg(scale + (per_row ? row : 0));
  const uint8_t* qr = q + row * ld_q;
  uint16_t* yr = y + row * ld_y;
  for (long long j = threadIdx.x; j < cols; j += kRowThreads) yr[j] = out16<YK>(dec1<QK>(qr[j]) * s);
}

// ---------------------------------------------------------------- launch helpers

// Shared memory of an SM (sm_100 family).
constexpr long long kSmSmem = 228 * 1024;

template <int XK, int QK>
cudaError_t launch_rows(const QuantArgs& a, cudaStream_t st) {
  const uint16_t* x = static_cast<const uint16_t*>(a.x);
  uint8_t* q = static_cast<uint8_t*>(a.q);
  const long long nvec = a.cols / 8;
  const long long per_thread = (nvec + kRowThreads - 1) / kRowThreads;
  const dim3 grid(static_cast<unsigned>(a.rows)), block(kRowThreads);
  if (a.vec && a.cols % 8 == 0 && a.ld_x % 8 == 0 && a.cols <= kBulkRowMaxCols) {
    const size_t smem = static_cast<size_t>(a.cols) * 2;
    auto kern = quant_row_bulk_kernel<XK, QK>;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    return launch_pdl_smem(kern, grid, block, smem, st, x, a.ld_x, a.cols, q, a.ld_q, a.scale, a.per_row, a.dynamic);
  }
#define W8A8_ROWS(V) \
  launch_pdl(quant_rows_kernel<XK, QK, V>, grid, block, st, x, a.ld_x, a.cols, q, a.ld_q, a.scale, a.per_row, a.dynamic)
  if (!a.vec) return W8A8_ROWS(0);
  if (per_thread <= 1) return W8A8_ROWS(1);
  if (per_thread <= 2) return W8A8_ROWS(2);
  if (per_thread <= 4) return W8A8_ROWS(4);
  if (per_thread <= 8) return W8A8_ROWS(8);
  return W8A8_ROWS(16);
#undef W8A8_ROWS
}

int flat_blocks(long long work_items, int num_sms) {
  long long b = (work_items + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

template <int XK, int QK>
cudaError_t launch_quant_t(const QuantArgs& a, int num_sms, cudaStream_t st) {
  const uint16_t* x = static_cast<const uint16_t*>(a.x);
  uint8_t* q = static_cast<uint8_t*>(a.q);
  const bool contiguous = (a.ld_x == a.cols && a.ld_q == a.cols) || a.rows == 1;
  const dim3 b256(256);
  if (a.per_row) return launch_rows<XK, QK>(a, st);
  // CTAs per SM: as many as the pass's chunk ring in shared memory allows
  // (<= 8: 2048 threads), all resident at once
  auto bulk_grid = [&](long long n, long long ring_bytes) {
    const long long chunks = (n + kQzChunk - 1) / kQzChunk;
    long long per_sm = kSmSmem / (ring_bytes + 1024);
    per_sm = per_sm < 1 ? 1 : (per_sm > 8 ? 8 : per_sm);
    const long long cap = static_cast<long long>(num_sms) * per_sm;
    return dim3(static_cast<unsigned>(chunks < cap ? chunks : cap));
  };
  const long long abs_ring = static_cast<long long>(kQzAbsStages) * kQzChunk * 2;
  const long long cvt_ring = static_cast<long long>(kQzCvtStages) * kQzChunk * 2 + 2 * kQzChunk;
  if (!a.dynamic) {
    if (contiguous && a.vec) {
      const long long n = a.rows * a.cols;
      if (n % 16 == 0)
        return launch_pdl(quant_bulk_kernel<XK, QK>, bulk_grid(n, cvt_ring), b256, st, x, n, q, a.scale,
                          static_cast<const unsigned*>(nullptr), 0);
      return launch_pdl(quant_flat_kernel<XK, QK>, dim3(flat_blocks(n / 16, num_sms)), b256, st, x, n, q, a.scale,
                        static_cast<const unsigned*>(nullptr), 0);
    }
    return launch_rows<XK, QK>(a, st);
  }
  // dynamic per-tensor: absmax pass, then quantise pass
  cudaError_t e = cudaMemsetAsync(a.amax_word, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  if (contiguous && a.vec && (a.rows * a.cols) % 16 == 0) {
    const long long n = a.rows * a.cols;
    e = launch_pdl(absmax_bulk_kernel<XK>, bulk_grid(n, abs_ring), b256, st, x, n, a.amax_word);
    if (e != cudaSuccess) return e;
    return launch_pdl(quant_bulk_kernel<XK, QK>, bulk_grid(n, cvt_ring), b256, st, x, n, q, a.scale,
                      static_cast<const unsigned*>(a.amax_word), 1);
  }
  if (contiguous && a.vec) {
    const long long n = a.rows * a.cols;
    e = launch_pdl(absmax_flat_kernel<XK>, dim3(flat_blocks(n / 8, num_sms)), b256, st, x, n, a.amax_word);
    if (e != cudaSuccess) return e;
    return launch_pdl(quant_flat_kernel<XK, QK>, dim3(flat_blocks(n / 16, num_sms)), b256, st, x, n, q, a.scale,
                      static_cast<const unsigned*>(a.amax_word), 1);
  }
  const dim3 grid(static_cast<unsigned>(a.rows)), block(kRowThreads);
  e = launch_pdl(absmax_rows_kernel<XK>, grid, block, st, x, a.ld_x, a.cols, a.amax_word);
  if (e != cudaSuccess) return e;
  return launch_pdl(quant_rows_from_word_kernel<XK, QK>, grid, block, st, x, a.ld_x, a.cols, q, a.ld_q, a.scale,
                    static_cast<const unsigned*>(a.amax_word));
}

template <int QK, int YK>
cudaError_t launch_dequant_t(const DequantArgs& a, int num_sms, cudaStream_t st) {
  const uint8_t* q = static_cast<const uint8_t*>(a.q);
  uint16_t* y = static_cast<uint16_t*>(a.y);
  const bool contiguous = (a.ld_q == a.cols && a.ld_y == a.cols) || a.rows == 1;
  if (!a.per_row && contiguous && a.vec) {
    const long long n = a.rows * a.cols;
    if (n % 16 == 0) {
      const long long chunks = (n + kDqChunk - 1) / kDqChunk;
      const long long cap = static_cast<long long>(num_sms) * 8;
      return launch_pdl(dequant_bulk_kernel<QK, YK>, dim3(static_cast<unsigned>(chunks < cap ? chunks : cap)),
                        dim3(256), st, q, n, a.scale, y);
    }
    return launch_pdl(dequant_flat_kernel<QK, YK>, dim3(flat_blocks(n / 16, num_sms)), dim3(256), st, q, n, a.scale, y);
  }
  return launch_pdl(dequant_rows_kernel<QK, YK>, dim3(static_cast<unsigned>(a.rows)), dim3(kRowThreads), st, q, a.ld_q,
                    a.cols, a.scale, a.per_row, y, a.ld_y);
}

}  // namespace

cudaError_t read_clear_quant_status(int* flags) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
  *flags = v;
  return e;
}

cudaError_t launch_quant(const QuantArgs& a, int num_sms, cudaStream_t st) {
  if (a.x_kind == 0)
    return a.q_kind == 0 ? launch_quant_t<0, 0>(a, num_sms, st) : launch_quant_t<0, 1>(a, num_sms, st);
  return a.q_kind == 0 ? launch_quant_t<1, 0>(a, num_sms, st) : launch_quant_t<1, 1>(a, num_sms, st);
}

cudaError_t launch_dequant(const DequantArgs& a, int num_sms, cudaStream_t st) {
  if (a.q_kind == 0)
    return a.y_kind == 0 ? launch_dequant_t<0, 0>(a, num_sms, st) : launch_dequant_t<0, 1>(a, num_sms, st);
  return a.y_kind == 0 ? launch_dequant_t<1, 0>(a, num_sms, st) : launch_dequant_t<1, 1>(a, num_sms, st);
}

}  // namespace w8a8
