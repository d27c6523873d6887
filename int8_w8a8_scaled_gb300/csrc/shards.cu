// shards.cu -- merged-layer helpers (sm_103a).
//
// A merged QKV or gate-up weight is stored [N, K] as consecutive row shards
// that may carry their own scales.  "[Kernel] Support Fp8 Checkpoints
// (Dynamic + Static)" lists two ways to run it as one GEMM:
//  - per-shard scales in the fused epilogue (the PR's next step): a shard
//    scale is a per-output-channel scale that is constant over the shard, so
//    expand_shard_scales writes the [N] per-channel vector once and the
//    ordinary per-channel scaled_mm does the rest;
//  - requantise every shard to the largest shard scale (review discussion):
//    q' = encode(decode(q) * (s_i / s_max)), one shared per-tensor scale.
#include <cuda_fp8.h>

#include "internal.h"

namespace w8a8 {

namespace {

__device__ __forceinline__ int shard_of(long long row, const ShardTable& t) {
  int i = 0;
  while (i + 1 < t.n && row >= t.end[i]) ++i;
  return i;
}

__device__ __forceinline__ float max_scale(const float* s, int n) {
  float m = __ldg(s);
  for (int i = 1; i < n; ++i) m = fmaxf(m, __ldg(s + i));
  return m;
}

__global__ void expand_shard_scales_kernel(const float* __restrict__ shard_scales, ShardTable t,
                                           float* __restrict__ out) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long total = t.end[t.n - 1];
  for (long long r = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; r < total;
       r += static_cast<long long>(gridDim.x) * blockDim.x)
    out[r] = __ldg(shard_scales + shard_of(r, t));
}

template <int QK>
__device__ __forceinline__ float dec(uint8_t c) {
  if (QK == 0) {
    __nv_fp8_e4m3 v;
    v.__x = c;
    return static_cast<float>(v);
  }
  return static_cast<float>(static_cast<int8_t>(c));
}

template <int QK>
__device__ __forceinline__ uint8_t enc(float v) {
  if (QK == 0) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
    return (v != v) ? static_cast<uint8_t>(0x7F) : static_cast<uint8_t>(r & 0xFF);
  }
  int i;
  asm("cvt.rni.s32.f32 %0, %1;" : "=r"(i) : "f"(v));
  return static_cast<uint8_t>(max(-128, min(127, i)));
}

// One CTA per row; ratio = s_i / s_max (IEEE division), v = decode * ratio.
template <int QK>
__global__ void requant_shards_kernel(const uint8_t* __restrict__ q, long long cols, long long ld,
                                      const float* __restrict__ shard_scales, ShardTable t,
                                      uint8_t* __restrict__ out, long long ld_out, float* __restrict__ scale_out) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long row = blockIdx.x;
  const float smax = max_scale(shard_scales, t.n);
  if (row == 0 && threadIdx.x == 0) *scale_out = smax;
  const float ratio = __fdiv_rn(__ldg(shard_scales + shard_of(row, t)), smax);
  const uint8_t* src = q + row * ld;
  uint8_t* dst = out + row * ld_out;
  for (long long j = threadIdx.x; j < cols; j += blockDim.x) dst[j] = enc<QK>(dec<QK>(src[j]) * ratio);
}

}  // namespace

cudaError_t launch_expand_shard_scales(const float* shard_scales, const ShardTable& t, float* out,
                                       cudaStream_t stream) {
  const long long total = t.end[t.n - 1];
  int blocks = static_cast<int>(min(1024LL, (total + 255) / 256));
  expand_shard_scales_kernel<<<max(blocks, 1), 256, 0, stream>>>(shard_scales, t, out);
  return cudaGetLastError();
}

cudaError_t launch_requant_shards(const void* q, int q_kind, long long cols, long long ld,
                                  const float* shard_scales, const ShardTable& t, void* out, long long ld_out,
                                  float* scale_out, cudaStream_t stream) {
  const long long rows = t.end[t.n - 1];
  const dim3 grid(static_cast<unsigned>(rows));
  if (q_kind == 0)
    requant_shards_kernel<0><<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(q), cols, ld, shard_scales, t,
                                                       static_cast<uint8_t*>(out), ld_out, scale_out);
  else
    requant_shards_kernel<1><<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(q), cols, ld, shard_scales, t,
                                                       static_cast<uint8_t*>(out), ld_out, scale_out);
  return cudaGetLastError();
}

}  // namespace w8a8
