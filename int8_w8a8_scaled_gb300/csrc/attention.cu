// attention.cu -- decode attention over an fp8 (e4m3) KV cache (sm_103a).
//
// "Enable scaled FP8 (e4m3fn) KV cache on ROCm (AMD GPU)": the K and V
// caches hold e4m3 codes with one per-tensor scaling factor each (the
// kv_scale of the paged attention kernel), and dequantisation is
// decode(code) * scaling_factor ("Scaling semantics").  The attention kernel
// reads the codes and dequantises them as it goes, so the cache costs one
// byte per element of HBM traffic.
//
// One query token per sequence (decode); the G = Hq / Hkv query heads of a
// KV head share every K and V read (grouped-query attention).  Flash
// decoding: a sequence's tokens are cut into chunks, and one CTA per
// (chunk, KV head, sequence) computes for each of its G heads the chunk's
// score maximum m (log2 domain), l = sum 2^(s - m) and the unnormalised
// o = sum 2^(s - m) * decode(v); a second kernel combines the chunks:
// out = (sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c) * v_scale.
//
// Work split inside a CTA (128 threads): 8 lanes per token, 16 head dims
// (16 code bytes) per lane, so a warp's load covers four whole 128-byte
// cache rows.  Scores: each lane multiplies its 16 dims by the G query rows
// (kept in registers) and the 8 lanes of a token add their partial sums
// with shuffles.  Output: each lane accumulates its 16 dims for the G heads
// over its tokens; lanes with the same dims then add up across tokens.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"

namespace w8a8 {

namespace {

constexpr int kHeadDim = 128;
constexpr int kAttnThreads = 128;
constexpr int kLanesPerToken = 8;                              // 16 dims per lane
constexpr int kTokPerPass = kAttnThreads / kLanesPerToken;    // 16 tokens per pass of the CTA
constexpr int kUnroll = 4;                                     // passes whose loads are in flight together
constexpr int kMaxChunk = 256;
constexpr int kPartStride = kHeadDim + 4;                      // o[128], m, l, 2 pad (floats)

// 16 e4m3 codes -> 16 floats (exact: e4m3 -> f16 -> f32 widen)
__device__ __forceinline__ void decode16(const uint4& w, float (&f)[16]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[i] >> 16), __NV_E4M3);
    const float2 a = __half22float2(__half2(lo));
    const float2 b = __half22float2(__half2(hi));
    f[4 * i + 0] = a.x;
    f[4 * i + 1] = a.y;
    f[4 * i + 2] = b.x;
    f[4 * i + 3] = b.y;
  }
}

__device__ __forceinline__ float load_q(const void* q, int q_fp16, size_t i) {
  if (q_fp16) return __half2float(static_cast<const __half*>(q)[i]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(q)[i]);
}

// Cache row (token slot) of token t of sequence b, or -1 if its block id is
// outside the cache (the token is then skipped).
__device__ __forceinline__ long long slot_of(const AttnParams& p, int b, int t) {
  if (!p.block_table) return static_cast<long long>(b) * p.max_seq_len + t;
  const int blk = __ldg(p.block_table + static_cast<size_t>(b) * p.max_blocks + t / p.block_size);
  if (blk < 0 || blk >= p.num_blocks) return -1;
  return static_cast<long long>(blk) * p.block_size + t % p.block_size;
}

__device__ __forceinline__ int seq_len_of(const AttnParams& p, int b) {
  const int len = __ldg(p.seq_lens + b);
  return len < 0 ? 0 : (len > p.max_seq_len ? p.max_seq_len : len);
}

// Up to 4 heads per KV head the kernel fits 96 registers without spilling,
// so 5 CTAs (20 warps) share an SM instead of 4; at 8 heads a cap spills.
template <int G>
__global__ void __launch_bounds__(kAttnThreads, G <= 4 ? 5 : 1) fp8kv_attn_chunk_kernel(const AttnParams p) {
  const int b = blockIdx.z;
  const int kvh = blockIdx.y;
  const int ch = blockIdx.x;
  const int len = seq_len_of(p, b);
  const int t0 = ch * p.chunk;
  if (t0 >= len) return;  // uniform: the combine reads only chunks that hold tokens
  const int n = min(len - t0, p.chunk);

  __shared__ float qs[G][kHeadDim];          // query rows * (sm_scale * k_scale * log2 e)
  __shared__ float ps[G][kMaxChunk];         // scores, then 2^(s - m)
  __shared__ float red[kAttnThreads / 32][G][kHeadDim];
  __shared__ float s_m[G], s_l[G];

  const float c = p.sm_scale * __ldg(p.k_scale) * 1.4426950408889634f;  // log2(e)
  for (int i = threadIdx.x; i < G * kHeadDim; i += kAttnThreads) {
    const int g = i / kHeadDim, d = i - g * kHeadDim;
    qs[g][d] = load_q(p.q, p.q_fp16, (static_cast<size_t>(b) * p.num_q_heads + kvh * G + g) * kHeadDim + d) * c;
  }
  __syncthreads();

  const int sub = threadIdx.x % kLanesPerToken;  // dims sub*16 .. +15
  const int tok = threadIdx.x / kLanesPerToken;  // token within a pass
  const uint8_t* kbase = static_cast<const uint8_t*>(p.k_cache) + kvh * kHeadDim + sub * 16;
  const uint8_t* vbase = static_cast<const uint8_t*>(p.v_cache) + kvh * kHeadDim + sub * 16;
  const long long row_bytes = static_cast<long long>(p.num_kv_heads) * kHeadDim;

  // ---- scores
  {
    float qr[G][16];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < 16; ++j) qr[g][j] = qs[g][sub * 16 + j];
    for (int i0 = 0; i0 < n; i0 += kTokPerPass * kUnroll) {
      uint4 w[kUnroll];
      bool valid[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = i0 + u * kTokPerPass + tok;
        const long long slot = i < n ? slot_of(p, b, t0 + i) : -1;
        valid[u] = slot >= 0;
        w[u] = valid[u] ? __ldg(reinterpret_cast<const uint4*>(kbase + slot * row_bytes)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        float f[16];
        decode16(w[u], f);
        float s[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float a = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) a = fmaf(f[j], qr[g][j], a);
          s[g] = a;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          s[g] += __shfl_xor_sync(0xffffffffu, s[g], 4);
          s[g] += __shfl_xor_sync(0xffffffffu, s[g], 2);
          s[g] += __shfl_xor_sync(0xffffffffu, s[g], 1);
        }
        const int i = i0 + u * kTokPerPass + tok;
        if (sub == 0 && i < n)
#pragma unroll
          for (int g = 0; g < G; ++g) ps[g][i] = valid[u] ? s[g] : -INFINITY;
      }
    }
  }
  __syncthreads();

  // ---- chunk maximum and 2^(s - m), per head (warp w takes heads w, w+4)
  {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int g = warp; g < G; g += kAttnThreads / 32) {
      float m = -INFINITY;
      for (int i = lane; i < n; i += 32) m = fmaxf(m, ps[g][i]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float l = 0.f;
      for (int i = lane; i < n; i += 32) {
        const float e = (m == -INFINITY) ? 0.f : exp2f(ps[g][i] - m);
        ps[g][i] = e;
        l += e;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      if (lane == 0) {
        s_m[g] = m;
        s_l[g] = l;
      }
    }
  }
  __syncthreads();

  // ---- o = sum_t 2^(s_t - m) * decode(v_t), per head
  float o[G][16];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int j = 0; j < 16; ++j) o[g][j] = 0.f;
  for (int i0 = 0; i0 < n; i0 += kTokPerPass * kUnroll) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kTokPerPass + tok;
      const long long slot = i < n ? slot_of(p, b, t0 + i) : -1;
      w[u] = slot >= 0 ? __ldg(reinterpret_cast<const uint4*>(vbase + slot * row_bytes)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kTokPerPass + tok;
      if (i >= n) continue;
      float f[16];
      decode16(w[u], f);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pg = ps[g][i];
#pragma unroll
        for (int j = 0; j < 16; ++j) o[g][j] = fmaf(pg, f[j], o[g][j]);
      }
    }
  }
  // lanes with the same dims (sub) in a warp: tokens differ by lane bits 3, 4
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[g][j] += __shfl_xor_sync(0xffffffffu, o[g][j], 8);
      o[g][j] += __shfl_xor_sync(0xffffffffu, o[g][j], 16);
    }
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (lane < kLanesPerToken)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int j = 0; j < 16; ++j) red[warp][g][lane * 16 + j] = o[g][j];
  __syncthreads();

  // ---- the chunk's partial result of each head: o[128], m, l
  const int nch = (p.max_seq_len + p.chunk - 1) / p.chunk;
  for (int g = 0; g < G; ++g) {
    float* part = p.partial + ((static_cast<size_t>(b) * p.num_q_heads + kvh * G + g) * nch + ch) * kPartStride;
    const int d = threadIdx.x;
    float acc = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kAttnThreads / 32; ++w2) acc += red[w2][g][d];
    part[d] = acc;
    if (d == 0) {
      part[kHeadDim] = s_m[g];
      part[kHeadDim + 1] = s_l[g];
    }
  }
}

// One CTA per (query head, sequence), one thread per head dim.
__global__ void __launch_bounds__(kHeadDim) fp8kv_attn_combine_kernel(const AttnParams p) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int len = seq_len_of(p, b);
  const size_t oi = (static_cast<size_t>(b) * p.num_q_heads + h) * kHeadDim + d;
  float y = 0.f;  // an empty sequence gives zeros
  if (len > 0) {
    const int nch = (p.max_seq_len + p.chunk - 1) / p.chunk;
    const int used = (len + p.chunk - 1) / p.chunk;
    const float* part = p.partial + (static_cast<size_t>(b) * p.num_q_heads + h) * nch * kPartStride;
    float mx = -INFINITY;
    for (int c = 0; c < used; ++c) mx = fmaxf(mx, part[c * kPartStride + kHeadDim]);
    float l = 0.f, o = 0.f;
    if (mx != -INFINITY) {
      for (int c = 0; c < used; ++c) {
        const float* pc = part + c * kPartStride;
        const float wgt = exp2f(pc[kHeadDim] - mx);
        l = fmaf(wgt, pc[kHeadDim + 1], l);
        o = fmaf(wgt, pc[d], o);
      }
    }
    y = l > 0.f ? (o / l) * __ldg(p.v_scale) : 0.f;
  }
  if (p.out_fp16)
    static_cast<__half*>(p.out)[oi] = __float2half_rn(y);
  else
    static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(y);
}

template <int G>
cudaError_t launch_chunks(const AttnParams& p, cudaStream_t stream) {
  const dim3 grid((p.max_seq_len + p.chunk - 1) / p.chunk, p.num_kv_heads, p.batch);
  fp8kv_attn_chunk_kernel<G><<<grid, kAttnThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int attn_part_stride() { return kPartStride; }
int attn_max_chunk() { return kMaxChunk; }

cudaError_t launch_fp8kv_attention(const AttnParams& p, cudaStream_t stream) {
  const int G = p.num_q_heads / p.num_kv_heads;
  cudaError_t e;
  switch (G) {
    case 1: e = launch_chunks<1>(p, stream); break;
    case 2: e = launch_chunks<2>(p, stream); break;
    case 4: e = launch_chunks<4>(p, stream); break;
    case 8: e = launch_chunks<8>(p, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  fp8kv_attn_combine_kernel<<<dim3(p.num_q_heads, p.batch), kHeadDim, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace w8a8
