// gemm_common.cuh -- constants and epilogue helpers shared by the scaled
// matmul kernels (gemm.cu: one CTA per 128-row tile; gemm2sm.cu: a CTA pair
// per 256-row tile).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace w8a8 {
namespace {  // each translation unit keeps its own copy

constexpr int kThreads = 192;     // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kEpiThreads = 128;
constexpr int kMaxSplits = 16;   // split_k limit of the reduction (host enforces)
constexpr int kMaxClusterSplits = kMaxClusterSplit;  // split_k limit of the cluster reduction
constexpr int kTileP = 128;       // rows of the P operand per tile (MMA M)
constexpr int kRowBytes = 128;    // bytes of K per stage row (one swizzle row)
constexpr int kPBytes = kTileP * kRowBytes;
constexpr int kBarBlockBytes = 256;  // mbarriers and the TMEM slot after the stage ring

// e4m3: accumulation units alternate between two fp32 accumulators (columns
// 0 and bn) so the epilogue of one unit overlaps the next unit's MMAs.
// int8: fp32 chunk accumulators (columns 0, bn) and the int32 total after
// them.  Up to 160 columns two chunk accumulators and the total fit the 512
// TMEM columns (3 * bn), so one chunk's MMAs run while the previous chunk
// drains; at 256 columns one chunk accumulator and the total fill TMEM and
// the MMAs wait for each drain.
__host__ __device__ constexpr int acc_bufs(int bn, bool int8) { return (int8 && 3 * bn > 512) ? 1 : 2; }

__host__ __device__ constexpr int tmem_cols_for(int bn, bool int8) {
  const int need = acc_bufs(bn, int8) * bn + (int8 ? bn : 0);
  int c = 32;
  while (c < need) c *= 2;
  return c;
}

// Output element conversion.  16-bit outputs round to nearest even; FP32
// stores y = (acc * s_a) * s_b unrounded; INT32 stores the raw accumulator
// (scales not applied).
template <typename OutT>
struct OutConv;
template <>
struct OutConv<__nv_bfloat16> {
  template <typename V>
  __device__ __forceinline__ static __nv_bfloat16 conv(V v, float sa, float sb) {
    return __float2bfloat16_rn((static_cast<float>(v) * sa) * sb);
  }
};
template <>
struct OutConv<__half> {
  template <typename V>
  __device__ __forceinline__ static __half conv(V v, float sa, float sb) {
    return __float2half_rn((static_cast<float>(v) * sa) * sb);
  }
};
template <>
struct OutConv<float> {
  template <typename V>
  __device__ __forceinline__ static float conv(V v, float sa, float sb) {
    return (static_cast<float>(v) * sa) * sb;
  }
};
template <>
struct OutConv<int> {
  template <typename V>
  __device__ __forceinline__ static int conv(V v, float, float) {
    return static_cast<int>(v);
  }
};

// Map a linear tile id to (tile_p, tile_q): tiles are walked in groups of
// `group` P-tiles, Q fastest inside a group, so concurrently running CTAs
// share operand tiles in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_p, int tiles_q, int group, int& tp,
                                            int& tq) {
  const int per_group = group * tiles_q;
  const int g = t / per_group;
  const int first = g * group;
  const int gsz = min(group, tiles_p - first);
  const int local = t - g * per_group;
  tp = first + local % gsz;
  tq = local / gsz;
}

// Epilogue store of 16 consecutive accumulator columns of one TMEM lane.
// Without swap the lane is an output row m and the columns are n; with swap
// the lane is an output column n and the columns are rows m.  The scale
// order is always (acc * scale_a) * scale_b.  s_lane is the lane's P-side
// scale; sq the unit's Q-side scales, staged in shared memory and indexed
// from the tile's first column (col0 - q0 = local column).
template <bool SWAP, typename OutT, typename V>
__device__ __forceinline__ void store16(const MmParams& prm, int lane_idx, int col0, int lcol0, const V (&v)[16],
                                        float s_lane, const float* sq) {
  OutT* out = reinterpret_cast<OutT*>(prm.out);
  if (!SWAP) {
    const int m = lane_idx;
    if (m >= prm.M) return;
    OutT* row = out + static_cast<long long>(m) * prm.ldc;
    if (prm.out_vec_ok && col0 + 16 <= prm.N) {
      alignas(16) OutT o[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j] = OutConv<OutT>::conv(v[j], s_lane, sq[lcol0 + j]);
      uint4* dst = reinterpret_cast<uint4*>(row + col0);
      const uint4* src = reinterpret_cast<const uint4*>(o);
#pragma unroll
      for (int j = 0; j < static_cast<int>(sizeof(o) / 16); ++j) dst[j] = src[j];
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int n = col0 + j;
        if (n < prm.N) row[n] = OutConv<OutT>::conv(v[j], s_lane, sq[lcol0 + j]);
      }
    }
  } else {
    const int n = lane_idx;
    if (n >= prm.N) return;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int m = col0 + j;
      if (m < prm.M) out[static_cast<long long>(m) * prm.ldc + n] = OutConv<OutT>::conv(v[j], sq[lcol0 + j], s_lane);
    }
  }
}

// Store of four reduced accumulators at P row p and Q columns q..q+3 (the
// first `nvalid` inside the problem), with the scales in registers: s_p for
// P row p, s_q[j] for Q column q + j.  The product order stays
// (acc * scale_a) * scale_b.
template <bool SWAP, typename OutT, typename V>
__device__ __forceinline__ void store4s(const MmParams& prm, int p, int q, int nvalid, const V (&v)[4], float s_p,
                                        const float (&s_q)[4]) {
  OutT* out = reinterpret_cast<OutT*>(prm.out);
  if (p >= (SWAP ? prm.N : prm.M)) return;
  if (!SWAP && nvalid >= 4 && prm.out_vec_ok) {
    // four consecutive outputs of one row in one store (q is a multiple of
    // 4 and the rows are 16-byte aligned)
    alignas(16) OutT o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = OutConv<OutT>::conv(v[j], s_p, s_q[j]);
    OutT* dst = out + static_cast<long long>(p) * prm.ldc + q;
    if (sizeof(OutT) == 2)
      *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(o);
    else
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(o);
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j < nvalid) {
      if (!SWAP)
        out[static_cast<long long>(p) * prm.ldc + q + j] = OutConv<OutT>::conv(v[j], s_p, s_q[j]);
      else
        out[static_cast<long long>(q + j) * prm.ldc + p] = OutConv<OutT>::conv(v[j], s_q[j], s_p);
    }
  }
}

__device__ __forceinline__ void epi_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

// Programmatic dependent launch: allow the next kernel to be scheduled; wait
// for the preceding kernel in the stream (and its memory) before touching
// global memory.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// int8 drain: 16-column groups per batch, the largest count <= cap that
// divides the tile's groups (160 columns: 10 groups, batches of 2)
__host__ __device__ constexpr int drain_batch(int groups, int cap) {
  return cap <= 1 ? 1 : (groups % cap == 0 ? cap : drain_batch(groups, cap - 1));
}

}  // namespace
}  // namespace w8a8
