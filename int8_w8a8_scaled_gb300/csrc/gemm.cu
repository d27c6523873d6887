// gemm.cu -- the scaled matmul kernels (sm_103a).
//
// out[m, n] = round16(((float)sum_k A[m, k] B[n, k]) * scale_a[m|0] * scale_b[n|0])
// ("[Kernel] Add w8a8 CUTLASS kernels", feature list of cutlass_scaled_mm_dq:
// per-tensor / per-token activation scales, per-tensor / per-channel weight
// scales, bf16 / fp16 output, dequantisation fused into the GEMM epilogue so
// the output is written once.)
//
// A persistent kernel: each CTA of 192 threads walks a list of work units
// (one 128 x BN output tile, or one K slice of it):
//   warp 0, one lane : TMA producer -- loads 128-byte-wide K blocks of both
//                      operands into a ring of shared-memory stages
//                      (128-byte swizzle), signalling a "full" mbarrier;
//   warp 1           : allocates TMEM; one lane issues tcgen05.mma for each
//                      K block and commits to the stage's "empty" mbarrier so
//                      the producer can refill it, and to a per-accumulator
//                      "full" mbarrier at the end of a unit;
//   warps 2..5       : epilogue -- tcgen05.ld of the accumulator lanes (warp
//                      w owns TMEM lanes 32(w%4)..32(w%4)+31), scale, round,
//                      store; then release the accumulator to the MMA warp.
// With small M the operands swap roles (weights on the 128-row MMA side, the
// few tokens on the BN side) so the narrow dimension costs no padding.
//
// fp8 e4m3 operands go straight to tcgen05 kind::f8f6f4 with an fp32
// accumulator.  int8 operands (tcgen05 kind::i8 is not available on sm_103a)
// arrive as f16 planes (int8 -> f16 is exact) and use kind::f16.  Products
// are at most 2^14, so an fp32 accumulator holds the exact integer sum for up
// to 1024 K; the MMA issuer accumulates one K chunk of <= 1024 at a time and
// the epilogue warps drain each finished chunk into an exact int32 total kept
// in a second TMEM region (2 * block_n columns, so two CTAs share an SM).
//
// Split-K (used when there are too few output tiles to fill the GPU, i.e.
// small-M decode): every slice writes its partial tile to the workspace; the
// last slice to arrive (atomic counter per tile) sums the partials in slice
// order 0..S-1 -- a fixed order, so results do not depend on scheduling --
// applies the epilogue and resets the counter to zero.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_common.cuh"
#include "internal.h"
#include "quant_math.cuh"
#include "sm103_ptx.cuh"

namespace w8a8 {

namespace {

// Split-K partial of one TMEM lane: 16 consecutive accumulator columns
// starting at col0 of row `row`, as float4s (those wholly past the valid
// columns are not written).  The layout of a partial tile follows the
// output's: with swap the P rows are output columns, and the tile is
// float4-column-major -- float4 (row, c4) at c4 * 128 + row -- so a warp (32
// consecutive rows) writes 512 contiguous bytes per store and the final sum
// walks down rows; without swap it is row-major -- (row, c4) at row * vpr +
// c4, vpr = valid columns / 4 rounded up -- and the final sum walks along
// rows, matching the output rows it stores.
template <bool SWAP>
__device__ __forceinline__ size_t partial_index(int row, int c4, int vpr) {
  return SWAP ? static_cast<size_t>(c4) * kTileP + row : static_cast<size_t>(row) * vpr + c4;
}

template <bool SWAP>
__device__ __forceinline__ void write_partial16(uint32_t* tile, int row, int col0, int qvalid,
                                                const uint32_t (&v)[16]) {
  uint4* t4 = reinterpret_cast<uint4*>(tile);
  const int vpr = (qvalid + 3) / 4;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (col0 + 4 * j < qvalid)
      t4[partial_index<SWAP>(row, col0 / 4 + j, vpr)] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

// Epilogue store of four reduced accumulators at P row p and Q columns
// q..q+3 (only the first `nvalid` are inside the problem).
template <bool SWAP, typename OutT, typename V>
__device__ __forceinline__ void store4(const MmParams& prm, int p, int q, int nvalid, const V (&v)[4]) {
  OutT* out = reinterpret_cast<OutT*>(prm.out);
  if (!SWAP) {
    if (p >= prm.M) return;
    const float sa = prm.a_per_row ? __ldg(prm.scale_a + p) : __ldg(prm.scale_a);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j < nvalid) {
        const float sb = prm.b_per_row ? __ldg(prm.scale_b + q + j) : __ldg(prm.scale_b);
        out[static_cast<long long>(p) * prm.ldc + q + j] = OutConv<OutT>::conv(v[j], sa, sb);
      }
    }
  } else {
    if (p >= prm.N) return;
    const float sb = prm.b_per_row ? __ldg(prm.scale_b + p) : __ldg(prm.scale_b);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j < nvalid) {
        const float sa = prm.a_per_row ? __ldg(prm.scale_a + q + j) : __ldg(prm.scale_a);
        out[static_cast<long long>(q + j) * prm.ldc + p] = OutConv<OutT>::conv(v[j], sa, sb);
      }
    }
  }
}

// One work unit is a (K slice, output tile) pair; the persistent CTAs walk
// the units round-robin.  Units are numbered slice-major so that the slices
// of a tile are spread over different CTAs.
struct Unit {
  int p0, q0, tile_lin, split, kb_begin, nkb;
};

__device__ __forceinline__ Unit unit_of(int w, const MmParams& prm, int group, int bn) {
  const int tiles = prm.tiles_p * prm.tiles_q;
  Unit u;
  u.split = w / tiles;
  int tp, tq;
  tile_coords(w - u.split * tiles, prm.tiles_p, prm.tiles_q, group, tp, tq);
  u.tile_lin = tp * prm.tiles_q + tq;
  u.p0 = tp * kTileP;
  u.q0 = tq * bn;
  u.kb_begin = u.split * prm.kb_per_split;
  u.nkb = min(prm.num_kb, u.kb_begin + prm.kb_per_split) - u.kb_begin;
  return u;
}

// Optional per-CTA phase trace (debug): kTraceSlots 64-bit %globaltimer
// stamps per CTA, written only when a trace buffer is set.
constexpr int kTraceSlots = 16;
enum TraceSlot {
  T_START = 0, T_PROLOGUE, T_DEP_RELEASED, T_FIRST_DATA, T_MMA_ISSUED, T_EPI_DONE, T_END, T_SMID,
  T_ACC_READY, T_DRAINED, T_SYNCED, T_REDUCED, T_FQ_AMAX, T_FQ_SCALES, T_FQ_STAGE0
};

__device__ __forceinline__ void trace_stamp(const MmParams& prm, int slot) {
  if (prm.trace && blockIdx.x < prm.trace_ctas)
    prm.trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + slot] = global_timer_ns();
}

// Persistent, warp-specialised scaled matmul.
//   warp 0 (one lane)  TMA producer over all units of this CTA;
//   warp 1             TMEM owner; one lane issues the MMAs;
//   warps 2..5         epilogue; warp w reads TMEM lanes 32*(w%4)...
// Accumulation units (one per work unit for e4m3, one per <= 1024-K chunk
// for int8) alternate between two TMEM accumulators, so the epilogue of one
// unit overlaps the MMAs of the next.
// Split-K, final sum of rows [r0, r0 + nrows) of a tile (both reductions):
// the vector -> (row, float4 column) map that walks the partial tiles in
// their storage order (see write_partial16), so that a warp's loads and its
// output stores are both contiguous.
template <bool SWAP>
__device__ __forceinline__ void reduce_pos(int v, int nrows, int vpr, int& rr, int& c4) {
  if (SWAP) {
    rr = v % nrows;
    c4 = v / nrows;
  } else {
    rr = v / vpr;
    c4 = v - rr * vpr;
  }
}

// Epilogue of one reduced float4 (four outputs at row r0 + rr, column c4*4).
template <int BN, bool SWAP, bool INT8, typename OutT, typename V>
__device__ __forceinline__ void reduce_store(const MmParams& prm, const Unit& un, int row, int c4, int qvalid,
                                             const V (&acc)[4], const float* s_scale_p, const float* s_scale_q) {
  const int col = c4 * 4;
  float s_q[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) s_q[j] = s_scale_q[min(col + j, BN - 1)];
  store4s<SWAP, OutT>(prm, un.p0 + row, un.q0 + col, qvalid - col, acc, s_scale_p[row], s_q);
}

// Each epilogue thread takes B float4 vectors per pass and requests all
// B * S partial vectors (L2; the slices' partial tiles are `slice_stride`
// words apart from `tile0`, float4-column-major) before using any, then sums
// each in slice order 0..S-1 from zero -- the order of both reductions, so
// they give the same bits -- and stores its four outputs with the staged
// scales.
template <int S, int B, int BN, bool SWAP, bool INT8, typename OutT>
__device__ __forceinline__ void reduce_rows(const MmParams& prm, const Unit& un, const uint32_t* tile0,
                                            size_t slice_stride, int r0, int nrows, int qvalid, int et,
                                            const float* s_scale_p, const float* s_scale_q) {
  const int vpr = (qvalid + 3) / 4;  // valid float4 columns
  const int nvec = nrows * vpr;
  for (int v0 = et; v0 < nvec; v0 += B * kEpiThreads) {
    uint4 x[B][S];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int v = v0 + b * kEpiThreads;
      int rr, c4;
      reduce_pos<SWAP>(v < nvec ? v : v0, nrows, vpr, rr, c4);  // past the end: an in-range load, no store
      const size_t idx = partial_index<SWAP>(r0 + rr, c4, vpr);
#pragma unroll
      for (int s2 = 0; s2 < S; ++s2) x[b][s2] = __ldcg(reinterpret_cast<const uint4*>(tile0 + s2 * slice_stride) + idx);
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int v = v0 + b * kEpiThreads;
      if (v >= nvec) break;
      int rr, c4;
      reduce_pos<SWAP>(v, nrows, vpr, rr, c4);
      if (INT8) {
        int acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
          acc[0] += static_cast<int>(x[b][s2].x);
          acc[1] += static_cast<int>(x[b][s2].y);
          acc[2] += static_cast<int>(x[b][s2].z);
          acc[3] += static_cast<int>(x[b][s2].w);
        }
        reduce_store<BN, SWAP, INT8, OutT>(prm, un, r0 + rr, c4, qvalid, acc, s_scale_p, s_scale_q);
      } else {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
          acc[0] += __uint_as_float(x[b][s2].x);
          acc[1] += __uint_as_float(x[b][s2].y);
          acc[2] += __uint_as_float(x[b][s2].z);
          acc[3] += __uint_as_float(x[b][s2].w);
        }
        reduce_store<BN, SWAP, INT8, OutT>(prm, un, r0 + rr, c4, qvalid, acc, s_scale_p, s_scale_q);
      }
    }
  }
}

// Any slice count: a running sum per vector in slice order (the loop is
// unrolled so several slices' loads are in flight).
template <int BN, bool SWAP, bool INT8, typename OutT>
__device__ __forceinline__ void reduce_rows_n(const MmParams& prm, const Unit& un, const uint32_t* tile0,
                                              size_t slice_stride, int S, int r0, int nrows, int qvalid, int et,
                                              const float* s_scale_p, const float* s_scale_q) {
  const int vpr = (qvalid + 3) / 4;
  const int nvec = nrows * vpr;
  for (int v = et; v < nvec; v += kEpiThreads) {
    int rr, c4;
    reduce_pos<SWAP>(v, nrows, vpr, rr, c4);
    const uint4* src = reinterpret_cast<const uint4*>(tile0) + partial_index<SWAP>(r0 + rr, c4, vpr);
    if (INT8) {
      int acc[4] = {0, 0, 0, 0};
#pragma unroll 4
      for (int s2 = 0; s2 < S; ++s2) {
        const uint4 x = __ldcg(src + s2 * (slice_stride / 4));
        acc[0] += static_cast<int>(x.x);
        acc[1] += static_cast<int>(x.y);
        acc[2] += static_cast<int>(x.z);
        acc[3] += static_cast<int>(x.w);
      }
      reduce_store<BN, SWAP, INT8, OutT>(prm, un, r0 + rr, c4, qvalid, acc, s_scale_p, s_scale_q);
    } else {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int s2 = 0; s2 < S; ++s2) {
        const uint4 x = __ldcg(src + s2 * (slice_stride / 4));
        acc[0] += __uint_as_float(x.x);
        acc[1] += __uint_as_float(x.y);
        acc[2] += __uint_as_float(x.z);
        acc[3] += __uint_as_float(x.w);
      }
      reduce_store<BN, SWAP, INT8, OutT>(prm, un, r0 + rr, c4, qvalid, acc, s_scale_p, s_scale_q);
    }
  }
}

// Dispatch on the slice count: 2, 4 and 8 keep every load of a pass in
// registers (fewer vectors per pass where two CTAs share the SM's registers).
template <int BN, bool SWAP, bool INT8, typename OutT>
__device__ __forceinline__ void reduce_rows_any(const MmParams& prm, const Unit& un, const uint32_t* tile0,
                                                size_t slice_stride, int S, int r0, int nrows, int qvalid, int et,
                                                const float* s_scale_p, const float* s_scale_q);

// ---------------------------------------------------------------- fused activation quantiser
// The decode matmul that quantises its own activations (swap-AB, e4m3, all
// M tokens in one tile).  The per-token dynamic scale is absmax / 448 over
// the token's whole row and every code is the quantiser's own arithmetic
// (quant_math.cuh), so the result equals the two calls quantiser + scaled
// matmul bit for bit ("[Kernel] Support Fp8 Checkpoints (Dynamic + Static)",
// dynamic per-token activation scales).  The epilogue warps, idle during the
// main loop, compute the scales and then fill the token slot of each stage
// with codes in the layout a 128-byte-swizzled TMA load would have written,
// while TMA streams the weights into the other slot.

// 16 consecutive x[m, k..k+15] (16-byte aligned: ld_x and K multiples of 16)
__device__ __forceinline__ void fq_load16(const MmParams& prm, int m, int k, uint4& a, uint4& b) {
  const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(prm.x) +
                                                  static_cast<size_t>(m) * prm.ld_x + k);
  a = p[0];
  b = p[1];
}

template <int XK>
__device__ __forceinline__ float fq_absmax16(const uint4& a, const uint4& b) {
  float f[8], g[8];
  unpack8<XK>(a, f);
  unpack8<XK>(b, g);
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) m = fmaxf(m, fmaxf(fabsf(f[j]), fabsf(g[j])));
  return m;
}

template <int XK>
__device__ __forceinline__ uint4 fq_quant16(const uint4& a, const uint4& b, float s, float y, bool ok) {
  float f[8], g[8];
  unpack8<XK>(a, f);
  unpack8<XK>(b, g);
  // dynamic per-token scales: the quotients stay within the code range
  const uint2 a8 = quant8<0>(f, s, y, ok, true), b8 = quant8<0>(g, s, y, ok, true);
  return make_uint4(a8.x, a8.y, b8.x, b8.y);
}

// Per-token scales of the CTA's token tile (rows 0..M-1), by the 128
// epilogue threads: absmax over this CTA's K range, combined over the
// cluster's K slices (each CTA arrives on every peer's `amax_bar` and reads
// the peers' partial maxima from distributed shared memory: BN words each),
// then scale = absmax / 448 (1 for an all-zero row).  The reciprocal and its
// validity feed the correctly rounded quotient (div_by).  False if a wait
// timed out.
template <int BN>
__device__ bool fq_token_scales(const MmParams& prm, const Unit& un, bool cl, int et, uint32_t amax_bar,
                                uint32_t* s_amax, float* s_tok, float* s_rcp, int* s_rok) {
  const int M = prm.M;
  const int k_lo = un.kb_begin * 128;
  const int k_hi = min(prm.K, (un.kb_begin + un.nkb) * 128);
  const int n16 = (k_hi - k_lo) / 16;
  const int total = M * n16;
  for (int m = et; m < BN; m += kEpiThreads) s_amax[m] = 0u;
  epi_bar_sync();
  for (int base = et; base < total; base += 4 * kEpiThreads) {
    uint4 a[4], b[4];
    int mm[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int idx = base + j * kEpiThreads;
      mm[j] = -1;
      if (idx < total) {
        const int m = idx / n16;
        mm[j] = m;
        fq_load16(prm, m, k_lo + (idx - m * n16) * 16, a[j], b[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (mm[j] >= 0) {
        const float v = prm.x_fp16 ? fq_absmax16<1>(a[j], b[j]) : fq_absmax16<0>(a[j], b[j]);
        atomicMax(s_amax + mm[j], __float_as_uint(v));  // non-negative floats order as their bits
      }
  }
  epi_bar_sync();
  if (et == 0) trace_stamp(prm, T_FQ_AMAX);
  bool ok = true;
  if (cl) {
    if (et == 0) {
      fence_acq_rel_cluster();
      for (int r = 0; r < prm.splits; ++r) mbar_arrive_remote(mapa_shared(amax_bar, static_cast<uint32_t>(r)));
    }
    ok = mbar_wait_cluster(amax_bar, 0);
  }
  for (int m = et; m < BN; m += kEpiThreads) {
    float s = 1.f;
    if (m < M) {
      uint32_t bits = s_amax[m];
      if (cl) {
        bits = 0u;
        for (int r = 0; r < prm.splits; ++r)
          bits = max(bits, ld_dsmem_u32(mapa_shared(smem_addr(s_amax + m), static_cast<uint32_t>(r))));
      }
      s = scale_from_amax<0>(__uint_as_float(bits));
    }
    float y;
    s_rok[m] = recip_ok(s, &y) ? 1 : 0;
    s_tok[m] = s;
    s_rcp[m] = y;
  }
  epi_bar_sync();
  if (et == 0) trace_stamp(prm, T_FQ_SCALES);
  if (prm.scale_a_out && (cl ? (cluster_ctarank() == 0 && cluster_id_x() == 0) : blockIdx.x == 0))
    for (int m = et; m < M; m += kEpiThreads) prm.scale_a_out[m] = s_tok[m];
  return ok;
}

// One warp fills the token slot of a stage (K block kb, BN rows x 128 codes,
// 128-byte swizzle: 16-byte chunk c of row r at r * 128 + (c ^ (r & 7)) * 16)
// with codes; rows >= M and columns >= K are zero.
template <int BN>
__device__ __forceinline__ void fq_fill_stage(const MmParams& prm, int kb, uint8_t* dst, const float* s_tok,
                                              const float* s_rcp, const int* s_rok, int lane) {
  constexpr int kPer = BN * 8 / 32;  // 16-code chunks per lane: 4 (BN 16) .. 16 (BN 64)
  constexpr int kBatch = kPer < 8 ? kPer : 8;
  const int k0 = kb * 128;
#pragma unroll
  for (int j0 = 0; j0 < kPer; j0 += kBatch) {
    uint4 a[kBatch], b[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int ch = lane + 32 * (j0 + j);
      const int r = ch >> 3;
      const int k = k0 + (ch & 7) * 16;
      if (r < prm.M && k < prm.K) fq_load16(prm, r, k, a[j], b[j]);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int ch = lane + 32 * (j0 + j);
      const int r = ch >> 3;
      const int c = ch & 7;
      const int k = k0 + c * 16;
      uint4 q = make_uint4(0u, 0u, 0u, 0u);
      if (r < prm.M && k < prm.K)
        q = prm.x_fp16 ? fq_quant16<1>(a[j], b[j], s_tok[r], s_rcp[r], s_rok[r] != 0)
                       : fq_quant16<0>(a[j], b[j], s_tok[r], s_rcp[r], s_rok[r] != 0);
      *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = q;
    }
  }
}

// Single-token decode variant of the token scales: the CTA's tokens' whole
// rows sit in shared memory (xs, row stride K elements, one bulk copy per
// row after the dependency wait), so the absmax is the full row's -- no
// exchange between the K slices of a cluster -- and the token stages are
// written from shared memory.  One global round trip in all.
template <int BN>
__device__ bool fq_token_scales_rows(const MmParams& prm, int et, uint32_t x_bar, const uint16_t* xs,
                                     uint32_t* s_amax, float* s_tok, float* s_rcp, int* s_rok) {
  const int M = prm.M;
  const int n16 = prm.K / 16;
  const int total = M * n16;
  for (int m = et; m < BN; m += kEpiThreads) s_amax[m] = 0u;
  if (et == 0) {
    mbar_arrive_expect_tx(x_bar, static_cast<uint32_t>(M * prm.K * 2));
    for (int m = 0; m < M; ++m)
      bulk_load(smem_addr(xs + static_cast<size_t>(m) * prm.K),
                static_cast<const uint16_t*>(prm.x) + static_cast<size_t>(m) * prm.ld_x,
                static_cast<uint32_t>(prm.K * 2), x_bar);
  }
  epi_bar_sync();
  if (!mbar_wait(x_bar, 0)) return false;
  if (et == 0) trace_stamp(prm, T_FQ_AMAX);
  float mx = 0.f;
  int cur = -1;
  for (int idx = et; idx < total; idx += kEpiThreads) {
    const int m = idx / n16;
    const uint4* p = reinterpret_cast<const uint4*>(xs + static_cast<size_t>(m) * prm.K + (idx - m * n16) * 16);
    const float v = prm.x_fp16 ? fq_absmax16<1>(p[0], p[1]) : fq_absmax16<0>(p[0], p[1]);
    if (m != cur) {
      if (cur >= 0) atomicMax(s_amax + cur, __float_as_uint(mx));
      cur = m;
      mx = 0.f;
    }
    mx = fmaxf(mx, v);
  }
  if (cur >= 0) atomicMax(s_amax + cur, __float_as_uint(mx));
  epi_bar_sync();
  for (int m = et; m < BN; m += kEpiThreads) {
    const float s = m < M ? scale_from_amax<0>(__uint_as_float(s_amax[m])) : 1.f;
    float y;
    s_rok[m] = recip_ok(s, &y) ? 1 : 0;
    s_tok[m] = s;
    s_rcp[m] = y;
  }
  epi_bar_sync();
  if (et == 0) trace_stamp(prm, T_FQ_SCALES);
  if (prm.scale_a_out && (prm.cluster ? (cluster_ctarank() == 0 && cluster_id_x() == 0) : blockIdx.x == 0))
    for (int m = et; m < M; m += kEpiThreads) prm.scale_a_out[m] = s_tok[m];
  return true;
}

// fq_fill_stage with the tokens' rows in shared memory.
template <int BN>
__device__ __forceinline__ void fq_fill_stage_rows(const MmParams& prm, int kb, uint8_t* dst, const uint16_t* xs,
                                                   const float* s_tok, const float* s_rcp, const int* s_rok,
                                                   int lane) {
  constexpr int kPer = BN * 8 / 32;
  const int k0 = kb * 128;
#pragma unroll 4
  for (int j = 0; j < kPer; ++j) {
    const int ch = lane + 32 * j;
    const int r = ch >> 3;
    const int c = ch & 7;
    const int k = k0 + c * 16;
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    if (r < prm.M && k < prm.K) {
      const uint4* p = reinterpret_cast<const uint4*>(xs + static_cast<size_t>(r) * prm.K + k);
      q = prm.x_fp16 ? fq_quant16<1>(p[0], p[1], s_tok[r], s_rcp[r], s_rok[r] != 0)
                     : fq_quant16<0>(p[0], p[1], s_tok[r], s_rcp[r], s_rok[r] != 0);
    }
    *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = q;
  }
}

// Split-K partial tiles kept in shared memory (distributed-shared-memory
// reduction): row-major in the idle stage ring, BN + 4 floats per row (the
// pad spreads a warp's 16-byte stores of 32 consecutive rows over the banks).
template <int BN>
__device__ __forceinline__ void write_partial16_smem(uint32_t* tile, int row, int col0, const uint32_t (&v)[16]) {
  uint4* dst = reinterpret_cast<uint4*>(tile + static_cast<size_t>(row) * (BN + 4) + col0);
#pragma unroll
  for (int j = 0; j < 4; ++j) dst[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

// Final sum of rows [r0, r0 + nrows) of a cluster-split tile from the S
// partial tiles in the cluster's shared memory (slice s in the CTA of rank
// s, at the same offset `tile_saddr`): B float4 vectors per pass, all B * S
// loads requested before any is used, each vector summed in slice order
// 0..S-1 from zero -- the order of the global reductions, so every form
// gives the same bits.
template <int S, int B, int BN, bool SWAP, bool INT8, typename OutT>
__device__ __forceinline__ void reduce_rows_dsmem(const MmParams& prm, const Unit& un, uint32_t tile_saddr, int r0,
                                                  int nrows, int qvalid, int et, const float* s_scale_p,
                                                  const float* s_scale_q) {
  const int vpr = (qvalid + 3) / 4;
  const int nvec = nrows * vpr;
  uint32_t peer[S];
#pragma unroll
  for (int s2 = 0; s2 < S; ++s2) peer[s2] = mapa_shared(tile_saddr, static_cast<uint32_t>(s2));
  for (int v0 = et; v0 < nvec; v0 += B * kEpiThreads) {
    uint4 x[B][S];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int v = v0 + b * kEpiThreads;
      int rr, c4;
      reduce_pos<SWAP>(v < nvec ? v : v0, nrows, vpr, rr, c4);
      const uint32_t off = static_cast<uint32_t>(((r0 + rr) * (BN + 4) + 4 * c4) * 4);
#pragma unroll
      for (int s2 = 0; s2 < S; ++s2) x[b][s2] = ld_dsmem_v4(peer[s2] + off);
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int v = v0 + b * kEpiThreads;
      if (v >= nvec) break;
      int rr, c4;
      reduce_pos<SWAP>(v, nrows, vpr, rr, c4);
      if (INT8) {
        int acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
          acc[0] += static_cast<int>(x[b][s2].x);
          acc[1] += static_cast<int>(x[b][s2].y);
          acc[2] += static_cast<int>(x[b][s2].z);
          acc[3] += static_cast<int>(x[b][s2].w);
        }
        reduce_store<BN, SWAP, INT8, OutT>(prm, un, r0 + rr, c4, qvalid, acc, s_scale_p, s_scale_q);
      } else {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
          acc[0] += __uint_as_float(x[b][s2].x);
          acc[1] += __uint_as_float(x[b][s2].y);
          acc[2] += __uint_as_float(x[b][s2].z);
          acc[3] += __uint_as_float(x[b][s2].w);
        }
        reduce_store<BN, SWAP, INT8, OutT>(prm, un, r0 + rr, c4, qvalid, acc, s_scale_p, s_scale_q);
      }
    }
  }
}

template <int BN, bool SWAP, bool INT8, typename OutT>
__device__ __forceinline__ void reduce_rows_dsmem_any(const MmParams& prm, const Unit& un, uint32_t tile_saddr, int S,
                                                      int r0, int nrows, int qvalid, int et, const float* s_scale_p,
                                                      const float* s_scale_q) {
  switch (S) {
    case 2: reduce_rows_dsmem<2, 4, BN, SWAP, INT8, OutT>(prm, un, tile_saddr, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
    case 3: reduce_rows_dsmem<3, 2, BN, SWAP, INT8, OutT>(prm, un, tile_saddr, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
    case 4: reduce_rows_dsmem<4, 2, BN, SWAP, INT8, OutT>(prm, un, tile_saddr, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
    case 5: reduce_rows_dsmem<5, 1, BN, SWAP, INT8, OutT>(prm, un, tile_saddr, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
    case 6: reduce_rows_dsmem<6, 1, BN, SWAP, INT8, OutT>(prm, un, tile_saddr, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
    case 7: reduce_rows_dsmem<7, 1, BN, SWAP, INT8, OutT>(prm, un, tile_saddr, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
    default: reduce_rows_dsmem<8, 1, BN, SWAP, INT8, OutT>(prm, un, tile_saddr, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
  }
}

// Narrow tiles run two CTAs per SM (the dispatch sizes their shared memory
// for that); cap their registers so that two fit (<= 168 per thread).
__host__ __device__ constexpr int min_ctas_for(int bn, bool) { return bn <= 64 ? 2 : 1; }
// int8 with one chunk accumulator (256 columns: the MMAs wait while a chunk
// drains into the int32 total) adds four drain-helper warps (6..9), one per
// TMEM lane quarter: each intermediate drain is split between the epilogue
// warp and the helper of a quarter, half of the 16-column groups each.
__host__ __device__ constexpr bool drain_helpers(int bn, bool int8) { return int8 && acc_bufs(bn, int8) == 1; }
__host__ __device__ constexpr int threads_for(int bn, bool int8) { return drain_helpers(bn, int8) ? 320 : 192; }

template <int BN, bool SWAP, bool INT8, typename OutT>
__device__ __forceinline__ void reduce_rows_any(const MmParams& prm, const Unit& un, const uint32_t* tile0,
                                                size_t slice_stride, int S, int r0, int nrows, int qvalid, int et,
                                                const float* s_scale_p, const float* s_scale_q) {
  // loads per pass: 16 (one CTA per SM) or 8 (two share the registers);
  // 32 measured slower (the decode M = 256 down projection's reduction took
  // 11 us instead of 8)
  constexpr int kLoads = 16;
  switch (S) {
    case 2: reduce_rows<2, kLoads / 2, BN, SWAP, INT8, OutT>(prm, un, tile0, slice_stride, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
    case 4: reduce_rows<4, kLoads / 4, BN, SWAP, INT8, OutT>(prm, un, tile0, slice_stride, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
    case 8: reduce_rows<8, kLoads / 8, BN, SWAP, INT8, OutT>(prm, un, tile0, slice_stride, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
    default: reduce_rows_n<BN, SWAP, INT8, OutT>(prm, un, tile0, slice_stride, S, r0, nrows, qvalid, et, s_scale_p, s_scale_q); break;
  }
}

template <int BN, bool SWAP, bool INT8, typename OutT, bool FQ = false>
__global__ void __launch_bounds__(threads_for(BN, INT8), min_ctas_for(BN, INT8))
    w8a8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_p,
                     const __grid_constant__ CUtensorMap tmap_q, const MmParams prm, int stages,
                     int group) {
  constexpr int kQBytes = BN * kRowBytes;
  constexpr int kStageBytes = kPBytes + kQBytes;
  constexpr int kKbElems = INT8 ? 64 : 128;  // elements per 128-byte K block
  constexpr uint32_t kIdesc = make_idesc(kTileP, BN, 0);
  constexpr int kTmemCols = tmem_cols_for(BN, INT8);
  constexpr int kGroups = BN / 16;
  static_assert((INT8 ? acc_bufs(BN, INT8) + 1 : acc_bufs(BN, INT8)) * BN <= kTmemCols && kTmemCols <= 512,
                "accumulators must fit the TMEM allocation");
  static_assert(!FQ || (SWAP && !INT8 && BN <= 64), "the fused quantiser is the swap-AB e4m3 decode path");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sp = smem;
  uint8_t* sq = smem + stages * kPBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sq + stages * kQBytes);
  // bars: full[stages], empty[stages], unit_full[2], unit_empty[2], amax, x,
  // mma_drain (failure path only)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * stages + 7);
  // fused quantiser, rows mode: the tokens' rows after the barrier block
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(reinterpret_cast<uint8_t*>(bars) + kBarBlockBytes);
  __shared__ int s_is_last;
  // fused quantiser: per-token partial absmax (float bits), scales, reciprocals
  __shared__ uint32_t s_amax[FQ ? BN : 1];
  __shared__ float s_tok[FQ ? BN : 1];
  __shared__ float s_rcp[FQ ? BN : 1];
  __shared__ int s_rok[FQ ? BN : 1];
  __shared__ float s_scale_p[kTileP];  // the unit's P-side row scales
  __shared__ float s_scale_q[BN];      // the unit's Q-side column scales

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int units = prm.tiles_p * prm.tiles_q * prm.splits;
  // Units this CTA walks.  Persistent: blockIdx.x, +gridDim.x, ...  With a
  // cluster split the grid is one CTA per unit: the CTA of rank r in cluster
  // c takes K slice r of tile c (units are numbered slice-major).
  const bool cl = prm.cluster != 0;
  const int w_first = cl ? static_cast<int>(cluster_ctarank()) * (prm.tiles_p * prm.tiles_q) +
                               static_cast<int>(cluster_id_x())
                         : static_cast<int>(blockIdx.x);
  const int w_step = cl ? units : static_cast<int>(gridDim.x);
  if (threadIdx.x == 0) trace_stamp(prm, T_START);

  // Warm L2 with the weight tiles of this CTA's first work unit before
  // waiting on the preceding kernel: a prefetch only reads (coherent) global
  // memory into L2, so it is safe whatever that kernel writes, and the
  // weight stream starts while the preceding kernel is still running.
  if (threadIdx.x == 0 && w_first < units) {
    const Unit un = unit_of(w_first, prm, group, BN);
    if constexpr (FQ) {
      // the activations this CTA quantises go first: once the weight stream
      // fills the HBM queues, a read behind it waits microseconds
      const int k_lo = un.kb_begin * 128;
      const int k_hi = min(prm.K, (un.kb_begin + un.nkb) * 128);
      for (int m = 0; m < prm.M; ++m)
        bulk_prefetch_l2(static_cast<const uint16_t*>(prm.x) + static_cast<size_t>(m) * prm.ld_x + k_lo,
                         static_cast<uint32_t>((k_hi - k_lo) * 2));
    }
    const CUtensorMap* wmap = SWAP ? &tmap_p : &tmap_q;
    const int w_row = SWAP ? un.p0 : un.q0;
    const int n_pf = min(un.nkb, prm.prefetch_kb);
    for (int i = 0; i < n_pf; ++i) tma_prefetch_l2_2d(wmap, (un.kb_begin + i) * kKbElems, w_row);
  }

  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + stages + s); };
  auto ufull_bar = [&](int b) { return smem_addr(bars + 2 * stages + b); };
  auto uempty_bar = [&](int b) { return smem_addr(bars + 2 * stages + 2 + b); };
  const uint32_t amax_bar = smem_addr(bars + 2 * stages + 4);
  const uint32_t x_bar = smem_addr(bars + 2 * stages + 5);
  const uint32_t drain_bar = smem_addr(bars + 2 * stages + 6);

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmap_p);
    prefetch_tensormap(&tmap_q);
    for (int s = 0; s < stages; ++s) {
      // fused quantiser: the weights' TMA and the warp writing the codes
      mbar_init(full_bar(s), FQ ? 2 : 1);
      mbar_init(empty_bar(s), 1);
    }
    if (FQ) {
      mbar_init(amax_bar, cl ? prm.splits : 1);
      mbar_init(x_bar, 1);
    }
    mbar_init(drain_bar, 1);
    mbar_init(ufull_bar(0), 1);
    mbar_init(ufull_bar(1), 1);
    // the epilogue threads (and the drain helpers) release an accumulator
    mbar_init(uempty_bar(0), drain_helpers(BN, INT8) ? 2 * kEpiThreads : kEpiThreads);
    mbar_init(uempty_bar(1), drain_helpers(BN, INT8) ? 2 * kEpiThreads : kEpiThreads);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the cluster's peers arrive on amax_bar: its initialisation must be
  // visible to them first
  if (FQ && cl && !prm.fq_rows) cluster_sync();
  if (threadIdx.x == 0) trace_stamp(prm, T_PROLOGUE);
  // Let the next kernel be scheduled (after this CTA holds its TMEM, so a
  // later kernel never takes TMEM ahead of an earlier one), then wait for the
  // preceding kernel's results.
  griddep_launch();
  griddep_wait();
  if (threadIdx.x == 0) trace_stamp(prm, T_DEP_RELEASED);

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      // The token tiles are reused by every weight tile (of a
      // rasterisation group) while the weights stream past once: keep the
      // former in L2 ahead of the latter.  Tokens are the P side without
      // swap, the Q side with it.
      const uint64_t pol_p = SWAP ? policy_evict_first() : policy_evict_last();
      const uint64_t pol_q = SWAP ? policy_evict_last() : policy_evict_first();
      for (int w = w_first; w < units && ok; w += w_step) {
        const Unit un = unit_of(w, prm, group, BN);
        for (int i = 0; i < un.nkb; ++i, ++it) {
          const int s = it % stages;
          const uint32_t ph = (it / stages) & 1;
          if (!mbar_wait(empty_bar(s), ph ^ 1)) { ok = false; break; }
          mbar_arrive_expect_tx(full_bar(s), FQ ? kPBytes : kStageBytes);
          const int kx = (un.kb_begin + i) * kKbElems;
          tma_load_2d_hint(smem_addr(sp + s * kPBytes), &tmap_p, full_bar(s), kx, un.p0, pol_p);
          if (!FQ) tma_load_2d_hint(smem_addr(sq + s * kQBytes), &tmap_q, full_bar(s), kx, un.q0, pol_q);
        }
      }
      if (!ok) {
        // a wait gave up: let the stage loads still in flight land (bounded)
        // before the CTA leaves and its shared memory is released
        for (uint32_t j = it > static_cast<uint32_t>(stages) ? it - stages : 0u; j < it; ++j)
          mbar_wait(full_bar(static_cast<int>(j % stages)), (j / stages) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, u = 0;
      bool ok = true;
      for (int w = w_first; w < units && ok; w += w_step) {
        const Unit un = unit_of(w, prm, group, BN);
        const int chunk = INT8 ? prm.kchunk_kb : un.nkb;
        const int nch = (un.nkb + chunk - 1) / chunk;
        for (int c = 0; c < nch && ok; ++c, ++u) {
          constexpr int kBufs = acc_bufs(BN, INT8);
          const int b = static_cast<int>(u % kBufs);
          if (u >= static_cast<uint32_t>(kBufs)) {
            if (!mbar_wait(uempty_bar(b), ((u - kBufs) / kBufs) & 1)) { ok = false; break; }
            tc_fence_after();
          }
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
          const int i_end = min(un.nkb, (c + 1) * chunk);
          for (int i = c * chunk; i < i_end; ++i, ++it) {
            const int s = it % stages;
            const uint32_t ph = (it / stages) & 1;
            if (!mbar_wait(full_bar(s), ph)) { ok = false; break; }
            if (it == 0) trace_stamp(prm, T_FIRST_DATA);
            tc_fence_after();
            const uint64_t da = smem_desc_sw128(smem_addr(sp + s * kPBytes));
            const uint64_t db = smem_desc_sw128(smem_addr(sq + s * kQBytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = (i == c * chunk && kk == 0) ? 0u : 1u;
              if (INT8)
                mma_f16(d_tmem, da + 2 * kk, db + 2 * kk, kIdesc, acc);
              else
                mma_f8f6f4(d_tmem, da + 2 * kk, db + 2 * kk, kIdesc, acc);
            }
            mma_commit(empty_bar(s));
          }
          mma_commit(ufull_bar(b));
        }
      }
      if (!ok) {
        // a wait gave up: the MMAs already issued finish (bounded wait on a
        // commit behind them) before the accumulators' TMEM is released
        mma_commit(drain_bar);
        mbar_wait(drain_bar, 0);
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // TMEM lane == tile row on the P side
    const int et = threadIdx.x - 2 * 32;  // 0..127
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const size_t tile_elems = static_cast<size_t>(kTileP) * BN;
    uint32_t u = 0;
    uint32_t ait = 0;  // fused quantiser: stage iterations so far (the producer's count)
    bool ok = true;
    if constexpr (FQ) {
      // every unit of this CTA has the same tokens (one token tile) and the
      // same K range (one slice per CTA, or the whole K)
      if (w_first < units)
        ok = prm.fq_rows ? fq_token_scales_rows<BN>(prm, et, x_bar, xs, s_amax, s_tok, s_rcp, s_rok)
                         : fq_token_scales<BN>(prm, unit_of(w_first, prm, group, BN), cl, et, amax_bar, s_amax, s_tok,
                                               s_rcp, s_rok);
    }
    for (int w = w_first; w < units && ok; w += w_step) {
      const Unit un = unit_of(w, prm, group, BN);
      if constexpr (FQ) {
        // warp `quarter` writes the token codes of K blocks quarter, +4, ...
        for (int i = quarter; i < un.nkb; i += 4) {
          const uint32_t itg = ait + static_cast<uint32_t>(i);
          const int s = static_cast<int>(itg % stages);
          if (!mbar_wait(empty_bar(s), ((itg / stages) & 1) ^ 1)) { ok = false; break; }
          if (prm.fq_rows)
            fq_fill_stage_rows<BN>(prm, un.kb_begin + i, sq + s * kQBytes, xs, s_tok, s_rcp, s_rok, lane);
          else
            fq_fill_stage<BN>(prm, un.kb_begin + i, sq + s * kQBytes, s_tok, s_rcp, s_rok, lane);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(s));
          if (itg == 0 && lane == 0) trace_stamp(prm, T_FQ_STAGE0);
        }
        ait += static_cast<uint32_t>(un.nkb);
      }
      const int chunk = INT8 ? prm.kchunk_kb : un.nkb;
      const int nch = (un.nkb + chunk - 1) / chunk;
      const int lane_idx = un.p0 + row;  // global P row of this thread
      // columns of this tile inside the problem (the Q side is M with swap)
      const int qvalid = min(BN, (SWAP ? prm.M : prm.N) - un.q0);
      const int qv4 = (qvalid + 3) & ~3;  // row stride of a partial tile (floats)
      // Stage this unit's scales in shared memory now, while its MMAs run:
      // P-side row scales and Q-side column scales (clamped to the problem;
      // out-of-range rows/columns are never stored).  The previous unit's
      // readers are done (barrier), and the tile's scales are ready before
      // the accumulator is.
      epi_bar_sync();
      {
        const float* ps = SWAP ? prm.scale_b : prm.scale_a;
        const int pp = SWAP ? prm.b_per_row : prm.a_per_row;
        const int plim = SWAP ? prm.N : prm.M;
        const float* qs = SWAP ? prm.scale_a : prm.scale_b;
        const int qp = SWAP ? prm.a_per_row : prm.b_per_row;
        const int qlim = SWAP ? prm.M : prm.N;
        s_scale_p[et] = pp ? __ldg(ps + min(un.p0 + et, plim - 1)) : __ldg(ps);
        if constexpr (FQ) {
          for (int i = et; i < BN; i += kEpiThreads) s_scale_q[i] = s_tok[i];  // the tokens' own scales
        } else {
          for (int i = et; i < BN; i += kEpiThreads) s_scale_q[i] = qp ? __ldg(qs + min(un.q0 + i, qlim - 1)) : __ldg(qs);
        }
      }
      epi_bar_sync();
      const float s_lane = s_scale_p[row];
      // Partial tile of a split unit in the workspace, row-major, row stride
      // = valid columns rounded up to 4 (coalesced float4 rows).
      uint32_t* part = nullptr;
      if (prm.splits > 1)
        part = reinterpret_cast<uint32_t*>(prm.partial) +
               (static_cast<size_t>(un.tile_lin) * prm.splits + un.split) * tile_elems;

      for (int c = 0; c < nch; ++c, ++u) {
        constexpr int kBufs = acc_bufs(BN, INT8);
        const int b = static_cast<int>(u % kBufs);
        if (!mbar_wait(ufull_bar(b), (u / kBufs) & 1)) { ok = false; break; }
        tc_fence_after();
        const bool last = (c == nch - 1);
        if (last && et == 0) trace_stamp(prm, T_ACC_READY);
        const uint32_t acc_addr = lane_base + static_cast<uint32_t>(b * BN);
        const uint32_t tot_addr = lane_base + static_cast<uint32_t>(kBufs * BN);
        if (INT8) {
          // drain in batches of up to four (two when two CTAs share the SM)
          // 16-column groups: all TMEM loads
          // of a batch are in flight together (one wait per batch), so the
          // drain of a 1024-K chunk stays shorter than the next chunk's MMAs
          constexpr int kBatch = drain_batch(kGroups, min_ctas_for(BN, INT8) == 2 ? 2 : 4);  // register budget
          // with drain helpers an intermediate drain covers the first half
          // of the groups here (the helpers take the rest); the last chunk
          // is drained and stored here in full
          const int g_end = (drain_helpers(BN, INT8) && !last) ? kGroups / 2 : kGroups;
#pragma unroll 1
          for (int g0 = 0; g0 < g_end; g0 += kBatch) {
            uint32_t r[kBatch][16], t[kBatch][16];
#pragma unroll
            for (int bb = 0; bb < kBatch; ++bb) {
              tmem_ld16(acc_addr + (g0 + bb) * 16, r[bb]);
              if (c > 0) tmem_ld16(tot_addr + (g0 + bb) * 16, t[bb]);
            }
            tmem_ld_wait();
#pragma unroll
            for (int bb = 0; bb < kBatch; ++bb) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int prev = (c > 0) ? static_cast<int>(t[bb][j]) : 0;
                t[bb][j] = static_cast<uint32_t>(prev + __float2int_rn(__uint_as_float(r[bb][j])));
              }
              const int g = g0 + bb;
              if (!last) {
                tmem_st16(tot_addr + g * 16, t[bb]);
              } else if (prm.splits > 1) {
                if (prm.dsmem_reduce)
                  write_partial16_smem<BN>(reinterpret_cast<uint32_t*>(smem), row, g * 16, t[bb]);
                else
                  write_partial16<SWAP>(part, row, g * 16, qvalid, t[bb]);
              } else {
                int v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = static_cast<int>(t[bb][j]);
                store16<SWAP, OutT>(prm, lane_idx, un.q0 + g * 16, g * 16, v, s_lane, s_scale_q);
              }
            }
          }
        } else {
#pragma unroll 1
          for (int g = 0; g < kGroups; ++g) {
            uint32_t r[16];
            tmem_ld16(acc_addr + g * 16, r);
            tmem_ld_wait();
            if (prm.splits > 1) {
              if (prm.dsmem_reduce)
                write_partial16_smem<BN>(reinterpret_cast<uint32_t*>(smem), row, g * 16, r);
              else
                write_partial16<SWAP>(part, row, g * 16, qvalid, r);
            } else {
              float v[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
              store16<SWAP, OutT>(prm, lane_idx, un.q0 + g * 16, g * 16, v, s_lane, s_scale_q);
            }
          }
        }
        if (INT8 && !last) tmem_st_wait();
        tc_fence_before();
        mbar_arrive(uempty_bar(b));
        if (last && et == 0) trace_stamp(prm, T_DRAINED);
      }
      if (!ok) break;

      if (prm.splits > 1 && !cl) {
        // the last slice to arrive sums all partials in slice order
        __threadfence();
        epi_bar_sync();
        if (et == 0) {
          const unsigned old = atomicAdd(prm.counters + un.tile_lin, 1u);
          s_is_last = (old == static_cast<unsigned>(prm.splits - 1));
        }
        epi_bar_sync();
        if (s_is_last) {
          __threadfence();
          // the 128 epilogue threads sum the whole tile over the slices
          const uint32_t* tile0 = reinterpret_cast<const uint32_t*>(prm.partial) +
                                  static_cast<size_t>(un.tile_lin) * prm.splits * tile_elems;
          reduce_rows_any<BN, SWAP, INT8, OutT>(prm, un, tile0, tile_elems, prm.splits, 0, kTileP, qvalid, et,
                                                s_scale_p, s_scale_q);
          if (et == 0) prm.counters[un.tile_lin] = 0u;
        }
      }
    }
  } else if constexpr (drain_helpers(BN, INT8)) {
    // ------------------------------------------------------ drain helpers
    // Same units and chunks as the epilogue warps; every intermediate drain
    // adds the second half of the chunk's columns into the int32 total.  On
    // the last chunk they only release the accumulator (the epilogue warps
    // read the whole total and store).
    const int quarter = warp & 3;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr int kBufs = acc_bufs(BN, INT8);
    constexpr int kBatch = drain_batch(kGroups, 4);
    uint32_t u = 0;
    bool ok = true;
    for (int w = w_first; w < units && ok; w += w_step) {
      const Unit un = unit_of(w, prm, group, BN);
      const int chunk = prm.kchunk_kb;
      const int nch = (un.nkb + chunk - 1) / chunk;
      for (int c = 0; c < nch; ++c, ++u) {
        const int b = static_cast<int>(u % kBufs);
        if (!mbar_wait(ufull_bar(b), (u / kBufs) & 1)) { ok = false; break; }
        tc_fence_after();
        if (c < nch - 1) {
          const uint32_t acc_addr = lane_base + static_cast<uint32_t>(b * BN);
          const uint32_t tot_addr = lane_base + static_cast<uint32_t>(kBufs * BN);
#pragma unroll 1
          for (int g0 = kGroups / 2; g0 < kGroups; g0 += kBatch) {
            uint32_t r[kBatch][16], t[kBatch][16];
#pragma unroll
            for (int bb = 0; bb < kBatch; ++bb) {
              tmem_ld16(acc_addr + (g0 + bb) * 16, r[bb]);
              if (c > 0) tmem_ld16(tot_addr + (g0 + bb) * 16, t[bb]);
            }
            tmem_ld_wait();
#pragma unroll
            for (int bb = 0; bb < kBatch; ++bb) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int prev = (c > 0) ? static_cast<int>(t[bb][j]) : 0;
                t[bb][j] = static_cast<uint32_t>(prev + __float2int_rn(__uint_as_float(r[bb][j])));
              }
              tmem_st16(tot_addr + (g0 + bb) * 16, t[bb]);
            }
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(uempty_bar(b));
      }
    }
  }

  if (warp == 1 && lane == 0) trace_stamp(prm, T_MMA_ISSUED);
  if (cl && prm.splits > 1) {
    // Cluster split-K: every slice has written its partial tile to the
    // workspace; the cluster barrier (release / acquire at cluster scope)
    // makes them visible to the other CTAs of the tile.  The CTA of rank r
    // then sums rows [r*128/S, (r+1)*128/S) over the S partials from L2
    // (slice order 0..S-1, so the result does not depend on scheduling) and
    // finishes those outputs.  The partials stay in the workspace: no CTA
    // waits for another after this point.
    cluster_sync();
    if (threadIdx.x == 2 * 32) trace_stamp(prm, T_SYNCED);
    if (warp >= 2 && warp < 6) {
      const int et = threadIdx.x - 2 * 32;
      const Unit un = unit_of(w_first, prm, group, BN);
      const int S = prm.splits;
      const int rank = static_cast<int>(cluster_ctarank());
      const int r0 = (rank * kTileP) / S;
      const int r1 = ((rank + 1) * kTileP) / S;
      const int qvalid = min(BN, (SWAP ? prm.M : prm.N) - un.q0);
      if (prm.dsmem_reduce) {
        reduce_rows_dsmem_any<BN, SWAP, INT8, OutT>(prm, un, smem_addr(smem), S, r0, r1 - r0, qvalid, et, s_scale_p,
                                                    s_scale_q);
      } else {
        const size_t tile_elems = static_cast<size_t>(kTileP) * BN;
        const uint32_t* tile0 = reinterpret_cast<const uint32_t*>(prm.partial) +
                                static_cast<size_t>(un.tile_lin) * S * tile_elems;
        reduce_rows_any<BN, SWAP, INT8, OutT>(prm, un, tile0, tile_elems, S, r0, r1 - r0, qvalid, et, s_scale_p,
                                              s_scale_q);
      }
    }
    if (threadIdx.x == 2 * 32) trace_stamp(prm, T_REDUCED);
    // the peers read this CTA's partial tile from its shared memory: it
    // stays allocated until every CTA of the cluster is done
    if (prm.dsmem_reduce) cluster_sync();
  }
  if (threadIdx.x == 2 * 32) trace_stamp(prm, T_EPI_DONE);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0 && prm.trace && blockIdx.x < prm.trace_ctas) {
    trace_stamp(prm, T_END);
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    prm.trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + T_SMID] = smid;
  }
}

template <int BN, bool SWAP, bool INT8, typename OutT, bool FQ = false>
cudaError_t launch_one(const CUtensorMap& tp, const CUtensorMap& tq, const MmParams& p, int stages,
                       cudaStream_t stream) {
  auto kern = w8a8_gemm_kernel<BN, SWAP, INT8, OutT, FQ>;
  // rows mode of the fused quantiser: the tokens' rows follow the barriers
  int smem = gemm_smem_bytes(BN, stages) + (FQ && p.fq_rows ? p.M * p.K * 2 : 0);
  // resident CTAs per SM from the kernel's own resources (shared memory,
  // registers, threads, TMEM columns)
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  int dev = 0, smem_sm = 0, reserved = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess) return e;
  // The block scheduler does not see TMEM: a CTA that finds its SM's columns
  // taken blocks in tcgen05.alloc until the holder exits.  Pad the shared
  // memory (few stages) so that no more CTAs fit an SM than its TMEM holds;
  // otherwise two CTAs of one split-K cluster could share an SM and the
  // one holding the columns would wait at the cluster barrier for the other.
  const int tmem_occ = 512 / tmem_cols_for(BN, INT8);
  const int fixed = static_cast<int>(fa.sharedSizeBytes) + reserved;
  if (smem_sm / (smem + fixed) > tmem_occ) smem = ((smem_sm / (tmem_occ + 1) + 1 - fixed) + 1023) & ~1023;
  // the attribute is per function and device; setting it again is harmless
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // all of the unified L1/shared storage as shared memory, so that two
  // CTAs of the narrow (decode) configurations fit on one SM
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  const int per_cta_smem = smem + fixed;
  const int regs_per_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
  int occ = smem_sm / per_cta_smem;
  constexpr int kCtaThreads = threads_for(BN, INT8);
  occ = min(occ, 65536 / (regs_per_warp * (kCtaThreads / 32)));
  occ = min(occ, 2048 / kCtaThreads);
  occ = max(1, min(occ, 512 / tmem_cols_for(BN, INT8)));
  if (p.max_ctas_per_sm > 0) occ = min(occ, p.max_ctas_per_sm);
  const int units = p.tiles_p * p.tiles_q * p.splits;
  const bool cl = p.cluster != 0 && p.splits > 1;
  if (cl && p.splits > kMaxClusterSplits) return cudaErrorInvalidValue;  // the host validates this first
  // persistent grid; with a cluster split one CTA per unit (clusters of
  // `splits` consecutive CTAs)
  const int grid = cl ? units : max(1, min(units, p.num_sms * occ));
  // Rasterisation: groups of `group` P tiles, Q tiles fastest within a group
  // (tile_coords).  Without swap the P side is the tokens: a group holds as
  // many 128-row token slabs as fit in 48 MB of L2, so they stay resident
  // while the weights stream past once per group (prefill: all 32 M tiles in
  // one group, the weights read once; int8 at M = 8192: 24 M tiles).  With
  // swap the P side is the weights, streamed once anyway.
  const long long slab = static_cast<long long>(kTileP) * p.K * (INT8 ? 2 : 1);
  long long g_tiles = (48LL << 20) / slab;
  if (g_tiles > p.tiles_p) g_tiles = p.tiles_p;
  if (g_tiles < 1) g_tiles = 1;
  const int group = SWAP ? 1 : static_cast<int>(g_tiles);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCtaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (p.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cl) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(p.splits);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  e = cudaLaunchKernelEx(&cfg, kern, tp, tq, p, stages, group);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BN, bool SWAP, bool INT8>
cudaError_t launch_out(const CUtensorMap& tp, const CUtensorMap& tq, const MmParams& p, int out_kind,
                       int stages, cudaStream_t stream) {
  switch (out_kind) {
    case OUT_BF16: return launch_one<BN, SWAP, INT8, __nv_bfloat16>(tp, tq, p, stages, stream);
    case OUT_FP16: return launch_one<BN, SWAP, INT8, __half>(tp, tq, p, stages, stream);
    case OUT_RAW:
      if (INT8) return launch_one<BN, SWAP, INT8, int>(tp, tq, p, stages, stream);
      return launch_one<BN, SWAP, INT8, float>(tp, tq, p, stages, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int BN, bool INT8>
cudaError_t launch_swap(const CUtensorMap& tp, const CUtensorMap& tq, const MmParams& p, bool swap,
                        int out_kind, int stages, cudaStream_t stream) {
  return swap ? launch_out<BN, true, INT8>(tp, tq, p, out_kind, stages, stream)
              : launch_out<BN, false, INT8>(tp, tq, p, out_kind, stages, stream);
}

template <bool INT8>
cudaError_t dispatch(const CUtensorMap& tp, const CUtensorMap& tq, const MmParams& p, int block_n,
                     bool swap, int out_kind, int stages, cudaStream_t stream) {
  switch (block_n) {
    case 16: return launch_swap<16, INT8>(tp, tq, p, swap, out_kind, stages, stream);
    case 32: return launch_swap<32, INT8>(tp, tq, p, swap, out_kind, stages, stream);
    case 64: return launch_swap<64, INT8>(tp, tq, p, swap, out_kind, stages, stream);
    case 128: return launch_swap<128, INT8>(tp, tq, p, swap, out_kind, stages, stream);
    case 256:
      // int8 at 256 columns: tokens on the 128-row side only
      if (INT8) return swap ? cudaErrorInvalidValue : launch_out<256, false, true>(tp, tq, p, out_kind, stages, stream);
      return launch_swap<256, false>(tp, tq, p, swap, out_kind, stages, stream);
    // wave-balancing widths for the large-M e4m3 regime (tokens on the
    // 128-row side only)
    case 160:
      if (swap) return cudaErrorInvalidValue;
      if (INT8) return launch_out<160, false, true>(tp, tq, p, out_kind, stages, stream);
      return launch_out<160, false, false>(tp, tq, p, out_kind, stages, stream);
    case 192:
      if (INT8 || swap) return cudaErrorInvalidValue;
      return launch_out<192, false, false>(tp, tq, p, out_kind, stages, stream);
    case 224:
      if (INT8 || swap) return cudaErrorInvalidValue;
      return launch_out<224, false, false>(tp, tq, p, out_kind, stages, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int BN>
cudaError_t launch_fq(const CUtensorMap& tp, const MmParams& p, int out_kind, int stages, cudaStream_t stream) {
  switch (out_kind) {
    case OUT_BF16: return launch_one<BN, true, false, __nv_bfloat16, true>(tp, tp, p, stages, stream);
    case OUT_FP16: return launch_one<BN, true, false, __half, true>(tp, tp, p, stages, stream);
    case OUT_RAW: return launch_one<BN, true, false, float, true>(tp, tp, p, stages, stream);
    default: return cudaErrorInvalidValue;
  }
}

// int8 [rows, K] (leading dim ld) -> f16 [rows, K] contiguous, exact.
__global__ void widen_int8_kernel(const int8_t* __restrict__ src, long long ld, int rows, int K,
                                  __half* __restrict__ dst) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int vpr = K / 16;  // K is a multiple of 16
  const long long total = static_cast<long long>(rows) * vpr;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / vpr;
    const int v = static_cast<int>(i - r * vpr);
    const int4 w = __ldcs(reinterpret_cast<const int4*>(src + r * ld) + v);
    const int8_t* b = reinterpret_cast<const int8_t*>(&w);
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      __half lo = __int2half_rn(b[2 * j]);
      __half hi = __int2half_rn(b[2 * j + 1]);
      o[j] = static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
    }
    uint4* d = reinterpret_cast<uint4*>(dst + r * K) + 2 * v;
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace

int gemm_smem_bytes(int block_n, int stages) {
  return stages * (kPBytes + block_n * kRowBytes) + 1024 /*alignment slack*/ + kBarBlockBytes;
}

int max_stages_for(int block_n, int smem_budget) {
  int s = (smem_budget - 1024 - 256) / (kPBytes + block_n * kRowBytes);
  return s;
}

cudaError_t launch_fp8_gemm(const CUtensorMap& tmap_p, const CUtensorMap& tmap_q, const MmParams& p,
                            int block_n, bool swap, int out_kind, int stages, cudaStream_t stream) {
  return dispatch<false>(tmap_p, tmap_q, p, block_n, swap, out_kind, stages, stream);
}

cudaError_t launch_fused_quant_gemm(const CUtensorMap& tmap_p, const MmParams& p, int block_n, int out_kind,
                                    int stages, cudaStream_t stream) {
  switch (block_n) {
    case 16: return launch_fq<16>(tmap_p, p, out_kind, stages, stream);
    case 32: return launch_fq<32>(tmap_p, p, out_kind, stages, stream);
    case 64: return launch_fq<64>(tmap_p, p, out_kind, stages, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_int8_gemm(const CUtensorMap& tmap_p, const CUtensorMap& tmap_q, const MmParams& p,
                             int block_n, bool swap, int out_kind, int stages, cudaStream_t stream) {
  return dispatch<true>(tmap_p, tmap_q, p, block_n, swap, out_kind, stages, stream);
}

cudaError_t read_clear_device_status(int* flags) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
  *flags = v;
  return e;
}

cudaError_t launch_int8_widen(const void* src, long long ld_src, int rows, int K, void* dst_f16,
                              cudaStream_t stream) {
  const long long total = static_cast<long long>(rows) * (K / 16);
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, widen_int8_kernel, static_cast<const int8_t*>(src), ld_src, rows, K,
                                     static_cast<__half*>(dst_f16));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace w8a8
