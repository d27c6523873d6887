// gemm2sm.cu -- the scaled matmul on CTA pairs (tcgen05.mma.cta_group::2), for
// large M with the tokens on the 128-row side of each CTA.
//
// out[m, n] = round16(((float)sum_k A[m, k] B[n, k]) * scale_a[m|0] * scale_b[n|0])
// ("[Kernel] Add w8a8 CUTLASS kernels", feature list of cutlass_scaled_mm_dq),
// computed exactly as the one-CTA kernel of gemm.cu does; only the tiling
// differs.
//
// Why pairs: a one-CTA tile of 128 x 256 writes (TMA) and reads (MMA)
// 2 * (16 KB + 32 KB) of shared memory per 128-deep K step, more than an SM's
// shared memory moves at the tensor pipe's rate.  A cluster of two CTAs on two
// SMs computes one 256 x BN tile with one MMA stream: each CTA holds its own
// 128 rows of A and half of the BN columns of B, and the pair's MMA reads the
// B halves of both (the pair, not each SM, holds B once), so each SM stages
// 16 + 16 KB per K step for the same work per SM.
//
// Roles (both CTAs run 192 threads):
//   warp 0, one lane   TMA producer of this CTA's A rows and B half.  The
//                      loads of both CTAs complete on the leader CTA's (rank
//                      0) full barrier, which expects the pair's bytes;
//   warp 1             allocates the pair's TMEM (cta_group::2); in the
//                      leader one lane issues the M = 256 MMAs and commits to
//                      both CTAs' barriers at once (multicast);
//   warps 2..5         epilogue of this CTA's 128 accumulator rows (its own
//                      TMEM), then a release arrival on the leader's barrier.
// Every wait is bounded (as in gemm.cu); a CTA whose wait gave up still meets
// its peer at the final cluster barrier, after the copies and MMAs it may
// have in flight have landed.
//
// The pairs walk the tiles round-robin, so a tile count just above a multiple
// of the pair count leaves a last round in which few pairs work for a whole
// tile's time.  With MmParams::tail_tiles > 0 (e4m3) the tiles of that round
// run as two K halves on two pairs each: every CTA writes its fp32 half to
// the workspace and the second half to arrive sums the two, half 0 first,
// and stores them -- the round then lasts about half as long.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_common.cuh"
#include "internal.h"
#include "sm103_ptx.cuh"

namespace w8a8 {

namespace {

// int8 with one chunk accumulator per CTA (256 columns) adds four
// drain-helper warps (6..9), one per TMEM lane quarter, that take half of
// each intermediate drain (as in the one-CTA kernel)
__host__ __device__ constexpr bool pair_drain_helpers(int bn, bool int8) { return int8 && acc_bufs(bn, int8) == 1; }
__host__ __device__ constexpr int pair_threads(int bn, bool int8) { return pair_drain_helpers(bn, int8) ? 320 : 192; }

// --- pair forms of the tcgen05 / TMA instructions (cta_group::2)

__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

template <bool INT8>
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  if (INT8)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on the mbarrier at this shared offset in both CTAs of the
// pair when the MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  const uint16_t both = 3;
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
               "h"(both)
               : "memory");
}

// 2-D tiled load into this CTA's shared memory, completing on an mbarrier of
// either CTA of the pair (a shared::cluster address), with an L2 cache
// policy.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t x,
                                                 int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

constexpr int kPairTileP = 2 * kTileP;  // 256 rows of A per pair tile

// Named barrier of the epilogue warps that also reduces a predicate: true
// when it holds in every epilogue thread.
__device__ __forceinline__ bool epi_bar_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kEpiThreads)
      : "memory");
  return r != 0;
}

// One work item of a pair: a whole tile, or one K half of a tile of the
// last round (prm.tail_tiles > 0).  Items [0, tiles - tail) are whole tiles
// in rasterised order; items [tiles - tail, tiles + tail) are the halves of
// the last `tail` tiles -- tail tile j = (item - first) % tail, half =
// (item - first) / tail -- so a tile's two halves run on two pairs in the
// same (last) round.
struct PairItem {
  int tile;      // linear tile id (tile_coords)
  int kb0, kb1;  // K blocks [kb0, kb1)
  int tail;      // index among the split tiles, -1 for a whole tile
  int half;      // 0: K blocks [0, tail_kb_half), 1: the rest
};

__device__ __forceinline__ PairItem pair_item(int w, const MmParams& prm, int tiles) {
  PairItem it;
  const int first = tiles - prm.tail_tiles;
  if (w < first) {
    it.tile = w;
    it.kb0 = 0;
    it.kb1 = prm.num_kb;
    it.tail = -1;
    it.half = 0;
    return it;
  }
  it.tail = (w - first) % prm.tail_tiles;
  it.half = (w - first) / prm.tail_tiles;
  it.tile = first + it.tail;
  it.kb0 = it.half ? prm.tail_kb_half : 0;
  it.kb1 = it.half ? prm.num_kb : prm.tail_kb_half;
  return it;
}

template <int BN, bool INT8, typename OutT>
__global__ void __launch_bounds__(pair_threads(BN, INT8), 1)
    w8a8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                          const MmParams prm, int stages, int group) {
  constexpr int kHalfN = BN / 2;                        // B rows (output columns) per CTA
  constexpr int kQBytes = kHalfN * kRowBytes;
  constexpr int kStageBytes = kPBytes + kQBytes;        // one CTA's share of a stage
  constexpr int kKbElems = INT8 ? 64 : 128;
  constexpr uint32_t kIdesc = make_idesc(kPairTileP, BN, 0);
  constexpr int kBufs = acc_bufs(BN, INT8);
  constexpr int kTmemCols = tmem_cols_for(BN, INT8);
  constexpr int kGroups = BN / 16;
  static_assert(BN % 32 == 0 && BN <= 256, "pair tile width");
  static_assert((INT8 ? kBufs + 1 : kBufs) * BN <= kTmemCols && kTmemCols <= 512, "TMEM");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + stages * kPBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb + stages * kQBytes);
  // bars: full[stages], empty[stages], ufull[2], uempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * stages + 5);
  __shared__ float s_scale_p[kTileP];
  __shared__ float s_scale_q[BN];
  __shared__ bool s_tail_last;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(gridDim.x / 2);
  const int tiles = prm.tiles_p * prm.tiles_q;  // pair tiles: 256 rows x BN columns
  const int items = tiles + prm.tail_tiles;      // work items (whole tiles and K halves)

  auto full_bar = [&](int s) { return smem_addr(bars + s); };
  auto empty_bar = [&](int s) { return smem_addr(bars + stages + s); };
  auto ufull_bar = [&](int b) { return smem_addr(bars + 2 * stages + b); };
  auto uempty_bar = [&](int b) { return smem_addr(bars + 2 * stages + 2 + b); };
  const uint32_t drain_bar = smem_addr(bars + 2 * stages + 4);

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmap_a);
    prefetch_tensormap(&tmap_b);
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_bar(s), 1);   // the leader's expect_tx arrival (+ both CTAs' bytes)
      mbar_init(empty_bar(s), 1);  // the pair MMA's commit
    }
    mbar_init(ufull_bar(0), 1);
    mbar_init(ufull_bar(1), 1);
    // both CTAs' epilogue threads (and drain helpers) release an accumulator
    // (the leader's copy)
    constexpr uint32_t kReleasers = (pair_drain_helpers(BN, INT8) ? 4 : 2) * kEpiThreads;
    mbar_init(uempty_bar(0), kReleasers);
    mbar_init(uempty_bar(1), kReleasers);
    mbar_init(drain_bar, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // the peer's barriers and TMEM exist before either CTA signals the other
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Request the first weight blocks of this CTA's first tile into L2 before
  // waiting on the preceding kernel (a prefetch only reads coherent global
  // memory, whatever that kernel writes), so the weight stream starts while
  // it finishes.
  if (threadIdx.x == 0 && pair < items) {
    const PairItem pi = pair_item(pair, prm, tiles);
    int tp, tq;
    tile_coords(pi.tile, prm.tiles_p, prm.tiles_q, group, tp, tq);
    const int b_row = tq * BN + static_cast<int>(rank) * kHalfN;
    const int kb_pf = min(pi.kb1, pi.kb0 + prm.prefetch_kb);
    for (int i = pi.kb0; i < kb_pf; ++i) tma_prefetch_l2_2d(&tmap_b, i * kKbElems, b_row);
  }
  griddep_launch();
  griddep_wait();

  // the leader's barriers as seen from this CTA
  const uint32_t full0 = mapa_shared(full_bar(0), 0);
  const uint32_t uempty0 = mapa_shared(uempty_bar(0), 0);

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      // token slabs are reused across the weight tiles of a group: kept in
      // L2 ahead of the weights, which stream past once
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_first();
      for (int w = pair; w < items && ok; w += npairs) {
        const PairItem pi = pair_item(w, prm, tiles);
        int tp, tq;
        tile_coords(pi.tile, prm.tiles_p, prm.tiles_q, group, tp, tq);
        const int a_row = tp * kPairTileP + static_cast<int>(rank) * kTileP;
        const int b_row = tq * BN + static_cast<int>(rank) * kHalfN;
        for (int i = pi.kb0; i < pi.kb1; ++i, ++it) {
          const int s = static_cast<int>(it % stages);
          const uint32_t ph = (it / stages) & 1;
          if (!mbar_wait(empty_bar(s), ph ^ 1)) { ok = false; break; }
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * kStageBytes);
          const uint32_t fb = full0 + static_cast<uint32_t>(s) * 8u;
          const int kx = i * kKbElems;
          tma_load_2d_pair(smem_addr(sa + s * kPBytes), &tmap_a, fb, kx, a_row, pol_a);
          tma_load_2d_pair(smem_addr(sb + s * kQBytes), &tmap_b, fb, kx, b_row, pol_b);
        }
      }
      if (!ok && leader) {
        // a wait gave up: let the pair's stage loads in flight land (bounded)
        for (uint32_t j = it > static_cast<uint32_t>(stages) ? it - stages : 0u; j < it; ++j)
          mbar_wait(full_bar(static_cast<int>(j % stages)), (j / stages) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (leader && lane == 0) {
      uint32_t it = 0, c_all = 0;
      bool ok = true;
      for (int w = pair; w < items && ok; w += npairs) {
        const PairItem pi = pair_item(w, prm, tiles);
        const int nkb = pi.kb1 - pi.kb0;
        const int chunk = INT8 ? prm.kchunk_kb : nkb;
        const int nch = (nkb + chunk - 1) / chunk;
        for (int c = 0; c < nch && ok; ++c, ++c_all) {
          const int b = static_cast<int>(c_all % kBufs);
          if (c_all >= static_cast<uint32_t>(kBufs)) {
            // both CTAs' epilogues released it (remote arrivals: acquire at cluster scope)
            if (!mbar_wait_cluster(uempty_bar(b), ((c_all - kBufs) / kBufs) & 1)) { ok = false; break; }
            tc_fence_after();
          }
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
          const int i_begin = pi.kb0 + c * chunk;
          const int i_end = min(pi.kb1, i_begin + chunk);
          for (int i = i_begin; i < i_end; ++i, ++it) {
            const int s = static_cast<int>(it % stages);
            if (!mbar_wait(full_bar(s), (it / stages) & 1)) { ok = false; break; }
            tc_fence_after();
            const uint64_t da = smem_desc_sw128(smem_addr(sa + s * kPBytes));
            const uint64_t db = smem_desc_sw128(smem_addr(sb + s * kQBytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_pair<INT8>(d_tmem, da + 2 * kk, db + 2 * kk, kIdesc, (i == i_begin && kk == 0) ? 0u : 1u);
            mma_commit_pair(empty_bar(s));
          }
          mma_commit_pair(ufull_bar(b));
        }
      }
      if (!ok) {
        // the MMAs already issued finish (bounded) before the TMEM is released
        mma_commit_pair(drain_bar);
        mbar_wait(drain_bar, 0);
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int et = threadIdx.x - 2 * 32;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t c_all = 0;
    bool ok = true;
    for (int w = pair; w < items && ok; w += npairs) {
      const PairItem pi = pair_item(w, prm, tiles);
      int tp, tq;
      tile_coords(pi.tile, prm.tiles_p, prm.tiles_q, group, tp, tq);
      const int p0 = tp * kPairTileP + static_cast<int>(rank) * kTileP;  // this CTA's 128 rows
      const int q0 = tq * BN;
      const int chunk = INT8 ? prm.kchunk_kb : (pi.kb1 - pi.kb0);
      const int nch = (pi.kb1 - pi.kb0 + chunk - 1) / chunk;
      // this CTA's fp32 half of a split tile, 128 rows x BN columns as
      // float4s (row, c4) at c4 * 128 + row: a warp's 32 rows of one float4
      // column are 512 contiguous bytes, written and read whole
      float* const part = pi.tail < 0 ? nullptr
                                      : prm.partial + static_cast<size_t>((pi.tail * 2 + pi.half) * 2 + rank) *
                                                          (kTileP * BN);
      uint32_t tail_acc = 0;  // TMEM address of the half's accumulator (kept for the sum)
      epi_bar_sync();
      s_scale_p[et] = prm.a_per_row ? __ldg(prm.scale_a + min(p0 + et, prm.M - 1)) : __ldg(prm.scale_a);
      for (int i = et; i < BN; i += kEpiThreads)
        s_scale_q[i] = prm.b_per_row ? __ldg(prm.scale_b + min(q0 + i, prm.N - 1)) : __ldg(prm.scale_b);
      epi_bar_sync();
      const float s_lane = s_scale_p[row];
      for (int c = 0; c < nch; ++c, ++c_all) {
        const int b = static_cast<int>(c_all % kBufs);
        if (!mbar_wait(ufull_bar(b), (c_all / kBufs) & 1)) { ok = false; break; }
        tc_fence_after();
        const bool last = (c == nch - 1);
        const uint32_t acc_addr = lane_base + static_cast<uint32_t>(b * BN);
        const uint32_t tot_addr = lane_base + static_cast<uint32_t>(kBufs * BN);
        if constexpr (INT8) {
          constexpr int kBatch = drain_batch(kGroups, 4);
          // with drain helpers an intermediate drain covers the first half
          // of the groups here; the last chunk is drained and stored here
          const int g_end = (pair_drain_helpers(BN, INT8) && !last) ? kGroups / 2 : kGroups;
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
              } else {
                int v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = static_cast<int>(t[bb][j]);
                store16<false, OutT>(prm, p0 + row, q0 + g * 16, g * 16, v, s_lane, s_scale_q);
              }
            }
          }
        } else if (part) {
          // a K half: the raw fp32 accumulator goes to the workspace
          uint4* dst = reinterpret_cast<uint4*>(part) + row;
          tail_acc = acc_addr;
#pragma unroll 1
          for (int g = 0; g < kGroups; ++g) {
            uint32_t r[16];
            tmem_ld16(acc_addr + g * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[(g * 4 + j) * kTileP] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          }
        } else {
#pragma unroll 1
          for (int g = 0; g < kGroups; ++g) {
            uint32_t r[16];
            tmem_ld16(acc_addr + g * 16, r);
            tmem_ld_wait();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
            store16<false, OutT>(prm, p0 + row, q0 + g * 16, g * 16, v, s_lane, s_scale_q);
          }
        }
        if (INT8 && !last) tmem_st_wait();
        // release the accumulator to the leader's MMA issuer; a K half keeps
        // it for the sum below (a pair's K half is its last item: nothing
        // waits for this accumulator any more)
        if (!part) {
          tc_fence_before();
          mbar_arrive_remote(uempty0 + static_cast<uint32_t>(b) * 8u);
        }
      }
      if constexpr (!INT8) {
        // every epilogue thread takes the same path through the barriers
        // below, even if one of them gave up on a wait
        if (part) ok = epi_bar_all(ok);
        if (ok && part) {
          // The second of the tile's two halves (for this CTA's 128 rows) to
          // arrive adds the other half's partial to its own accumulator, in
          // half order from zero -- (0 + half 0) + half 1 -- so the bits do
          // not depend on which pair finished first, and stores the rows as
          // the whole-tile epilogue does.  The other half's loads of a batch
          // are all requested before any is used.
          __threadfence();
          epi_bar_sync();
          if (et == 0) s_tail_last = atomicAdd(prm.counters + pi.tail * 2 + rank, 1u) == 1u;
          epi_bar_sync();
          if (s_tail_last) {
            __threadfence();
            const uint4* other = reinterpret_cast<const uint4*>(
                                     prm.partial + static_cast<size_t>((pi.tail * 2 + (pi.half ^ 1)) * 2 + rank) *
                                                       (kTileP * BN)) +
                                 row;
            constexpr int kB = drain_batch(kGroups, 4);
#pragma unroll 1
            for (int g0 = 0; g0 < kGroups; g0 += kB) {
              uint4 x[kB][4];
              uint32_t r[kB][16];
#pragma unroll
              for (int bb = 0; bb < kB; ++bb)
#pragma unroll
                for (int j = 0; j < 4; ++j) x[bb][j] = __ldcg(other + ((g0 + bb) * 4 + j) * kTileP);
#pragma unroll
              for (int bb = 0; bb < kB; ++bb) tmem_ld16(tail_acc + (g0 + bb) * 16, r[bb]);
              tmem_ld_wait();
#pragma unroll
              for (int bb = 0; bb < kB; ++bb) {
                float v[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const float o[4] = {__uint_as_float(x[bb][j].x), __uint_as_float(x[bb][j].y),
                                      __uint_as_float(x[bb][j].z), __uint_as_float(x[bb][j].w)};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const float mine = __uint_as_float(r[bb][4 * j + e]);
                    const float h0 = pi.half == 0 ? mine : o[e];
                    const float h1 = pi.half == 0 ? o[e] : mine;
                    v[4 * j + e] = (0.f + h0) + h1;
                  }
                }
                const int g = g0 + bb;
                store16<false, OutT>(prm, p0 + row, q0 + g * 16, g * 16, v, s_lane, s_scale_q);
              }
            }
            if (et == 0) prm.counters[pi.tail * 2 + rank] = 0u;
          }
        }
      }
    }
  } else if constexpr (pair_drain_helpers(BN, INT8)) {
    // ------------------------------------------------------ drain helpers
    // The epilogue's chunk sequence; each intermediate drain adds the second
    // half of the columns into the int32 total, the last chunk only releases.
    const int quarter = warp & 3;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr int kBatch = drain_batch(kGroups, 4);
    uint32_t c_all = 0;
    bool ok = true;
    for (int w = pair; w < items && ok; w += npairs) {
      const int chunk = prm.kchunk_kb;
      const int nch = (prm.num_kb + chunk - 1) / chunk;  // int8 items are whole tiles
      for (int c = 0; c < nch; ++c, ++c_all) {
        const int b = static_cast<int>(c_all % kBufs);
        if (!mbar_wait(ufull_bar(b), (c_all / kBufs) & 1)) { ok = false; break; }
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
        mbar_arrive_remote(uempty0 + static_cast<uint32_t>(b) * 8u);
      }
    }
  }

  tc_fence_before();
  // neither CTA leaves (nor frees the pair's TMEM) while its peer may still
  // read its shared memory or signal its barriers
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int BN, bool INT8, typename OutT>
cudaError_t launch_pair_t(const CUtensorMap& ta, const CUtensorMap& tb, const MmParams& p, int stages,
                          cudaStream_t stream) {
  auto kern = w8a8_gemm_pair_kernel<BN, INT8, OutT>;
  const int smem = stages * (kPBytes + (BN / 2) * kRowBytes) + 1024 + kBarBlockBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  const int npairs = pair_grid_pairs(static_cast<long long>(p.tiles_p) * p.tiles_q, p.num_sms);
  // rasterisation: groups of 256-row token slabs that fit in 48 MB of L2
  const long long slab = static_cast<long long>(kPairTileP) * p.K * (INT8 ? 2 : 1);
  long long g_tiles = (48LL << 20) / slab;
  if (g_tiles > p.tiles_p) g_tiles = p.tiles_p;
  if (g_tiles < 1) g_tiles = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * npairs);
  cfg.blockDim = dim3(pair_threads(BN, INT8));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int na = 1;
  if (p.pdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  e = cudaLaunchKernelEx(&cfg, kern, ta, tb, p, stages, static_cast<int>(g_tiles));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BN, bool INT8>
cudaError_t launch_pair_out(const CUtensorMap& ta, const CUtensorMap& tb, const MmParams& p, int out_kind, int stages,
                            cudaStream_t stream) {
  switch (out_kind) {
    case OUT_BF16: return launch_pair_t<BN, INT8, __nv_bfloat16>(ta, tb, p, stages, stream);
    case OUT_FP16: return launch_pair_t<BN, INT8, __half>(ta, tb, p, stages, stream);
    case OUT_RAW:
      if (INT8) return launch_pair_t<BN, INT8, int>(ta, tb, p, stages, stream);
      return launch_pair_t<BN, INT8, float>(ta, tb, p, stages, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int gemm_pair_smem_bytes(int block_n, int stages) {
  return stages * (kPBytes + (block_n / 2) * kRowBytes) + 1024 + kBarBlockBytes;
}

cudaError_t launch_gemm_pair(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const MmParams& p, int block_n,
                             bool int8, int out_kind, int stages, cudaStream_t stream) {
  if (int8) {
    switch (block_n) {
      case 256: return launch_pair_out<256, true>(tmap_a, tmap_b, p, out_kind, stages, stream);
      case 128: return launch_pair_out<128, true>(tmap_a, tmap_b, p, out_kind, stages, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (block_n) {
    case 256: return launch_pair_out<256, false>(tmap_a, tmap_b, p, out_kind, stages, stream);
    case 224: return launch_pair_out<224, false>(tmap_a, tmap_b, p, out_kind, stages, stream);
    case 192: return launch_pair_out<192, false>(tmap_a, tmap_b, p, out_kind, stages, stream);
    case 128: return launch_pair_out<128, false>(tmap_a, tmap_b, p, out_kind, stages, stream);
    case 96: return launch_pair_out<96, false>(tmap_a, tmap_b, p, out_kind, stages, stream);
    case 64: return launch_pair_out<64, false>(tmap_a, tmap_b, p, out_kind, stages, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w8a8
