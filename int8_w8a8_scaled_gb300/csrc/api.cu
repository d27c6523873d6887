// api.cu -- the C ABI (include/w8a8.h): argument validation, kernel
// configuration, TMA tensor maps and launches.  No call allocates device
// memory or synchronises the stream; every call returns a status and leaves a
// message for w8a8_last_error() on failure.
//
// Input validation instead of assertions follows the review of "[Kernel] Add
// w8a8 CUTLASS kernels" (no input may crash the caller; a B that is not
// column-major used to end in "misaligned address" -- here it is a status).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <mutex>
#include <string>

#include "../../include/w8a8.h"
#include "internal.h"

using namespace w8a8;

namespace {

thread_local std::string t_last_error;

// debug trace target (process-wide; set and read on the host only)
std::atomic<unsigned long long*> g_trace_buf{nullptr};
std::atomic<int> g_trace_ctas{0};

w8a8_status fail(w8a8_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

w8a8_status ok() {
  t_last_error.clear();
  return W8A8_OK;
}

w8a8_status cuda_fail(cudaError_t e, const char* what) {
  return fail(W8A8_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------------ device info

struct DeviceInfo {
  bool ready = false;
  int major = 0, minor = 0, sms = 0, smem_optin = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

w8a8_status device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(W8A8_ERR_NO_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.ready = true;
  }
  if (d.major != 10 || d.minor != 3)
    return fail(W8A8_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                d.major, d.minor);
  *out = d;
  return W8A8_OK;
}

// ------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D K-major operand [rows, K] (row stride ld_bytes), box of box_rows rows x
// 128 bytes, 128-byte swizzle, zero fill outside the tensor.
w8a8_status make_operand_map(CUtensorMap* map, const void* base, bool f16, long long rows, long long K,
                             long long ld_bytes, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(W8A8_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_bytes)};
  const cuuint32_t box[2] = {f16 ? 64u : 128u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(W8A8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return W8A8_OK;
}

// ------------------------------------------------------------------ GEMM configuration

// SM count of the current device; without a usable device (host-only size
// queries) a GB300's 152.
int sms_or_default() {
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
    else cudaGetLastError();
  } else {
    cudaGetLastError();
  }
  return sms;
}

// CTA-pair tiles with split_k 2: the tiles of the last, partial round of
// pairs are split into two K halves when that round would otherwise keep at
// most half of the pairs busy -- the halves then fill at most all of them and
// the round takes about half as long (e4m3; at least two K blocks).
int pair_tail_tiles(long long tiles, int kb, int sms, int split_k, int q_dtype) {
  if (split_k != 2 || q_dtype != W8A8_E4M3 || kb < 2) return 0;
  const long long pairs = pair_grid_pairs(tiles, sms);
  const long long rem = tiles % pairs;
  return (rem > 0 && 2 * rem <= pairs) ? static_cast<int>(rem) : 0;
}

constexpr int kSmemTwoPerSm = 113 * 1024;   // budget that lets two CTAs share an SM
constexpr int kInt8ChunkK = 1024;           // exact fp32 accumulation bound: 1024 * 128 * 128 = 2^24
constexpr long long kFusedRowsMaxBytes = 32768;  // one-kernel quant_scaled_mm: rows staged in shared memory
constexpr long long kPairMinM = 1024;            // e4m3 tokens from which CTA-pair tiles are used

bool valid_block_n(int bn, int q_dtype, int swap_ab) {
  if (bn == 16 || bn == 32 || bn == 64 || bn == 128) return true;
  if (q_dtype == W8A8_INT8) return (bn == 160 || bn == 256) && !swap_ab;
  if (bn == 256) return true;
  return !swap_ab && (bn == 160 || bn == 192 || bn == 224);
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

int num_kb(long long K, int q_dtype) { return static_cast<int>(ceil_div(K, q_dtype == W8A8_INT8 ? 64 : 128)); }

// Automatic configuration, fitted to the decode and prefill sweeps of
// `bench.py --sweep-decode / --sweep-large` on GB300:
//  - M <= 64: weights on the 128-row MMA side (swap), block_n the smallest of
//    16 / 32 / 64 that holds all M tokens -- one token tile, so every weight
//    byte crosses L2 once, and two CTAs resident per SM -- except for
//    32 < M <= 64 with enough weight tiles to fill the GPU unsplit (the
//    gate-up projection), where tokens on the 128-row side win (22.8 us
//    against 25.5 us at M = 64);
//  - M > 64: tokens on the 128-row side, the widest block_n in {256, 128, 64}
//    that still gives >= 0.6 tiles per SM;
//  - split-K: the largest power of two of K slices that fits one wave of
//    resident CTAs (<= slots / tiles), at least 4 K blocks per slice, at
//    most 8 (one portable cluster: the slices reduce through distributed
//    shared memory).  More waves or wider splits lose to the fixed cost of
//    each unit and of the reduction.
int one_wave_split(long long tiles, int kb, long long slots) {
  long long sp = slots / std::max<long long>(1, tiles);
  sp = std::min<long long>(sp, std::max(1, kb / 4));
  sp = std::min<long long>(sp, 8);
  // a power of two: clusters of 3, 5, 6 or 7 CTAs co-schedule poorly (the
  // decode sweep measured 6 slices of a 48-tile QKV at 13 us against 8.2 us
  // for 4)
  long long p2 = 1;
  while (p2 * 2 <= sp) p2 *= 2;
  return static_cast<int>(p2);
}

int resident_per_sm(int block_n, int q_dtype) {
  (void)q_dtype;
  return block_n <= 64 ? 2 : 1;
}

void auto_config(long long M, long long N, long long K, int q_dtype, int sms, w8a8_mm_config* c) {
  const int kb = num_kb(K, q_dtype);
  const long long slots2 = 2LL * sms;  // resident narrow-tile CTAs
  if (M <= 64 && !(M > 32 && ceil_div(N, 128) * 2 >= slots2)) {
    // all tokens in one narrow tile: the weights stream through L2 once
    c->swap_ab = 1;
    c->block_n = M <= 16 ? 16 : M <= 32 ? 32 : 64;
  } else {
    c->swap_ab = 0;
    if (q_dtype == W8A8_INT8) {
      // 256 columns (one fp32 chunk accumulator + the int32 total fill TMEM)
      // measured 939-979 TFLOP/s at the 70B shapes vs ~600-800 at 128
      c->block_n = 64;
      for (int bn = 256; bn >= 64; bn /= 2) {
        if (ceil_div(M, 128) * ceil_div(N, bn) * 10 >= 6LL * sms) {
          c->block_n = bn;
          break;
        }
      }
    } else {
      // widest tile first; prefer a narrower one only when it balances the
      // persistent waves clearly better (a wave of width-w tiles costs ~w)
      const int cands[5] = {256, 224, 192, 160, 128};
      double best = 1e30;
      c->block_n = 64;
      for (int i = 0; i < 5; ++i) {
        const int bn = cands[i];
        const long long tiles = ceil_div(M, 128) * ceil_div(N, bn);
        if (tiles * 10 < 6LL * sms) continue;
        const long long waves = (tiles + sms - 1) / sms;
        // time ~ waves * bn / efficiency(bn); narrower tiles lose a little
        // per-flop efficiency (operand re-reads), modelled as 3 % per step
        const double t = static_cast<double>(waves) * bn * (1.0 + 0.03 * i) /
                         static_cast<double>(std::min<long long>(N, ceil_div(N, bn) * bn));
        if (t < best - 1e-12) {
          best = t;
          c->block_n = bn;
        }
      }
    }
  }
  // few token tiles and a long K (the decode down projection, K = 14336 at
  // M = 256): the widest tile split over K beats narrow tiles, which re-read
  // every activation K block once per 64 output columns (sweep: 25.4 us for
  // 256 x 4 slices against 30.1 us for 64 x 2; in the decode step it also
  // beat all 256 tokens in one swap-AB tile, 28.2 against 31.4 us)
  if (!c->swap_ab && q_dtype == W8A8_E4M3 && M <= 256 && K >= 8192) c->block_n = 256;
  c->stages = 0;
  c->ctas_per_sm = 0;
  c->reduce = W8A8_REDUCE_AUTO;
  c->cta_pair = 0;
  // Large-M e4m3: 256 x block_n tiles on CTA pairs (each SM stages half of
  // B).  Measured at M = 4096 on the Llama-3-8B projections: 2438 / 2368 /
  // 3094 / 2751 TFLOP/s (QKV / O / gate-up / down) against 2326 / 2227 /
  // 2837 / 2599 on one-CTA tiles.  int8 stays on one-CTA tiles: its chunk
  // drains stall both CTAs of a pair (942-979 against 949-1003).
  // block_n: a round of pair tiles takes the same time at 192-256 columns
  // (its stages are bound by the operand round trip, not by the MMA width:
  // 256 and 224 columns measured 84.6 / 84.4 us for QKV, 58.0 / 58.0 O,
  // 174.8 / 174.4 down, all in six, four and four rounds), so the model
  // counts rounds; a last round that keeps at most half of the pairs busy
  // runs as K halves (split_k 2) and costs half a round plus the exchange
  // of the halves, measured at about 8 us, 20 K blocks' worth (so only long
  // K gains: the down projection 166.6 against 174.4-176.5 us; QKV and O
  // at K = 4096 measured even, 84.7 / 59.8 against 84.8 / 59.6).
  if (!c->swap_ab && q_dtype == W8A8_E4M3 && M >= kPairMinM) {
    const int cands[3] = {256, 224, 192};
    double best = 1e30;
    for (int i = 0; i < 3; ++i) {
      const int bn = cands[i];
      const long long tiles = ceil_div(M, 256) * ceil_div(N, bn);
      const long long pairs = pair_grid_pairs(tiles, sms);
      const long long full = tiles / pairs;
      const long long rem = tiles % pairs;
      const bool halves = pair_tail_tiles(tiles, kb, sms, 2, q_dtype) > 0 && 0.5 + 20.0 / kb < 1.0;
      // equal rounds: the narrower tile (less padding work, measured 84.8 /
      // 59.6 us at 224 against 85.7 / 59.9 at 256 for QKV / O)
      const double t =
          static_cast<double>(full) + (rem == 0 ? 0.0 : halves ? 0.5 + 20.0 / kb : 1.0) + 1e-3 * bn / 256;
      if (t < best - 1e-9) {
        best = t;
        c->block_n = bn;
        c->split_k = halves ? 2 : 1;
      }
    }
    c->cta_pair = 1;
    return;
  }
  const long long tiles = c->swap_ab ? ceil_div(N, 128) * ceil_div(M, c->block_n)
                                     : ceil_div(M, 128) * ceil_div(N, c->block_n);
  c->split_k = one_wave_split(tiles, kb, static_cast<long long>(sms) * resident_per_sm(c->block_n, q_dtype));
}

int auto_stages(int block_n, int q_dtype, int smem_optin) {
  const int budget = resident_per_sm(block_n, q_dtype) == 2 ? kSmemTwoPerSm : smem_optin;
  return std::max(2, std::min(8, max_stages_for(block_n, budget)));
}

// CTA-pair tiles: each CTA stages 128 rows of A and block_n / 2 of B per stage.
int auto_pair_stages(int block_n, int smem_optin) {
  int s = 8;
  while (s > 2 && gemm_pair_smem_bytes(block_n, s) > smem_optin) --s;
  return s;
}

struct Plan {
  w8a8_mm_config cfg;
  int kb, kb_per_split, splits, tiles_p, tiles_q, stages;
  bool cluster;    // split slices reduce through distributed shared memory
  int tail_tiles;  // CTA-pair tiles of the last round run as two K halves
  size_t off_counters, off_partial, off_a16, off_b16, total;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace layout.  The split-K arrival counters live in a fixed region at
// the head of every workspace (kCounterRegion) and nothing else is ever
// written there: each call that uses them leaves them zero, so a zero-filled
// workspace stays valid across calls of any shape and configuration (scratch
// data -- split-K partials, int8 f16 planes -- always lives after the region).

Plan make_plan(long long M, long long N, long long K, int q_dtype, const w8a8_mm_config& cfg, int smem_optin,
               int sms) {
  Plan p{};
  p.cfg = cfg;
  p.kb = num_kb(K, q_dtype);
  const long long P = cfg.swap_ab ? N : M;
  const long long Q = cfg.swap_ab ? M : N;
  p.tiles_p = static_cast<int>(ceil_div(P, cfg.cta_pair ? 256 : 128));
  p.tiles_q = static_cast<int>(ceil_div(Q, cfg.block_n));
  // CTA pairs take split_k only as the last round's K halves
  int sp = cfg.cta_pair ? 1 : std::max(1, std::min(cfg.split_k, p.kb));
  p.kb_per_split = static_cast<int>(ceil_div(p.kb, sp));
  p.splits = static_cast<int>(ceil_div(p.kb, p.kb_per_split));  // every slice non-empty
  p.stages = cfg.stages > 0 ? cfg.stages
                            : (cfg.cta_pair ? auto_pair_stages(cfg.block_n, smem_optin)
                                            : auto_stages(cfg.block_n, q_dtype, smem_optin));
  p.cluster = p.splits > 1 && cfg.reduce != W8A8_REDUCE_GLOBAL && p.splits <= kMaxClusterSplit;
  const size_t tiles = static_cast<size_t>(p.tiles_p) * p.tiles_q;
  p.tail_tiles = cfg.cta_pair ? pair_tail_tiles(static_cast<long long>(tiles), p.kb, sms, cfg.split_k, q_dtype) : 0;
  const bool need_ws = p.splits > 1 || p.tail_tiles > 0 || q_dtype == W8A8_INT8;
  size_t off = need_ws ? kCounterRegion : 0;
  p.off_counters = 0;
  if (p.splits > 1) {
    p.off_partial = off;
    off = align256(off + tiles * p.splits * 128 * cfg.block_n * sizeof(float));
  }
  if (p.tail_tiles > 0) {
    // [tail][half][rank] partial tiles of 128 x block_n fp32
    p.off_partial = off;
    off = align256(off + static_cast<size_t>(p.tail_tiles) * 4 * 128 * cfg.block_n * sizeof(float));
  }
  if (q_dtype == W8A8_INT8) {
    p.off_a16 = off;
    off = align256(off + static_cast<size_t>(M) * K * 2);
    p.off_b16 = off;
    off = align256(off + static_cast<size_t>(N) * K * 2);
  }
  p.total = off;
  return p;
}

w8a8_status validate_config(const w8a8_mm_config& c, int q_dtype, int smem_optin) {
  if (c.swap_ab != 0 && c.swap_ab != 1) return fail(W8A8_ERR_UNSUPPORTED, "swap_ab must be 0 or 1");
  if (!c.cta_pair && !valid_block_n(c.block_n, q_dtype, c.swap_ab))
    return fail(W8A8_ERR_UNSUPPORTED,
                "block_n %d not supported (16, 32, 64, 128, 256; 160/192/224 for e4m3 without swap; 160/256 for int8 without swap)",
                c.block_n);
  if (c.split_k < 1 || c.split_k > 16) return fail(W8A8_ERR_UNSUPPORTED, "split_k must be in [1, 16]");
  if (c.stages != 0 && (c.stages < 2 || c.stages > 8))
    return fail(W8A8_ERR_UNSUPPORTED, "stages must be 0 (auto) or in [2, 8]");
  if (c.ctas_per_sm < 0 || c.ctas_per_sm > 4)
    return fail(W8A8_ERR_UNSUPPORTED, "ctas_per_sm must be 0 (auto) or in [1, 4]");
  if (c.reduce < W8A8_REDUCE_AUTO || c.reduce > W8A8_REDUCE_CLUSTER)
    return fail(W8A8_ERR_UNSUPPORTED, "reduce must be W8A8_REDUCE_AUTO, _GLOBAL or _CLUSTER");
  const int st = c.stages > 0 ? c.stages : auto_stages(c.block_n, q_dtype, smem_optin);
  if (!c.cta_pair && gemm_smem_bytes(c.block_n, st) > smem_optin)
    return fail(W8A8_ERR_UNSUPPORTED, "stages=%d with block_n=%d needs %d bytes of shared memory (> %d)", st,
                c.block_n, gemm_smem_bytes(c.block_n, st), smem_optin);
  if (c.reduce == W8A8_REDUCE_CLUSTER && c.split_k > kMaxClusterSplit)
    return fail(W8A8_ERR_UNSUPPORTED, "the cluster reduction takes split_k <= %d", kMaxClusterSplit);
  if (c.cta_pair != 0 && c.cta_pair != 1) return fail(W8A8_ERR_UNSUPPORTED, "cta_pair must be 0 or 1");
  if (c.cta_pair) {
    if (c.swap_ab || c.split_k < 1 || c.split_k > (q_dtype == W8A8_E4M3 ? 2 : 1))
      return fail(W8A8_ERR_UNSUPPORTED,
                  "CTA-pair tiles take swap_ab = 0 and split_k = 1 (e4m3: or 2, the last round's tiles in K halves)");
    const bool bn_ok = q_dtype == W8A8_INT8 ? (c.block_n == 128 || c.block_n == 256)
                                            : (c.block_n == 64 || c.block_n == 96 || c.block_n == 128 ||
                                               c.block_n == 192 || c.block_n == 224 || c.block_n == 256);
    if (!bn_ok)
      return fail(W8A8_ERR_UNSUPPORTED,
                  "CTA-pair tiles take block_n 64, 96, 128, 192, 224 or 256 (int8: 128 or 256)");
    const int ps = c.stages > 0 ? c.stages : auto_pair_stages(c.block_n, smem_optin);
    if (gemm_pair_smem_bytes(c.block_n, ps) > smem_optin)
      return fail(W8A8_ERR_UNSUPPORTED, "stages=%d with block_n=%d needs more shared memory than a CTA has", ps,
                  c.block_n);
  }
  return W8A8_OK;
}

w8a8_status validate_mm(const void* a_q, long long lda, const void* b_q, long long ldb, const float* sa,
                        int a_gran, const float* sb, int b_gran, void* out, long long ldc, long long M,
                        long long N, long long K, int q_dtype, int out_dtype) {
  if (!a_q || !b_q || !sa || !sb || !out) return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
  if (q_dtype != W8A8_E4M3 && q_dtype != W8A8_INT8)
    return fail(W8A8_ERR_INVALID_ARG, "q_dtype must be W8A8_E4M3 or W8A8_INT8");
  if (out_dtype != W8A8_BF16 && out_dtype != W8A8_FP16 && out_dtype != W8A8_FP32 && out_dtype != W8A8_INT32)
    return fail(W8A8_ERR_INVALID_ARG, "out_dtype must be BF16, FP16, FP32 or INT32");
  if ((out_dtype == W8A8_FP32 && q_dtype != W8A8_E4M3) || (out_dtype == W8A8_INT32 && q_dtype != W8A8_INT8))
    return fail(W8A8_ERR_UNSUPPORTED, "FP32 output is for e4m3 operands and INT32 output for int8 operands");
  if ((a_gran != W8A8_PER_TENSOR && a_gran != W8A8_PER_ROW) || (b_gran != W8A8_PER_TENSOR && b_gran != W8A8_PER_ROW))
    return fail(W8A8_ERR_INVALID_ARG, "granularity must be W8A8_PER_TENSOR or W8A8_PER_ROW");
  if (M < 1 || N < 1 || K < 1) return fail(W8A8_ERR_INVALID_ARG, "M, N, K must be >= 1 (got %lld, %lld, %lld)", M, N, K);
  if (M >= (1LL << 31) || N >= (1LL << 31) || K >= (1LL << 31))
    return fail(W8A8_ERR_UNSUPPORTED, "M, N, K must be < 2^31");
  if (lda < K || ldb < K) return fail(W8A8_ERR_INVALID_ARG, "lda and ldb must be >= K (%lld)", K);
  if (ldc < N) return fail(W8A8_ERR_INVALID_ARG, "ldc must be >= N (%lld)", N);
  if (q_dtype == W8A8_INT8 && K > 131071)
    return fail(W8A8_ERR_UNSUPPORTED, "int8 needs K <= 131071 so that int32 cannot overflow");
  if (q_dtype == W8A8_INT8 && K % 16 != 0) return fail(W8A8_ERR_UNSUPPORTED, "int8 needs K to be a multiple of 16");
  if (!aligned(a_q, 16) || !aligned(b_q, 16))
    return fail(W8A8_ERR_MISALIGNED, "A and B must be 16-byte aligned (B must be stored [N, K], K contiguous)");
  if (lda % 16 != 0 || ldb % 16 != 0)
    return fail(W8A8_ERR_MISALIGNED, "lda and ldb must be multiples of 16 bytes (got %lld, %lld)", lda, ldb);
  if (!aligned(out, out_dtype >= W8A8_FP32 ? 4 : 2)) return fail(W8A8_ERR_MISALIGNED, "out is not element-aligned");
  if (!aligned(sa, 4) || !aligned(sb, 4)) return fail(W8A8_ERR_MISALIGNED, "scales must be 4-byte aligned");
  return W8A8_OK;
}

// Whether a cluster split keeps its partial tiles in the CTAs' shared memory
// and sums them through distributed shared memory: a 128 x block_n fp32 tile
// (rows padded by 16 bytes) must fit the stage ring, which is idle once the
// CTA's single unit is accumulated.  Only with tokens on the 128-row side:
// there a lane drains whole tile rows and the final sum walks along rows
// (measured at M = 256: the down projection 28.0 -> 23.6 us, O 14.8 -> 13.5
// us); the swap-AB decode tiles, whose final sum walks down the rows, were
// slower that way (M = 64 QKV 10.8 -> 13.9 us) and keep the L2 reduction.
bool dsmem_reduce_fits(const Plan& plan, int block_n, int stages) {
  if (!plan.cluster || plan.splits < 2 || plan.cfg.swap_ab) return false;
  const long long ring = static_cast<long long>(gemm_smem_bytes(block_n, stages)) - gemm_smem_bytes(block_n, 0);
  return ring >= 128LL * (block_n + 4) * 4;
}

// Activations the matmul quantises itself (dynamic per token, e4m3).
struct FusedAct {
  const void* x;
  long long ld_x;
  int x_fp16;
  float* scale_out;
};

// Whether the decode matmul can quantise its own activations under `cfg`:
// e4m3, swap-AB with every token in one tile, and K slices that one CTA or
// one cluster covers (the per-token absmax needs the whole row).
bool fused_quant_ok(const w8a8_mm_config& cfg, long long M, long long K, int q_dtype) {
  if (q_dtype != W8A8_E4M3 || !cfg.swap_ab || cfg.block_n > 64 || M > cfg.block_n || K % 16 != 0) return false;
  return cfg.split_k == 1 || (cfg.split_k <= kMaxClusterSplit && cfg.reduce != W8A8_REDUCE_GLOBAL);
}

// Whether w8a8_quant_scaled_mm's automatic route takes the one-kernel path.
// Measured on GB300 in the Llama-3-8B decode step, the one kernel is slower
// than quantiser + matmul even at M = 1: it removes the quantiser's launch
// and kernel boundary (2-4 us) but its own start -- the token scales (with a
// cluster exchange under split-K) and the first token stage written by the
// epilogue warps -- costs 4.6-9 us from the dependency release to the first
// MMA, against 1.5-2.3 us for a matmul whose codes arrive by TMA.  So the
// automatic route is the two-step one; the one-kernel route is there on
// request (W8A8_ROUTE_ONE_KERNEL).
bool fused_quant_preferred(const w8a8_mm_config&, long long, long long, int) { return false; }

w8a8_status run_mm(const void* a_q, long long lda, const void* b_q, long long ldb, const float* sa, int a_gran,
                   const float* sb, int b_gran, void* out, long long ldc, long long M, long long N, long long K,
                   int q_dtype, int out_dtype, void* ws, size_t ws_bytes, const w8a8_mm_config* user_cfg,
                   cudaStream_t stream, const FusedAct* fa = nullptr) {
  // with fused activations the A operand is x (validated by the caller): give
  // the operand checks a stand-in that passes them
  static const uint4 kAligned = {};
  w8a8_status st = validate_mm(fa ? static_cast<const void*>(&kAligned) : a_q, fa ? K : lda, b_q, ldb,
                               fa ? reinterpret_cast<const float*>(&kAligned) : sa, fa ? W8A8_PER_ROW : a_gran, sb,
                               b_gran, out, ldc, M, N, K, q_dtype, out_dtype);
  if (st != W8A8_OK) return st;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != W8A8_OK) return st;
  w8a8_mm_config cfg;
  if (user_cfg) {
    cfg = *user_cfg;
    w8a8_mm_config a;
    auto_config(M, N, K, q_dtype, dev.sms, &a);
    if (cfg.block_n == 0) cfg.block_n = a.block_n;
    if (cfg.split_k == 0)
      cfg.split_k = cfg.cta_pair ? (a.cta_pair && a.block_n == cfg.block_n ? a.split_k : 1) : a.split_k;
  } else {
    auto_config(M, N, K, q_dtype, dev.sms, &cfg);
  }
  if ((st = validate_config(cfg, q_dtype, dev.smem_optin)) != W8A8_OK) return st;
  if (fa && !fused_quant_ok(cfg, M, K, q_dtype))
    return fail(W8A8_ERR_UNSUPPORTED, "this configuration cannot quantise the activations inside the matmul");
  const Plan plan = make_plan(M, N, K, q_dtype, cfg, dev.smem_optin, dev.sms);
  if (plan.splits > 1 && !plan.cluster && static_cast<size_t>(plan.tiles_p) * plan.tiles_q > kCounterSlots)
    return fail(W8A8_ERR_UNSUPPORTED, "split_k > 1 supports at most %zu output tiles (got %d)", kCounterSlots,
                plan.tiles_p * plan.tiles_q);
  if (plan.total > 0) {
    if (!ws) return fail(W8A8_ERR_WORKSPACE, "this problem needs %zu bytes of workspace", plan.total);
    if (ws_bytes < plan.total)
      return fail(W8A8_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, plan.total);
    if (!aligned(ws, 256)) return fail(W8A8_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  }
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  const bool i8 = (q_dtype == W8A8_INT8);
  const void* a_op = a_q;
  const void* b_op = b_q;
  long long lda_b = lda, ldb_b = ldb;
  cudaError_t e;
  if (i8) {
    // exact int8 -> f16 widening of both operands into the workspace
    if ((e = launch_int8_widen(a_q, lda, static_cast<int>(M), static_cast<int>(K), wsb + plan.off_a16, stream)) !=
        cudaSuccess)
      return cuda_fail(e, "int8 widen (A) launch");
    if ((e = launch_int8_widen(b_q, ldb, static_cast<int>(N), static_cast<int>(K), wsb + plan.off_b16, stream)) !=
        cudaSuccess)
      return cuda_fail(e, "int8 widen (B) launch");
    a_op = wsb + plan.off_a16;
    b_op = wsb + plan.off_b16;
    lda_b = K * 2;
    ldb_b = K * 2;
  }
  CUtensorMap tp, tq;
  const void* p_base = cfg.swap_ab ? b_op : a_op;
  const void* q_base = cfg.swap_ab ? a_op : b_op;
  const long long p_rows = cfg.swap_ab ? N : M;
  const long long q_rows = cfg.swap_ab ? M : N;
  const long long p_ld = cfg.swap_ab ? ldb_b : lda_b;
  const long long q_ld = cfg.swap_ab ? lda_b : ldb_b;
  if ((st = make_operand_map(&tp, p_base, i8, p_rows, K, p_ld, 128)) != W8A8_OK) return st;
  if (!fa && (st = make_operand_map(&tq, q_base, i8, q_rows, K, q_ld, cfg.cta_pair ? cfg.block_n / 2 : cfg.block_n)) !=
                 W8A8_OK)
    return st;

  MmParams prm{};
  prm.M = static_cast<int>(M);
  prm.N = static_cast<int>(N);
  prm.K = static_cast<int>(K);
  prm.tiles_p = plan.tiles_p;
  prm.tiles_q = plan.tiles_q;
  prm.num_kb = plan.kb;
  prm.kb_per_split = plan.kb_per_split;
  prm.splits = plan.splits;
  prm.scale_a = sa;
  prm.a_per_row = (a_gran == W8A8_PER_ROW);
  prm.scale_b = sb;
  prm.b_per_row = (b_gran == W8A8_PER_ROW);
  prm.out = out;
  prm.ldc = ldc;
  const long long out_elem = out_dtype >= W8A8_FP32 ? 4 : 2;
  prm.out_vec_ok = aligned(out, 16) && ((ldc * out_elem) % 16 == 0);
  prm.cluster = plan.cluster ? 1 : 0;
  prm.partial = plan.splits > 1 ? reinterpret_cast<float*>(wsb + plan.off_partial) : nullptr;
  prm.counters = plan.splits > 1 && !plan.cluster ? reinterpret_cast<unsigned*>(wsb + plan.off_counters) : nullptr;
  prm.kchunk_kb = kInt8ChunkK / 64;
  prm.num_sms = dev.sms;
  if (plan.tail_tiles > 0) {
    prm.tail_tiles = plan.tail_tiles;
    prm.tail_kb_half = plan.kb / 2;
    prm.partial = reinterpret_cast<float*>(wsb + plan.off_partial);
    prm.counters = reinterpret_cast<unsigned*>(wsb + plan.off_counters);
  }
  prm.pdl = 1;
  // up to 256 KB of each CTA's first weight slice (16 KB per K block of 128
  // weight rows)
  prm.prefetch_kb = 16;
  prm.max_ctas_per_sm = cfg.ctas_per_sm;
  prm.trace = g_trace_buf.load();
  prm.trace_ctas = g_trace_ctas.load();
  const int out_kind = out_dtype == W8A8_BF16 ? OUT_BF16 : out_dtype == W8A8_FP16 ? OUT_FP16 : OUT_RAW;
  if (fa) {
    prm.scale_a = nullptr;
    prm.x = fa->x;
    prm.ld_x = fa->ld_x;
    prm.x_fp16 = fa->x_fp16;
    prm.scale_a_out = fa->scale_out;
    // rows mode: the tokens' whole rows (<= 32 KB) go to shared memory once,
    // at the cost of stages where the budget requires it
    int stages = plan.stages;
    const long long x_bytes = M * K * 2;
    if (x_bytes <= kFusedRowsMaxBytes) {
      const int budget = resident_per_sm(cfg.block_n, q_dtype) == 2 ? kSmemTwoPerSm : dev.smem_optin;
      const int stage_bytes = gemm_smem_bytes(cfg.block_n, 2) - gemm_smem_bytes(cfg.block_n, 1);
      const int fit = (budget - static_cast<int>(x_bytes) - gemm_smem_bytes(cfg.block_n, 0)) / stage_bytes;
      if (fit >= 2) {
        prm.fq_rows = 1;
        stages = std::min(stages, fit);
      }
    }
    prm.dsmem_reduce = dsmem_reduce_fits(plan, cfg.block_n, stages);
    e = launch_fused_quant_gemm(tp, prm, cfg.block_n, out_kind, stages, stream);
  } else {
    prm.dsmem_reduce = dsmem_reduce_fits(plan, cfg.block_n, plan.stages);
    if (cfg.cta_pair)
      e = launch_gemm_pair(tp, tq, prm, cfg.block_n, i8, out_kind, plan.stages, stream);
    else
      e = i8 ? launch_int8_gemm(tp, tq, prm, cfg.block_n, cfg.swap_ab != 0, out_kind, plan.stages, stream)
           : launch_fp8_gemm(tp, tq, prm, cfg.block_n, cfg.swap_ab != 0, out_kind, plan.stages, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "scaled_mm kernel launch");
  return ok();
}

}  // namespace

void w8a8::set_last_error(const char* msg) { t_last_error = msg ? msg : ""; }

size_t w8a8::mm_counter_bytes(long long M, long long N, long long K, int q_dtype, const w8a8_mm_config& cfg) {
  DeviceInfo dev;
  if (device_info(&dev) != W8A8_OK) return kCounterRegion;  // unknown: the whole region
  const Plan plan = make_plan(M, N, K, q_dtype, cfg, dev.smem_optin, dev.sms);
  if (plan.tail_tiles > 0) return static_cast<size_t>(plan.tail_tiles) * 2 * sizeof(unsigned);
  if (plan.splits <= 1 || plan.cluster) return 0;
  return std::min(kCounterRegion, static_cast<size_t>(plan.tiles_p) * plan.tiles_q * sizeof(unsigned));
}

extern "C" {

const char* w8a8_last_error(void) { return t_last_error.c_str(); }

int w8a8_version(void) { return 100; }

size_t w8a8_scaled_quant_workspace_size(int64_t rows, int64_t cols, int gran, int mode) {
  (void)rows;
  (void)cols;
  return (gran == W8A8_PER_TENSOR && mode == W8A8_DYNAMIC) ? 16 : 0;
}

w8a8_status w8a8_scaled_quant(const void* x, int x_dtype, int64_t rows, int64_t cols, int64_t ld_x, void* q,
                              int q_dtype, int64_t ld_q, float* scale, int gran, int mode, void* workspace,
                              size_t workspace_bytes, w8a8_stream_t stream) {
  if (!x || !q || !scale) return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
  if (x_dtype != W8A8_BF16 && x_dtype != W8A8_FP16) return fail(W8A8_ERR_INVALID_ARG, "x_dtype must be BF16 or FP16");
  if (q_dtype != W8A8_E4M3 && q_dtype != W8A8_INT8) return fail(W8A8_ERR_INVALID_ARG, "q_dtype must be E4M3 or INT8");
  if (gran != W8A8_PER_TENSOR && gran != W8A8_PER_ROW) return fail(W8A8_ERR_INVALID_ARG, "bad granularity");
  if (mode != W8A8_DYNAMIC && mode != W8A8_STATIC) return fail(W8A8_ERR_INVALID_ARG, "bad mode");
  if (rows < 1 || cols < 1) return fail(W8A8_ERR_INVALID_ARG, "rows and cols must be >= 1");
  if (rows >= (1LL << 31) || rows * cols >= (1LL << 40)) return fail(W8A8_ERR_UNSUPPORTED, "tensor too large");
  if (ld_x < cols || ld_q < cols) return fail(W8A8_ERR_INVALID_ARG, "leading dimensions must be >= cols");
  if (!aligned(x, 2)) return fail(W8A8_ERR_MISALIGNED, "x must be 2-byte aligned");
  if (!aligned(scale, 4)) return fail(W8A8_ERR_MISALIGNED, "scale must be 4-byte aligned");
  const size_t need = w8a8_scaled_quant_workspace_size(rows, cols, gran, mode);
  if (need > 0) {
    if (!workspace || workspace_bytes < need)
      return fail(W8A8_ERR_WORKSPACE, "dynamic per-tensor quantisation needs %zu bytes of workspace", need);
    if (!aligned(workspace, 4)) return fail(W8A8_ERR_MISALIGNED, "workspace must be 4-byte aligned");
  }
  DeviceInfo dev;
  w8a8_status st = device_info(&dev);
  if (st != W8A8_OK) return st;
  QuantArgs a{};
  a.x = x;
  a.x_kind = (x_dtype == W8A8_BF16) ? 0 : 1;
  a.rows = rows;
  a.cols = cols;
  a.ld_x = ld_x;
  a.q = q;
  a.q_kind = (q_dtype == W8A8_E4M3) ? 0 : 1;
  a.ld_q = ld_q;
  a.scale = scale;
  a.per_row = (gran == W8A8_PER_ROW);
  a.dynamic = (mode == W8A8_DYNAMIC);
  a.amax_word = static_cast<unsigned*>(workspace);
  a.vec = aligned(x, 16) && (ld_x % 8 == 0) && aligned(q, 16) && (ld_q % 8 == 0);
  cudaError_t e = launch_quant(a, dev.sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "scaled_quant launch");
  return ok();
}

w8a8_status w8a8_scaled_dequant(const void* q, int q_dtype, int64_t rows, int64_t cols, int64_t ld_q,
                                const float* scale, int gran, void* y, int y_dtype, int64_t ld_y,
                                w8a8_stream_t stream) {
  if (!q || !scale || !y) return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
  if (q_dtype != W8A8_E4M3 && q_dtype != W8A8_INT8) return fail(W8A8_ERR_INVALID_ARG, "q_dtype must be E4M3 or INT8");
  if (y_dtype != W8A8_BF16 && y_dtype != W8A8_FP16) return fail(W8A8_ERR_INVALID_ARG, "y_dtype must be BF16 or FP16");
  if (gran != W8A8_PER_TENSOR && gran != W8A8_PER_ROW) return fail(W8A8_ERR_INVALID_ARG, "bad granularity");
  if (rows < 1 || cols < 1) return fail(W8A8_ERR_INVALID_ARG, "rows and cols must be >= 1");
  if (rows >= (1LL << 31) || rows * cols >= (1LL << 40)) return fail(W8A8_ERR_UNSUPPORTED, "tensor too large");
  if (ld_q < cols || ld_y < cols) return fail(W8A8_ERR_INVALID_ARG, "leading dimensions must be >= cols");
  if (!aligned(y, 2)) return fail(W8A8_ERR_MISALIGNED, "y must be 2-byte aligned");
  if (!aligned(scale, 4)) return fail(W8A8_ERR_MISALIGNED, "scale must be 4-byte aligned");
  DeviceInfo dev;
  w8a8_status st = device_info(&dev);
  if (st != W8A8_OK) return st;
  DequantArgs a{};
  a.q = q;
  a.q_kind = (q_dtype == W8A8_E4M3) ? 0 : 1;
  a.rows = rows;
  a.cols = cols;
  a.ld_q = ld_q;
  a.scale = scale;
  a.per_row = (gran == W8A8_PER_ROW);
  a.y = y;
  a.y_kind = (y_dtype == W8A8_BF16) ? 0 : 1;
  a.ld_y = ld_y;
  a.vec = aligned(q, 16) && aligned(y, 16);
  cudaError_t e = launch_dequant(a, dev.sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "scaled_dequant launch");
  return ok();
}

w8a8_status w8a8_scaled_mm_pick_config(int64_t M, int64_t N, int64_t K, int q_dtype, w8a8_mm_config* cfg) {
  if (!cfg) return fail(W8A8_ERR_INVALID_ARG, "cfg is null");
  if (M < 1 || N < 1 || K < 1) return fail(W8A8_ERR_INVALID_ARG, "M, N, K must be >= 1");
  if (q_dtype != W8A8_E4M3 && q_dtype != W8A8_INT8) return fail(W8A8_ERR_INVALID_ARG, "bad q_dtype");
  auto_config(M, N, K, q_dtype, sms_or_default(), cfg);
  return ok();
}

size_t w8a8_scaled_mm_config_workspace_size(int64_t M, int64_t N, int64_t K, int q_dtype,
                                            const w8a8_mm_config* cfg) {
  if (!cfg || M < 1 || N < 1 || K < 1) return 0;
  w8a8_mm_config c = *cfg;
  if (c.block_n == 0 || c.split_k == 0) {
    w8a8_mm_config a;
    w8a8_scaled_mm_pick_config(M, N, K, q_dtype, &a);
    if (c.block_n == 0) c.block_n = a.block_n;
    if (c.split_k == 0)
      c.split_k = c.cta_pair ? (a.cta_pair && a.block_n == c.block_n ? a.split_k : 1) : a.split_k;
  }
  if (c.split_k < 1) c.split_k = 1;
  return make_plan(M, N, K, q_dtype, c, 227 * 1024, sms_or_default()).total;
}

size_t w8a8_scaled_mm_workspace_size(int64_t M, int64_t N, int64_t K, int q_dtype) {
  w8a8_mm_config c;
  if (w8a8_scaled_mm_pick_config(M, N, K, q_dtype, &c) != W8A8_OK) return 0;
  return w8a8_scaled_mm_config_workspace_size(M, N, K, q_dtype, &c);
}

w8a8_status w8a8_scaled_mm(const void* a_q, int64_t lda, const void* b_q, int64_t ldb, const float* scale_a,
                           int a_gran, const float* scale_b, int b_gran, void* out, int64_t ldc, int64_t M,
                           int64_t N, int64_t K, int q_dtype, int out_dtype, void* workspace,
                           size_t workspace_bytes, w8a8_stream_t stream) {
  return run_mm(a_q, lda, b_q, ldb, scale_a, a_gran, scale_b, b_gran, out, ldc, M, N, K, q_dtype, out_dtype,
                workspace, workspace_bytes, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

// Activation quantiser + scaled matmul in one call.  The decode shapes (e4m3,
// every token in one narrow tile) run as one kernel that quantises its own
// activations; the rest run the quantiser into the workspace, then the
// matmul.  Both give the bits of w8a8_scaled_quant (dynamic, per row)
// followed by w8a8_scaled_mm.
size_t w8a8_quant_scaled_mm_workspace_size(int64_t M, int64_t N, int64_t K, int q_dtype) {
  if (M < 1 || N < 1 || K < 1) return 0;
  const size_t mm = w8a8_scaled_mm_workspace_size(M, N, K, q_dtype);
  const size_t ldq = static_cast<size_t>((K + 15) & ~15LL);
  const size_t two_step = align256(static_cast<size_t>(M) * ldq) + align256(static_cast<size_t>(M) * 4) + mm;
  return std::max(mm, two_step);
}

w8a8_status w8a8_quant_scaled_mm(const void* x, int x_dtype, int64_t ld_x, const void* b_q, int64_t ldb,
                                 const float* scale_b, int b_gran, void* out, int64_t ldc, int64_t M, int64_t N,
                                 int64_t K, int q_dtype, int out_dtype, float* scale_a_out, int route,
                                 void* workspace, size_t workspace_bytes, w8a8_stream_t stream) {
  if (!x) return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
  if (x_dtype != W8A8_BF16 && x_dtype != W8A8_FP16) return fail(W8A8_ERR_INVALID_ARG, "x_dtype must be BF16 or FP16");
  if (M < 1 || N < 1 || K < 1) return fail(W8A8_ERR_INVALID_ARG, "M, N, K must be >= 1 (got %lld, %lld, %lld)",
                                           static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K));
  if (ld_x < K) return fail(W8A8_ERR_INVALID_ARG, "ld_x must be >= K");
  if (!aligned(x, 2) || (scale_a_out && !aligned(scale_a_out, 4))) return fail(W8A8_ERR_MISALIGNED, "x or scale_a_out misaligned");
  if (route != W8A8_ROUTE_AUTO && route != W8A8_ROUTE_ONE_KERNEL && route != W8A8_ROUTE_TWO_STEP)
    return fail(W8A8_ERR_INVALID_ARG, "route must be W8A8_ROUTE_AUTO, _ONE_KERNEL or _TWO_STEP");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (route != W8A8_ROUTE_TWO_STEP) {
    DeviceInfo dev;
    w8a8_status s0 = device_info(&dev);
    if (s0 != W8A8_OK) return s0;
    w8a8_mm_config cfg;
    auto_config(M, N, K, q_dtype, dev.sms, &cfg);
    const bool possible = q_dtype == W8A8_E4M3 && aligned(x, 16) && (ld_x * 2) % 16 == 0 &&
                          fused_quant_ok(cfg, M, K, q_dtype);
    if (route == W8A8_ROUTE_ONE_KERNEL && !possible)
      return fail(W8A8_ERR_UNSUPPORTED,
                  "the one-kernel route needs e4m3, M <= 64 in one token tile, K %% 16 == 0 and 16-byte aligned x rows");
    if (possible && (route == W8A8_ROUTE_ONE_KERNEL || fused_quant_preferred(cfg, M, K, q_dtype))) {
      const FusedAct fa{x, static_cast<long long>(ld_x), x_dtype == W8A8_FP16 ? 1 : 0, scale_a_out};
      return run_mm(nullptr, K, b_q, ldb, nullptr, W8A8_PER_ROW, scale_b, b_gran, out, ldc, M, N, K, q_dtype,
                    out_dtype, workspace, workspace_bytes, &cfg, st, &fa);
    }
  }
  // two steps: codes (rows padded to 16 bytes) and per-token scales into the
  // workspace, then the matmul
  const long long ldq = (K + 15) & ~15LL;
  const size_t a_bytes = align256(static_cast<size_t>(M) * static_cast<size_t>(ldq));
  const size_t s_bytes = align256(static_cast<size_t>(M) * 4);
  if (!workspace || workspace_bytes < a_bytes + s_bytes)
    return fail(W8A8_ERR_WORKSPACE, "this problem needs %zu bytes of workspace",
                w8a8_quant_scaled_mm_workspace_size(M, N, K, q_dtype));
  if (!aligned(workspace, 256)) return fail(W8A8_ERR_MISALIGNED, "workspace must be 256-byte aligned");
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  float* sa = scale_a_out ? scale_a_out : reinterpret_cast<float*>(wsb + a_bytes);
  w8a8_status s1 = w8a8_scaled_quant(x, x_dtype, M, K, ld_x, wsb, q_dtype, ldq, sa, W8A8_PER_ROW, W8A8_DYNAMIC,
                                     nullptr, 0, stream);
  if (s1 != W8A8_OK) return s1;
  return run_mm(wsb, ldq, b_q, ldb, sa, W8A8_PER_ROW, scale_b, b_gran, out, ldc, M, N, K, q_dtype, out_dtype,
                wsb + a_bytes + s_bytes, workspace_bytes - a_bytes - s_bytes, nullptr, st);
}

w8a8_status w8a8_scaled_mm_with_config(const void* a_q, int64_t lda, const void* b_q, int64_t ldb,
                                       const float* scale_a, int a_gran, const float* scale_b, int b_gran,
                                       void* out, int64_t ldc, int64_t M, int64_t N, int64_t K, int q_dtype,
                                       int out_dtype, void* workspace, size_t workspace_bytes,
                                       const w8a8_mm_config* cfg, w8a8_stream_t stream) {
  if (!cfg) return fail(W8A8_ERR_INVALID_ARG, "cfg is null");
  return run_mm(a_q, lda, b_q, ldb, scale_a, a_gran, scale_b, b_gran, out, ldc, M, N, K, q_dtype, out_dtype,
                workspace, workspace_bytes, cfg, reinterpret_cast<cudaStream_t>(stream));
}

namespace {
w8a8_status shard_table(const int64_t* shard_rows, int nshards, ShardTable* t) {
  if (!shard_rows) return fail(W8A8_ERR_INVALID_ARG, "shard_rows is null");
  if (nshards < 1 || nshards > kMaxShards)
    return fail(W8A8_ERR_UNSUPPORTED, "nshards must be in [1, %d]", kMaxShards);
  t->n = nshards;
  long long acc = 0;
  for (int i = 0; i < nshards; ++i) {
    if (shard_rows[i] < 0) return fail(W8A8_ERR_INVALID_ARG, "shard_rows must be >= 0");
    acc += shard_rows[i];
    if (acc >= (1LL << 31)) return fail(W8A8_ERR_UNSUPPORTED, "too many rows");
    t->end[i] = acc;
  }
  if (acc < 1) return fail(W8A8_ERR_INVALID_ARG, "the shards hold no rows");
  return W8A8_OK;
}
}  // namespace

w8a8_status w8a8_expand_shard_scales(const float* shard_scales, const int64_t* shard_rows, int nshards,
                                     float* scale_b, w8a8_stream_t stream) {
  if (!shard_scales || !scale_b) return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(shard_scales, 4) || !aligned(scale_b, 4)) return fail(W8A8_ERR_MISALIGNED, "scales must be 4-byte aligned");
  ShardTable t;
  w8a8_status st = shard_table(shard_rows, nshards, &t);
  if (st != W8A8_OK) return st;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != W8A8_OK) return st;
  cudaError_t e = launch_expand_shard_scales(shard_scales, t, scale_b, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "expand_shard_scales launch");
  return ok();
}

w8a8_status w8a8_requant_shards(const void* q, int q_dtype, int64_t cols, int64_t ld_q, const float* shard_scales,
                                const int64_t* shard_rows, int nshards, void* q_out, int64_t ld_out,
                                float* scale_out, w8a8_stream_t stream) {
  if (!q || !shard_scales || !q_out || !scale_out) return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
  if (q_dtype != W8A8_E4M3 && q_dtype != W8A8_INT8) return fail(W8A8_ERR_INVALID_ARG, "q_dtype must be E4M3 or INT8");
  if (cols < 1) return fail(W8A8_ERR_INVALID_ARG, "cols must be >= 1");
  if (ld_q < cols || ld_out < cols) return fail(W8A8_ERR_INVALID_ARG, "leading dimensions must be >= cols");
  if (q == q_out && ld_q != ld_out) return fail(W8A8_ERR_INVALID_ARG, "in-place requantisation needs ld_out == ld_q");
  if (!aligned(shard_scales, 4) || !aligned(scale_out, 4)) return fail(W8A8_ERR_MISALIGNED, "scales must be 4-byte aligned");
  ShardTable t;
  w8a8_status st = shard_table(shard_rows, nshards, &t);
  if (st != W8A8_OK) return st;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != W8A8_OK) return st;
  cudaError_t e = launch_requant_shards(q, q_dtype == W8A8_E4M3 ? 0 : 1, cols, ld_q, shard_scales, t, q_out, ld_out,
                                        scale_out, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "requant_shards launch");
  return ok();
}

namespace {
// Tokens per CTA of the attention: the largest of 256 / 128 / 64 that still
// gives two CTAs per SM; the workspace is sized for 64.
int attn_chunk_for(long long batch, long long kv_heads, long long max_seq, int sms) {
  int chunk = w8a8::attn_max_chunk();
  while (chunk > 64 && batch * kv_heads * ((max_seq + chunk - 1) / chunk) < 2LL * sms) chunk /= 2;
  return chunk;
}
}  // namespace

size_t w8a8_fp8_kv_attention_workspace_size(int64_t batch, int64_t num_q_heads, int64_t max_seq_len) {
  if (batch < 1 || num_q_heads < 1 || max_seq_len < 1) return 0;
  // 0 as well when the size does not fit 2^62 bytes (no wrap-around)
  const long double bytes = static_cast<long double>(batch) * num_q_heads * ((max_seq_len + 63) / 64) *
                            w8a8::attn_part_stride() * sizeof(float);
  if (bytes > static_cast<long double>(1ULL << 62)) return 0;
  return static_cast<size_t>(batch) * num_q_heads * ((max_seq_len + 63) / 64) * w8a8::attn_part_stride() *
         sizeof(float);
}

w8a8_status w8a8_fp8_kv_decode_attention(const void* q, int q_dtype, int64_t batch, int64_t num_q_heads,
                                         int64_t num_kv_heads, int64_t head_dim, const void* k_cache,
                                         const void* v_cache, int64_t max_seq_len, const int32_t* block_table,
                                         int64_t block_size, int64_t max_blocks, int64_t num_blocks,
                                         const int32_t* seq_lens, const float* k_scale, const float* v_scale,
                                         float sm_scale, void* out, int out_dtype, void* workspace,
                                         size_t workspace_bytes, w8a8_stream_t stream) {
  if (!q || !k_cache || !v_cache || !seq_lens || !k_scale || !v_scale || !out)
    return fail(W8A8_ERR_INVALID_ARG, "null pointer argument");
  if ((q_dtype != W8A8_BF16 && q_dtype != W8A8_FP16) || (out_dtype != W8A8_BF16 && out_dtype != W8A8_FP16))
    return fail(W8A8_ERR_INVALID_ARG, "q and out must be BF16 or FP16");
  if (head_dim != 128) return fail(W8A8_ERR_INVALID_ARG, "head_dim must be 128");
  if (batch < 1 || num_q_heads < 1 || num_kv_heads < 1 || max_seq_len < 1)
    return fail(W8A8_ERR_INVALID_ARG, "batch, head counts and max_seq_len must be >= 1");
  if (batch > 65535 || num_kv_heads > 65535 || max_seq_len > (1LL << 30) || num_q_heads > 65535 ||
      ((max_seq_len + 63) / 64) * num_kv_heads >= (1LL << 31))
    return fail(W8A8_ERR_INVALID_ARG, "sizes exceed the launch grid");
  if (num_q_heads % num_kv_heads != 0) return fail(W8A8_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  const long long G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return fail(W8A8_ERR_INVALID_ARG, "num_q_heads / num_kv_heads must be 1, 2, 4 or 8");
  if (block_table && (block_size < 1 || max_blocks < 1 || num_blocks < 1 || max_blocks * block_size < max_seq_len))
    return fail(W8A8_ERR_INVALID_ARG, "a block table needs block_size, max_blocks, num_blocks >= 1 and "
                                      "max_blocks * block_size >= max_seq_len");
  if (block_table && (block_size > (1 << 30) || max_blocks > (1 << 30) || num_blocks > (1LL << 31) / block_size))
    return fail(W8A8_ERR_INVALID_ARG, "block table sizes out of range");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return fail(W8A8_ERR_MISALIGNED, "caches must be 16-byte aligned");
  if (!aligned(seq_lens, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4) || (block_table && !aligned(block_table, 4)) ||
      !aligned(q, 2) || !aligned(out, 2))
    return fail(W8A8_ERR_MISALIGNED, "misaligned q, out, scale, length or block table pointer");
  const size_t need = w8a8_fp8_kv_attention_workspace_size(batch, num_q_heads, max_seq_len);
  if (need == 0) return fail(W8A8_ERR_INVALID_ARG, "batch x heads x max_seq_len too large");
  if (!workspace || workspace_bytes < need || !aligned(workspace, 16))
    return fail(W8A8_ERR_WORKSPACE, "workspace must be 16-byte aligned and hold %zu bytes", need);
  w8a8_status st;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != W8A8_OK) return st;
  w8a8::AttnParams p{};
  p.q = q;
  p.q_fp16 = q_dtype == W8A8_FP16;
  p.q_vec = aligned(q, 8) ? 1 : 0;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_table = block_table;
  p.block_size = block_table ? static_cast<int>(block_size) : 1;
  p.max_blocks = block_table ? static_cast<int>(max_blocks) : 1;
  p.num_blocks = block_table ? static_cast<int>(num_blocks) : 1;
  p.seq_lens = seq_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.sm_scale = sm_scale;
  p.out = out;
  p.out_fp16 = out_dtype == W8A8_FP16;
  p.partial = static_cast<float*>(workspace);
  p.batch = static_cast<int>(batch);
  p.num_q_heads = static_cast<int>(num_q_heads);
  p.num_kv_heads = static_cast<int>(num_kv_heads);
  p.max_seq_len = static_cast<int>(max_seq_len);
  p.chunk = attn_chunk_for(batch, num_kv_heads, max_seq_len, dev.sms);
  // bulk-tensor copies of the 16-token blocks where the cache rows of a block
  // are consecutive: a contiguous cache, or a paged one with 16 | block_size
  CUtensorMap mk, mv;
  const long long rows = block_table ? num_blocks * block_size : batch * max_seq_len;
  bool tma = (!block_table || block_size % 16 == 0) && rows < (1LL << 31);
  if (tma) {
    tma = make_operand_map(&mk, k_cache, false, rows, num_kv_heads * 128, num_kv_heads * 128, 16) == W8A8_OK &&
          make_operand_map(&mv, v_cache, false, rows, num_kv_heads * 128, num_kv_heads * 128, 16) == W8A8_OK;
    if (!tma) t_last_error.clear();  // the per-lane path needs no tensor map
  }
  cudaError_t e = w8a8::launch_fp8kv_attention(p, tma ? &mk : nullptr, tma ? &mv : nullptr,
                                               reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fp8 KV attention launch");
  return ok();
}

w8a8_status w8a8_debug_mm_trace(void* buf, size_t bytes) {
  if (buf && !aligned(buf, 8)) return fail(W8A8_ERR_MISALIGNED, "trace buffer must be 8-byte aligned");
  const size_t per_cta = 16 * sizeof(unsigned long long);
  g_trace_ctas.store(buf ? static_cast<int>(std::min<size_t>(bytes / per_cta, 1u << 20)) : 0);
  g_trace_buf.store(buf ? static_cast<unsigned long long*>(buf) : nullptr);
  return ok();
}

w8a8_status w8a8_device_status(int* flags) {
  if (!flags) return fail(W8A8_ERR_INVALID_ARG, "flags is null");
  cudaError_t e = read_clear_device_status(flags);
  if (e != cudaSuccess) return cuda_fail(e, "device status read");
  int qf = 0;
  e = read_clear_quant_status(&qf);
  if (e != cudaSuccess) return cuda_fail(e, "device status read");
  *flags |= qf;
  e = read_clear_attn_status(&qf);
  if (e != cudaSuccess) return cuda_fail(e, "device status read");
  *flags |= qf;
  return ok();
}

}  // extern "C"
