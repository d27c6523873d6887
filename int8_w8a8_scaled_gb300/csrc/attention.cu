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
// Both products run on the tensor cores (mma.sync m16n8k16, f16 operands,
// fp32 accumulation), 16 tokens at a time per warp:
//   scores  S^T[16 tokens x 8 heads] = K[16 tokens x 128] . q^T[128 x 8]
//   output  O^T[128 dims x 8 heads] += V^T[128 x 16 tokens] . P^T[16 tokens x 8]
// e4m3 codes convert exactly to f16 (one cvt per two codes).  The query is
// scaled by a power of two 2^e before its conversion to f16, so that its
// largest element lies in [2^14, 2^15): every bf16 query element down to
// 2^-31 of the largest converts exactly (f16 carries bf16's 8 significant
// bits over that range), and the scores are multiplied by 2^-e after.  The
// softmax weights p = 2^(s - m) <= 1 are carried as p * 2^15 = hi + lo, two
// f16 values (hi = f16(p * 2^15), lo = f16(p * 2^15 - hi)), so a weight
// keeps ~22 significant bits: for G <= 4 the lo halves take the four
// padding columns of the 8-column MMA (no extra MMA), for G = 8 a second
// MMA adds them.  For G <= 4 the query rows are also duplicated into those
// columns, so the score MMA already gives the lanes that carry the lo
// halves their heads' scores.
//
// Register layout (lane = 4 g + t):
//  - scores: A = K tile, rows g and g + 8 are tokens g and g + 8; thread t
//    reads bytes [16t, 16t + 16) and [64 + 16t, 64 + 16t + 16) of a 128-byte
//    cache row (the 8 lanes t = 0..3 of two instructions read whole rows),
//    and k-block j (16 dims) takes 4 of those 32 bytes.  The dot product
//    does not depend on the order of the dims, so q's fragment is laid out
//    with the same permutation.
//  - output: A = V^T tile, rows are dims; thread g reads bytes
//    [16g, 16g + 16) of the rows of tokens 2t, 2t+1, 2t+8, 2t+9 and
//    m-block i (16 dims) takes dims 16g + 2i (row g) and 16g + 2i + 1
//    (row g + 8): byte permutes pair two tokens' codes of one dim.
//  - P^T: the scores' accumulator layout transposed in registers
//    (movmatrix), which is exactly the B fragment of the output MMA.
//
// Work split: a CTA of 4 warps takes one (chunk, KV head, sequence); each
// warp takes a quarter of the chunk's tokens, 16 at a time, into a per-warp
// shared-memory ring of 16-token blocks filled while the current block is
// used: by two bulk-tensor copies per block (K and V rows, 128-byte swizzle)
// when every 16-token block is contiguous in the cache (no block table, or
// 16 dividing the block size), else by the lanes' own 16-byte cp.async
// pieces.  The 4 warps' (m, l, o) are combined in shared memory at the end.
// The KV heads of a chunk are consecutive CTAs, so they read the same cache
// rows (each its 128-byte slice) at about the same time.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace w8a8 {

namespace {

constexpr int kHeadDim = 128;
constexpr int kWarps = 4;                         // warps per CTA; each takes chunk / 4 tokens
constexpr int kAttnThreads = 32 * kWarps;
// Resident CTAs per SM the register budget is fitted to (4: <= 128
// registers, 16 warps per SM), with a ring of 2 blocks per warp: measured
// best (a third slot, or 3 CTAs with deeper rings, ran 5-7 % slower).
#ifndef W8A8_ATTN_MIN_CTAS
#define W8A8_ATTN_MIN_CTAS 4
#endif
#ifndef W8A8_ATTN_MAX_CHUNK
#define W8A8_ATTN_MAX_CHUNK 512
#endif
constexpr int kMaxChunk = W8A8_ATTN_MAX_CHUNK;
constexpr int kPartStride = kHeadDim + 4;         // o[128], m, l, 2 pad (floats)
constexpr int kOStride = kHeadDim + kHeadDim / 16;  // a warp's o per head in shared memory (padded)
constexpr float kPScale = 32768.f;                // weights enter the output MMA as p * 2^15

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

__device__ __forceinline__ void cvt4(uint32_t four_codes, uint32_t& lo, uint32_t& hi) {
  e4m3x4_to_f16x2x2(four_codes, lo, hi);
}

// D += A . B for one m16n8k16 tile: f16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit elements held one row pair per lane
// (lane 4r + c holds row r, columns 2c and 2c + 1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t smem_addr_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// Two weights a, b as f16 pairs hi = (RN(a), RN(b)) and lo = (RN(a - hi.a),
// RN(b - hi.b)), a in the low half; a - hi.a is exact in fp32.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 2^x by the hardware approximation (relative error about 2^-22; results
// below 2^-126 flush to zero, a softmax weight that no sum can see).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The codes one lane holds for a block of 16 tokens: K rows g and g + 8
// (bytes 16t and 64 + 16t) and whether they are tokens of the sequence;
// V rows 2t, 2t + 1, 2t + 8, 2t + 9 (bytes 16g) are read from the ring slot
// only once the score MMAs have taken K (fewer registers live at once):
// `vsrc` is the slot, `vlim` the number of its leading rows that hold tokens
// (rows past it read as zero codes).
struct KvBlock {
  uint4 k[2][2];
  bool kval[2];
  const uint8_t* vsrc;
  int vlim;
};

// Ring of blocks in flight per warp (shared memory, filled by cp.async).  A
// lane copies its own eight 16-byte chunks of a block and later reads them
// back itself, so the ring needs no synchronisation between lanes; chunk j
// of lane L sits at (j * 32 + L) * 16 within the block's 4 KB, so a warp's
// 16-byte reads of one chunk index touch 32 consecutive 16-byte words.
#ifndef W8A8_ATTN_RING
#define W8A8_ATTN_RING 2
#endif
constexpr int kRing = W8A8_ATTN_RING;
static_assert(kRing >= 2 && kRing <= 8, "ring depth");
constexpr int kBlockBytes = 32 * 8 * 16;  // one 16-token block of K and V codes

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  // invalid: no read, the 16 bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Requests the block at chunk position ib into ring slot `slot` (tokens past
// `end` or in padding blocks are not read: zeros) and returns the validity
// bits of K rows g, g + 8.
__device__ __forceinline__ uint32_t issue_block(const AttnParams& p, int b, int t0, int ib, int end, int g, int t,
                                                int lane, const uint8_t* kbase, const uint8_t* vbase,
                                                long long row_bytes, uint32_t slot_addr) {
  uint32_t kv = 0u;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = ib + g + 8 * r;
    const long long slot = i < end ? slot_of(p, b, t0 + i) : -1;
    const bool ok = slot >= 0;
    kv |= ok ? (1u << r) : 0u;
    const uint8_t* row = kbase + (ok ? slot : 0) * row_bytes;
    cp_async16(slot_addr + ((2 * r + 0) * 32 + lane) * 16, row + 16 * t, ok);
    cp_async16(slot_addr + ((2 * r + 1) * 32 + lane) * 16, row + 64 + 16 * t, ok);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = ib + 2 * t + (r & 1) + 8 * (r >> 1);
    const long long slot = i < end ? slot_of(p, b, t0 + i) : -1;
    const bool ok = slot >= 0;
    cp_async16(slot_addr + ((4 + r) * 32 + lane) * 16, vbase + (ok ? slot : 0) * row_bytes + 16 * g, ok);
  }
  return kv;
}

// The lane's chunks of a block, back from its ring slot.
__device__ __forceinline__ void read_block(const uint8_t* slot_ptr, int lane, uint32_t kv, KvBlock& x) {
  const uint4* c = reinterpret_cast<const uint4*>(slot_ptr) + lane;
  x.k[0][0] = c[0 * 32];
  x.k[0][1] = c[1 * 32];
  x.k[1][0] = c[2 * 32];
  x.k[1][1] = c[3 * 32];
  x.kval[0] = (kv & 1u) != 0u;
  x.kval[1] = (kv & 2u) != 0u;
  x.vsrc = slot_ptr;
  x.vlim = 16;  // the copies zero-filled every V chunk that is not a token
}


// ---- the bulk-tensor path: per 16-token block two TMA copies (the K and the
// V rows of this KV head, 16 x 128 bytes each, 128-byte swizzled) into the
// warp's ring slot, one mbarrier per slot.  Per-lane 16-byte copies keep at
// most ~64 KB per SM in flight, whatever the ring depth; bulk copies do not
// have that limit.  Chunk c of tile row r sits at r * 128 + (c ^ (r & 7)) * 16,
// so a quarter-warp's fragment reads hit different banks.

// Cache row of the 16-token block starting at token tb of sequence b (16 |
// block_size with a table), or -1 for a padding block.
__device__ __forceinline__ long long block_row(const AttnParams& p, int b, int tb) {
  if (!p.block_table) return static_cast<long long>(b) * p.max_seq_len + tb;
  const int blk = __ldg(p.block_table + static_cast<size_t>(b) * p.max_blocks + tb / p.block_size);
  if (blk < 0 || blk >= p.num_blocks) return -1;
  return static_cast<long long>(blk) * p.block_size + tb % p.block_size;
}

// lane 0: the two copies of the block at chunk position ib into slot `dst`
__device__ __forceinline__ void tma_issue_block(const AttnParams& p, const CUtensorMap* mk, const CUtensorMap* mv,
                                                int b, int t0, int ib, int kvh, uint32_t dst, uint32_t bar) {
  const long long row = block_row(p, b, t0 + ib);
  if (row < 0) {
    mbar_arrive(bar);  // a padding block: nothing to copy
    return;
  }
  mbar_arrive_expect_tx(bar, kBlockBytes);
  // the cache is read once per call: ahead of it in L2 go the queries and
  // the partial results
  const uint64_t pol = policy_evict_first();
  tma_load_2d_hint(dst, mk, bar, kvh * kHeadDim, static_cast<int32_t>(row), pol);
  tma_load_2d_hint(dst + kBlockBytes / 2, mv, bar, kvh * kHeadDim, static_cast<int32_t>(row), pol);
}

__device__ __forceinline__ uint32_t swz(int r, int c) { return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4)); }

// The lane's fragments of a block from its (swizzled) slot; tokens past
// `end` or in a padding block are invalid: their K rows masked by kval,
// their V codes zeroed (whatever the cache holds there, their weight is 0).
__device__ __forceinline__ void read_block_tma(const uint8_t* slot, const AttnParams& p, int b, int t0, int ib,
                                               int end, int g, int t, KvBlock& x) {
  const bool blk_ok = block_row(p, b, t0 + ib) >= 0;
  const uint8_t* kt = slot;
  const uint8_t* vt = slot + kBlockBytes / 2;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = g + 8 * r;
    x.k[r][0] = *reinterpret_cast<const uint4*>(kt + swz(row, t));
    x.k[r][1] = *reinterpret_cast<const uint4*>(kt + swz(row, 4 + t));
    x.kval[r] = blk_ok && ib + row < end;
  }
  x.vsrc = slot;
  x.vlim = blk_ok ? min(16, end - ib) : 0;
  (void)vt;
}

// The lane's V chunks of a block (see KvBlock), from a per-lane ring slot
// (kTma false: chunk r of lane L at (4 + r) * 32 + L) or a swizzled bulk-copy
// slot (rows 2t, 2t+1, 2t+8, 2t+9, chunk g).
template <bool kTma>
__device__ __forceinline__ void read_v(const KvBlock& x, int lane, int g, int t, uint4 (&v)[4]) {
  if (!kTma) {
    const uint4* c = reinterpret_cast<const uint4*>(x.vsrc) + lane;
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = c[(4 + r) * 32];
    return;
  }
  const uint8_t* vt = x.vsrc + kBlockBytes / 2;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = 2 * t + (r & 1) + 8 * (r >> 1);
    v[r] = *reinterpret_cast<const uint4*>(vt + swz(row, g));
    if (x.vlim < 16 && row >= x.vlim) v[r] = make_uint4(0u, 0u, 0u, 0u);  // warp-uniform test first
  }
}

// Running softmax state of one lane: maxima and (lane-partial) sums of its
// two columns, and the O^T accumulators of the 8 dim blocks.
struct SoftmaxState {
  float m[2], l[2];
  float o[8][4];
};

// Scores, online softmax and output update for one block of 16 tokens.
template <bool kPack, bool kTma>
__device__ __forceinline__ void attend_block(const KvBlock& x, const uint32_t (&qf)[8][2], float cs, bool lo_lane,
                                             int lane, int g, int t, SoftmaxState& st) {
  // scores S^T[token g / g+8][column 2t / 2t+1]: four independent
  // accumulator chains of two k-blocks each (a single chain of eight MMAs
  // would make the block wait for eight MMA latencies), summed after
  float sp[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c) sp[c][0] = sp[c][1] = sp[c][2] = sp[c][3] = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t w0r = word_of(x.k[0][j >> 2], j & 3);
    const uint32_t w1r = word_of(x.k[1][j >> 2], j & 3);
    uint32_t a0, a1, a2, a3;
    cvt4(w0r, a0, a2);
    cvt4(w1r, a1, a3);
    mma16816(sp[j & 3], a0, a1, a2, a3, qf[j][0], qf[j][1]);
  }
  // V's codes, now that the score MMAs hold K
  uint4 v[4];
  read_v<kTma>(x, lane, g, t, v);
  float s[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) s[k] = (sp[0][k] + sp[1][k]) + (sp[2][k] + sp[3][k]);
  // (with packing, lanes t >= 2 hold duplicates of their partner's
  // columns: the query rows are duplicated); invalid tokens -inf
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float y = x.kval[k >> 1] ? s[k] * cs : -INFINITY;
    s[k] = y;
    mx[k & 1] = fmaxf(mx[k & 1], y);
  }
  // The running maxima only move when some score of the block exceeds them
  // (rare once the first blocks are seen): then the new maxima are reduced
  // over the 8 lanes of each column and the state rescaled by 2^(m_old -
  // m_new); otherwise the factor would be exactly 1 and all of it is skipped.
  float m_new[2] = {st.m[0], st.m[1]};
  if (__any_sync(0xffffffffu, mx[0] > st.m[0] || mx[1] > st.m[1])) {
    float alpha[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], off));
      m_new[c] = fmaxf(st.m[c], mx[c]);
      alpha[c] = m_new[c] == -INFINITY ? 1.f : ex2_fast(st.m[c] - m_new[c]);
      st.m[c] = m_new[c];
      st.l[c] *= alpha[c];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.o[i][0] *= alpha[0];
      st.o[i][1] *= alpha[1];
      st.o[i][2] *= alpha[0];
      st.o[i][3] *= alpha[1];
    }
  }
  float pw[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float mc = m_new[k & 1];
    pw[k] = (mc == -INFINITY) ? 0.f : ex2_fast(s[k] - mc);
    st.l[k & 1] += pw[k];
  }
  // P^T fragments (tokens 2t.., column g) by transposing the accumulator layout
  uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
  {
    uint32_t h01, l01, h23, l23;
    split_pair(pw[0] * kPScale, pw[1] * kPScale, h01, l01);
    split_pair(pw[2] * kPScale, pw[3] * kPScale, h23, l23);
    if (kPack) {
      bh0 = movmatrix_t(lo_lane ? l01 : h01);
      bh1 = movmatrix_t(lo_lane ? l23 : h23);
    } else {
      bh0 = movmatrix_t(h01);
      bh1 = movmatrix_t(h23);
      bl0 = movmatrix_t(l01);
      bl1 = movmatrix_t(l23);
    }
  }
  // O^T[dims 16g+2i, 16g+2i+1][columns] += V^T . P^T
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
    const uint32_t p01 = __byte_perm(word_of(v[0], i >> 1), word_of(v[1], i >> 1), sel);
    const uint32_t p23 = __byte_perm(word_of(v[2], i >> 1), word_of(v[3], i >> 1), sel);
    uint32_t a0, a1, a2, a3;
    cvt4(p01, a0, a1);
    cvt4(p23, a2, a3);
    mma16816(st.o[i], a0, a1, a2, a3, bh0, bh1);
    if (!kPack) mma16816(st.o[i], a0, a1, a2, a3, bl0, bl1);
  }
}

template <int G, bool kTma>
__global__ void __launch_bounds__(kAttnThreads, W8A8_ATTN_MIN_CTAS)
    fp8kv_attn_chunk_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v) {
  // G <= 4: the lo halves of the weights ride in the padding columns 4..7
  constexpr bool kPack = G <= 4;
  // the KV heads of a chunk are consecutive CTAs: they run side by side and
  // read the same cache rows (each its 128-byte slice) at about the same time
  // programmatic dependent launch: let the combine kernel be scheduled, then
  // wait for the preceding kernel (and its memory) before reading anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.y;
  const int kvh = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.num_kv_heads));
  const int ch = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.num_kv_heads));
  const int len = seq_len_of(p, b);
  const int t0 = ch * p.chunk;
  if (t0 >= len) return;  // uniform: the combine reads only chunks that hold tokens
  const int n = min(len - t0, p.chunk);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane >> 2, t = lane & 3;

  __shared__ __align__(16) __half qs[8][kHeadDim];   // q * 2^e in f16; zero rows for padding heads
  __shared__ float s_qmax[kWarps];
  __shared__ float s_m[kWarps][8], s_l[kWarps][8];
  extern __shared__ __align__(128) uint8_t ring_raw[];  // [kWarps][kRing][kBlockBytes], 1024-byte aligned
  __shared__ uint64_t s_bar[kWarps][kRing];             // bulk-tensor path: one per ring slot
  uint8_t* ring_smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ring_raw) + 1023) &
                                                  ~static_cast<uintptr_t>(1023));

  // this warp's tokens of the chunk, in blocks of 16; the first kRing - 1
  // blocks are requested before the query is prepared
  const uint8_t* kbase = static_cast<const uint8_t*>(p.k_cache) + kvh * kHeadDim;
  const uint8_t* vbase = static_cast<const uint8_t*>(p.v_cache) + kvh * kHeadDim;
  const long long row_bytes = static_cast<long long>(p.num_kv_heads) * kHeadDim;
  const int per_warp = p.chunk / kWarps;
  const int w0 = warp * per_warp;
  const int w1 = min(n, w0 + per_warp);
  const int nblk = w1 > w0 ? (w1 - w0 + 15) / 16 : 0;
  uint8_t* ring = ring_smem + static_cast<size_t>(warp) * kRing * kBlockBytes;
  const uint32_t ring_addr = smem_addr_u32(ring);
  uint32_t kvbits = 0u;  // K-row validity, two bits per ring slot (per-lane copies)
  if (kTma) {
    if (lane == 0) {
      for (int j = 0; j < kRing; ++j) mbar_init(smem_addr(&s_bar[warp][j]), 1);
      fence_barrier_init();
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
      for (int j = 0; j < kRing - 1 && j < nblk; ++j)
        tma_issue_block(p, &tmap_k, &tmap_v, b, t0, w0 + 16 * j, kvh, ring_addr + j * kBlockBytes,
                        smem_addr(&s_bar[warp][j]));
    }
    __syncwarp();
  } else {
#pragma unroll
    for (int j = 0; j < kRing - 1; ++j) {
      if (j < nblk)
        kvbits |= issue_block(p, b, t0, w0 + 16 * j, w1, g, t, lane, kbase, vbase, row_bytes,
                              ring_addr + j * kBlockBytes) << (2 * j);
      cp_async_commit();  // one group per block, empty past the end
    }
  }

  // ---- the query rows of the G heads, scaled by 2^e into [2^14, 2^15) and
  // converted to f16: one pass of 8-byte loads (G * 128 values, 4 per thread
  // and pass), the values kept in registers for the conversion
  const size_t q0 = (static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(kvh) * G) * kHeadDim;
  constexpr int kQPer = (G * kHeadDim) / (4 * kAttnThreads) > 0 ? (G * kHeadDim) / (4 * kAttnThreads) : 1;
  float qv[kQPer][4];
  float qmax = 0.f;
#pragma unroll
  for (int u = 0; u < kQPer; ++u) {
    const int i = 4 * (threadIdx.x + u * kAttnThreads);
    if (i < G * kHeadDim) {
      if (p.q_vec) {  // q 8-byte aligned
        const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.q) + q0 + i);
        const uint16_t e4[4] = {static_cast<uint16_t>(w.x), static_cast<uint16_t>(w.x >> 16),
                                static_cast<uint16_t>(w.y), static_cast<uint16_t>(w.y >> 16)};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          qv[u][c] = p.q_fp16 ? __half2float(__ushort_as_half(e4[c])) : __bfloat162float(__ushort_as_bfloat16(e4[c]));
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) qv[u][c] = load_q(p.q, p.q_fp16, q0 + i + c);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) qmax = fmaxf(qmax, fabsf(qv[u][c]));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
  if (lane == 0) s_qmax[warp] = qmax;
  // padding heads' rows of the fragment are zero (with packing, rows 4..7
  // repeat rows 0..3)
  for (int i = threadIdx.x; i < 8 * kHeadDim; i += kAttnThreads) {
    const int r = i / kHeadDim;
    if ((kPack ? (r & 3) : r) >= G) qs[r][i % kHeadDim] = __float2half_rn(0.f);
  }
  __syncthreads();
  qmax = s_qmax[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) qmax = fmaxf(qmax, s_qmax[w]);
  int e = 0;
  if (qmax > 0.f && qmax <= 3.0e38f) {
    int ex;
    frexpf(qmax, &ex);  // qmax in [2^(ex-1), 2^ex)
    e = min(100, max(-100, 15 - ex));
  }
#pragma unroll
  for (int u = 0; u < kQPer; ++u) {
    const int i = 4 * (threadIdx.x + u * kAttnThreads);
    if (i < G * kHeadDim) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const __half h = __float2half_rn(ldexpf(qv[u][c], e));
        qs[(i + c) / kHeadDim][(i + c) % kHeadDim] = h;
        if (kPack) qs[(i + c) / kHeadDim + 4][(i + c) % kHeadDim] = h;
      }
    }
  }
  __syncthreads();
  // B fragment of k-block j: dims L_t[4j .. 4j+3] of head g, L_t = [16t, 16t+16) ++ [64+16t, 64+16t+16)
  uint32_t qf[8][2];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int d = (j < 4 ? 16 * t : 64 + 16 * t) + 4 * (j & 3);
    qf[j][0] = *reinterpret_cast<const uint32_t*>(&qs[g][d]);
    qf[j][1] = *reinterpret_cast<const uint32_t*>(&qs[g][d + 2]);
  }
  // scores in the log2 domain: S' * (sm_scale * k_scale * log2 e) * 2^-e
  const float cs = ldexpf(p.sm_scale * __ldg(p.k_scale) * 1.4426950408889634f, -e);

  // columns 2t and 2t+1 of this lane: heads hc, hc + 1 (with packing the
  // lanes t >= 2 hold the lo parts of the heads of lane t - 2)
  const bool lo_lane = kPack && t >= 2;
  SoftmaxState st;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;

  // blocks of 16 tokens, kRing - 1 blocks in flight ahead of the one used
  bool ok = true;
  int issued = kTma ? min(kRing - 1, nblk) : 0, consumed = 0;
  for (int i = 0; i < nblk; ++i) {
    const int jn = i + kRing - 1;  // its slot held block i - 1, already read back
    const int sn = jn % kRing;
    const int si = i % kRing;
    KvBlock x;
    if (kTma) {
      __syncwarp();  // every lane is done with block i - 1's slot
      if (lane == 0 && jn < nblk) {
        fence_proxy_async_shared();  // its reads before the copy that overwrites it
        tma_issue_block(p, &tmap_k, &tmap_v, b, t0, w0 + 16 * jn, kvh, ring_addr + sn * kBlockBytes,
                        smem_addr(&s_bar[warp][sn]));
      }
      if (jn < nblk) ++issued;
      if (!mbar_wait(smem_addr(&s_bar[warp][si]), (i / kRing) & 1)) {
        ok = false;
        break;
      }
      consumed = i + 1;
      read_block_tma(ring + si * kBlockBytes, p, b, t0, w0 + 16 * i, w1, g, t, x);
    } else {
      kvbits &= ~(3u << (2 * sn));
      if (jn < nblk)
        kvbits |= issue_block(p, b, t0, w0 + 16 * jn, w1, g, t, lane, kbase, vbase, row_bytes,
                              ring_addr + sn * kBlockBytes) << (2 * sn);
      cp_async_commit();
      cp_async_wait<kRing - 1>();  // block i's group has landed
      read_block(ring + si * kBlockBytes, lane, (kvbits >> (2 * si)) & 3u, x);
    }
    attend_block<kPack, kTma>(x, qf, cs, lo_lane, lane, g, t, st);
  }
  if (kTma && !ok && lane == 0) {
    // a wait gave up (flagged in the device status): let the copies still in
    // flight land, bounded, before the CTA's shared memory is released
    for (int j = consumed; j < issued; ++j) mbar_wait(smem_addr(&s_bar[warp][j % kRing]), (j / kRing) & 1);
  }
  if (!kTma) cp_async_wait<0>();
  // every copy into this warp's ring has landed and been read: the ring now
  // holds the warp's o per head, [G][128 + 8] floats (one pad word per 16
  // dims keeps the 8 lanes of a store on different banks)
  __syncwarp();
  float* s_o_w = reinterpret_cast<float*>(ring);
  static_assert(G * kOStride * 4 <= kRing * kBlockBytes, "o fits the warp's ring");
  float (&o)[8][4] = st.o;
  float (&m_run)[2] = st.m;
  float (&l_run)[2] = st.l;

  // ---- this warp's (m, l, o) per head into shared memory
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l_run[c] += __shfl_xor_sync(0xffffffffu, l_run[c], off);
  if (kPack) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[i][k] += __shfl_xor_sync(0xffffffffu, o[i][k], 2);  // hi + lo
  }
  const int hc = kPack ? 2 * (t & 1) : 2 * t;
  if (!lo_lane) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int h = hc + c;
      if (h < G) {
        if (g == 0) {
          s_m[warp][h] = m_run[c];
          s_l[warp][h] = l_run[c];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d = 16 * g + 2 * i;
          s_o_w[h * kOStride + d + g] = o[i][c];  // d + d / 16
          s_o_w[h * kOStride + d + 1 + g] = o[i][2 + c];
        }
      }
    }
  }
  __syncthreads();

  // ---- the chunk's partial result of each head: o[128], m, l (warps combined in order)
  const int nch = (p.max_seq_len + p.chunk - 1) / p.chunk;
  for (int idx = threadIdx.x; idx < G * kHeadDim; idx += kAttnThreads) {
    const int h = idx / kHeadDim, d = idx % kHeadDim;
    float M = s_m[0][h];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_m[w][h]);
    float acc = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(s_m[w][h] - M);
        acc = fmaf(f, reinterpret_cast<const float*>(ring_smem + static_cast<size_t>(w) * kRing * kBlockBytes)
                              [h * kOStride + d + d / 16],
                   acc);
        l = fmaf(f, s_l[w][h], l);
      }
    }
    float* part = p.partial + ((static_cast<size_t>(b) * p.num_q_heads + kvh * G + h) * nch + ch) * kPartStride;
    part[d] = acc * (1.f / kPScale);
    if (d == 0) {
      part[kHeadDim] = M;
      part[kHeadDim + 1] = l;
    }
  }
}

// One CTA per (query head, sequence), one thread per head dim.
__global__ void __launch_bounds__(kHeadDim) fp8kv_attn_combine_kernel(const AttnParams p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the chunks' partials are complete
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

// Launch with programmatic stream serialisation (both attention kernels wait
// for their predecessor with griddepcontrol.wait before touching memory).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int G, bool kTma>
cudaError_t launch_chunks_t(const AttnParams& p, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t stream) {
  const long long nch = (p.max_seq_len + p.chunk - 1) / p.chunk;
  const dim3 grid(static_cast<unsigned>(nch * p.num_kv_heads), p.batch);
  constexpr int smem = kWarps * kRing * kBlockBytes + 1024;  // + alignment slack
  auto kern = fp8kv_attn_chunk_kernel<G, kTma>;
  // the attribute is per function and device; setting it again is harmless
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(kAttnThreads), smem, stream, p, mk, mv);
}

template <int G>
cudaError_t launch_chunks(const AttnParams& p, const CUtensorMap* mk, const CUtensorMap* mv, cudaStream_t stream) {
  if (mk) return launch_chunks_t<G, true>(p, *mk, *mv, stream);
  CUtensorMap none;
  memset(&none, 0, sizeof(none));
  return launch_chunks_t<G, false>(p, none, none, stream);
}

}  // namespace

int attn_part_stride() { return kPartStride; }
int attn_max_chunk() { return kMaxChunk; }

cudaError_t read_clear_attn_status(int* flags) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
  *flags = v;
  return e;
}

cudaError_t launch_fp8kv_attention(const AttnParams& p, const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                   cudaStream_t stream) {
  const int G = p.num_q_heads / p.num_kv_heads;
  cudaError_t e;
  switch (G) {
    case 1: e = launch_chunks<1>(p, tmap_k, tmap_v, stream); break;
    case 2: e = launch_chunks<2>(p, tmap_k, tmap_v, stream); break;
    case 4: e = launch_chunks<4>(p, tmap_k, tmap_v, stream); break;
    case 8: e = launch_chunks<8>(p, tmap_k, tmap_v, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_pdl(fp8kv_attn_combine_kernel, dim3(p.num_q_heads, p.batch), dim3(kHeadDim), 0, stream, p);
}

}  // namespace w8a8
