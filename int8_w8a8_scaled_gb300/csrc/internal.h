// internal.h -- declarations shared by the library's translation units (not
// part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/w8a8.h"

namespace w8a8 {

// Parameters of one scaled-matmul launch.  "P" is the operand on the
// 128-row MMA side, "Q" the operand on the narrow (block_n) side.  Without
// swap P = activations [M, K] and Q = weights [N, K]; with swap the roles
// are exchanged, which keeps small-M (decode) problems on the tensor cores
// with M padded only up to block_n.
struct MmParams {
  int M, N, K;
  int tiles_p, tiles_q;  // tiles along the P rows (128 each) and Q rows (block_n each)
  int num_kb;            // K blocks of 128 bytes
  int kb_per_split;      // K blocks per split
  int splits;            // >= 1; > 1 reduces fp32 partials in split order
  int cluster;           // 1: the splits of a tile form one thread-block cluster;
                         // after a cluster barrier each CTA sums 1/splits of the
                         // tile's rows from the workspace partials
  int dsmem_reduce;      // cluster split whose partial tiles stay in each CTA's
                         // shared memory (stage ring) and are summed from there
                         // through distributed shared memory
  const float* scale_a;
  int a_per_row;
  const float* scale_b;
  int b_per_row;
  void* out;
  long long ldc;
  int out_vec_ok;        // 16-byte vector stores allowed along n
  float* partial;        // [tiles][splits][128 * block_n] fp32 / int32 (splits > 1)
  unsigned* counters;    // [tiles] arrival counters (splits > 1, no cluster), left zero
  int kchunk_kb;         // int8 path: K blocks per exact fp32 chunk
  int num_sms;           // persistent grid = min(units, num_sms * resident CTAs per SM)
  int pdl;               // launch with programmatic stream serialisation
  int prefetch_kb;       // weight K blocks of the first unit prefetched into L2 early
  // CTA-pair tiles only: the last, partial round of pair tiles, when it
  // would leave at least half of the pairs idle, is run as two K halves per
  // tile ([0, tail_kb_half) and [tail_kb_half, num_kb)) on two pairs; each
  // CTA writes its fp32 half into `partial` ([tail][half][rank][128 *
  // block_n]) and the last of the tile's two halves to arrive on
  // counters[tail * 2 + rank] sums them in half order
  int tail_tiles;        // 0: every tile whole
  int tail_kb_half;
  int max_ctas_per_sm;   // 0: as many as fit; else cap the persistent grid per SM
  // fused activation quantiser (swap-AB e4m3 decode, one token tile): the
  // kernel quantises x itself (scale_a is then unused)
  const void* x;         // [M, K] bf16 / fp16 activations
  long long ld_x;        // row stride of x in elements
  int x_fp16;            // 1: x is fp16, 0: bf16
  float* scale_a_out;    // [M] per-token scales the kernel computed (nullable)
  int fq_rows;           // 1: the tokens' whole rows are staged in shared memory
  unsigned long long* trace;  // debug: per-CTA phase stamps (null = off)
  int trace_ctas;             // CTAs the trace buffer has room for
};

// Debug trace buffer for subsequent scaled_mm launches (null disables).
void set_mm_trace(unsigned long long* buf, int ctas);
void get_mm_trace(unsigned long long** buf, int* ctas);

// OUT_RAW: fp32 y = (acc * s_a) * s_b for the fp8 path, raw int32
// accumulators for the int8 path.
enum OutKind { OUT_BF16 = 0, OUT_FP16 = 1, OUT_RAW = 2 };

// fp8 e4m3 GEMM (tcgen05 kind::f8f6f4).  Tensor maps are uint8 [rows, K]
// with a 128x128 box for P and a block_n x 128 box for Q, 128-byte swizzle.
cudaError_t launch_fp8_gemm(const CUtensorMap& tmap_p, const CUtensorMap& tmap_q,
                            const MmParams& p, int block_n, bool swap, int out_kind,
                            int stages, cudaStream_t stream);

// Pairs in the persistent CTA-pair grid: one per two SMs, at most one per
// tile.
inline int pair_grid_pairs(long long tiles, int num_sms) {
  const long long p = tiles < num_sms / 2 ? tiles : num_sms / 2;
  return p < 1 ? 1 : static_cast<int>(p);
}
// The same matmul on CTA pairs (gemm2sm.cu): 256 x block_n tiles, tokens on
// the 128-row side of each CTA (no swap; split-K only as the last round's K
// halves, p.tail_tiles).  tmap_a boxes 128 rows, tmap_b block_n / 2 rows.
cudaError_t launch_gemm_pair(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const MmParams& p, int block_n,
                             bool int8, int out_kind, int stages, cudaStream_t stream);
int gemm_pair_smem_bytes(int block_n, int stages);

// int8 GEMM.  Operands are first widened to f16 planes (exact), then
// multiplied with tcgen05 kind::f16 in K chunks small enough that the fp32
// accumulator is exact; each chunk is drained into an int32 total.
cudaError_t launch_int8_widen(const void* src, long long ld_src, int rows, int K,
                              void* dst_f16, cudaStream_t stream);
// The decode matmul that quantises its own activations (prm.x); tmap_p maps
// the weights (swap-AB).  block_n 16 / 32 / 64, e4m3 weights.
cudaError_t launch_fused_quant_gemm(const CUtensorMap& tmap_p, const MmParams& p, int block_n, int out_kind,
                                    int stages, cudaStream_t stream);
cudaError_t launch_int8_gemm(const CUtensorMap& tmap_p, const CUtensorMap& tmap_q,
                             const MmParams& p, int block_n, bool swap, int out_kind,
                             int stages, cudaStream_t stream);

// Synchronises the device, then reads and clears the device status word.
cudaError_t read_clear_device_status(int* flags);
// Reads and clears the quantiser kernels' status word (call after a sync).
cudaError_t read_clear_quant_status(int* flags);

// Shared-memory bytes a GEMM launch needs (ring + barriers + alignment).
int gemm_smem_bytes(int block_n, int stages);
// Largest split_k the cluster reduction takes (one portable cluster).
constexpr int kMaxClusterSplit = 8;
int max_stages_for(int block_n, int smem_budget);

// Decode attention over an e4m3 KV cache (attention.cu).  Caches hold
// token rows of num_kv_heads * 128 codes; token t of sequence b sits in row
// b * max_seq_len + t, or with a block table in row
// block_table[b * max_blocks + t / block_size] * block_size + t % block_size.
struct AttnParams {
  const void* q;        // [batch, num_q_heads, 128] bf16 / fp16
  int q_fp16;
  int q_vec;            // q is 8-byte aligned (vector loads)
  const void* k_cache;  // e4m3 rows
  const void* v_cache;
  const int* block_table;  // null: contiguous per-sequence rows
  int block_size, max_blocks, num_blocks;
  const int* seq_lens;  // [batch], clamped to [0, max_seq_len]
  const float* k_scale; // [1]
  const float* v_scale; // [1]
  float sm_scale;
  void* out;            // [batch, num_q_heads, 128] bf16 / fp16
  int out_fp16;
  float* partial;       // [batch, num_q_heads, chunks, attn_part_stride()] fp32
  int batch, num_q_heads, num_kv_heads, max_seq_len;
  int chunk;            // tokens per CTA, <= attn_max_chunk()
};
int attn_part_stride();
int attn_max_chunk();
// tmap_k / tmap_v: 2-D uint8 tensor maps over the caches ({num_kv_heads *
// 128, rows}, box {128, 16}, 128-byte swizzle) for the bulk-tensor path
// (contiguous caches, or 16 | block_size), or null for per-lane copies.
cudaError_t launch_fp8kv_attention(const AttnParams& p, const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                   cudaStream_t stream);
// Reads and clears the attention kernels' status word (call after a sync).
cudaError_t read_clear_attn_status(int* flags);

// Quantiser / dequantiser launchers.
struct QuantArgs {
  const void* x;
  int x_kind;  // 0 bf16, 1 fp16
  long long rows, cols, ld_x;
  void* q;
  int q_kind;  // 0 e4m3, 1 int8
  long long ld_q;
  float* scale;
  int per_row;
  int dynamic;
  unsigned* amax_word;  // dynamic per-tensor only
  int vec;              // 16-byte vector path allowed
};
cudaError_t launch_quant(const QuantArgs& a, int num_sms, cudaStream_t stream);

struct DequantArgs {
  const void* q;
  int q_kind;
  long long rows, cols, ld_q;
  const float* scale;
  int per_row;
  void* y;
  int y_kind;
  long long ld_y;
  int vec;
};
cudaError_t launch_dequant(const DequantArgs& a, int num_sms, cudaStream_t stream);

// Sets the message returned by w8a8_last_error() on this host thread.
void set_last_error(const char* msg);

// Split-K arrival counters: a fixed region at the head of every matmul
// workspace (one 32-bit counter per output tile), left zero by every call
// that uses it.  Scratch data always lives after the region.
constexpr size_t kCounterSlots = 16384;
constexpr size_t kCounterRegion = kCounterSlots * sizeof(unsigned);

// Bytes at the head of the workspace whose counters this matmul uses under
// `cfg` (complete: no automatic fields) on the current device, 0 when it
// uses none.
size_t mm_counter_bytes(long long M, long long N, long long K, int q_dtype, const w8a8_mm_config& cfg);

// Row shards of a merged weight: cumulative row ends.
constexpr int kMaxShards = 16;
struct ShardTable {
  int n;
  long long end[kMaxShards];
};
cudaError_t launch_expand_shard_scales(const float* shard_scales, const ShardTable& t, float* out,
                                       cudaStream_t stream);
cudaError_t launch_requant_shards(const void* q, int q_kind, long long cols, long long ld,
                                  const float* shard_scales, const ShardTable& t, void* out, long long ld_out,
                                  float* scale_out, cudaStream_t stream);

}  // namespace w8a8
