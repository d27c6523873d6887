/*
 * w8a8.h -- C ABI of the GB300 (sm_103a) w8a8 scaled quantiser and scaled
 * matrix multiply.
 *
 * What it computes (sources are web pages, cited by title and section):
 *
 *  - Quantiser, "Enable scaled FP8 (e4m3fn) KV cache on ROCm (AMD GPU)",
 *    section "Scaling semantics": scale = AbsMax(x) / 448 for e4m3fn (the OCP
 *    MAXNORM), q = fp8(x / scale), x' = dequant(q) * scale.  The int8 variant
 *    uses 127.  Dynamic (runtime absmax) and static (given scale) modes, and
 *    per-tensor / per-token granularity, follow "[Kernel] Support Fp8
 *    Checkpoints (Dynamic + Static)" (PR description) and "[Kernel] Add w8a8
 *    CUTLASS kernels" (feature list).
 *  - Scaled matmul, "[Kernel] Add w8a8 CUTLASS kernels", feature list of
 *    cutlass_scaled_mm_dq: out = scale_a * scale_b * (A_q @ B_q) with
 *    symmetric fp8-e4m3 or int8 operands, per-tensor or per-token scale_a,
 *    per-tensor or per-output-channel scale_b, bf16 or fp16 output; B is
 *    "column-major" (stored [N, K], K contiguous) as the review thread of the
 *    same page requires.
 *
 * Exact rules where the pages are silent:
 *  - x / scale is a correctly rounded fp32 division;
 *  - e4m3: round to nearest, ties to the even code, saturate to +-448
 *    (+-inf included), NaN -> 0x7F, the sign of zero is kept;
 *  - int8: round half to even, saturate to [-128, 127], NaN -> 0;
 *  - absmax ignores NaN; an all-zero row or tensor gets scale 1.0;
 *  - epilogue: y = ((float)acc * scale_a[m|0]) * scale_b[n|0] in fp32, then
 *    round-to-nearest-even to bf16/fp16.  The fp8 path accumulates in fp32
 *    on the tensor cores; the int8 path accumulates exactly in int32.
 *
 * Conventions for every entry point:
 *  - All data pointers are DEVICE pointers (cudaMalloc'd or equivalent) on
 *    the current device, unless noted.  The caller owns every buffer; the
 *    library keeps no pointer after a call returns.
 *  - Matrices are row-major with a leading dimension in ELEMENTS (ld >= cols);
 *    sub-matrix views (ld > cols) are allowed.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream);
 *    they never synchronise, never allocate device memory and are safe to
 *    capture in a CUDA graph.  The first call on a device does a one-time
 *    host-side set-up (driver entry-point lookup, device attributes); make it
 *    before any stream capture.
 *  - Errors are reported by the return status; a status other than W8A8_OK
 *    means nothing was launched (except W8A8_ERR_CUDA, which reports a launch
 *    failure) and w8a8_last_error() holds a message.  Inputs are validated,
 *    never asserted on: no input makes the library abort the process.
 *  - Thread-safety: calls from several host threads are safe; the last-error
 *    message is per host thread.
 */
#ifndef W8A8_GB300_H
#define W8A8_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W8A8_API __attribute__((visibility("default")))
#else
#define W8A8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* w8a8_stream_t;

/* Element types. */
enum {
  W8A8_E4M3 = 0, /* OCP float8 e4m3fn, 1 byte */
  W8A8_INT8 = 1, /* signed 8-bit integer */
  W8A8_BF16 = 2, /* bfloat16, 2 bytes */
  W8A8_FP16 = 3, /* IEEE binary16, 2 bytes */
  W8A8_FP32 = 4, /* scaled_mm output for e4m3 only: y = (acc*scale_a)*scale_b, unrounded */
  W8A8_INT32 = 5 /* scaled_mm output for int8 only: the exact int32 accumulators, unscaled */
};

/* Scale granularity.  PER_ROW is per-token for activations [M, K] and
 * per-output-channel for weights stored [N, K]. */
enum { W8A8_PER_TENSOR = 0, W8A8_PER_ROW = 1 };

/* Quantiser mode: DYNAMIC computes the scales from absmax and writes them;
 * STATIC reads the given scales. */
enum { W8A8_DYNAMIC = 0, W8A8_STATIC = 1 };

/* Status codes. */
typedef int w8a8_status;
enum {
  W8A8_OK = 0,
  W8A8_ERR_INVALID_ARG = 1, /* null pointer, bad enum, size <= 0, ld < cols */
  W8A8_ERR_UNSUPPORTED = 2, /* dtype combination or size outside the limits */
  W8A8_ERR_MISALIGNED = 3,  /* base pointer or row stride not 16-byte aligned */
  W8A8_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
  W8A8_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  W8A8_ERR_NO_DEVICE = 6    /* current device is not an sm_103 GPU */
};

/* Device status bits reported by w8a8_device_status().
 *
 * No call returns a timeout status: calls only enqueue work and never wait
 * for the GPU, so a call cannot see a kernel's wait give up.  Every wait
 * inside a kernel is bounded instead (about 2 s); one that gives up lets its
 * kernel finish without hanging the GPU and sets W8A8_DEVICE_TIMEOUT in the
 * device status word, which w8a8_device_status() reads. */
enum { W8A8_DEVICE_TIMEOUT = 1 };

/* Message for the last failing call on this host thread ("" if none).
 * The string is owned by the library and valid until the next call. */
W8A8_API const char* w8a8_last_error(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
W8A8_API int w8a8_version(void);

/* ------------------------------------------------------------------------
 * Quantiser
 *
 * q[i, j] = encode(x[i, j] / scale[i or 0])
 *
 *  x        device, [rows, cols] of x_dtype (W8A8_BF16 or W8A8_FP16), leading
 *           dimension ld_x elements.
 *  q        device, [rows, cols] of q_dtype (W8A8_E4M3 or W8A8_INT8), leading
 *           dimension ld_q bytes.
 *  scale    device fp32, length rows (PER_ROW) or 1 (PER_TENSOR).  DYNAMIC
 *           writes absmax/448 (e4m3) or absmax/127 (int8), or 1.0 for an
 *           all-zero row/tensor; STATIC reads it.
 *  workspace, workspace_bytes
 *           device scratch of at least w8a8_scaled_quant_workspace_size()
 *           bytes (0 for every mode except DYNAMIC + PER_TENSOR, which uses
 *           16 bytes and clears them itself).  May be NULL when 0 is required.
 *  Alignment: the vectorised path is used when x, q, ld_x*2 and ld_q are
 *  16-byte aligned; other layouts are accepted and run a scalar path.
 *  Limits: rows, cols >= 1; rows * cols < 2^40.
 * ---------------------------------------------------------------------- */
W8A8_API size_t w8a8_scaled_quant_workspace_size(int64_t rows, int64_t cols, int gran,
                                        int mode);

W8A8_API w8a8_status w8a8_scaled_quant(const void* x, int x_dtype, int64_t rows,
                              int64_t cols, int64_t ld_x, void* q, int q_dtype,
                              int64_t ld_q, float* scale, int gran, int mode,
                              void* workspace, size_t workspace_bytes,
                              w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * Dequantiser (the KV-cache page's "scaled_fr_fp8_dequant")
 *
 * y[i, j] = round16(float(decode(q[i, j])) * scale[i or 0])
 *
 *  q      device [rows, cols] of q_dtype (E4M3 or INT8), leading dim ld_q.
 *  scale  device fp32, length rows (PER_ROW) or 1 (PER_TENSOR).
 *  y      device [rows, cols] of y_dtype (BF16 or FP16), leading dim ld_y.
 *  NaN codes decode to NaN.
 * ---------------------------------------------------------------------- */
W8A8_API w8a8_status w8a8_scaled_dequant(const void* q, int q_dtype, int64_t rows,
                                int64_t cols, int64_t ld_q, const float* scale,
                                int gran, void* y, int y_dtype, int64_t ld_y,
                                w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * Scaled matmul with a dequantising epilogue (cutlass_scaled_mm_dq)
 *
 * out[m, n] = round16(((float)sum_k A_q[m, k] * B_q[n, k]) * scale_a[m|0]
 *                     * scale_b[n|0])
 *
 *  a_q      device [M, K] codes of q_dtype, row-major, leading dim lda bytes.
 *  b_q      device weights stored [N, K] (K contiguous; the "column-major
 *           [K, N]" B of the CUTLASS page), leading dim ldb bytes.
 *  scale_a  device fp32, length M (a_gran = PER_ROW) or 1 (PER_TENSOR).
 *  scale_b  device fp32, length N (b_gran = PER_ROW) or 1 (PER_TENSOR); a
 *           merged QKV / gate-up weight shares one PER_TENSOR scale.
 *  out      device [M, N] of out_dtype, leading dim ldc (elements).
 *           out_dtype is BF16 or FP16 (the method's outputs), or for
 *           inspection FP32 (e4m3 only: y before the 16-bit rounding) or
 *           INT32 (int8 only: raw accumulators, scales ignored).
 *  q_dtype  W8A8_E4M3 (fp32 accumulation) or W8A8_INT8 (exact int32).
 *  workspace, workspace_bytes
 *           device scratch of at least w8a8_scaled_mm_workspace_size() bytes
 *           (0 for e4m3 without split-K or K halves), 256-byte aligned.  Its
 *           first 64 KiB hold split-K arrival counters that must be
 *           zero-filled before the first use; every call leaves them zero
 *           again and writes its other scratch (split-K partials, the K
 *           halves of CTA-pair tiles, int8 f16 planes) only after them, so one zero-filled buffer serves any sequence of
 *           scaled_mm calls of any shape on one stream.  Use it for nothing
 *           else, and give calls that may overlap on the GPU separate
 *           workspaces.
 *  Alignment (the CUTLASS page's "misaligned address" crash turned into a
 *  status): a_q and b_q 16-byte aligned and lda, ldb multiples of 16
 *  (W8A8_ERR_MISALIGNED otherwise).  out needs element alignment only.
 *  Limits: M, N, K >= 1 and < 2^31; for int8 also K % 16 == 0 and
 *  K <= 131071 (the int32 range).
 * ---------------------------------------------------------------------- */
W8A8_API size_t w8a8_scaled_mm_workspace_size(int64_t M, int64_t N, int64_t K,
                                     int q_dtype);

W8A8_API w8a8_status w8a8_scaled_mm(const void* a_q, int64_t lda, const void* b_q,
                           int64_t ldb, const float* scale_a, int a_gran,
                           const float* scale_b, int b_gran, void* out,
                           int64_t ldc, int64_t M, int64_t N, int64_t K,
                           int q_dtype, int out_dtype, void* workspace,
                           size_t workspace_bytes, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * w8a8_quant_scaled_mm -- dynamic per-token activation quantiser and scaled
 * matmul in one call: scale_a[m] = absmax_k |x[m, k]| / 448 (e4m3) or / 127
 * (int8), 1 for an all-zero row; A_q = sat_round(x / scale_a); then
 * out = w8a8_scaled_mm(A_q, b_q, scale_a (per row), scale_b).  The result
 * is bit for bit that of w8a8_scaled_quant (W8A8_PER_ROW, W8A8_DYNAMIC)
 * followed by w8a8_scaled_mm.  ("[Kernel] Support Fp8 Checkpoints (Dynamic
 * + Static)": dynamic per-token activation scales; "[Kernel] Add w8a8
 * CUTLASS kernels": the scaled matmul.)
 *
 *  x         [M, K] BF16 or FP16 activations (x_dtype), row stride ld_x
 *            elements (ld_x >= K).
 *  b_q, ldb, scale_b, b_gran, out, ldc, M, N, K, q_dtype, out_dtype
 *            as for w8a8_scaled_mm.
 *  scale_a_out  [M] fp32, receives the per-token scales; may be NULL.
 *  route     W8A8_ROUTE_AUTO: one kernel where it pays (below), else two
 *            steps; W8A8_ROUTE_ONE_KERNEL: one kernel, W8A8_ERR_UNSUPPORTED
 *            where it cannot run; W8A8_ROUTE_TWO_STEP: quantiser, then
 *            matmul.
 *  workspace   device scratch of at least
 *            w8a8_quant_scaled_mm_workspace_size(M, N, K, q_dtype) bytes,
 *            256-byte aligned (the quantised activations when the two
 *            steps run separately, split-K partials).  Split-K arrival
 *            counters live at its head: zero-fill it once before first use;
 *            every call leaves them zero.
 *
 * The one-kernel route (e4m3, every token in one narrow matmul tile, x 16-byte
 * aligned with ld_x * 2 a multiple of 16, K a multiple of 16) quantises the
 * activations inside the matmul.  The two-step route runs the quantiser into
 * the workspace and then the matmul; AUTO takes it (measured faster on
 * GB300 at every decode shape).  Errors as for w8a8_scaled_mm and
 * w8a8_scaled_quant.
 * ---------------------------------------------------------------------- */
#define W8A8_ROUTE_AUTO 0
#define W8A8_ROUTE_ONE_KERNEL 1
#define W8A8_ROUTE_TWO_STEP 2

W8A8_API size_t w8a8_quant_scaled_mm_workspace_size(int64_t M, int64_t N, int64_t K, int q_dtype);

W8A8_API w8a8_status w8a8_quant_scaled_mm(const void* x, int x_dtype, int64_t ld_x, const void* b_q,
                                 int64_t ldb, const float* scale_b, int b_gran, void* out,
                                 int64_t ldc, int64_t M, int64_t N, int64_t K, int q_dtype,
                                 int out_dtype, float* scale_a_out, int route, void* workspace,
                                 size_t workspace_bytes, w8a8_stream_t stream);

/* Kernel configuration of one scaled_mm call (tests and tuning).
 *  swap_ab   1: the weight rows N are the 128-row MMA side and the tokens M
 *            the narrow side (small-M / decode regime); 0: tokens M on the
 *            128-row side (large-M regime).
 *  block_n   width of the narrow MMA side: 16..256, multiple of 16.
 *  split_k   number of K slices reduced in a fixed order (1..16).
 *  stages    depth of the shared-memory ring (2..8); 0 = automatic.
 *  ctas_per_sm  cap on the persistent CTAs per SM (1..4); 0 = as many as
 *            the kernel's shared memory, registers and TMEM allow.
 *  reduce    how split_k > 1 slices are summed (both in slice order 0..S-1,
 *            so the result does not depend on scheduling):
 *            W8A8_REDUCE_GLOBAL  partial tiles in the workspace, the last
 *                                slice to arrive sums them;
 *            W8A8_REDUCE_CLUSTER the slices of a tile run as one
 *                                thread-block cluster: each writes its
 *                                partial tile to the workspace and, after
 *                                a cluster barrier, sums 1/split_k of the
 *                                tile's rows over all partials (split_k
 *                                <= 8);
 *            W8A8_REDUCE_AUTO    the cluster reduction when split_k <= 8,
 *                                else the global one.
 *  cta_pair  1: tiles of 256 token rows computed by a pair of CTAs on two SMs
 *            with one tcgen05 MMA stream (cta_group::2): each CTA stages its
 *            128 rows of A and half of the block_n columns of B (swap_ab 0;
 *            block_n 64, 96, 128, 192, 224 or 256 for e4m3, 128 or 256 for
 *            int8); 0: one CTA per 128-row tile.  With pairs split_k is 1,
 *            or 2 (e4m3): when the tiles leave a last round that keeps at
 *            most half of the pairs (one per two SMs) busy, each tile of
 *            that round is computed as two K halves on two pairs, whose fp32
 *            partial tiles go through the workspace and are summed in half
 *            order (deterministic) by the second to finish.
 * Fields set to 0 (except swap_ab and cta_pair) mean "choose automatically". */
#define W8A8_REDUCE_AUTO 0
#define W8A8_REDUCE_GLOBAL 1
#define W8A8_REDUCE_CLUSTER 2

typedef struct {
  int swap_ab;
  int block_n;
  int split_k;
  int stages;
  int ctas_per_sm;
  int reduce;
  int cta_pair;
} w8a8_mm_config;

/* The configuration w8a8_scaled_mm() picks for this problem (host only). */
W8A8_API w8a8_status w8a8_scaled_mm_pick_config(int64_t M, int64_t N, int64_t K,
                                       int q_dtype, w8a8_mm_config* cfg);

/* Workspace bytes needed by an explicit configuration. */
W8A8_API size_t w8a8_scaled_mm_config_workspace_size(int64_t M, int64_t N, int64_t K,
                                            int q_dtype,
                                            const w8a8_mm_config* cfg);

/* w8a8_scaled_mm with an explicit configuration (validated: W8A8_ERR_
 * UNSUPPORTED for a block_n / split_k / stages value outside the limits). */
W8A8_API w8a8_status w8a8_scaled_mm_with_config(
    const void* a_q, int64_t lda, const void* b_q, int64_t ldb,
    const float* scale_a, int a_gran, const float* scale_b, int b_gran,
    void* out, int64_t ldc, int64_t M, int64_t N, int64_t K, int q_dtype,
    int out_dtype, void* workspace, size_t workspace_bytes,
    const w8a8_mm_config* cfg, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * Merged-layer (QKV / gate-up) helpers
 *
 * A merged weight stored [N, K] consists of nshards consecutive row shards
 * (shard_rows[i] rows each, HOST array, 1 <= nshards <= 16, sum = N) that may
 * have been quantised with their own per-tensor scales shard_scales[i]
 * (DEVICE fp32 array).  "[Kernel] Support Fp8 Checkpoints (Dynamic +
 * Static)" runs such a layer as one GEMM either with the shard scales fused
 * into the epilogue or after rewriting every shard to one shared scale.
 * ---------------------------------------------------------------------- */

/* scale_b[n] = shard_scales[shard of row n]  (device fp32 [N]).  Passing the
 * result as a PER_ROW scale_b to w8a8_scaled_mm applies each shard's scale in
 * the fused epilogue. */
W8A8_API w8a8_status w8a8_expand_shard_scales(const float* shard_scales,
                                              const int64_t* shard_rows,
                                              int nshards, float* scale_b,
                                              w8a8_stream_t stream);

/* q_out[r, j] = encode(decode(q[r, j]) * (s_i / s_max)) with s_max the
 * largest shard scale (written to scale_out[0], device fp32 [1]); the ratio
 * is one IEEE fp32 division, the product one fp32 multiplication, the encode
 * the quantiser's rounding and saturation.  q and q_out are [N, cols] codes
 * of q_dtype with leading dimensions ld_q / ld_out bytes; q_out may equal q
 * (in place, same leading dimension). */
W8A8_API w8a8_status w8a8_requant_shards(const void* q, int q_dtype, int64_t cols,
                                         int64_t ld_q, const float* shard_scales,
                                         const int64_t* shard_rows, int nshards,
                                         void* q_out, int64_t ld_out,
                                         float* scale_out, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * Decode attention over an fp8 (e4m3) KV cache
 *
 * "Enable scaled FP8 (e4m3fn) KV cache on ROCm (AMD GPU)", section
 * "Scaling semantics": the cache holds e4m3 codes written with one
 * per-tensor scaling factor for K and one for V (absmax / 448), and the
 * paged attention kernel dequantises as decode(code) * kv_scale.  For one
 * query token per sequence and every query head h (KV head h / G,
 * G = num_q_heads / num_kv_heads):
 *   s_t = sm_scale * sum_d q[b,h,d] * (decode(K[t,d]) * k_scale)
 *   out[b,h,:] = sum_t softmax(s)_t * (decode(V[t,:]) * v_scale)
 * over the tokens t < seq_lens[b] (an empty sequence gives zeros).
 *
 * Layouts (all DEVICE memory, caller-owned, 16-byte aligned caches):
 *   q, out        [batch, num_q_heads, 128] contiguous, bf16 or fp16
 *   k/v_cache     e4m3 token rows of num_kv_heads * 128 bytes.  Without a
 *                 block table (block_table NULL) token t of sequence b is
 *                 row b * max_seq_len + t.  With one (int32
 *                 [batch, max_blocks], the paged cache) it is row
 *                 block_table[b * max_blocks + t / block_size] * block_size
 *                 + t % block_size, and num_blocks blocks exist; tokens
 *                 whose block id is outside [0, num_blocks) are skipped.
 *   seq_lens      int32 [batch], clamped to [0, max_seq_len]
 *   k_scale, v_scale  fp32 [1]
 * head_dim must be 128 and G one of 1, 2, 4, 8.  The workspace holds the
 * per-chunk partial results (w8a8_fp8_kv_attention_workspace_size).  Its
 * size is an upper bound on purpose: it assumes chunks of 64 tokens, the
 * smallest the kernel picks, so one size serves every call with the same
 * batch, heads and max_seq_len whatever the GPU (the kernel takes chunks of
 * up to 512 tokens, and then uses an eighth of it).  No
 * allocation, no synchronisation; graph-capturable.  Errors: INVALID_ARG
 * (null pointer, sizes, head_dim, G), MISALIGNED (cache base not 16-byte
 * aligned), WORKSPACE (too small), CUDA (launch).  The workspace size is
 * 0 for invalid sizes, including a size beyond 2^62 bytes. */
W8A8_API size_t w8a8_fp8_kv_attention_workspace_size(int64_t batch, int64_t num_q_heads,
                                                     int64_t max_seq_len);

W8A8_API w8a8_status w8a8_fp8_kv_decode_attention(
    const void* q, int q_dtype, int64_t batch, int64_t num_q_heads, int64_t num_kv_heads,
    int64_t head_dim, const void* k_cache, const void* v_cache, int64_t max_seq_len,
    const int32_t* block_table, int64_t block_size, int64_t max_blocks, int64_t num_blocks,
    const int32_t* seq_lens, const float* k_scale, const float* v_scale, float sm_scale,
    void* out, int out_dtype, void* workspace, size_t workspace_bytes, w8a8_stream_t stream);

/* ------------------------------------------------------------------------
 * Scaled matmul without a caller-provided workspace
 *
 * No counterpart on the source pages: this entry point exists for callers
 * that cannot allocate device memory where they run the matmul -- code
 * running inside an allocator hook or a CUDA-graph-capturing runtime that
 * forbids new allocations, plug-ins handed only their operand and output
 * buffers, or processes whose memory is fully reserved by another runtime.
 *
 * Same arguments and results as w8a8_scaled_mm, minus the workspace.  The
 * scratch the matmul needs (split-K arrival counters and partial tiles)
 * lives in one fixed array of w8a8_scaled_mm_noalloc_max_scratch() bytes
 * (8 MiB + 64 KiB) that the library defines in device memory: every GPU that
 * loads the library holds it until the process exits.  Nothing is allocated
 * or freed by the call, not even through a library routine.
 *
 *  - It runs the configuration w8a8_scaled_mm_pick_config() gives, except
 *    that CTA-pair tiles whose last-round K halves (split_k 2) need more
 *    scratch than the array holds run whole (split_k 1).  Problems whose
 *    scratch need still exceeds the array are rejected with
 *    W8A8_ERR_WORKSPACE and a message; in practice this covers e4m3 at
 *    every size and int8 only where its widened operand planes fit.
 *  - The array is shared by every call on a device and keeps the previous
 *    call's contents.  A call that uses split-K arrival counters clears
 *    them first (an asynchronous memset of those counters on `stream`);
 *    every other byte it reads it has written itself.  Calls that may
 *    overlap on the GPU (different streams without ordering) race on the
 *    array: serialise them.
 *  - The first call on a device (and again after the device's context has
 *    been replaced, e.g. by cudaDeviceReset) looks up the array's device
 *    address with a host query, with that device current; make that first
 *    call before any stream capture.
 */
W8A8_API size_t w8a8_scaled_mm_noalloc_max_scratch(void);

W8A8_API w8a8_status w8a8_scaled_mm_noalloc(const void* a_q, int64_t lda, const void* b_q,
                                            int64_t ldb, const float* scale_a, int a_gran,
                                            const float* scale_b, int b_gran, void* out,
                                            int64_t ldc, int64_t M, int64_t N, int64_t K,
                                            int q_dtype, int out_dtype,
                                            w8a8_stream_t stream);

/* Debug: per-CTA phase trace of subsequent scaled_mm launches (process
 * wide).  buf is a device buffer of `bytes` bytes; each CTA c < bytes / 128
 * writes sixteen 64-bit words at buf[16c..16c+15]: %globaltimer (ns) at
 * kernel entry [0], after its prologue (barriers, TMEM) [1], when the
 * preceding kernel's dependency was released [2], when its first operand
 * stage landed [3], when its last MMA was issued [4], when its epilogue
 * finished [5], at exit [6], its SM id [7], and for its last unit: when the
 * accumulator was complete [8] and drained [9], and with a cluster split,
 * after the cluster barrier [10] and its share of the reduction [11]; in a
 * matmul that quantises its own activations, when the token maxima [12],
 * the token scales [13] and the first token stage [14] were ready; unused
 * words are left as they were.  Each launch overwrites the buffer.  Launches
 * on CTA pairs (cta_pair = 1) write no stamps.  NULL turns tracing off (the
 * default).  A diagnostic aid, not part of the hot path: concurrent launches
 * share the buffer. */
W8A8_API w8a8_status w8a8_debug_mm_trace(void* buf, size_t bytes);

/* Reads and clears the library's device-side status word on the current
 * device (W8A8_DEVICE_* bits; a kernel sets W8A8_DEVICE_TIMEOUT when one of
 * its bounded pipeline waits gave up instead of hanging).  This call
 * synchronises the device; use it in tests and diagnostics, not on a hot
 * path. */
W8A8_API w8a8_status w8a8_device_status(int* flags);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_GB300_H */
