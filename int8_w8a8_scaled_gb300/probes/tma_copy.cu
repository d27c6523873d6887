// tma_copy.cu -- throughput of 2-D bulk-tensor copies (cp.async.bulk.tensor)
// into shared memory, the operand path of the scaled matmul, as a function
// of who issues them: one thread with a ring of copies in flight, several
// issuing warps per CTA, several CTAs per SM, box sizes, and a burst of
// copies waited for together.  Standalone (not part of the library):
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        int8_w8a8_scaled_gb300/probes/tma_copy.cu -o tma_copy && ./tma_copy
//
// Each CTA copies 128-byte-wide boxes of a 1 GiB buffer (128-byte swizzle,
// the matmul's layout) either from a 512-box set that stays in L2, or
// streaming through distinct boxes (DRAM).  Every wait is bounded (2 s of
// %globaltimer) and reported in the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

namespace {

__device__ int g_timeouts;

__device__ __forceinline__ uint32_t saddr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool bar_done(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = now_ns();
  for (uint32_t n = 0;; ++n) {
    if (bar_done(bar, parity)) return true;
    if ((n & 255u) == 255u && now_ns() - t0 > 2000000000ull) {
      atomicAdd(&g_timeouts, 1);
      return false;
    }
  }
}

__device__ __forceinline__ void load_box(uint32_t dst, const CUtensorMap* map, uint32_t bar, int row, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(row)
      : "memory");
}

struct Case {
  int box_rows;   // 64, 128 or 256 rows of 128 B
  int ring;       // copies in flight per CTA (ring slots)
  int producers;  // issuing warps per CTA (one lane each), every producers-th slot each
  int per_sm;     // CTAs per SM
  int stream;     // 1: distinct boxes (DRAM), 0: a 512-box set resident in L2
  int burst;      // 1: issue `ring` copies back to back, then wait for all of them
  int grid;       // 0: SMs x per_sm
};

__global__ void copy_kernel(const __grid_constant__ CUtensorMap map, Case c, int iters, long long nboxes,
                            unsigned long long* stamps) {
  extern __shared__ uint8_t raw[];
  __shared__ uint64_t bars[16];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const uint32_t box_bytes = c.box_rows * 128u;
  if (threadIdx.x == 0) {
    for (int r = 0; r < c.ring; ++r)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&bars[r])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int w = threadIdx.x / 32;
  if (threadIdx.x % 32 != 0 || w >= c.producers) return;
  auto box_of = [&](long long i) {
    const long long b = c.stream ? blockIdx.x * static_cast<long long>(iters) + i : (blockIdx.x * 37LL + i) % 512;
    return static_cast<int>((b % nboxes) * c.box_rows);
  };
  const uint64_t t0 = now_ns();
  if (c.burst) {
    for (int round = 0; round < iters / c.ring; ++round) {
      for (int s = 0; s < c.ring; ++s)
        load_box(saddr(ring + s * box_bytes), &map, saddr(&bars[s]), box_of(round * c.ring + s), box_bytes);
      const uint64_t t_issued = now_ns();
      bool ok = true;
      for (int s = 0; s < c.ring && ok; ++s) ok = bar_wait(saddr(&bars[s]), round & 1);
      if (blockIdx.x == 0 && round < 2) {
        stamps[1 + 2 * round] = t_issued - t0;
        stamps[2 + 2 * round] = now_ns() - t0;
      }
      if (!ok) return;
    }
  } else {
    int i = w;
    for (; i < iters; i += c.producers) {
      const int s = i % c.ring;
      if (i >= c.ring && !bar_wait(saddr(&bars[s]), ((i / c.ring) - 1) & 1)) break;
      load_box(saddr(ring + s * box_bytes), &map, saddr(&bars[s]), box_of(i), box_bytes);
    }
    // this producer's copies still in flight land before the CTA exits
    for (int j = i - c.producers; j >= 0 && j >= i - c.ring; j -= c.producers)
      bar_wait(saddr(&bars[j % c.ring]), (j / c.ring) & 1);
  }
  if (blockIdx.x == 0 && w == 0) stamps[0] = now_ns() - t0;
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

int main() {
  const long long rows = 8LL << 20;  // 1 GiB of 128-byte rows
  void* buf = nullptr;
  unsigned long long* stamps = nullptr;
  if (cudaMalloc(&buf, rows * 128) != cudaSuccess || cudaMalloc(&stamps, 16 * sizeof(unsigned long long)) != cudaSuccess) {
    printf("allocation failed\n");
    return 1;
  }
  cudaMemset(buf, 1, rows * 128);
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
      qr != cudaDriverEntryPointSuccess) {
    printf("cuTensorMapEncodeTiled unavailable\n");
    return 1;
  }
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const Case cases[] = {
      // box, ring, producers, per_sm, stream, burst, grid
      {128, 8, 1, 1, 0, 0, 0},  {128, 4, 1, 1, 0, 0, 0},  {128, 12, 1, 1, 0, 0, 0}, {64, 16, 1, 1, 0, 0, 0},
      {256, 4, 1, 1, 0, 0, 0},  {128, 8, 2, 1, 0, 0, 0},  {128, 8, 4, 1, 0, 0, 0},  {128, 4, 1, 2, 0, 0, 0},
      {128, 2, 1, 4, 0, 0, 0},  {128, 12, 1, 1, 0, 1, 0}, {128, 12, 1, 1, 0, 1, 1}, {128, 8, 1, 1, 0, 0, 1},
      {128, 8, 1, 1, 1, 0, 0},  {128, 8, 2, 1, 1, 0, 0},  {128, 2, 1, 4, 1, 0, 0}};
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  printf("%-6s %4s %4s %4s %4s %5s %5s %10s %10s %s\n", "source", "box", "ring", "prod", "CTA/SM", "burst", "grid",
         "GB/s", "GB/s/CTA", "burst issued/landed (ns)");
  for (const Case& c : cases) {
    CUtensorMap map;
    const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(c.box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    if (reinterpret_cast<EncodeFn>(fn)(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, buf, dims, strides, box, estr,
                                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      printf("tensor map encoding failed\n");
      return 1;
    }
    const int box_bytes = c.box_rows * 128;
    const int iters = (4 << 20) / box_bytes;  // 4 MiB per CTA
    const int smem = c.ring * box_bytes + 1024;
    const int grid = c.grid ? c.grid : sms * c.per_sm;
    cudaFuncSetAttribute(copy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    const long long nboxes = rows / c.box_rows;
    for (int r = 0; r < 2; ++r) copy_kernel<<<grid, 32 * c.producers, smem>>>(map, c, iters, nboxes, stamps);
    const int reps = 5;
    cudaEventRecord(e0);
    for (int r = 0; r < reps; ++r) copy_kernel<<<grid, 32 * c.producers, smem>>>(map, c, iters, nboxes, stamps);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    unsigned long long st[5] = {};
    cudaMemcpy(st, stamps, sizeof(st), cudaMemcpyDeviceToHost);
    const double gbs = static_cast<double>(grid) * iters * box_bytes * reps / (ms * 1e-3) / 1e9;
    printf("%-6s %4d %4d %4d %4d %5d %5d %10.1f %10.1f", c.stream ? "DRAM" : "L2", c.box_rows, c.ring, c.producers,
           c.per_sm, c.burst, grid, gbs, gbs / grid);
    if (c.burst) printf(" %llu/%llu, %llu/%llu", st[1], st[2], st[3], st[4]);
    printf("%s\n", cudaGetLastError() == cudaSuccess ? "" : "  (launch error)");
  }
  int timeouts = 0;
  cudaMemcpyFromSymbol(&timeouts, g_timeouts, sizeof(int));
  printf("bounded waits that gave up: %d\n", timeouts);
  return timeouts == 0 ? 0 : 1;
}
