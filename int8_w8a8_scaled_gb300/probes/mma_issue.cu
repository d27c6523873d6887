// mma_issue.cu -- rate of tcgen05.mma issued back to back on operands already
// in shared memory (no copies, no epilogue): the ceiling of the scaled
// matmul's MMA stream per SM.  One CTA per SM; one thread issues 4 MMAs per
// 128-deep K step (K = 32 each for e4m3, 16 for f16) into one accumulator,
// or alternates two accumulators, or two threads (in different warps) each
// feed their own accumulator.  Standalone (not part of the library):
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        int8_w8a8_scaled_gb300/probes/mma_issue.cu -o mma_issue && ./mma_issue
#include <cstdio>

#include "../csrc/sm103_ptx.cuh"
using namespace w8a8;

__global__ void __launch_bounds__(128, 1) mma_probe(int rounds, int mode, int n, int kind16, unsigned long long* out) {
  extern __shared__ uint8_t raw[];
  __shared__ uint64_t done_bar[2];
  __shared__ uint32_t tmem_slot;
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  for (int i = tid; i < (48 * 1024) / 16; i += 128) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    mbar_init(smem_addr(&done_bar[0]), 1);
    mbar_init(smem_addr(&done_bar[1]), 1);
    fence_barrier_init();
  }
  fence_proxy_async_shared();
  __syncthreads();
  if (warp == 1) { tmem_alloc(smem_addr(&tmem_slot), 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  // A and B format 0: e4m3 for kind::f8f6f4, f16 for kind::f16; fp32 accumulator
  const uint32_t idesc = make_idesc(128, n, 0);
  const uint64_t da = smem_desc_sw128(smem_addr(sm)), db = smem_desc_sw128(smem_addr(sm + 16384));
  const uint64_t t0 = global_timer_ns();
  // mode 0: one issuer, one accumulator; 1: one issuer, two accumulators alternating per K step;
  // 2: two issuers (warps 0 and 2), one accumulator each
  const bool issuer = lane == 0 && (warp == 0 || (mode == 2 && warp == 2));
  if (issuer) {
    const int which = warp == 0 ? 0 : 1;
    const int my = mode == 2 ? rounds / 2 : rounds;
    for (int r = 0; r < my; ++r) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t d = tbase + (mode == 1 ? ((kk & 1) * 256) : which * 256);
        const uint32_t acc = (r > 0 || kk >= (mode == 1 ? 2 : 1)) ? 1u : 0u;
        if (kind16) mma_f16(d, da + 2 * kk, db + 2 * kk, idesc, acc);
        else mma_f8f6f4(d, da + 2 * kk, db + 2 * kk, idesc, acc);
      }
    }
    mma_commit(smem_addr(&done_bar[which]));
    mbar_wait(smem_addr(&done_bar[which]), 0);
  }
  __syncthreads();
  if (tid == 0 && blockIdx.x == 0) out[0] = global_timer_ns() - t0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long* out;
  cudaMalloc(&out, 64);
  const int smem = 160 * 1024;  // one CTA per SM
  cudaFuncSetAttribute(mma_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  const int rounds = 2048;
  struct C { int mode, n, k16; const char* name; };
  const C cases[] = {{0, 256, 0, "f8f6f4 N=256, 1 issuer, 1 acc"}, {1, 256, 0, "f8f6f4 N=256, 1 issuer, 2 accs"},
                     {2, 256, 0, "f8f6f4 N=256, 2 issuers"}, {0, 128, 0, "f8f6f4 N=128, 1 issuer, 1 acc"},
                     {1, 128, 0, "f8f6f4 N=128, 1 issuer, 2 accs"}, {0, 64, 0, "f8f6f4 N=64, 1 issuer, 1 acc"},
                     {0, 256, 1, "f16 N=256, 1 issuer, 1 acc"}, {1, 256, 1, "f16 N=256, 1 issuer, 2 accs"}};
  for (const C& c : cases) {
    mma_probe<<<sms, 128, smem>>>(64, c.mode, c.n, c.k16, out);
    cudaEventRecord(e0);
    mma_probe<<<sms, 128, smem>>>(rounds, c.mode, c.n, c.k16, out);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms;
    cudaEventElapsedTime(&ms, e0, e1);
    unsigned long long ns;
    cudaMemcpy(&ns, out, 8, cudaMemcpyDeviceToHost);
    const double flop = 2.0 * 128 * c.n * (c.k16 ? 16 : 32) * 4.0 * rounds * sms;
    printf("%-34s: %8.1f us, %7.1f TFLOP/s, %6.1f ns per MMA (CTA 0: %llu ns) err=%s\n", c.name, ms * 1e3,
           flop / (ms * 1e-3) / 1e12, ms * 1e6 / (4.0 * rounds), ns, cudaGetErrorString(cudaGetLastError()));
  }
  int st = 0;
  cudaMemcpyFromSymbol(&st, g_device_status, sizeof(int));
  printf("device status %d\n", st);
  return 0;
}
