// int8_routes.cu -- throughput of the warp-level MMA instructions an int8
// GEMM could use on this GPU, with register operands and no memory traffic
// (8 independent accumulator tiles per warp, 8 warps per CTA): mma.sync
// m16n8k32 s8 -> s32, and m16n8k16 f16 -> f32 for comparison.  The tcgen05
// routes are measured by the library's own matmul (bench.py).
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

template <int KIND>
__global__ void __launch_bounds__(256) mma_loop(int iters, int* out) {
  uint32_t a0 = threadIdx.x, a1 = a0 * 3u, a2 = a0 * 5u, a3 = a0 * 7u, b0 = a0 ^ 0x55u, b1 = a0 ^ 0x33u;
  float f[8][4] = {};
  int s[8][4] = {};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (KIND == 0) {
        asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+r"(s[j][0]), "+r"(s[j][1]), "+r"(s[j][2]), "+r"(s[j][3])
                     : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      } else {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                     : "+f"(f[j][0]), "+f"(f[j][1]), "+f"(f[j][2]), "+f"(f[j][3])
                     : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      }
    }
  }
  int acc = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) acc += s[j][0] + s[j][3] + static_cast<int>(f[j][0] + f[j][3]);
  if (acc == 123456789) out[0] = acc;
}

int main() {
  int* out;
  cudaMalloc(&out, 4);
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  for (int kind = 0; kind < 2; ++kind) {
    for (int per_sm : {2, 4, 8}) {
      const int iters = 4096;
      dim3 grid(sms * per_sm), block(256);
      cudaEvent_t e0, e1;
      cudaEventCreate(&e0); cudaEventCreate(&e1);
      if (kind == 0) mma_loop<0><<<grid, block>>>(16, out); else mma_loop<1><<<grid, block>>>(16, out);
      cudaEventRecord(e0);
      if (kind == 0) mma_loop<0><<<grid, block>>>(iters, out); else mma_loop<1><<<grid, block>>>(iters, out);
      cudaEventRecord(e1);
      cudaEventSynchronize(e1);
      float ms; cudaEventElapsedTime(&ms, e0, e1);
      const double mmas = double(grid.x) * 8 /*warps*/ * iters * 8;
      const double ops = mmas * 2.0 * 16 * 8 * (kind == 0 ? 32 : 16);
      printf("%s  %d CTAs/SM: %.1f T(FL)OP/s  (%s)\n", kind == 0 ? "mma.sync s8 m16n8k32 " : "mma.sync f16 m16n8k16",
             per_sm, ops / (ms * 1e-3) / 1e12, cudaGetErrorString(cudaGetLastError()));
    }
  }
  return 0;
}
