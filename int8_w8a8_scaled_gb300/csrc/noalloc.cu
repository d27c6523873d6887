// noalloc.cu -- a scaled_mm entry point that needs no caller-provided
// workspace and allocates nothing.
//
// Some callers cannot allocate device memory at the point where they run a
// matmul: code that executes inside a framework's own allocator hook, a
// plug-in that is handed only the operand and output buffers, or a runtime
// that has already reserved all device memory for itself.  For them this
// file keeps the matmul's scratch (the split-K arrival counters and the
// split-K partial tiles) in one file-scope device array of fixed size, which
// the CUDA runtime creates when the library is loaded on a device and keeps
// until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/w8a8.h"

#include "internal.h"

// 8 MiB of split-K partials plus the counter region at the head.
static constexpr size_t kScratchBytes = (8u << 20) + w8a8::kCounterRegion;

// The scratch itself: one per device that loads the library, zero at load.
static __device__ __align__(256) unsigned char g_w8a8_static_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

// Device address of the array, per device, remembered together with the
// context it was looked up in: a context created later on the same device
// (after cudaDeviceReset, say) holds the array at another address, and the
// lookup is then made again.
struct ScratchAddr {
  CUcontext ctx = nullptr;
  void* ptr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch array on the current device.  The array's
// name in host code is only a host-side handle, so its address is looked up
// with cudaGetSymbolAddress, with the device current, the first time a
// device (in a given context) is used.
w8a8_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    w8a8::set_last_error("scaled_mm_noalloc: no usable current CUDA device");
    return W8A8_ERR_NO_DEVICE;
  }
  CtxGetCurrentFn get = ctx_get_current_fn();
  if (!get) {
    w8a8::set_last_error("scaled_mm_noalloc: cuCtxGetCurrent is not available from the driver");
    return W8A8_ERR_CUDA;
  }
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) ctx = nullptr;  // none yet: the lookup below creates the runtime's
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& s = g_scratch[dev];
  if (!ctx || !s.ptr || s.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_w8a8_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      w8a8::set_last_error("scaled_mm_noalloc: cudaGetSymbolAddress of the scratch array failed");
      return W8A8_ERR_CUDA;
    }
    if (get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    s.ptr = p;
    s.ctx = ctx;
  }
  *out = s.ptr;
  return W8A8_OK;
}

}  // namespace

extern "C" {

size_t w8a8_scaled_mm_noalloc_max_scratch(void) { return kScratchBytes; }

w8a8_status w8a8_scaled_mm_noalloc(const void* a_q, int64_t lda, const void* b_q, int64_t ldb,
                                   const float* scale_a, int a_gran, const float* scale_b, int b_gran,
                                   void* out, int64_t ldc, int64_t M, int64_t N, int64_t K, int q_dtype,
                                   int out_dtype, w8a8_stream_t stream) {
  if (M < 1 || N < 1 || K < 1) {
    // let the regular entry point produce the message
    return w8a8_scaled_mm(a_q, lda, b_q, ldb, scale_a, a_gran, scale_b, b_gran, out, ldc, M, N, K, q_dtype,
                          out_dtype, nullptr, 0, stream);
  }
  w8a8_mm_config cfg;
  if (w8a8_scaled_mm_pick_config(M, N, K, q_dtype, &cfg) != W8A8_OK) {
    // an invalid q_dtype: the regular entry point produces the message
    return w8a8_scaled_mm(a_q, lda, b_q, ldb, scale_a, a_gran, scale_b, b_gran, out, ldc, M, N, K, q_dtype,
                          out_dtype, nullptr, 0, stream);
  }
  size_t need = w8a8_scaled_mm_config_workspace_size(M, N, K, q_dtype, &cfg);
  if (need > kScratchBytes && cfg.cta_pair && cfg.split_k > 1) {
    // K halves of the last round's CTA-pair tiles only shorten that round;
    // where their partial tiles do not fit the array, the tiles run whole
    cfg.split_k = 1;
    need = w8a8_scaled_mm_config_workspace_size(M, N, K, q_dtype, &cfg);
  }
  if (need > kScratchBytes) {
    w8a8::set_last_error("scaled_mm_noalloc: this problem needs more scratch than the library's fixed array");
    return W8A8_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  w8a8_status st = scratch_address(&scratch);
  if (st != W8A8_OK) return st;
  // The array keeps whatever the previous call left.  The split-K arrival
  // counters this problem uses must start at zero: a successful call leaves
  // them zero, but a call whose kernel gave up on a wait may not, so they
  // are cleared (only they, and only when the plan uses them).
  const size_t ctr = need > 0 ? w8a8::mm_counter_bytes(M, N, K, q_dtype, cfg) : 0;
  if (ctr > 0 && cudaMemsetAsync(scratch, 0, ctr, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    w8a8::set_last_error("scaled_mm_noalloc: clearing the split-K counters failed");
    return W8A8_ERR_CUDA;
  }
  return w8a8_scaled_mm_with_config(a_q, lda, b_q, ldb, scale_a, a_gran, scale_b, b_gran, out, ldc, M, N, K, q_dtype,
                                    out_dtype, need > 0 ? scratch : nullptr, need > 0 ? kScratchBytes : 0, &cfg,
                                    stream);
}

}  // extern "C"
