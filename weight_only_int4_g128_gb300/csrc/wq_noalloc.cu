// wq_noalloc.cu -- wq_gemm_w4a16_noalloc: the W4A16 GEMM for callers that
// cannot hand the library a workspace.
//
// Some callers cannot allocate device memory where they call the GEMM: code
// that runs inside a framework which forbids allocations outside its own
// caching allocator, host code that runs while a stream is being captured
// into a CUDA graph (cudaMalloc is not a capturable operation), or
// latency-critical loops where a cudaMalloc may synchronize the device.  This
// entry point needs no workspace argument: the scratch the GEMM may need (the
// correction columns of the large-M path and, for bf16 activations, the
// per-token scaled fp16 copy of X that path reads) lives in one fixed-size array of
// device memory that is part of the library image, so every GPU that loads the
// library holds it until the process exits.  Nothing here allocates.
#include <cuda_runtime.h>

#include <mutex>

#include "wq.h"
#include "wq_internal.h"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;  // 16 MiB

// Shared by every call on a device: it keeps whatever the last call left in
// it (no call needs any of it to start at zero), and calls whose kernels
// overlap on the GPU (different streams) race on it.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {};   // device address of g_scratch, per device
wq::PerContextOnce g_looked_up;  // ... valid for the context it was looked up in

// The array's name in host code is only a stand-in for the symbol; the device
// address has to be looked up (once per device, with that device current, and
// again if the device's context has been rebuilt, e.g. after cudaDeviceReset)
// before a kernel can be given it.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return wq::set_last_error(WQ_ERR_CUDA, "wq_gemm_w4a16_noalloc: cudaGetDevice: %s",
                                                  cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return wq::set_last_error(WQ_ERR_CUDA, "wq_gemm_w4a16_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev] || g_looked_up.needed(dev)) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p)
      return wq::set_last_error(WQ_ERR_CUDA, "wq_gemm_w4a16_noalloc: cudaGetSymbolAddress: %s",
                                cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
    g_looked_up.done(dev);
  }
  *out = g_scratch_addr[dev];
  return WQ_OK;
}

}  // namespace

extern "C" int wq_gemm_w4a16_noalloc(const void* X, int x_dtype, const uint32_t* Bpacked, const void* S,
                                     const float* delta, void* Y, int y_dtype, int M, int N, int K,
                                     int group_size, void* stream) {
  const int variant = delta ? WQ_VARIANT_W4A16 : WQ_VARIANT_W4A16_SYM;
  // 0 for shapes the GEMM rejects; wq_gemm_w4a16 below reports those itself.
  const size_t need = (M > 0) ? wq::gemm_workspace_bytes(variant, x_dtype, M, N, K, group_size) : 0;
  if (need > kScratchBytes) {
    // Too large for the array.  The arguments are still checked first, as the
    // workspace entry checks them: without a workspace wq_gemm_w4a16 returns its
    // argument errors, and otherwise WQ_ERR_WORKSPACE before it launches anything.
    const int rc = wq_gemm_w4a16(X, x_dtype, Bpacked, S, delta, Y, y_dtype, M, N, K, group_size, nullptr, 0,
                                 stream);
    if (rc != WQ_ERR_WORKSPACE) return rc;
    return wq::set_last_error(WQ_ERR_WORKSPACE,
                              "wq_gemm_w4a16_noalloc: this problem needs %zu bytes of scratch; the built-in "
                              "scratch holds %zu (use wq_gemm_w4a16 with a workspace)",
                              need, kScratchBytes);
  }
  void* scratch = nullptr;
  if (need > 0) {
    const int rc = scratch_address(&scratch);
    if (rc != WQ_OK) return rc;
  }
  return wq_gemm_w4a16(X, x_dtype, Bpacked, S, delta, Y, y_dtype, M, N, K, group_size, scratch,
                       need > 0 ? kScratchBytes : 0, stream);
}
