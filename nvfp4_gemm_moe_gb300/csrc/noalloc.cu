// noalloc.cu -- bsg_gemm_amax_noalloc: the dense GEMM + amax without a caller workspace.
//
// Some callers cannot hand the library any device memory of their own at the call site:
// code that runs under a memory plan fixed at start-up (an arena that forbids allocations
// afterwards) and latency-critical paths that cannot afford cudaMalloc's implicit device
// synchronisation.  For them this entry point takes the GEMM's scratch (the device error
// word the kernel writes) from a static device array that the library itself owns.  Every
// GPU that loads the library keeps that array until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "bsg.h"

namespace {

// The scratch of every bsg_gemm_amax_noalloc call on a device.  Host code must not pass
// this symbol to a kernel (on the host it is only a stand-in, not a device address); it
// uses the address cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BSG_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

}  // namespace

extern "C" bsg_status bsg_gemm_amax_noalloc(const void* a, const void* b, const uint8_t* sfa, const uint8_t* sfb,
                                            bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype, int sf_vec_size, int64_t m,
                                            int64_t n, int64_t k, int64_t l, void* c, bsg_dtype c_dtype,
                                            float* amax, const bsg_gemm_opts* opts, void* stream) {
  const size_t need = bsg_workspace_size();
  if (need > BSG_NOALLOC_SCRATCH_BYTES) return BSG_ERR_WORKSPACE;  // the kernel's scratch outgrew the array
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSG_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BSG_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    // one-time set-up per device, with that device current: the array's device address
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return BSG_ERR_CUDA;
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  // bsg_gemm_amax clears the error word on `stream` before the kernel runs, so the previous
  // call's contents never leak into this one.
  return bsg_gemm_amax(a, b, sfa, sfb, ab_dtype, sf_dtype, sf_vec_size, m, n, k, l, c, c_dtype, amax, opts,
                       scratch, BSG_NOALLOC_SCRATCH_BYTES, stream);
}
