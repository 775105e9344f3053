// noalloc.cu -- bsg_gemm_amax_noalloc: the dense GEMM + amax without a caller workspace.
//
// Some callers cannot hand the library any device memory of their own at the call site:
// code that runs under a memory plan fixed at start-up (an arena that forbids allocations
// afterwards) and latency-critical paths that cannot afford cudaMalloc's implicit device
// synchronisation.  For them this entry point takes the GEMM's scratch (the device error
// record and the amax reduction the kernel keeps) from a static device array that the library
// itself owns.  Every GPU that loads the library keeps that array until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "bsg.h"
#include "internal.h"

static_assert(bsg::kWorkspaceBytes <= BSG_NOALLOC_SCRATCH_BYTES,
              "the GEMM's scratch must fit the library's static array");

namespace {

// The scratch of every bsg_gemm_amax_noalloc call on a device.  Host code must not pass
// this symbol to a kernel (on the host it is only a stand-in, not a device address); it
// uses the address cudaGetSymbolAddress returns for the current device and context.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BSG_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Identity of the calling thread's current context (unique within the process, never reused:
// a context re-created after a device reset gets a new one); 0 when none is current yet.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

struct ScratchSlot {
  unsigned long long ctx_id = 0;  // context the address belongs to
  void* addr = nullptr;
};

std::mutex g_noalloc_mu;
ScratchSlot g_noalloc_slot[64];

// The array's device address on the current device, looked up again whenever the current
// context is not the one the cached address was taken in (after a device reset the module is
// loaded anew and the old address is dead).  nullptr on a CUDA error.
void* scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  ScratchSlot& s = g_noalloc_slot[dev];
  const unsigned long long id = current_context_id();
  if (s.addr != nullptr && id != 0 && id == s.ctx_id) return s.addr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
  s.addr = p;
  s.ctx_id = current_context_id();  // the lookup makes the device's context current if none was
  return p;
}

bsg_status current_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSG_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BSG_ERR_UNSUPPORTED;
  *out = scratch_address(dev);
  return *out ? BSG_OK : BSG_ERR_CUDA;
}

}  // namespace

extern "C" bsg_status bsg_gemm_amax_noalloc(const void* a, const void* b, const uint8_t* sfa, const uint8_t* sfb,
                                            bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype, int sf_vec_size, int64_t m,
                                            int64_t n, int64_t k, int64_t l, void* c, bsg_dtype c_dtype,
                                            float* amax, const bsg_gemm_opts* opts, void* stream) {
  const size_t need = bsg_workspace_size();
  if (need > BSG_NOALLOC_SCRATCH_BYTES) return BSG_ERR_WORKSPACE;  // the kernel's scratch outgrew the array
  void* scratch = nullptr;
  const bsg_status st = current_scratch(&scratch);
  if (st != BSG_OK) return st;
  // bsg_gemm_amax tags the error record and the amax reduction in the array with a number
  // unique to the call, so the previous call's contents never leak into this one.
  return bsg_gemm_amax(a, b, sfa, sfb, ab_dtype, sf_dtype, sf_vec_size, m, n, k, l, c, c_dtype, amax, opts,
                       scratch, BSG_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" bsg_status bsg_gemm_amax_noalloc_read_error(void* stream, uint32_t* error_bits) {
  if (!error_bits) return BSG_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const bsg_status st = current_scratch(&scratch);
  if (st != BSG_OK) return st;
  return bsg_read_device_error(scratch, stream, error_bits);
}
