// selftest.cu -- a device-side failure-detection self-test: one bounded wait that runs out.
//
// The GEMM kernels never wait unboundedly: every mbarrier wait gives up after kWaitLimitNs,
// records BSG_DEVERR_TIMEOUT in the caller's workspace and lets the CTA drain and exit.  This
// kernel exercises that wait (the same wait_bounded the GEMM roles use) on a barrier that
// nothing ever arrives on, so the timeout path runs on a real GPU without faulting, trapping
// or hanging it; the context stays usable afterwards.
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsg.h"
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr uint32_t kErrSelftestCompleted = 0x80000000u;  // the wait completed: it must not

__global__ void selftest_wait_kernel(uint32_t* ws, uint32_t epoch) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const bsg::ErrSink err{ws, epoch};
  if (threadIdx.x == 0) {
    bsg::mark_call(err);
    bsg::mbar_init(&bar, 1);
    abort_flag = 0;
    bsg::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 of `bar` never completes (its one expected arrival never comes)
    if (bsg::wait_bounded(&bar, 0, &abort_flag, err)) bsg::report_error(err, kErrSelftestCompleted);
  }
}

}  // namespace

extern "C" bsg_status bsg_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < bsg_workspace_size()) return BSG_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return BSG_ERR_ALIGNMENT;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return BSG_ERR_CUDA;
  if (major != 10 || minor != 3) return BSG_ERR_ARCH;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selftest_wait_kernel<<<1, 32, 0, s>>>(static_cast<uint32_t*>(workspace), bsg::next_call_epoch());
  return cudaGetLastError() == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
}
