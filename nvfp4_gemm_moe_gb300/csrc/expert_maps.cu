// expert_maps.cu -- the TMA descriptors of per-expert weight allocations, built on the device.
//
// "Grouped GEMM + sReLU (SM100)", Shapes: with discrete weights, B and SFB of expert g are
// separate allocations addressed by the device arrays b_ptrs[g] / sfb_ptrs[g].  Every expert's
// B has the same shape (n, k) and strides, so its tensor map differs from a template, encoded
// on the host for that shape, only in the global address.  One thread per expert copies the
// template into the workspace and replaces the address with tensormap.replace, so the call
// never reads the pointer arrays on the host (no synchronisation; it can be captured in a CUDA
// graph).  Invalid entries are reported through the device error record.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace bsg {
namespace {

__global__ void expert_maps_kernel(const __grid_constant__ CUtensorMap tmpl, const int64_t* b_ptrs,
                                   const int64_t* sfb_ptrs, int num_experts, CUtensorMap* maps, uint32_t* ws,
                                   uint32_t epoch) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= num_experts) return;
  const ErrSink es{ws, epoch};
  const int64_t b = b_ptrs[g];
  const int64_t sf = sfb_ptrs[g];
  if (b == 0 || sf == 0 || (b & 15) != 0 || (sf & 15) != 0) {
    report_error(es, kErrBadPointers);
    *reinterpret_cast<volatile uint32_t*>(ws + kWsBadPointersWord) = epoch;
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(&tmpl);
  uint4* dst = reinterpret_cast<uint4*>(maps + g);
#pragma unroll
  for (int i = 0; i < 8; ++i) dst[i] = src[i];
  asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(
                   reinterpret_cast<uint64_t>(maps + g)),
               "l"(b)
               : "memory");
  // the GEMM kernel's producers acquire the descriptor through the tensor-map proxy before use
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

}  // namespace

cudaError_t launch_expert_maps(const CUtensorMap& tmpl, const int64_t* b_ptrs, const int64_t* sfb_ptrs,
                               int num_experts, CUtensorMap* maps, uint32_t* ws, uint32_t epoch, cudaStream_t s) {
  const int threads = 128;
  expert_maps_kernel<<<(num_experts + threads - 1) / threads, threads, 0, s>>>(tmpl, b_ptrs, sfb_ptrs, num_experts,
                                                                                 maps, ws, epoch);
  return cudaGetLastError();
}

}  // namespace bsg
