// gemm_dense.cu -- instantiations of the persistent GEMM kernel with the dense C + amax epilogue.
#include "gemm_kernel.cuh"

namespace bsg {

cudaError_t launch_gemm_dense(const GemmConfig& cfg, const CUtensorMap& ta, const CUtensorMap& tb,
                              const GemmParams& p, int grid, cudaStream_t stream) {
  if (cfg.fmt == kMXFP8 && cfg.bn == 256) return launch_gemm_t<kMXFP8, 256, kEpiDense>(ta, tb, p, grid, stream);
  if (cfg.fmt == kMXFP8 && cfg.bn == 224) return launch_gemm_t<kMXFP8, 224, kEpiDense>(ta, tb, p, grid, stream);
  if (cfg.fmt == kMXFP8 && cfg.bn == 192) return launch_gemm_t<kMXFP8, 192, kEpiDense>(ta, tb, p, grid, stream);
  if (cfg.fmt == kMXFP8 && cfg.bn == 128) return launch_gemm_t<kMXFP8, 128, kEpiDense>(ta, tb, p, grid, stream);
  if (cfg.fmt == kNVFP4 && cfg.bn == 256) return launch_gemm_t<kNVFP4, 256, kEpiDense>(ta, tb, p, grid, stream);
  if (cfg.fmt == kNVFP4 && cfg.bn == 128) return launch_gemm_t<kNVFP4, 128, kEpiDense>(ta, tb, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bsg
