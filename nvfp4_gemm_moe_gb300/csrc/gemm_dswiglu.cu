// gemm_dswiglu.cu -- instantiations of the persistent GEMM kernel with the grouped dSwiGLU
// backward epilogue ("Grouped GEMM + dSwiGLU (SM100)"): float D with per-expert (|ab|, |dswiglu|)
// amax, or E4M3 D with row and column MXFP8 scale factors.
#include "gemm_kernel.cuh"

namespace bsg {

cudaError_t launch_gemm_dswiglu(const GemmConfig& cfg, const CUtensorMap& ta, const CUtensorMap& tb,
                                const GemmParams& p, int grid, cudaStream_t stream) {
  if (cfg.epi == kEpiDswigluF) {
    if (cfg.fmt == kMXFP8 && cfg.bn == 256) return launch_gemm_t<kMXFP8, 256, kEpiDswigluF>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 224) return launch_gemm_t<kMXFP8, 224, kEpiDswigluF>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 128) return launch_gemm_t<kMXFP8, 128, kEpiDswigluF>(ta, tb, p, grid, stream);
    if (cfg.fmt == kNVFP4 && cfg.bn == 256) return launch_gemm_t<kNVFP4, 256, kEpiDswigluF>(ta, tb, p, grid, stream);
    if (cfg.fmt == kNVFP4 && cfg.bn == 128) return launch_gemm_t<kNVFP4, 128, kEpiDswigluF>(ta, tb, p, grid, stream);
  } else if (cfg.epi == kEpiDswigluFP8) {
    if (cfg.fmt == kMXFP8 && cfg.bn == 256) return launch_gemm_t<kMXFP8, 256, kEpiDswigluFP8>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 224) return launch_gemm_t<kMXFP8, 224, kEpiDswigluFP8>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 128) return launch_gemm_t<kMXFP8, 128, kEpiDswigluFP8>(ta, tb, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsg
