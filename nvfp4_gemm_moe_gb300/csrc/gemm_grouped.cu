// gemm_grouped.cu -- instantiations of the persistent GEMM kernel with the grouped MoE epilogues
// (alpha, C, prob-gated sReLU / tanh clamp, bf16 D + per-expert amax, or E4M3 D with row and
// column MXFP8 scale factors).
#include "gemm_kernel.cuh"

namespace bsg {

cudaError_t launch_gemm_grouped(const GemmConfig& cfg, const CUtensorMap& ta, const CUtensorMap& tb,
                                const GemmParams& p, int grid, cudaStream_t stream) {
  if (cfg.epi == kEpiGroupedBF16) {
    if (cfg.fmt == kMXFP8 && cfg.bn == 256) return launch_gemm_t<kMXFP8, 256, kEpiGroupedBF16>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 224) return launch_gemm_t<kMXFP8, 224, kEpiGroupedBF16>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 192) return launch_gemm_t<kMXFP8, 192, kEpiGroupedBF16>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 128) return launch_gemm_t<kMXFP8, 128, kEpiGroupedBF16>(ta, tb, p, grid, stream);
    if (cfg.fmt == kNVFP4 && cfg.bn == 256) return launch_gemm_t<kNVFP4, 256, kEpiGroupedBF16>(ta, tb, p, grid, stream);
    if (cfg.fmt == kNVFP4 && cfg.bn == 128) return launch_gemm_t<kNVFP4, 128, kEpiGroupedBF16>(ta, tb, p, grid, stream);
  } else if (cfg.epi == kEpiGroupedFP8) {
    if (cfg.fmt == kMXFP8 && cfg.bn == 256) return launch_gemm_t<kMXFP8, 256, kEpiGroupedFP8>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 224) return launch_gemm_t<kMXFP8, 224, kEpiGroupedFP8>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 192) return launch_gemm_t<kMXFP8, 192, kEpiGroupedFP8>(ta, tb, p, grid, stream);
    if (cfg.fmt == kMXFP8 && cfg.bn == 128) return launch_gemm_t<kMXFP8, 128, kEpiGroupedFP8>(ta, tb, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsg
