// gemm_pair_dswiglu.cu -- instantiations of the CTA-pair GEMM kernel with the grouped dSwiGLU
// backward epilogue.
#include "gemm_pair_kernel.cuh"

namespace bsg {

cudaError_t launch_gemm_pair_dswiglu(const GemmConfig& cfg, const CUtensorMap& ta, const CUtensorMap& tb,
                                     const GemmParams& p, int max_pairs, cudaStream_t stream) {
  if (cfg.fmt == kMXFP8 && cfg.bn == 256) {
    if (cfg.epi == kEpiDswigluF) return launch_gemm_pair_t<kMXFP8, 256, kEpiDswigluF>(ta, tb, p, max_pairs, stream);
    if (cfg.epi == kEpiDswigluFP8) return launch_gemm_pair_t<kMXFP8, 256, kEpiDswigluFP8>(ta, tb, p, max_pairs, stream);
  } else if (cfg.fmt == kMXFP8 && cfg.bn == 224) {
    if (cfg.epi == kEpiDswigluF) return launch_gemm_pair_t<kMXFP8, 224, kEpiDswigluF>(ta, tb, p, max_pairs, stream);
    if (cfg.epi == kEpiDswigluFP8) return launch_gemm_pair_t<kMXFP8, 224, kEpiDswigluFP8>(ta, tb, p, max_pairs, stream);
  } else if (cfg.fmt == kNVFP4 && cfg.bn == 256) {
    if (cfg.epi == kEpiDswigluF) return launch_gemm_pair_t<kNVFP4, 256, kEpiDswigluF>(ta, tb, p, max_pairs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsg
