// gemm_pair.cu -- instantiations of the CTA-pair GEMM kernel (256 x 256 and 256 x 224 tiles): dense and grouped.
#include "gemm_pair_kernel.cuh"

namespace bsg {

cudaError_t launch_gemm_pair(const GemmConfig& cfg, const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                             int max_pairs, cudaStream_t stream, const CUtensorMap* tc, const CUtensorMap* td) {
  if (cfg.fmt == kMXFP8 && cfg.bn == 256) {
    if (cfg.epi == kEpiDense) return launch_gemm_pair_t<kMXFP8, 256, kEpiDense>(ta, tb, p, max_pairs, stream);
    if (cfg.epi == kEpiGroupedBF16)
      return launch_gemm_pair_t<kMXFP8, 256, kEpiGroupedBF16>(ta, tb, p, max_pairs, stream, tc, td);
    if (cfg.epi == kEpiGroupedFP8) return launch_gemm_pair_t<kMXFP8, 256, kEpiGroupedFP8>(ta, tb, p, max_pairs, stream);
  } else if (cfg.fmt == kMXFP8 && cfg.bn == 224) {
    if (cfg.epi == kEpiDense) return launch_gemm_pair_t<kMXFP8, 224, kEpiDense>(ta, tb, p, max_pairs, stream);
    if (cfg.epi == kEpiGroupedBF16)
      return launch_gemm_pair_t<kMXFP8, 224, kEpiGroupedBF16>(ta, tb, p, max_pairs, stream, tc, td);
    if (cfg.epi == kEpiGroupedFP8) return launch_gemm_pair_t<kMXFP8, 224, kEpiGroupedFP8>(ta, tb, p, max_pairs, stream);
  } else if (cfg.fmt == kNVFP4 && cfg.bn == 256) {
    if (cfg.epi == kEpiDense) return launch_gemm_pair_t<kNVFP4, 256, kEpiDense>(ta, tb, p, max_pairs, stream);
    if (cfg.epi == kEpiGroupedBF16)
      return launch_gemm_pair_t<kNVFP4, 256, kEpiGroupedBF16>(ta, tb, p, max_pairs, stream, tc, td);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsg
