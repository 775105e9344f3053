// gemm_pair.cu -- instantiations of the CTA-pair (256 x 256 tile) GEMM kernel.
#include "gemm_pair_kernel.cuh"

namespace bsg {

cudaError_t launch_gemm_pair(const GemmConfig& cfg, const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                             int max_pairs, cudaStream_t stream) {
  if (cfg.fmt == kMXFP8) {
    if (cfg.epi == kEpiDense) return launch_gemm_pair_t<kMXFP8, kEpiDense>(ta, tb, p, max_pairs, stream);
    if (cfg.epi == kEpiGroupedBF16)
      return launch_gemm_pair_t<kMXFP8, kEpiGroupedBF16>(ta, tb, p, max_pairs, stream);
    if (cfg.epi == kEpiGroupedFP8)
      return launch_gemm_pair_t<kMXFP8, kEpiGroupedFP8>(ta, tb, p, max_pairs, stream);
  } else {
    if (cfg.epi == kEpiDense) return launch_gemm_pair_t<kNVFP4, kEpiDense>(ta, tb, p, max_pairs, stream);
    if (cfg.epi == kEpiGroupedBF16)
      return launch_gemm_pair_t<kNVFP4, kEpiGroupedBF16>(ta, tb, p, max_pairs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bsg
