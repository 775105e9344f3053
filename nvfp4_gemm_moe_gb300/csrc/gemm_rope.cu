// gemm_rope.cu -- the persistent GEMM kernel with the RoPE + dual-direction MXFP8 projection
// epilogue ("GEMM + RoPE + MXFP8 Projection (SM100)"), and the plain-to-atom scale repack it
// uses for callers that hold plain row-major E8M0 scales.
#include "gemm_kernel.cuh"
#include "gemm_pair_kernel.cuh"

namespace bsg {

cudaError_t launch_gemm_rope(const GemmConfig& cfg, const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                             int grid, cudaStream_t stream) {
  if (cfg.fmt == kMXFP8 && cfg.bn == 192 && cfg.epi == kEpiRope)
    return launch_gemm_t<kMXFP8, 192, kEpiRope>(ta, tb, p, grid, stream);
  if (cfg.fmt == kBF16 && cfg.bn == 192 && cfg.epi == kEpiRope)
    return launch_gemm_t<kBF16, 192, kEpiRope>(ta, tb, p, grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_pair_rope(const GemmConfig& cfg, const CUtensorMap& ta, const CUtensorMap& tb,
                                  const GemmParams& p, int max_pairs, cudaStream_t stream) {
  if (cfg.fmt == kMXFP8 && cfg.bn == 256 && cfg.epi == kEpiRope)
    return launch_gemm_pair_t<kMXFP8, 256, kEpiRope>(ta, tb, p, max_pairs, stream);
  if (cfg.fmt == kMXFP8 && cfg.bn == 192 && cfg.epi == kEpiRope)
    return launch_gemm_pair_t<kMXFP8, 192, kEpiRope>(ta, tb, p, max_pairs, stream);
  if (cfg.fmt == kBF16 && cfg.bn == 192 && cfg.epi == kEpiRope)
    return launch_gemm_pair_t<kBF16, 192, kEpiRope>(ta, tb, p, max_pairs, stream);
  return cudaErrorInvalidValue;
}

// One thread per scale byte: src is (rows, blocks) row-major, dst the atom layout of a
// (1, rows, 32 * blocks) operand.
__global__ void sf_pack_kernel(const uint8_t* __restrict__ src, int64_t rows, int blocks, int mt, int kt,
                               uint8_t* __restrict__ dst) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * blocks) return;
  const int r = static_cast<int>(i / blocks);
  const int kb = static_cast<int>(i - static_cast<int64_t>(r) * blocks);
  dst[sf_offset(r, kb, 0, mt, kt)] = src[i];
}

cudaError_t launch_sf_pack(const uint8_t* src, int64_t rows, int64_t blocks, uint8_t* dst, cudaStream_t stream) {
  const int mt = static_cast<int>((rows + 127) / 128);
  const int kt = static_cast<int>((blocks + 3) / 4);
  cudaError_t e = cudaMemsetAsync(dst, 0, static_cast<size_t>(mt) * kt * 512, stream);
  if (e != cudaSuccess) return e;
  const int64_t n = rows * blocks;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  sf_pack_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0, stream>>>(
      src, rows, static_cast<int>(blocks), mt, kt, dst);
  return cudaGetLastError();
}

}  // namespace bsg
