// internal.h -- launch interfaces between the C ABI (bsg_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bsg {

// Bytes of the per-call scratch every GEMM entry point needs (the device error word and the
// words next to it); bsg_workspace_size() returns it.
constexpr size_t kWorkspaceBytes = 256;
// Byte offsets in it: 0-11 the device error record (ErrSink in common.cuh); 16-31 the dense
// kernel's amax record: the call's epoch, the count of finished CTAs and the running maximum
// (32 bits each, one unused), updated together by one 128-bit compare-and-swap, so a record a
// previous call left behind is recognised by its epoch and no call has to clear it first.
// Word 3 (bytes 12-15): set to the call's epoch by the per-expert descriptor kernel when a weight
// pointer is invalid; the GEMM kernel then computes nothing.
constexpr int kWsAmaxRecordByte = 16;
constexpr int kWsBadPointersWord = 3;

// A fresh nonzero tag for the next call's device-side records (process-wide counter).
uint32_t next_call_epoch();

enum Fmt : int { kMXFP8 = 0, kNVFP4 = 1, kBF16 = 2 };  // kBF16: plain bf16 operands, no scale factors
// Element types of the C / D outputs.  E4M3 and E2M1 here are plain conversions (round to
// nearest even, saturating), without block scales; E2M1 packs two values per byte, element 2j
// in the low nibble.
enum OutKind : int { kOutNone = 0, kOutF32 = 1, kOutBF16 = 2, kOutE4M3 = 3, kOutF16 = 4, kOutE2M1 = 5 };
enum EpiKind : int {
  kEpiDense = 0,        // C + global amax
  kEpiGroupedBF16 = 1,  // grouped sReLU, float D (bf16 / f16 / f32) + per-expert amax
  kEpiGroupedFP8 = 2,   // grouped sReLU, E4M3 D with row and column scale factors
  kEpiDswigluF = 3,     // grouped dSwiGLU backward, float D + per-expert (|ab|, |dswiglu|) amax
  kEpiDswigluFP8 = 4,   // grouped dSwiGLU backward, E4M3 D with row and column scale factors
  kEpiRope = 5          // dense projection + per-head RoPE + row / column MXFP8 (plain scale layouts)
};
__host__ __device__ constexpr bool epi_is_grouped(int epi) {
  return epi == kEpiGroupedBF16 || epi == kEpiGroupedFP8 || epi == kEpiDswigluF || epi == kEpiDswigluFP8;
}
__host__ __device__ constexpr bool epi_is_dswiglu(int epi) { return epi == kEpiDswigluF || epi == kEpiDswigluFP8; }
__host__ __device__ constexpr bool epi_has_fp8_d(int epi) { return epi == kEpiGroupedFP8 || epi == kEpiDswigluFP8; }

// Everything a GEMM kernel needs besides the two tensor maps.
struct GemmParams {
  // problem
  int m, n, k;           // rows of A, rows of B (N), K in elements
  int l;                 // batch (dense) or number of experts (grouped)
  int m_tiles, n_tiles;  // ceil(m/128), ceil(n/BN)
  int k_tiles;           // ceil(K / elements per 128-byte K tile)
  int num_tiles;         // l*m_tiles*n_tiles (dense) or m_tiles*n_tiles (grouped)
  // scale factors
  const uint8_t* sfa;
  const uint8_t* sfb;
  const CUtensorMap* b_maps;   // grouped with per-expert weights: one B tensor map per expert (global)
  const int64_t* sfb_ptrs;     // grouped with per-expert weights: one SFB pointer per expert
  int b_mn_major;              // FP8 B stored N-major, (k, n) with n contiguous, per expert (128 N per CTA)
  int sfa_mt, sfb_mt;    // ceil(m/128), ceil(n/128)
  int sf_kt;             // ceil(K / (4 v)) atoms along K
  // dense epilogue
  void* c;
  int c_kind;            // OutKind
  float* amax;           // dense: 1 float; grouped bf16 D: num_experts floats
  // grouped epilogue
  const int32_t* offsets;
  const float* alpha;
  const float* prob;
  int d_kind;            // OutKind of D for the bf16 / f16 / f32 grouped epilogue
  float clamp_s;         // <= 0: no tanh clamp
  int tanh_approx;
  const float* norm_const;
  void* d;
  void* d_col;
  uint8_t* sfd_row;
  uint8_t* sfd_col;
  int sfd_row_kt;        // ceil(n / 128): atoms along N of SFD_row
  int sfd_col_mt;        // ceil(n / 128): 128-row groups of SFD_col
  int sfd_col_kt;        // ceil(valid_m / 128): atoms along M of SFD_col
  // dSwiGLU backward: C is an input of 2N columns (32-column input / gate blocks), D is 2N wide
  const void* c_in;
  int c_in_kind;         // OutKind of C (f32 / bf16 / f16 / E4M3 values)
  const float* beta;     // per-expert scale of C
  float* dprob;          // (valid_m,) accumulated with atomic adds
  // RoPE projection: bf16 rotary tables (m, qk_rope); d / d_col / sfd_row / sfd_col hold the
  // row- and column-quantised outputs with plain (row-major) scale arrays
  const uint16_t* rope_cos;
  const uint16_t* rope_sin;
  int qk_rope;
  // the rows of C (c_v8) or of D and D_col (d_v8) are written as whole 32-byte sectors, one
  // 256-bit store per thread and row, instead of through the transpose block (addresses and row
  // pitch 32-byte aligned)
  int c_v8;
  int d_v8;
  // grouped bf16 D (and bf16 or no C) on 256-wide CTA pairs: the epilogue stages each 32 x 32
  // block of C and D in shared memory and stores it with a TMA tensor store (the output tensor
  // maps are kernel parameters) instead of per-thread global stores
  int out_tma;
  // device error record (workspace) and this call's epoch (see ErrSink)
  uint32_t* err;
  uint32_t epoch;
};

struct GemmConfig {
  int fmt;       // Fmt
  int bn;        // 128 or 256
  int epi;       // EpiKind
};

// Launches the persistent GEMM kernel for `cfg`; returns cudaSuccess or the launch error.
cudaError_t launch_gemm(const GemmConfig& cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                        const GemmParams& p, int grid, cudaStream_t stream);
cudaError_t launch_gemm_dense(const GemmConfig& cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                              const GemmParams& p, int grid, cudaStream_t stream);
cudaError_t launch_gemm_grouped(const GemmConfig& cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                const GemmParams& p, int grid, cudaStream_t stream);

// Launches the CTA-pair kernel (256 x 256 tiles on clusters of two CTAs) with at most
// `max_pairs` clusters.  tmap_c / tmap_d: the output tensor maps when p.out_tma is set (else
// unused and may be null).
cudaError_t launch_gemm_pair(const GemmConfig& cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                             const GemmParams& p, int max_pairs, cudaStream_t stream,
                             const CUtensorMap* tmap_c = nullptr, const CUtensorMap* tmap_d = nullptr);

// The dSwiGLU backward epilogue kernels (one-CTA and CTA-pair tiles).
cudaError_t launch_gemm_dswiglu(const GemmConfig& cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                const GemmParams& p, int grid, cudaStream_t stream);
cudaError_t launch_gemm_pair_dswiglu(const GemmConfig& cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                     const GemmParams& p, int max_pairs, cudaStream_t stream);

// The GEMM + RoPE + MXFP8 projection kernels: one-CTA tiles of 128 tokens x one head, or CTA
// pairs on 256 x 256 tiles spanning heads.
cudaError_t launch_gemm_rope(const GemmConfig& cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                             const GemmParams& p, int grid, cudaStream_t stream);
cudaError_t launch_gemm_pair_rope(const GemmConfig& cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                  const GemmParams& p, int max_pairs, cudaStream_t stream);

// Per-expert weights: writes maps[g] = `tmpl` with its global address replaced by b_ptrs[g], for
// every expert g (device arrays b_ptrs / sfb_ptrs).  A null or misaligned entry records
// BSG_DEVERR_BAD_POINTERS and tags workspace word kWsBadPointersWord with `epoch`.
cudaError_t launch_expert_maps(const CUtensorMap& tmpl, const int64_t* b_ptrs, const int64_t* sfb_ptrs,
                               int num_experts, CUtensorMap* maps, uint32_t* ws, uint32_t epoch, cudaStream_t s);

// Scatters plain row-major scale bytes (rows, blocks) into the 128x4 atom layout (dst zeroed
// first, so padding bytes hold the finite scale 0).
cudaError_t launch_sf_pack(const uint8_t* src, int64_t rows, int64_t blocks, uint8_t* dst, cudaStream_t stream);

// Launches the block quantiser.
// x: fp32, or bf16 when x_bf16 (widened exactly to fp32 on load).
cudaError_t launch_quantize(int fmt, const void* x, bool x_bf16, int64_t batch, int64_t rows, int64_t k, uint8_t* q,
                            uint8_t* sf, int num_sms, cudaStream_t stream);

}  // namespace bsg
