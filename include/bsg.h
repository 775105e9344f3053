/*
 * bsg.h -- C ABI of the block-scaled GEMM library for GB300 (sm_103a).
 *
 * Three operations, each one asynchronous launch sequence on the caller's
 * CUDA stream:
 *
 *   bsg_quantize_mx[_bf16]  fp32 (or bf16) -> MXFP8 / NVFP4 codes + scale factors in the
 *                           128x4 scale-factor atom layout (produces the GEMM operands);
 *   bsg_gemm_amax           dense / batched block-scaled GEMM + global amax
 *                           ("GEMM + Amax (SM100)", Overview and Equations);
 *   bsg_grouped_gemm_srelu  grouped MoE block-scaled GEMM + prob-gated sReLU with
 *                           optional tanh soft clamp, per-expert amax or FP8 D with
 *                           row/column MXFP8 scale factors
 *                           ("Grouped GEMM + sReLU (SM100)", Overview, Equations,
 *                           Tanh soft clamp); bsg_grouped_gemm_srelu_discrete takes
 *                           the experts' weights as separate allocations;
 *   bsg_grouped_gemm_dswiglu grouped MoE block-scaled GEMM + dSwiGLU backward epilogue
 *                           ("Grouped GEMM + dSwiGLU (SM100)", Equations);
 *   bsg_gemm_rope_mxfp8     MXFP8 projection GEMM + per-head RoPE + row and column MXFP8
 *                           ("GEMM + RoPE + MXFP8 Projection (SM100)", Equations).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named as device pointers must be device memory of the current CUDA
 *   device (or managed memory); the library never allocates, frees or retains
 *   them.  All tensors are caller-owned.
 * - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *   stream.  Every entry point only enqueues work (memsets, copies and kernel
 *   launches) and returns; results are valid once the stream reaches that point.
 *   Two calls synchronise `stream` first, as their comments say: a grouped call
 *   with opts->validate_offsets, and bsg_read_device_error.
 * - CUDA graphs: every other compute call enqueues only kernels and memsets on
 *   `stream`, so it can be captured into a graph and replayed (inputs read, outputs
 *   written at replay time through the captured pointers).  Make one eager call of
 *   each kernel configuration first: the first launch of a kernel sets its
 *   shared-memory limit and, for CTA pairs, queries the resident cluster count.
 * - Sizes are element counts, not bytes, unless the name says bytes.
 * - Errors: invalid arguments are detected on the host before anything is
 *   enqueued and reported as a bsg_status; nothing is thrown across the ABI.
 *   Each compute call opens an NVTX range named after itself.
 *   Errors detected on the device (a pipeline wait that exceeded its time limit,
 *   invalid padded_offsets contents) set bits in the caller's workspace; read
 *   them with bsg_read_device_error.
 * - Scale-factor (SF) layout ("GEMM + Amax (SM100)", Shapes and "Using JAX
 *   arrays"): for a (batch, rows, K) operand with block size v the SF buffer is
 *   the C-contiguous physical array (batch, ceil(rows/128), ceil(K/(4v)), 32, 4, 4)
 *   of one byte per scale; the byte of row r, block kb, batch l is
 *       ((((l*MT + r/128)*KT + kb/4)*32 + r%32)*4 + (r%128)/32)*4 + kb%4
 *   with MT = ceil(rows/128), KT = ceil(K/(4v)).  Padding bytes (rows >= rows or
 *   blocks >= ceil(K/v)) must hold a finite scale (bsg_quantize_mx writes 0).
 * - Formats: MXFP8 = E4M3 codes (1 byte) with UE8M0 scales and v = 32; NVFP4 =
 *   E2M1 codes packed two per byte (element 2j in the low nibble) with UE4M3
 *   scales and v = 16 ("GEMM + Amax (SM100)", Support surface: E4M3 scales
 *   only with v = 16, FP8 operands only with v = 32).
 * - Operands A (rows, K) and B are K-major (row-major with K contiguous);
 *   outputs C, D, D_col are N-major (row-major with N contiguous).  Every
 *   base pointer must be 16-byte aligned and every row pitch a multiple of 16
 *   bytes ("GEMM + Amax (SM100)", Layouts and strides).
 * - Requires a device of compute capability 10.3 (GB300); the library carries
 *   sm_103a code only.
 */
#ifndef BSG_H
#define BSG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bsg_status {
  BSG_OK = 0,
  BSG_ERR_INVALID_ARG = 1,   /* null pointer, bad size or inconsistent arguments */
  BSG_ERR_UNSUPPORTED = 2,   /* a valid combination this library does not implement */
  BSG_ERR_ALIGNMENT = 3,     /* a pointer or pitch breaks the 16-byte rule */
  BSG_ERR_ARCH = 4,          /* current device is not compute capability 10.3 */
  BSG_ERR_CUDA = 5,          /* a CUDA runtime / driver call failed */
  BSG_ERR_DEVICE = 6,        /* bsg_read_device_error found device-side error bits */
  BSG_ERR_BAD_OFFSETS = 7,   /* host-validated padded_offsets are invalid */
  BSG_ERR_WORKSPACE = 8      /* workspace missing or smaller than bsg_workspace_size() */
} bsg_status;

typedef enum bsg_dtype {
  BSG_E4M3 = 0,  /* float8_e4m3fn */
  BSG_E5M2 = 1,  /* float8_e5m2 (not implemented) */
  BSG_E2M1 = 2,  /* float4_e2m1fn, two per byte */
  BSG_F32 = 3,
  BSG_BF16 = 4,
  BSG_F16 = 5
} bsg_dtype;

typedef enum bsg_sf_dtype {
  BSG_SF_UE8M0 = 0, /* float8_e8m0fnu: 2^(code-127) */
  BSG_SF_UE4M3 = 1  /* float8_e4m3fn used as an unsigned scale */
} bsg_sf_dtype;

/* Device error bits written to the workspace. */
#define BSG_DEVERR_TIMEOUT 0x1u      /* a pipeline wait exceeded its time limit; the kernel gave up */
#define BSG_DEVERR_BAD_OFFSETS 0x2u  /* padded_offsets not non-decreasing multiples of 256 ending at valid_m */
#define BSG_DEVERR_BAD_POINTERS 0x4u /* a null or misaligned b_ptrs / sfb_ptrs entry (per-expert weights) */

/* Optional launch options; pass NULL for the defaults (all fields 0). */
typedef struct bsg_gemm_opts {
  int tile_n;            /* output tile width: 0 = automatic, else 128 or 256 (MXFP8 also 192 or
                            224: two accumulators in TMEM); other values mean automatic */
  int max_ctas;          /* 0 = up to one persistent CTA per SM, else at most this many CTAs; the
                            launch uses the fewest CTAs (CTA pairs) that take the tiles in the
                            same number of rounds */
  int tanh_approx;       /* grouped only: 1 = tanh.approx.f32 in the soft clamp, 0 = tanhf */
  int validate_offsets;  /* grouped only: 1 = copy padded_offsets to the host and check them
                            before launching (synchronises the stream) */
  int cta_pair;          /* 0 = automatic (GEMMs: CTA pairs, widths as for 2, when tile_n is 0,
                            M >= 256, N > 128 and there are at least #SMs/2 256 x 256 tiles),
                            1 = one CTA per 128 x tile_n tile,
                            2 = CTA pairs on 256-row tiles, 256 wide, or 224 wide (MXFP8) with
                            tile_n == 224 or, when tile_n is 0, an E4M3-D or dSwiGLU epilogue;
                            the RoPE projections describe their own choices */
  int b_major;           /* bsg_grouped_gemm_srelu_discrete with MXFP8 operands: 0 = each expert's
                            B is (n, k) K-major, 1 = (k, n) N-major (n contiguous, n % 16 == 0);
                            N-major B runs on 256-wide CTA-pair or 128-wide one-CTA tiles */
  int reserved[2];
} bsg_gemm_opts;

/* Bytes of scratch the GEMM entry points need in `workspace` (device memory,
 * 256-byte aligned).  The calls keep their device error record and the dense amax
 * reduction there, each tagged with a number unique to the call, so a call never clears
 * it first (no memset before the kernel).  Zero-fill a new workspace once before reading
 * errors from it with bsg_read_device_error; do not share one workspace between calls
 * that may run concurrently.  A CUDA graph replays the tag it captured: the error bits of
 * a replayed call accumulate over its replays until another call uses the workspace. */
size_t bsg_workspace_size(void);

/* Bytes of the SF buffer for a (batch, rows, K) operand with block size v. */
size_t bsg_sf_bytes(int64_t batch, int64_t rows, int64_t k, int sf_vec_size);

/*
 * bsg_quantize_mx -- block quantiser that produces GEMM operands.
 *
 * x       device, fp32 (batch, rows, k) row-major (k contiguous).
 * q       device output: E4M3 -> (batch, rows, k) bytes; E2M1 -> (batch, rows, k/2)
 *         bytes, element 2j in the low nibble of byte j.
 * sf      device output: bsg_sf_bytes(batch, rows, k, sf_vec_size) bytes in the SF
 *         layout above; every byte is written, padding bytes as 0.
 * Formats (the workloads' recipes for the operands of "GEMM + Amax (SM100)"):
 *   q_dtype = BSG_E4M3, sf_vec_size = 32, sf_dtype = BSG_SF_UE8M0 (MXFP8): per block
 *     of 32 the scale is 2^e, e the smallest integer with blockamax <= 448*2^e
 *     (E8M0 code clamped to [0, 254]); code = RNE_satfinite_E4M3(x / 2^e).
 *   q_dtype = BSG_E2M1, sf_vec_size = 16, sf_dtype = BSG_SF_UE4M3 (NVFP4): scale
 *     s = RNE_UE4M3(blockamax / 6); code = RNE_satfinite_E2M1(x / s), decided on the
 *     exact quotient; s = 0 gives zero codes.
 * Requirements: k % sf_vec_size == 0, rows >= 1, batch >= 1, sf_vec_size <= k <= 2^30
 *   (else BSG_ERR_INVALID_ARG).
 * Returns BSG_OK after enqueueing; x must not contain NaN or infinities.
 */
bsg_status bsg_quantize_mx(const float* x, int64_t batch, int64_t rows, int64_t k,
                           bsg_dtype q_dtype, int sf_vec_size, bsg_sf_dtype sf_dtype,
                           void* q, uint8_t* sf, void* stream);

/*
 * bsg_quantize_mx_bf16 -- bsg_quantize_mx on bf16 input: x is device bf16 (batch, rows, k)
 * row-major, 16-byte aligned.  Each value is taken exactly (bf16 widens to fp32 without
 * rounding), so the codes and scales equal those bsg_quantize_mx gives for the same values in
 * fp32; the kernel reads half the bytes.  Arguments, requirements and errors as bsg_quantize_mx.
 */
bsg_status bsg_quantize_mx_bf16(const void* x, int64_t batch, int64_t rows, int64_t k,
                                bsg_dtype q_dtype, int sf_vec_size, bsg_sf_dtype sf_dtype,
                                void* q, uint8_t* sf, void* stream);

/*
 * bsg_gemm_amax -- dense batched block-scaled GEMM with fused global amax
 * ("GEMM + Amax (SM100)", Equations):
 *     C[m, n, l] = sum_k Ahat[m, k, l] * Bhat[n, k, l],   *amax = max |C|,
 * Ahat/Bhat the codes times their block scales, accumulated in fp32.
 *
 * a, b      device codes: A (l, m, k) and B (l, n, k), K-major; E4M3 one byte per
 *           element or E2M1 packed (k/2 bytes per row).
 * sfa, sfb  device SF buffers for A (rows m) and B (rows n).
 * ab_dtype / sf_dtype / sf_vec_size: (BSG_E4M3, BSG_SF_UE8M0, 32) or (BSG_E2M1, BSG_SF_UE4M3, 16).
 * c         device output (l, m, n), N-major: c_dtype BSG_F32, BSG_BF16 or BSG_F16 (RNE from
 *           fp32); with E2M1 operands also BSG_E4M3 or BSG_E2M1 ("GEMM + Amax (SM100)",
 *           Parameters: FP8 C with FP8 operands is disabled, FP4 C needs FP4 operands), a
 *           plain RNE_satfinite conversion of the fp32 C without block scales, E2M1 packed two
 *           per byte with element 2j in the low nibble.
 * amax      device output, one float: the max of |C| taken on the fp32 accumulator
 *           before rounding to c_dtype.  Written by the kernel itself (the last CTA to finish
 *           writes the maximum of all CTAs), so the call launches one kernel and nothing else.
 * workspace device scratch of bsg_workspace_size() bytes (see bsg_read_device_error).
 * Requirements: m, n, k, l >= 1; k*bytes_per_element % 16 == 0 (k % 16 for E4M3,
 * k % 32 for E2M1); k % sf_vec_size == 0; the bytes of a row of C a multiple of 16
 * (n % 4, % 8, % 16, % 32 for 4-, 2-, 1-, half-byte elements).  Other C types return
 * BSG_ERR_UNSUPPORTED.
 */
bsg_status bsg_gemm_amax(const void* a, const void* b, const uint8_t* sfa, const uint8_t* sfb,
                         bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype, int sf_vec_size,
                         int64_t m, int64_t n, int64_t k, int64_t l,
                         void* c, bsg_dtype c_dtype, float* amax,
                         const bsg_gemm_opts* opts, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * bsg_grouped_gemm_srelu -- grouped MoE block-scaled GEMM + prob-gated sReLU
 * ("Grouped GEMM + sReLU (SM100)", Equations and Tanh soft clamp).  Rows
 * [padded_offsets[g-1], padded_offsets[g]) (0 for g = 0) belong to expert g
 * ("Grouped GEMM (SM100 BF16)", Operation):
 *     C[m, n] = alpha[g] * sum_k Ahat[m, k] * Bhat[n, k, g]
 *     D[m, n] = prob[m] * relu(C[m, n])^2                          (tanh_clamp_scale <= 0)
 *     D[m, n] = prob[m] * (s * min(tanh(relu(C[m, n]) / s), 1))^2  (s = tanh_clamp_scale > 0)
 * evaluated in fp32 from the fp32 accumulator.
 *
 * a               device codes (valid_m, k), K-major.
 * b               device codes (num_experts, n, k), K-major.
 * sfa, sfb        device SF buffers: A with rows valid_m, B with batch num_experts, rows n.
 * padded_offsets  device int32 (num_experts,): cumulative ends, non-decreasing multiples
 *                 of 256, the last equal to valid_m.  Caller's responsibility; with
 *                 opts->validate_offsets the host checks them first (and syncs), otherwise
 *                 the kernel checks them, sets BSG_DEVERR_BAD_OFFSETS and computes nothing.
 * alpha           device fp32 (num_experts,).
 * prob            device fp32 (valid_m,).
 * norm_const      device fp32 (1,); required iff d_dtype == BSG_E4M3.
 * c               optional device output (valid_m, n) f32, bf16 or f16 (c_dtype); NULL skips C.
 * d               device output (valid_m, n): d_dtype BSG_BF16, BSG_F16 or BSG_F32 (RNE of the
 *                 fp32 D), or BSG_E4M3 (row-quantised D; E4M3 operands only).
 * d_col           device output (valid_m, n) E4M3 (column-quantised D); required iff
 *                 d_dtype == BSG_E4M3, else must be NULL.
 * sfd_row         device output, SF layout with rows valid_m and K = n (blocks of 32 columns).
 * sfd_col         device output, SF layout with rows n and K = valid_m (blocks of 32 rows).
 *                 For E4M3 D the scale of a block is 2^e, e the smallest integer with
 *                 norm_const * blockamax(|D|) <= 448 * 2^e, and the code is
 *                 RNE_satfinite_E4M3(D * norm_const / 2^e) ("Grouped GEMM + dSwiGLU (SM100)",
 *                 Step 3, with the scale rounded up to a power of two).
 * amax            device fp32 (num_experts,): max |D| over each expert's rows (0 for an
 *                 empty expert); required iff d_dtype is not BSG_E4M3.  Zeroed by the call.
 * Requirements: valid_m % 256 == 0, 1 <= num_experts <= 1024, sf as for bsg_gemm_amax,
 * n % 32 == 0 for E4M3 D, the bytes of a row of C and of D a multiple of 16.  With valid_m == 0
 * only padded_offsets and (float D) amax are used: amax is zeroed, nothing else is touched, and
 * the other pointers may be null.
 */
bsg_status bsg_grouped_gemm_srelu(const void* a, const void* b, const uint8_t* sfa, const uint8_t* sfb,
                                  bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype, int sf_vec_size,
                                  int64_t valid_m, int64_t n, int64_t k, int64_t num_experts,
                                  const int32_t* padded_offsets, const float* alpha, const float* prob,
                                  float tanh_clamp_scale, const float* norm_const,
                                  void* c, bsg_dtype c_dtype,
                                  void* d, void* d_col, bsg_dtype d_dtype,
                                  uint8_t* sfd_row, uint8_t* sfd_col, float* amax,
                                  const bsg_gemm_opts* opts, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * bsg_grouped_gemm_dswiglu -- grouped MoE block-scaled GEMM + dSwiGLU backward epilogue
 * ("Grouped GEMM + dSwiGLU (SM100)", Shapes, Equations Steps 1-3).  Rows
 * [padded_offsets[g-1], padded_offsets[g]) belong to expert g.  C is the stored forward
 * intermediate (valid_m, 2N): 32-column blocks alternating input, gate, input, gate, ...; ref
 * column n (block j = n / 32, i = n % 32) pairs with C columns 64 j + i (input) and 64 j + 32 + i
 * (gate).  With x = beta[g] * input, gt = beta[g] * gate, s = 1 / (1 + exp(-gt)):
 *     ref[m, n]          = alpha[g] * sum_k Ahat[m, k] * Bhat[n, k, g]
 *     D[m, 64 j + i]      = ab      = ref * prob[m] * gt * s
 *     D[m, 64 j + 32 + i] = dswiglu = ref * prob[m] * x * s * (1 + gt * (1 - s))
 *     dprob[m]           += sum_n gt * s * x * ref
 * evaluated in fp32 from the fp32 accumulator (the sigmoid from the fast exponential and
 * division, within a few ulp).  The page's Step 1 prints alpha_g squared while its diagram and
 * the grouped sReLU page scale by alpha_g once: alpha is applied once here (pass the squares for
 * the other reading).
 *
 * a, b, sfa, sfb  as for bsg_grouped_gemm_srelu (b: (num_experts, n, k)).
 * alpha, beta     device fp32 (num_experts,).
 * prob            device fp32 (valid_m,).
 * c               device input (valid_m, 2n), c_dtype BSG_BF16, BSG_F16, BSG_F32 or BSG_E4M3
 *                 (plain E4M3 values; beta carries any scale).
 * d_row           device output (valid_m, 2n): d_dtype BSG_BF16 / BSG_F16 / BSG_F32 (RNE of the
 *                 fp32 values), or BSG_E4M3 (row-quantised, MXFP8 operands only).
 * d_col           E4M3 D only: device output (valid_m, 2n), column-quantised; else NULL.
 * sfd_row, sfd_col E4M3 D only: SF layout with rows valid_m and K = 2n (sfd_row), rows 2n and
 *                 K = valid_m (sfd_col); scales and codes as for bsg_grouped_gemm_srelu.
 * norm_const      device fp32 (1,); required iff d_dtype == BSG_E4M3.
 * dprob           device fp32 (valid_m,): the call ADDS each row's sum (atomic adds in an
 *                 unspecified order); zero it first for the plain gradient.
 * amax            device fp32 (num_experts, 2): [g][0] = max |ab|, [g][1] = max |dswiglu| over
 *                 expert g's rows (0 for an empty expert); required iff d_dtype is not E4M3.
 *                 Zeroed by the call.
 * Requirements: valid_m % 256 == 0, n % 32 == 0, 1 <= num_experts <= 512, k a multiple of the
 * scale block, operand rows a multiple of 16 bytes.  opts->tile_n may be 128, 224 (MXFP8) or 256.
 * With valid_m == 0 only padded_offsets and (float D) amax are used, as for the sReLU call.
 */
bsg_status bsg_grouped_gemm_dswiglu(const void* a, const void* b, const uint8_t* sfa, const uint8_t* sfb,
                                    bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype, int sf_vec_size,
                                    int64_t valid_m, int64_t n, int64_t k, int64_t num_experts,
                                    const int32_t* padded_offsets, const float* alpha, const float* beta,
                                    const float* prob, const void* c, bsg_dtype c_dtype, const float* norm_const,
                                    void* d_row, void* d_col, bsg_dtype d_dtype, uint8_t* sfd_row,
                                    uint8_t* sfd_col, float* dprob, float* amax, const bsg_gemm_opts* opts,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * bsg_gemm_rope_mxfp8 -- projection GEMM + per-head RoPE + dual-direction MXFP8
 * ("GEMM + RoPE + MXFP8 Projection (SM100)", Overview, Shapes, Equations; MXFP8 input path).
 * With N = num_heads * head_dim and P = head_dim - qk_rope:
 *     Y[t, h, f] = sum_k xhat[t, k] * what[h * head_dim + f, k]              (fp32 accumulator)
 *     features f >= P of each head are interleaved pairs (a_j, b_j) = (Y[P + 2j], Y[P + 2j + 1])
 *     rotated into halves: out[P + j] = a_j cos[t, j] - b_j sin[t, j],
 *                          out[P + R/2 + j] = b_j cos[t, R/2 + j] + a_j sin[t, R/2 + j]  (R = qk_rope)
 *     (the page's "interleaved-in / halves-out" RoPE; YARN scaling is in the caller's tables);
 *     out_fp8_row / out_scales_row: MXFP8 of Y in blocks of 32 features of a head,
 *     out_fp8_col / out_scales_col: MXFP8 of Y in blocks of 32 tokens of a feature; each block's
 *     E8M0 scale is the smallest 2^e with blockamax <= 448 * 2^e, codes RNE_satfinite(Y / 2^e).
 *
 * x               device E4M3 codes (tokens, q_lora), K-major.
 * w               device E4M3 codes (N, q_lora): the [out, in] weight layout.
 * x_scale, w_scale device E8M0 block scales along q_lora: scale_layout 0 = the 128x4 atom layout
 *                 of bsg_quantize_mx (rows tokens / N); 1 = plain row-major (rows, q_lora / 32) (the
 *                 page's layout; repacked into the workspace on the device).
 * cos, sin        device bf16 (tokens, qk_rope).
 * out_fp8_row, out_fp8_col   device E4M3 (tokens, num_heads, head_dim).
 * out_scales_row  device E8M0 (tokens, num_heads, head_dim / 32), plain row-major.
 * out_scales_col  device E8M0 (tokens / 32, num_heads, head_dim), plain row-major.
 * workspace       bsg_workspace_size() bytes for scale_layout 0, bsg_rope_workspace_size(...) for 1.
 * Requirements: tokens % 128 == 0, q_lora % 32 == 0, head_dim == 192 and qk_rope == 64 (one head
 * per CTA tile; other head shapes return BSG_ERR_UNSUPPORTED).  Tiles: opts->cta_pair == 0 takes
 * CTA pairs on 256 x 192 tiles when tokens % 256 == 0, else one-CTA 128 x 192 tiles; 1 forces the
 * one-CTA tiles; 2 selects CTA pairs, on 256 x 192 tiles with opts->tile_n == 192 (needs tokens %
 * 256 == 0), otherwise on 256 x 256 tiles spanning heads (needs tokens % 256 == 0 and N % 256 ==
 * 0); an ineligible shape returns BSG_ERR_INVALID_ARG.
 */
size_t bsg_rope_workspace_size(int64_t tokens, int64_t num_heads, int64_t head_dim, int64_t q_lora);
bsg_status bsg_gemm_rope_mxfp8(const uint8_t* x, const uint8_t* x_scale, const uint8_t* w, const uint8_t* w_scale,
                               int scale_layout, const void* cos, const void* sin, int64_t tokens, int64_t q_lora,
                               int64_t num_heads, int64_t head_dim, int64_t qk_rope, uint8_t* out_fp8_row,
                               uint8_t* out_scales_row, uint8_t* out_fp8_col, uint8_t* out_scales_col,
                               const bsg_gemm_opts* opts, void* workspace, size_t workspace_bytes, void* stream);

/*
 * bsg_gemm_rope_bf16 -- the BF16-input path of the projection GEMM + RoPE + MXFP8
 * ("GEMM + RoPE + MXFP8 Projection (SM100)", Overview: the GEMM in bf16).  As
 * bsg_gemm_rope_mxfp8 with x (tokens, q_lora) and w (num_heads * head_dim, q_lora) bf16 values
 * (K-major; tcgen05 kind::f16 MMAs, fp32 accumulation) and no scales.  Requirements: q_lora % 8
 * == 0 (16-byte rows), the rest as bsg_gemm_rope_mxfp8.  opts->cta_pair == 2 selects CTA pairs on
 * 256 x 192 tiles (needs tokens % 256 == 0, else BSG_ERR_INVALID_ARG).  Workspace:
 * bsg_workspace_size() bytes.
 */
bsg_status bsg_gemm_rope_bf16(const void* x, const void* w, const void* cos, const void* sin, int64_t tokens,
                              int64_t q_lora, int64_t num_heads, int64_t head_dim, int64_t qk_rope,
                              uint8_t* out_fp8_row, uint8_t* out_scales_row, uint8_t* out_fp8_col,
                              uint8_t* out_scales_col, const bsg_gemm_opts* opts, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * bsg_grouped_gemm_srelu_discrete -- bsg_grouped_gemm_srelu with per-expert weight allocations
 * ("Grouped GEMM + sReLU (SM100)", Shapes: B and SFB given as per-expert tensors addressed by
 * pointer arrays; API usage, discrete input B and SFB pointers).
 *
 * Arguments and results are those of bsg_grouped_gemm_srelu except:
 * b_ptrs     device int64 (num_experts,): b_ptrs[g] is the device address of expert g's codes,
 *            (n, k) K-major, C-contiguous, 16-byte aligned; with MXFP8 operands and
 *            opts->b_major == 1, (k, n) N-major instead ("Grouped GEMM + sReLU (SM100)", Support
 *            surface and constraints: discrete B in K-major or, for FP8, N-major form).
 * sfb_ptrs   device int64 (num_experts,): sfb_ptrs[g] is the device address of expert g's SF
 *            buffer for a (1, n, k) operand (bsg_sf_bytes(1, n, k, v) bytes), 16-byte aligned.
 * workspace  at least bsg_grouped_discrete_workspace_size(num_experts) bytes, 64-byte aligned:
 *            besides the error word it holds one TMA descriptor per expert.
 * The call never reads b_ptrs / sfb_ptrs on the host: a small kernel enqueued before the GEMM
 * writes each expert's TMA descriptor into the workspace from a template (the shape is the same
 * for every expert) by replacing its global address with b_ptrs[g], so the call does not
 * synchronise and can be captured into a CUDA graph.  A null or misaligned pointer entry sets
 * BSG_DEVERR_BAD_POINTERS (read it with bsg_read_device_error) and the GEMM then computes and
 * writes nothing (the per-expert amax stays zeroed).  The weight buffers must stay allocated
 * until the kernel has completed.
 */
size_t bsg_grouped_discrete_workspace_size(int64_t num_experts);
bsg_status bsg_grouped_gemm_srelu_discrete(const void* a, const int64_t* b_ptrs, const uint8_t* sfa,
                                           const int64_t* sfb_ptrs, bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype,
                                           int sf_vec_size, int64_t valid_m, int64_t n, int64_t k,
                                           int64_t num_experts, const int32_t* padded_offsets,
                                           const float* alpha, const float* prob, float tanh_clamp_scale,
                                           const float* norm_const, void* c, bsg_dtype c_dtype,
                                           void* d, void* d_col, bsg_dtype d_dtype,
                                           uint8_t* sfd_row, uint8_t* sfd_col, float* amax,
                                           const bsg_gemm_opts* opts, void* workspace, size_t workspace_bytes,
                                           void* stream);

/*
 * bsg_gemm_amax_noalloc -- bsg_gemm_amax for callers that cannot provide device memory.
 *
 * The pages have no counterpart of this call.  It exists for callers that cannot hand the
 * library device memory of their own at the call site: code running under a memory plan
 * fixed at start-up that forbids later allocations, and latency-critical paths that cannot
 * afford cudaMalloc's implicit device synchronisation.  Arguments and results are those of
 * bsg_gemm_amax without `workspace` / `workspace_bytes`; the call allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine) and instead uses a static device
 * array of BSG_NOALLOC_SCRATCH_BYTES bytes owned by the library (every GPU that loads the
 * library holds it until the process exits).
 * - The first call on a device looks up that array's address on the current device; make
 *   that first call before any stream capture.  The address is kept with the context it was
 *   taken in: after a device reset (a new context) the next call looks it up again, so the
 *   first call after a reset must also come before any stream capture.
 * - All calls on a device share the one array: calls that may overlap on the GPU (other
 *   streams, other threads) race on it.  Each call tags what it writes there, so what a
 *   previous call left behind never leaks into the next one.
 * - Returns BSG_ERR_WORKSPACE if the GEMM's scratch (bsg_workspace_size()) is larger than
 *   BSG_NOALLOC_SCRATCH_BYTES (the library also checks this when it is compiled).
 * - Device-side errors of the last call on the current device are read with
 *   bsg_gemm_amax_noalloc_read_error.
 */
#define BSG_NOALLOC_SCRATCH_BYTES 256
bsg_status bsg_gemm_amax_noalloc(const void* a, const void* b, const uint8_t* sfa, const uint8_t* sfb,
                                 bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype, int sf_vec_size,
                                 int64_t m, int64_t n, int64_t k, int64_t l,
                                 void* c, bsg_dtype c_dtype, float* amax,
                                 const bsg_gemm_opts* opts, void* stream);

/* Synchronises `stream` and returns in *error_bits the device error bits of the last
 * bsg_gemm_amax_noalloc call on the current device (the error word of the library's static
 * array); BSG_ERR_DEVICE if any bit is set, BSG_ERR_CUDA if the array cannot be found. */
bsg_status bsg_gemm_amax_noalloc_read_error(void* stream, uint32_t* error_bits);

/*
 * bsg_selftest_wait_timeout -- failure-detection self-test of the device-side bounded waits.
 * Launches one warp whose wait on an mbarrier that nothing arrives on runs out after the
 * library's wait limit (2 s), records BSG_DEVERR_TIMEOUT in `workspace` (bsg_workspace_size()
 * bytes, 256-byte aligned) as this call's error and returns; the GEMM kernels use the same wait.  No
 * fault, trap or hang: the context stays usable.  Read the result with bsg_read_device_error;
 * bit 31 set means the wait completed, which it must not.
 */
bsg_status bsg_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream` and returns the device error bits of the last call that
 * used `workspace` in *error_bits; BSG_ERR_DEVICE if any bit is set. */
bsg_status bsg_read_device_error(const void* workspace, void* stream, uint32_t* error_bits);

/* Static string naming a status code. */
const char* bsg_status_string(bsg_status status);

#ifdef __cplusplus
}
#endif

#endif /* BSG_H */
