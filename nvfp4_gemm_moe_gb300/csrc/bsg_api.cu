// bsg_api.cu -- the C ABI: argument validation, TMA descriptor encoding, launch configuration.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "bsg.h"
#include "internal.h"

namespace {

using bsg::GemmConfig;
using bsg::GemmParams;
using bsg::kWorkspaceBytes;

// One NVTX range per C ABI call, named after the entry point (shown by Nsight tools; without a
// tool attached the calls return at once).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int num_sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[64];

std::atomic<uint32_t> g_epoch{0};

bsg_status current_device(int* dev_out, DeviceInfo* info_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSG_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BSG_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BSG_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.probed = true;
  }
  if (dev_out) *dev_out = dev;
  if (info_out) *info_out = d;
  return d.supported ? BSG_OK : BSG_ERR_ARCH;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// K-major operand (batch, rows, row_bytes) of bytes, loaded as 128-byte x box_rows boxes with
// the 128-byte swizzle; out-of-range rows / K bytes read as zero.
bool make_operand_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint64_t batch,
                      uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {row_bytes, rows, batch};
  const cuuint64_t strides[2] = {row_bytes, row_bytes * rows};
  const cuuint32_t box[3] = {128, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// N-major 8-bit operand (k rows of n bytes), loaded as 128-byte (N) x 128-row (K) boxes with the
// 128-byte swizzle: one 128-element swizzle row of N per K row.
bool make_operand_map_mn(CUtensorMap* m, const void* base, uint64_t n, uint64_t k) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {n, k, 1};
  const cuuint64_t strides[2] = {n, n * k};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bf16 output (rows x cols, cols % 8 == 0) stored by the grouped epilogue as 32 x 32
// boxes (64 bytes of a row each) from shared-memory blocks in the 64-byte swizzled layout.
bool make_output_map_bf16(CUtensorMap* m, void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Operand format from the (ab_dtype, sf_dtype, sf_vec_size) triple.
bsg_status operand_format(bsg_dtype ab, bsg_sf_dtype sf, int v, int* fmt) {
  if (ab == BSG_E4M3 && sf == BSG_SF_UE8M0 && v == 32) { *fmt = bsg::kMXFP8; return BSG_OK; }
  if (ab == BSG_E2M1 && sf == BSG_SF_UE4M3 && v == 16) { *fmt = bsg::kNVFP4; return BSG_OK; }
  if (v != 16 && v != 32) return BSG_ERR_INVALID_ARG;
  if (sf != BSG_SF_UE8M0 && sf != BSG_SF_UE4M3) return BSG_ERR_INVALID_ARG;
  // couplings the operation forbids: E4M3 scales need v = 16, FP8 operands need v = 32
  if (sf == BSG_SF_UE4M3 && v == 32) return BSG_ERR_INVALID_ARG;
  if ((ab == BSG_E4M3 || ab == BSG_E5M2) && v == 16) return BSG_ERR_INVALID_ARG;
  if (ab != BSG_E4M3 && ab != BSG_E5M2 && ab != BSG_E2M1) return BSG_ERR_INVALID_ARG;
  return BSG_ERR_UNSUPPORTED;  // E5M2 operands, MXFP4 (E2M1 with E8M0 scales)
}

bool fits_int32(int64_t v) { return v >= 0 && v < (int64_t(1) << 31); }

int out_kind(bsg_dtype t) {
  switch (t) {
    case BSG_F32: return bsg::kOutF32;
    case BSG_BF16: return bsg::kOutBF16;
    case BSG_F16: return bsg::kOutF16;
    case BSG_E4M3: return bsg::kOutE4M3;
    case BSG_E2M1: return bsg::kOutE2M1;
    default: return bsg::kOutNone;
  }
}

// Bits per element of an output kind.
int64_t out_bits(int kind) {
  return kind == bsg::kOutF32 ? 32 : (kind == bsg::kOutBF16 || kind == bsg::kOutF16) ? 16 : kind == bsg::kOutE4M3 ? 8 : 4;
}

int choose_tile_n(int fmt, int64_t n, int64_t m_tiles_total, int num_sms, bool heavy_epilogue,
                  const bsg_gemm_opts* opts) {
  if (opts && (opts->tile_n == 128 || opts->tile_n == 256)) return opts->tile_n;
  if (opts && (opts->tile_n == 192 || opts->tile_n == 224) && fmt == bsg::kMXFP8) return opts->tile_n;
  if (n <= 128) return 128;
  // Heavy epilogues (E4M3 D with row and column re-quantisation; the dSwiGLU backward with its
  // C reads) run about as long as a tile's MMAs: 224-wide tiles keep two accumulators in TMEM so
  // they overlap the next tile's MMAs.  Lighter epilogues run faster on 256-wide tiles (fewer,
  // larger MMAs).
  if (fmt == bsg::kMXFP8 && heavy_epilogue) return 224;
  return (m_tiles_total * cdiv(n, 256) >= num_sms) ? 256 : 128;
}

// CTA pairs (256 x 256 tiles) when asked for, or when the problem still gives every pair a tile.
struct TilePlan {
  bool pairs;  // CTA-pair kernel (256-row tiles) or one-CTA kernel (128-row tiles)
  int bn;      // tile width
};

// Kernel and tile width for a GEMM with `m` rows (per batch), `n` columns and `l` batches.
// CTA pairs halve the B bytes each SM loads per K slice (the one-CTA kernel's TMA feed is its
// limit once the epilogue is overlapped); they need enough 256-row tiles to fill the GPU.  Heavy
// epilogues (E4M3 D, dSwiGLU) run about as long as a tile's MMAs, so they take 224-wide tiles
// with two TMEM accumulators, whose epilogue overlaps the next tile.
TilePlan plan_tiles(int fmt, int64_t m, int64_t n, int64_t l, int num_sms, bool heavy_epilogue,
                    const bsg_gemm_opts* opts) {
  const int cta_pair = opts ? opts->cta_pair : 0;
  const int tile_n = opts ? opts->tile_n : 0;
  const bool wide_ok = fmt == bsg::kMXFP8;
  if (cta_pair == 2) {
    const bool w224 = wide_ok && (tile_n == 224 || (tile_n == 0 && heavy_epilogue));
    return {true, w224 ? 224 : 256};
  }
  const int64_t tiles256 = l * cdiv(m, 256) * cdiv(n, 256);
  if (cta_pair == 0 && tile_n == 0 && m >= 256 && n > 128 && tiles256 >= num_sms / 2)
    return {true, (wide_ok && heavy_epilogue) ? 224 : 256};
  return {false, choose_tile_n(fmt, n, l * cdiv(m, 128), num_sms, heavy_epilogue, opts)};
}

int max_pairs(int64_t tiles, int num_sms, const bsg_gemm_opts* opts) {
  int64_t pairs = num_sms / 2;
  if (opts && opts->max_ctas > 0 && opts->max_ctas / 2 < pairs) pairs = opts->max_ctas / 2;
  if (tiles < pairs) pairs = tiles;
  return static_cast<int>(pairs < 1 ? 1 : pairs);
}

int grid_size(int64_t tiles, int num_sms, const bsg_gemm_opts* opts) {
  int64_t g = num_sms;
  if (opts && opts->max_ctas > 0 && opts->max_ctas < g) g = opts->max_ctas;
  if (tiles < g) g = tiles;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

uint32_t bsg::next_call_epoch() {
  uint32_t e = 0;
  while (e == 0) e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  return e;
}

extern "C" {

size_t bsg_workspace_size(void) { return kWorkspaceBytes; }

size_t bsg_sf_bytes(int64_t batch, int64_t rows, int64_t k, int sf_vec_size) {
  if (batch <= 0 || rows <= 0 || k <= 0 || sf_vec_size <= 0) return 0;
  return static_cast<size_t>(batch * cdiv(rows, 128) * cdiv(cdiv(k, sf_vec_size), 4) * 512);
}

const char* bsg_status_string(bsg_status s) {
  switch (s) {
    case BSG_OK: return "BSG_OK";
    case BSG_ERR_INVALID_ARG: return "BSG_ERR_INVALID_ARG";
    case BSG_ERR_UNSUPPORTED: return "BSG_ERR_UNSUPPORTED";
    case BSG_ERR_ALIGNMENT: return "BSG_ERR_ALIGNMENT";
    case BSG_ERR_ARCH: return "BSG_ERR_ARCH";
    case BSG_ERR_CUDA: return "BSG_ERR_CUDA";
    case BSG_ERR_DEVICE: return "BSG_ERR_DEVICE";
    case BSG_ERR_BAD_OFFSETS: return "BSG_ERR_BAD_OFFSETS";
    case BSG_ERR_WORKSPACE: return "BSG_ERR_WORKSPACE";
  }
  return "BSG_ERR_UNKNOWN";
}

namespace {

bsg_status quantize_impl(const void* x, bool x_bf16, int64_t batch, int64_t rows, int64_t k, bsg_dtype q_dtype,
                         int sf_vec_size, bsg_sf_dtype sf_dtype, void* q, uint8_t* sf, void* stream) {
  int fmt = 0;
  bsg_status st = operand_format(q_dtype, sf_dtype, sf_vec_size, &fmt);
  if (st != BSG_OK) return st;
  if (!x || !q || !sf) return BSG_ERR_INVALID_ARG;
  if (batch < 1 || rows < 1 || k < sf_vec_size || k % sf_vec_size != 0) return BSG_ERR_INVALID_ARG;
  if (k > (int64_t{1} << 30)) return BSG_ERR_INVALID_ARG;  // row offsets along K are 32-bit in the kernel
  if ((fmt == bsg::kMXFP8 && k % 16 != 0) || (fmt == bsg::kNVFP4 && k % 32 != 0)) return BSG_ERR_ALIGNMENT;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return BSG_ERR_ALIGNMENT;
  DeviceInfo info;
  st = current_device(nullptr, &info);
  if (st != BSG_OK) return st;
  cudaError_t e = bsg::launch_quantize(fmt, x, x_bf16, batch, rows, k, static_cast<uint8_t*>(q), sf, info.num_sms,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
}

}  // namespace

bsg_status bsg_quantize_mx(const float* x, int64_t batch, int64_t rows, int64_t k, bsg_dtype q_dtype,
                           int sf_vec_size, bsg_sf_dtype sf_dtype, void* q, uint8_t* sf, void* stream) {
  NvtxRange nvtx_range("bsg_quantize_mx");
  return quantize_impl(x, false, batch, rows, k, q_dtype, sf_vec_size, sf_dtype, q, sf, stream);
}

bsg_status bsg_quantize_mx_bf16(const void* x, int64_t batch, int64_t rows, int64_t k, bsg_dtype q_dtype,
                                int sf_vec_size, bsg_sf_dtype sf_dtype, void* q, uint8_t* sf, void* stream) {
  NvtxRange nvtx_range("bsg_quantize_mx_bf16");
  return quantize_impl(x, true, batch, rows, k, q_dtype, sf_vec_size, sf_dtype, q, sf, stream);
}

bsg_status bsg_gemm_amax(const void* a, const void* b, const uint8_t* sfa, const uint8_t* sfb, bsg_dtype ab_dtype,
                         bsg_sf_dtype sf_dtype, int sf_vec_size, int64_t m, int64_t n, int64_t k, int64_t l,
                         void* c, bsg_dtype c_dtype, float* amax, const bsg_gemm_opts* opts, void* workspace,
                         size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("bsg_gemm_amax");
  int fmt = 0;
  bsg_status st = operand_format(ab_dtype, sf_dtype, sf_vec_size, &fmt);
  if (st != BSG_OK) return st;
  if (!a || !b || !sfa || !sfb || !c || !amax) return BSG_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kWorkspaceBytes) return BSG_ERR_WORKSPACE;
  if (m < 1 || n < 1 || k < 1 || l < 1) return BSG_ERR_INVALID_ARG;
  if (opts && opts->b_major != 0) return BSG_ERR_INVALID_ARG;  // N-major B: per-expert weights only
  if (!fits_int32(m) || !fits_int32(n) || !fits_int32(k) || !fits_int32(l)) return BSG_ERR_INVALID_ARG;
  if (k % sf_vec_size != 0) return BSG_ERR_INVALID_ARG;
  // C: f32, bf16 or f16; with FP4 operands also plain E4M3 or packed E2M1 (the pages disable FP8
  // C with FP8 operands and allow FP4 C only with FP4 operands)
  const int c_kind = out_kind(c_dtype);
  if (c_kind == bsg::kOutNone) return BSG_ERR_UNSUPPORTED;
  if ((c_kind == bsg::kOutE4M3 || c_kind == bsg::kOutE2M1) && fmt != bsg::kNVFP4) return BSG_ERR_UNSUPPORTED;
  const int64_t row_bytes = fmt == bsg::kMXFP8 ? k : k / 2;
  if (row_bytes % 16 != 0 || (n * out_bits(c_kind)) % 128 != 0) return BSG_ERR_ALIGNMENT;
  if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(c) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || (reinterpret_cast<uintptr_t>(amax) & 3u) != 0)
    return BSG_ERR_ALIGNMENT;
  DeviceInfo info;
  st = current_device(nullptr, &info);
  if (st != BSG_OK) return st;

  const TilePlan plan = plan_tiles(fmt, m, n, l, info.num_sms, false, opts);
  const bool pairs = plan.pairs;
  const int bn = plan.bn;
  const int64_t m_tiles = pairs ? cdiv(m, 256) : cdiv(m, 128);
  const int64_t n_tiles = cdiv(n, bn);
  const int64_t tiles = l * m_tiles * n_tiles;
  const int elems_per_ktile = fmt == bsg::kMXFP8 ? 128 : 256;
  if (!fits_int32(tiles)) return BSG_ERR_INVALID_ARG;

  CUtensorMap ta, tb;
  if (!make_operand_map(&ta, a, row_bytes, m, l, 128) ||
      !make_operand_map(&tb, b, row_bytes, n, l, pairs ? bn / 2 : bn))
    return BSG_ERR_CUDA;
  const int64_t sf_kt = cdiv(k / sf_vec_size, 4);

  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.m = static_cast<int>(m);
  p.n = static_cast<int>(n);
  p.k = static_cast<int>(k);
  p.l = static_cast<int>(l);
  p.m_tiles = static_cast<int>(m_tiles);
  p.n_tiles = static_cast<int>(n_tiles);
  p.k_tiles = static_cast<int>(cdiv(k, elems_per_ktile));
  p.num_tiles = static_cast<int>(tiles);
  p.sfa = sfa;
  p.sfb = sfb;
  p.sfa_mt = static_cast<int>(cdiv(m, 128));
  p.sfb_mt = static_cast<int>(cdiv(n, 128));
  p.sf_kt = static_cast<int>(sf_kt);
  p.c = c;
  p.c_kind = c_kind;
  p.amax = amax;
  p.err = static_cast<uint32_t*>(workspace);
  p.epoch = bsg::next_call_epoch();

  // one launch and nothing else: the kernel tags its error record and amax accumulator in the
  // workspace with this call's epoch and writes *amax itself
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemmConfig cfg{fmt, bn, bsg::kEpiDense};
  cudaError_t e = pairs ? bsg::launch_gemm_pair(cfg, ta, tb, p, max_pairs(tiles, info.num_sms, opts), s)
                        : bsg::launch_gemm_dense(cfg, ta, tb, p, grid_size(tiles, info.num_sms, opts), s);
  return e == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
}

}  // extern "C"

namespace {

// The grouped GEMM for contiguous B / SFB (b, sfb) or per-expert pointer arrays (b_ptrs, sfb_ptrs,
// device int64 (num_experts,)); exactly one of the two forms is given.
bsg_status grouped_impl(const void* a, const void* b, const int64_t* b_ptrs, const uint8_t* sfa, const uint8_t* sfb,
                        const int64_t* sfb_ptrs, bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype, int sf_vec_size,
                        int64_t valid_m, int64_t n, int64_t k, int64_t num_experts, const int32_t* padded_offsets,
                        const float* alpha, const float* prob, float tanh_clamp_scale, const float* norm_const,
                        void* c, bsg_dtype c_dtype, void* d, void* d_col, bsg_dtype d_dtype, uint8_t* sfd_row,
                        uint8_t* sfd_col, float* amax, const bsg_gemm_opts* opts, void* workspace,
                        size_t workspace_bytes, void* stream) {
  int fmt = 0;
  bsg_status st = operand_format(ab_dtype, sf_dtype, sf_vec_size, &fmt);
  if (st != BSG_OK) return st;
  const bool discrete = b_ptrs != nullptr;
  // with valid_m == 0 nothing is read or written but the per-expert amax: the row-sized and
  // operand buffers may be null (empty tensors)
  const bool empty = valid_m == 0;
  if (!padded_offsets || (!empty && (!a || !sfa || !alpha || !prob || !d))) return BSG_ERR_INVALID_ARG;
  if (discrete ? (b || sfb || !sfb_ptrs) : (!empty && (!b || !sfb || sfb_ptrs))) return BSG_ERR_INVALID_ARG;
  const size_t ws_need = discrete ? bsg_grouped_discrete_workspace_size(num_experts) : kWorkspaceBytes;
  if (!workspace || workspace_bytes < ws_need) return BSG_ERR_WORKSPACE;
  if (valid_m < 0 || valid_m % 256 != 0 || n < 1 || k < 1 || num_experts < 1 || num_experts > 1024)
    return BSG_ERR_INVALID_ARG;
  if (!fits_int32(valid_m) || !fits_int32(n) || !fits_int32(k)) return BSG_ERR_INVALID_ARG;
  if (k % sf_vec_size != 0) return BSG_ERR_INVALID_ARG;
  const bool fp8_d = d_dtype == BSG_E4M3;
  const int d_kind = fp8_d ? bsg::kOutE4M3 : out_kind(d_dtype);
  if (!fp8_d && d_kind != bsg::kOutBF16 && d_kind != bsg::kOutF16 && d_kind != bsg::kOutF32) return BSG_ERR_UNSUPPORTED;
  if (fp8_d) {
    if (fmt != bsg::kMXFP8) return BSG_ERR_UNSUPPORTED;
    if (!empty && (!d_col || !sfd_row || !sfd_col || !norm_const)) return BSG_ERR_INVALID_ARG;
    if (n % 32 != 0) return BSG_ERR_INVALID_ARG;
  } else {
    if (!amax || d_col || sfd_row || sfd_col) return BSG_ERR_INVALID_ARG;
  }
  const int c_kind = c ? out_kind(c_dtype) : bsg::kOutNone;
  if (c && c_kind != bsg::kOutBF16 && c_kind != bsg::kOutF16 && c_kind != bsg::kOutF32) return BSG_ERR_UNSUPPORTED;
  if (!(tanh_clamp_scale == tanh_clamp_scale)) return BSG_ERR_INVALID_ARG;  // NaN
  const int64_t row_bytes = fmt == bsg::kMXFP8 ? k : k / 2;
  if (row_bytes % 16 != 0 || (n * out_bits(d_kind)) % 128 != 0 || (c && (n * out_bits(c_kind)) % 128 != 0))
    return BSG_ERR_ALIGNMENT;
  if (!aligned16(a) || (b && !aligned16(b)) || !aligned16(sfa) || (sfb && !aligned16(sfb)) || !aligned16(d) ||
      (reinterpret_cast<uintptr_t>(b_ptrs) & 7u) || (reinterpret_cast<uintptr_t>(sfb_ptrs) & 7u) ||
      (c && !aligned16(c)) || (d_col && !aligned16(d_col)) || (sfd_row && !aligned16(sfd_row)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || (reinterpret_cast<uintptr_t>(padded_offsets) & 3u))
    return BSG_ERR_ALIGNMENT;
  DeviceInfo info;
  st = current_device(nullptr, &info);
  if (st != BSG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (opts && opts->validate_offsets) {
    std::vector<int32_t> h(static_cast<size_t>(num_experts));
    if (cudaMemcpyAsync(h.data(), padded_offsets, h.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return BSG_ERR_CUDA;
    int32_t prev = 0;
    for (size_t i = 0; i < h.size(); ++i) {
      if (h[i] % 256 != 0 || h[i] < prev || h[i] > valid_m) return BSG_ERR_BAD_OFFSETS;
      prev = h[i];
    }
    if (prev != valid_m) return BSG_ERR_BAD_OFFSETS;
  }

  // N-major B (per-expert weights, FP8): one 128-element swizzle row of N per CTA and K row, so
  // 256-wide CTA-pair tiles or 128-wide one-CTA tiles
  const bool b_mn = discrete && opts && opts->b_major == 1;
  if (opts && opts->b_major != 0 && !b_mn) return BSG_ERR_INVALID_ARG;
  if (b_mn) {
    if (fmt != bsg::kMXFP8) return BSG_ERR_UNSUPPORTED;
    if (opts->tile_n != 0 && opts->tile_n != 128 && opts->tile_n != 256) return BSG_ERR_UNSUPPORTED;
    if (n % 16 != 0) return BSG_ERR_ALIGNMENT;  // the row pitch of a (k, n) B
  }

  // tiles and tensor maps (host only) before anything is enqueued
  TilePlan plan = plan_tiles(fmt, valid_m, n, 1, info.num_sms, fp8_d && !b_mn, opts);
  if (b_mn) plan.bn = plan.pairs ? 256 : 128;
  const bool pairs = plan.pairs;
  const int bn = plan.bn;
  const int64_t m_tiles = pairs ? valid_m / 256 : valid_m / 128;
  const int64_t n_tiles = cdiv(n, bn);
  const int64_t tiles = m_tiles * n_tiles;
  if (!fits_int32(tiles)) return BSG_ERR_INVALID_ARG;
  const int elems_per_ktile = fmt == bsg::kMXFP8 ? 128 : 256;
  CUtensorMap ta, tb;
  if (valid_m > 0) {
    if (!make_operand_map(&ta, a, row_bytes, valid_m, 1, 128)) return BSG_ERR_CUDA;
    // per-expert weights: a template for one expert's B, its address replaced per expert on the
    // device (the address encoded here, a's, is never read through it)
    const bool ok = b_mn ? make_operand_map_mn(&tb, a, n, k)
                         : make_operand_map(&tb, discrete ? a : b, row_bytes, n, discrete ? 1 : num_experts,
                                            pairs ? bn / 2 : bn);
    if (!ok) return BSG_ERR_CUDA;
  }

  if (!fp8_d && cudaMemsetAsync(amax, 0, sizeof(float) * num_experts, s) != cudaSuccess) return BSG_ERR_CUDA;
  if (fp8_d && n % 128 != 0 && !empty) {
    // SFD_col rows n .. ceil(n/128)*128 are padding the kernel never touches
    if (cudaMemsetAsync(sfd_col, 0, bsg_sf_bytes(1, n, valid_m, 32), s) != cudaSuccess) return BSG_ERR_CUDA;
  }
  // no kernel runs for an empty call: its error record is cleared instead
  if (empty) return cudaMemsetAsync(workspace, 0, 16, s) == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
  const uint32_t epoch = bsg::next_call_epoch();
  const CUtensorMap* b_maps = nullptr;
  if (discrete) {
    // one descriptor per expert after the 256-byte record, written by a kernel from the device
    // pointer arrays; the GEMM kernel reads them from global memory (tensor-map proxy acquire)
    CUtensorMap* dst = reinterpret_cast<CUtensorMap*>(static_cast<uint8_t*>(workspace) + kWorkspaceBytes);
    if (bsg::launch_expert_maps(tb, b_ptrs, sfb_ptrs, static_cast<int>(num_experts), dst,
                                static_cast<uint32_t*>(workspace), epoch, s) != cudaSuccess)
      return BSG_ERR_CUDA;
    b_maps = dst;
  }
  const int64_t sf_kt = cdiv(k / sf_vec_size, 4);

  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.m = static_cast<int>(valid_m);
  p.n = static_cast<int>(n);
  p.k = static_cast<int>(k);
  p.l = static_cast<int>(num_experts);
  p.m_tiles = static_cast<int>(m_tiles);
  p.n_tiles = static_cast<int>(n_tiles);
  p.k_tiles = static_cast<int>(cdiv(k, elems_per_ktile));
  p.num_tiles = static_cast<int>(tiles);
  p.sfa = sfa;
  p.sfb = sfb;
  p.b_maps = b_maps;
  p.sfb_ptrs = sfb_ptrs;
  p.b_mn_major = b_mn ? 1 : 0;
  p.sfa_mt = static_cast<int>(valid_m / 128);
  p.sfb_mt = static_cast<int>(cdiv(n, 128));
  p.sf_kt = static_cast<int>(sf_kt);
  p.c = c;
  p.c_kind = c_kind;
  p.d_kind = d_kind;
  p.amax = amax;
  p.offsets = padded_offsets;
  p.alpha = alpha;
  p.prob = prob;
  p.clamp_s = tanh_clamp_scale > 0.0f ? tanh_clamp_scale : 0.0f;
  p.tanh_approx = (opts && opts->tanh_approx) ? 1 : 0;
  p.norm_const = norm_const;
  p.d = d;
  p.d_col = d_col;
  p.sfd_row = sfd_row;
  p.sfd_col = sfd_col;
  p.sfd_row_kt = static_cast<int>(cdiv(n, 128));
  p.sfd_col_mt = static_cast<int>(cdiv(n, 128));
  p.sfd_col_kt = static_cast<int>(cdiv(valid_m, 128));
  // whole-sector row stores of C only beside the E4M3-D epilogue, which overlaps the next tile's
  // MMAs (measured 1.2-1.5 % faster there; the exposed bf16-D epilogue was 2.6 % slower with them)
  p.c_v8 = fp8_d && c_kind == bsg::kOutBF16 && aligned32(c) && n % 16 == 0;
  p.d_v8 = fp8_d && aligned32(d) && aligned32(d_col);
  p.err = static_cast<uint32_t*>(workspace);
  p.epoch = epoch;
  // bf16 D (and bf16 or no C) on 256-wide CTA pairs: the epilogue stores its 32 x 32 blocks with
  // TMA (row pitch a multiple of 16 bytes; the maps clip the blocks at valid_m rows and N columns)
  CUtensorMap tcm, tdm;
  p.out_tma = pairs && bn == 256 && d_kind == bsg::kOutBF16 && (c_kind == bsg::kOutNone || c_kind == bsg::kOutBF16) &&
              n % 8 == 0 && aligned16(d) && (c_kind == bsg::kOutNone || aligned16(c));
  if (p.out_tma) {
    if (!make_output_map_bf16(&tdm, d, n, valid_m)) return BSG_ERR_CUDA;
    tcm = tdm;  // not read without C
    if (c_kind == bsg::kOutBF16 && !make_output_map_bf16(&tcm, c, n, valid_m)) return BSG_ERR_CUDA;
  }

  GemmConfig cfg{fmt, bn, fp8_d ? bsg::kEpiGroupedFP8 : bsg::kEpiGroupedBF16};
  cudaError_t e = pairs ? bsg::launch_gemm_pair(cfg, ta, tb, p, max_pairs(tiles, info.num_sms, opts), s,
                                                p.out_tma ? &tcm : nullptr, p.out_tma ? &tdm : nullptr)
                        : bsg::launch_gemm_grouped(cfg, ta, tb, p, grid_size(tiles, info.num_sms, opts), s);
  if (e == cudaErrorInvalidValue) return BSG_ERR_UNSUPPORTED;
  return e == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
}

}  // namespace

extern "C" {

bsg_status bsg_grouped_gemm_srelu(const void* a, const void* b, const uint8_t* sfa, const uint8_t* sfb,
                                  bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype, int sf_vec_size, int64_t valid_m,
                                  int64_t n, int64_t k, int64_t num_experts, const int32_t* padded_offsets,
                                  const float* alpha, const float* prob, float tanh_clamp_scale,
                                  const float* norm_const, void* c, bsg_dtype c_dtype, void* d, void* d_col,
                                  bsg_dtype d_dtype, uint8_t* sfd_row, uint8_t* sfd_col, float* amax,
                                  const bsg_gemm_opts* opts, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  NvtxRange nvtx_range("bsg_grouped_gemm_srelu");
  if (!b || !sfb) return BSG_ERR_INVALID_ARG;
  return grouped_impl(a, b, nullptr, sfa, sfb, nullptr, ab_dtype, sf_dtype, sf_vec_size, valid_m, n, k, num_experts,
                      padded_offsets, alpha, prob, tanh_clamp_scale, norm_const, c, c_dtype, d, d_col, d_dtype,
                      sfd_row, sfd_col, amax, opts, workspace, workspace_bytes, stream);
}

size_t bsg_grouped_discrete_workspace_size(int64_t num_experts) {
  if (num_experts < 1) return kWorkspaceBytes;
  return kWorkspaceBytes + static_cast<size_t>(num_experts) * sizeof(CUtensorMap);
}

bsg_status bsg_grouped_gemm_srelu_discrete(const void* a, const int64_t* b_ptrs, const uint8_t* sfa,
                                           const int64_t* sfb_ptrs, bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype,
                                           int sf_vec_size, int64_t valid_m, int64_t n, int64_t k,
                                           int64_t num_experts, const int32_t* padded_offsets, const float* alpha,
                                           const float* prob, float tanh_clamp_scale, const float* norm_const,
                                           void* c, bsg_dtype c_dtype, void* d, void* d_col, bsg_dtype d_dtype,
                                           uint8_t* sfd_row, uint8_t* sfd_col, float* amax,
                                           const bsg_gemm_opts* opts, void* workspace, size_t workspace_bytes,
                                           void* stream) {
  NvtxRange nvtx_range("bsg_grouped_gemm_srelu_discrete");
  if (!b_ptrs || !sfb_ptrs) return BSG_ERR_INVALID_ARG;
  return grouped_impl(a, nullptr, b_ptrs, sfa, nullptr, sfb_ptrs, ab_dtype, sf_dtype, sf_vec_size, valid_m, n, k,
                      num_experts, padded_offsets, alpha, prob, tanh_clamp_scale, norm_const, c, c_dtype, d, d_col,
                      d_dtype, sfd_row, sfd_col, amax, opts, workspace, workspace_bytes, stream);
}

bsg_status bsg_grouped_gemm_dswiglu(const void* a, const void* b, const uint8_t* sfa, const uint8_t* sfb,
                                    bsg_dtype ab_dtype, bsg_sf_dtype sf_dtype, int sf_vec_size, int64_t valid_m,
                                    int64_t n, int64_t k, int64_t num_experts, const int32_t* padded_offsets,
                                    const float* alpha, const float* beta, const float* prob, const void* c,
                                    bsg_dtype c_dtype, const float* norm_const, void* d_row, void* d_col,
                                    bsg_dtype d_dtype, uint8_t* sfd_row, uint8_t* sfd_col, float* dprob,
                                    float* amax, const bsg_gemm_opts* opts, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  NvtxRange nvtx_range("bsg_grouped_gemm_dswiglu");
  int fmt = 0;
  bsg_status st = operand_format(ab_dtype, sf_dtype, sf_vec_size, &fmt);
  if (st != BSG_OK) return st;
  // with valid_m == 0 nothing is read or written but the per-expert amax: the row-sized and
  // operand buffers may be null (empty tensors)
  const bool empty = valid_m == 0;
  if (!padded_offsets ||
      (!empty && (!a || !b || !sfa || !sfb || !alpha || !beta || !prob || !c || !d_row || !dprob)))
    return BSG_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kWorkspaceBytes) return BSG_ERR_WORKSPACE;
  if (opts && opts->b_major != 0) return BSG_ERR_INVALID_ARG;  // N-major B: per-expert weights only
  // N a multiple of 32: C and D are 32-column input / gate (ab / dswiglu) blocks; 2 * num_experts
  // amax values are staged in the kernel's shared memory
  if (valid_m < 0 || valid_m % 256 != 0 || n < 32 || n % 32 != 0 || k < 1 || num_experts < 1 ||
      num_experts > 512)
    return BSG_ERR_INVALID_ARG;
  if (!fits_int32(valid_m) || !fits_int32(2 * n) || !fits_int32(k)) return BSG_ERR_INVALID_ARG;
  if (k % sf_vec_size != 0) return BSG_ERR_INVALID_ARG;
  const bool fp8_d = d_dtype == BSG_E4M3;
  const int d_kind = out_kind(d_dtype);
  if (!fp8_d && d_kind != bsg::kOutBF16 && d_kind != bsg::kOutF16 && d_kind != bsg::kOutF32) return BSG_ERR_UNSUPPORTED;
  if (fp8_d) {
    if (fmt != bsg::kMXFP8) return BSG_ERR_UNSUPPORTED;
    if (!empty && (!d_col || !sfd_row || !sfd_col || !norm_const)) return BSG_ERR_INVALID_ARG;
  } else {
    if (!amax || d_col || sfd_row || sfd_col) return BSG_ERR_INVALID_ARG;
  }
  const int c_kind = out_kind(c_dtype);
  if (c_kind != bsg::kOutBF16 && c_kind != bsg::kOutF16 && c_kind != bsg::kOutF32 && c_kind != bsg::kOutE4M3)
    return BSG_ERR_UNSUPPORTED;
  const int64_t row_bytes = fmt == bsg::kMXFP8 ? k : k / 2;
  if (row_bytes % 16 != 0 || (2 * n * out_bits(d_kind)) % 128 != 0 || (2 * n * out_bits(c_kind)) % 128 != 0)
    return BSG_ERR_ALIGNMENT;
  if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(c) || !aligned16(d_row) ||
      (d_col && !aligned16(d_col)) || (sfd_row && !aligned16(sfd_row)) || (sfd_col && !aligned16(sfd_col)) ||
      (reinterpret_cast<uintptr_t>(dprob) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      (reinterpret_cast<uintptr_t>(padded_offsets) & 3u))
    return BSG_ERR_ALIGNMENT;
  DeviceInfo info;
  st = current_device(nullptr, &info);
  if (st != BSG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (opts && opts->validate_offsets) {
    std::vector<int32_t> h(static_cast<size_t>(num_experts));
    if (cudaMemcpyAsync(h.data(), padded_offsets, h.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return BSG_ERR_CUDA;
    int32_t prev = 0;
    for (size_t i = 0; i < h.size(); ++i) {
      if (h[i] % 256 != 0 || h[i] < prev || h[i] > valid_m) return BSG_ERR_BAD_OFFSETS;
      prev = h[i];
    }
    if (prev != valid_m) return BSG_ERR_BAD_OFFSETS;
  }

  const int64_t n_d = 2 * n;
  // tiles and tensor maps (host only) before anything is enqueued
  const TilePlan plan = plan_tiles(fmt, valid_m, n, 1, info.num_sms, true, opts);
  const bool pairs = plan.pairs;
  const int bn = plan.bn;
  if (!pairs && bn == 192) return BSG_ERR_UNSUPPORTED;  // no 192-wide dSwiGLU kernel
  const int64_t m_tiles = pairs ? valid_m / 256 : valid_m / 128;
  const int64_t n_tiles = cdiv(n, bn);
  const int64_t tiles = m_tiles * n_tiles;
  if (!fits_int32(tiles)) return BSG_ERR_INVALID_ARG;
  const int elems_per_ktile = fmt == bsg::kMXFP8 ? 128 : 256;
  CUtensorMap ta, tb;
  if (valid_m > 0 && (!make_operand_map(&ta, a, row_bytes, valid_m, 1, 128) ||
                      !make_operand_map(&tb, b, row_bytes, n, num_experts, pairs ? bn / 2 : bn)))
    return BSG_ERR_CUDA;

  if (!fp8_d && cudaMemsetAsync(amax, 0, 2 * sizeof(float) * num_experts, s) != cudaSuccess) return BSG_ERR_CUDA;
  if (fp8_d && n_d % 128 != 0 && !empty) {
    // SFD_col rows 2N .. ceil(2N/128)*128 are padding the kernel never touches
    if (cudaMemsetAsync(sfd_col, 0, bsg_sf_bytes(1, n_d, valid_m, 32), s) != cudaSuccess) return BSG_ERR_CUDA;
  }
  // no kernel runs for an empty call: its error record is cleared instead
  if (empty) return cudaMemsetAsync(workspace, 0, 16, s) == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
  const int64_t sf_kt = cdiv(k / sf_vec_size, 4);

  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.m = static_cast<int>(valid_m);
  p.n = static_cast<int>(n);
  p.k = static_cast<int>(k);
  p.l = static_cast<int>(num_experts);
  p.m_tiles = static_cast<int>(m_tiles);
  p.n_tiles = static_cast<int>(n_tiles);
  p.k_tiles = static_cast<int>(cdiv(k, elems_per_ktile));
  p.num_tiles = static_cast<int>(tiles);
  p.sfa = sfa;
  p.sfb = sfb;
  p.sfa_mt = static_cast<int>(valid_m / 128);
  p.sfb_mt = static_cast<int>(cdiv(n, 128));
  p.sf_kt = static_cast<int>(sf_kt);
  p.c_kind = bsg::kOutNone;
  p.d_kind = d_kind;
  p.amax = fp8_d ? nullptr : amax;
  p.offsets = padded_offsets;
  p.alpha = alpha;
  p.prob = prob;
  p.norm_const = norm_const;
  p.d = d_row;
  p.d_col = d_col;
  p.d_v8 = fp8_d && aligned32(d_row) && aligned32(d_col);
  p.sfd_row = sfd_row;
  p.sfd_col = sfd_col;
  p.sfd_row_kt = static_cast<int>(cdiv(n_d, 128));
  p.sfd_col_mt = static_cast<int>(cdiv(n_d, 128));
  p.sfd_col_kt = static_cast<int>(cdiv(valid_m, 128));
  p.c_in = c;
  p.c_in_kind = c_kind;
  p.beta = beta;
  p.dprob = dprob;
  p.err = static_cast<uint32_t*>(workspace);
  p.epoch = bsg::next_call_epoch();

  GemmConfig cfg{fmt, bn, fp8_d ? bsg::kEpiDswigluFP8 : bsg::kEpiDswigluF};
  cudaError_t e = pairs ? bsg::launch_gemm_pair_dswiglu(cfg, ta, tb, p, max_pairs(tiles, info.num_sms, opts), s)
                        : bsg::launch_gemm_dswiglu(cfg, ta, tb, p, grid_size(tiles, info.num_sms, opts), s);
  if (e == cudaErrorInvalidValue) return BSG_ERR_UNSUPPORTED;
  return e == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
}

size_t bsg_rope_workspace_size(int64_t tokens, int64_t num_heads, int64_t head_dim, int64_t q_lora) {
  if (tokens < 0 || num_heads < 0 || head_dim < 0 || q_lora < 0) return kWorkspaceBytes;
  return kWorkspaceBytes + bsg_sf_bytes(1, tokens, q_lora, 32) + bsg_sf_bytes(1, num_heads * head_dim, q_lora, 32);
}

bsg_status bsg_gemm_rope_mxfp8(const uint8_t* x, const uint8_t* x_scale, const uint8_t* w, const uint8_t* w_scale,
                               int scale_layout, const void* cos, const void* sin, int64_t tokens, int64_t q_lora,
                               int64_t num_heads, int64_t head_dim, int64_t qk_rope, uint8_t* out_fp8_row,
                               uint8_t* out_scales_row, uint8_t* out_fp8_col, uint8_t* out_scales_col,
                               const bsg_gemm_opts* opts, void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("bsg_gemm_rope_mxfp8");
  if (!x || !x_scale || !w || !w_scale || !cos || !sin || !out_fp8_row || !out_scales_row || !out_fp8_col ||
      !out_scales_col)
    return BSG_ERR_INVALID_ARG;
  if (scale_layout != 0 && scale_layout != 1) return BSG_ERR_INVALID_ARG;
  if (tokens < 128 || tokens % 128 != 0 || q_lora < 32 || q_lora % 32 != 0 || num_heads < 1 || head_dim < 1 ||
      qk_rope < 1)
    return BSG_ERR_INVALID_ARG;
  // the kernel holds one head per 192-wide tile, the last 64 features rotary
  if (head_dim != 192 || qk_rope != 64) return BSG_ERR_UNSUPPORTED;
  const int64_t n = num_heads * head_dim;
  if (!fits_int32(tokens) || !fits_int32(n) || !fits_int32(q_lora) || !fits_int32(tokens * (n / 32)))
    return BSG_ERR_INVALID_ARG;
  // Tiles: one head per CTA, two accumulators (the dual E4M3 epilogue overlaps the next tile's
  // MMAs): CTA pairs on 256 x 192 tiles (automatic when tokens % 256 == 0: each SM loads half a
  // head of w per K slice; measured 8 % faster at the DeepSeek-V3 shapes) or one-CTA 128 x 192
  // tiles (cta_pair == 1, or tokens % 256 != 0).  cta_pair == 2 with tile_n != 192 selects pairs
  // on 256 x 256 tiles spanning heads (a head's rotary chunk pair never straddles a 256-column
  // tile); their single accumulator exposes the epilogue and measured slower.
  const int cta_pair = opts ? opts->cta_pair : 0;
  const bool pair192 = (cta_pair == 0 && tokens % 256 == 0) || (cta_pair == 2 && opts->tile_n == 192);
  const bool pair_ok = tokens % 256 == 0 && (pair192 || n % 256 == 0);
  if (cta_pair == 2 && !pair_ok) return BSG_ERR_INVALID_ARG;
  const size_t ws_need = scale_layout == 1 ? bsg_rope_workspace_size(tokens, num_heads, head_dim, q_lora)
                                           : kWorkspaceBytes;
  if (!workspace || workspace_bytes < ws_need) return BSG_ERR_WORKSPACE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(cos) || !aligned16(sin) || !aligned16(out_fp8_row) ||
      !aligned16(out_fp8_col) || (scale_layout == 0 && (!aligned16(x_scale) || !aligned16(w_scale))) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return BSG_ERR_ALIGNMENT;
  DeviceInfo info;
  bsg_status st = current_device(nullptr, &info);
  if (st != BSG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const uint8_t* sfa = x_scale;
  const uint8_t* sfb = w_scale;
  if (scale_layout == 1) {
    // plain (rows, q_lora / 32) scales: scattered into the atom layout in the workspace
    uint8_t* pa = static_cast<uint8_t*>(workspace) + kWorkspaceBytes;
    uint8_t* pb = pa + bsg_sf_bytes(1, tokens, q_lora, 32);
    if (bsg::launch_sf_pack(x_scale, tokens, q_lora / 32, pa, s) != cudaSuccess ||
        bsg::launch_sf_pack(w_scale, n, q_lora / 32, pb, s) != cudaSuccess)
      return BSG_ERR_CUDA;
    sfa = pa;
    sfb = pb;
  }

  const bool pairs = pair_ok && (cta_pair == 2 || pair192);
  const int bn = pairs && !pair192 ? 256 : 192;
  const int64_t m_tiles = pairs ? tokens / 256 : tokens / 128;
  const int64_t n_tiles = n / bn;
  const int64_t tiles = m_tiles * n_tiles;
  if (!fits_int32(tiles)) return BSG_ERR_INVALID_ARG;
  CUtensorMap ta, tb;
  // a pair CTA holds half of the tile's B rows
  if (!make_operand_map(&ta, x, q_lora, tokens, 1, 128) ||
      !make_operand_map(&tb, w, q_lora, n, 1, pairs ? bn / 2 : bn))
    return BSG_ERR_CUDA;

  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.m = static_cast<int>(tokens);
  p.n = static_cast<int>(n);
  p.k = static_cast<int>(q_lora);
  p.l = 1;
  p.m_tiles = static_cast<int>(m_tiles);
  p.n_tiles = static_cast<int>(n_tiles);
  p.k_tiles = static_cast<int>(cdiv(q_lora, 128));
  p.num_tiles = static_cast<int>(tiles);
  p.sfa = sfa;
  p.sfb = sfb;
  p.sfa_mt = static_cast<int>(tokens / 128);
  p.sfb_mt = static_cast<int>(cdiv(n, 128));
  p.sf_kt = static_cast<int>(cdiv(q_lora / 32, 4));
  p.c_kind = bsg::kOutNone;
  p.d = out_fp8_row;
  p.d_col = out_fp8_col;
  p.d_v8 = aligned32(out_fp8_row) && aligned32(out_fp8_col);
  p.sfd_row = out_scales_row;
  p.sfd_col = out_scales_col;
  p.rope_cos = static_cast<const uint16_t*>(cos);
  p.rope_sin = static_cast<const uint16_t*>(sin);
  p.qk_rope = static_cast<int>(qk_rope);
  p.err = static_cast<uint32_t*>(workspace);
  p.epoch = bsg::next_call_epoch();

  GemmConfig cfg{bsg::kMXFP8, bn, bsg::kEpiRope};
  cudaError_t e = pairs ? bsg::launch_gemm_pair_rope(cfg, ta, tb, p, max_pairs(tiles, info.num_sms, opts), s)
                        : bsg::launch_gemm_rope(cfg, ta, tb, p, grid_size(tiles, info.num_sms, opts), s);
  if (e == cudaErrorInvalidValue) return BSG_ERR_UNSUPPORTED;
  return e == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
}

bsg_status bsg_gemm_rope_bf16(const void* x, const void* w, const void* cos, const void* sin, int64_t tokens,
                              int64_t q_lora, int64_t num_heads, int64_t head_dim, int64_t qk_rope,
                              uint8_t* out_fp8_row, uint8_t* out_scales_row, uint8_t* out_fp8_col,
                              uint8_t* out_scales_col, const bsg_gemm_opts* opts, void* workspace,
                              size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_range("bsg_gemm_rope_bf16");
  if (!x || !w || !cos || !sin || !out_fp8_row || !out_scales_row || !out_fp8_col || !out_scales_col)
    return BSG_ERR_INVALID_ARG;
  // bf16 rows of q_lora values: a multiple of eight keeps every row 16-byte aligned for TMA
  if (tokens < 128 || tokens % 128 != 0 || q_lora < 8 || q_lora % 8 != 0 || num_heads < 1 || head_dim < 1 ||
      qk_rope < 1)
    return BSG_ERR_INVALID_ARG;
  if (head_dim != 192 || qk_rope != 64) return BSG_ERR_UNSUPPORTED;
  // one head per 128 x 192 one-CTA tile, or with opts->cta_pair == 2 per CTA of a 256 x 192 pair
  // tile (not faster with bf16 operands: there the 192-wide MMAs, not the loads, bound the loop)
  const bool pairs = opts && opts->cta_pair == 2;
  if (pairs && tokens % 256 != 0) return BSG_ERR_INVALID_ARG;
  const int64_t n = num_heads * head_dim;
  if (!fits_int32(tokens) || !fits_int32(n) || !fits_int32(q_lora) || !fits_int32(tokens * (n / 32)))
    return BSG_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kWorkspaceBytes) return BSG_ERR_WORKSPACE;
  const int64_t row_bytes = q_lora * 2;
  if (!aligned16(x) || !aligned16(w) || !aligned16(cos) || !aligned16(sin) ||
      !aligned16(out_fp8_row) || !aligned16(out_fp8_col) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return BSG_ERR_ALIGNMENT;
  DeviceInfo info;
  bsg_status st = current_device(nullptr, &info);
  if (st != BSG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int bn = 192;
  const int64_t m_tiles = pairs ? tokens / 256 : tokens / 128;
  const int64_t tiles = m_tiles * num_heads;
  if (!fits_int32(tiles)) return BSG_ERR_INVALID_ARG;
  CUtensorMap ta, tb;
  if (!make_operand_map(&ta, x, row_bytes, tokens, 1, 128) ||
      !make_operand_map(&tb, w, row_bytes, n, 1, pairs ? bn / 2 : bn))
    return BSG_ERR_CUDA;

  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.m = static_cast<int>(tokens);
  p.n = static_cast<int>(n);
  p.k = static_cast<int>(q_lora);
  p.l = 1;
  p.m_tiles = static_cast<int>(m_tiles);
  p.n_tiles = static_cast<int>(num_heads);
  p.k_tiles = static_cast<int>(cdiv(q_lora, 64));
  p.num_tiles = static_cast<int>(tiles);
  p.c_kind = bsg::kOutNone;
  p.d = out_fp8_row;
  p.d_col = out_fp8_col;
  p.d_v8 = aligned32(out_fp8_row) && aligned32(out_fp8_col);
  p.sfd_row = out_scales_row;
  p.sfd_col = out_scales_col;
  p.rope_cos = static_cast<const uint16_t*>(cos);
  p.rope_sin = static_cast<const uint16_t*>(sin);
  p.qk_rope = static_cast<int>(qk_rope);
  p.err = static_cast<uint32_t*>(workspace);
  p.epoch = bsg::next_call_epoch();

  GemmConfig cfg{bsg::kBF16, bn, bsg::kEpiRope};
  cudaError_t e = pairs ? bsg::launch_gemm_pair_rope(cfg, ta, tb, p, max_pairs(tiles, info.num_sms, opts), s)
                        : bsg::launch_gemm_rope(cfg, ta, tb, p, grid_size(tiles, info.num_sms, opts), s);
  if (e == cudaErrorInvalidValue) return BSG_ERR_UNSUPPORTED;
  return e == cudaSuccess ? BSG_OK : BSG_ERR_CUDA;
}

bsg_status bsg_read_device_error(const void* workspace, void* stream, uint32_t* error_bits) {
  if (!workspace || !error_bits) return BSG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return BSG_ERR_CUDA;
  // error bits, the epoch that set them, the epoch of the last call that ran: the bits are that
  // call's only when the two epochs agree
  uint32_t w[3] = {0, 0, 0};
  if (cudaMemcpy(w, workspace, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return BSG_ERR_CUDA;
  const uint32_t bits = w[1] == w[2] ? w[0] : 0u;
  *error_bits = bits;
  return bits ? BSG_ERR_DEVICE : BSG_OK;
}

}  // extern "C"
