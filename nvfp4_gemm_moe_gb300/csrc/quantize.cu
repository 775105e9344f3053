// quantize.cu -- fp32 or bf16 -> MXFP8 / NVFP4 block quantiser (memory-bound).
//
// A warp takes one row at a time and walks its "units" of 32 blocks (1024 values for MXFP8, 512
// for NVFP4), with 4 KB of loads in flight per warp.  Each lane owns one block, so its maximum
// and its scale are decided once, without shuffles.  The scale bytes of 4 consecutive blocks are
// adjacent in the atom layout and leave as one 32-bit store.  Units of the padding rows of the
// last 128-row atom produce zero scale bytes.
// bf16 inputs are widened to fp32 (exactly) when a block is processed, so both input types share
// the arithmetic; their units are the same element counts at half the bytes, two units in flight.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace bsg {
namespace {

constexpr int kThreads = 256;

// RNE_UE4M3(a / 6) decided exactly: candidate from an fp32 approximation of the quotient
// (a times the rounded 1/6, within two ulps of a/6, so the candidate is at most one code
// off), then moved by at most one code after comparing a with 6 * (neighbouring midpoints),
// products that are exact in fp32 (a midpoint has at most 5 significant bits).  Saturates
// at 448.
__device__ __forceinline__ uint32_t ue4m3_code_of_amax_over_6(float a) {
  if (!(a > 0.0f)) return 0;
  const float q = a * (1.0f / 6.0f);
  uint32_t c = cvt_e4m3x2(q, 0.0f) & 0x7Fu;
  if (c > 0x7Eu) c = 0x7Eu;
  if (c < 0x7Eu) {
    const float t = 6.0f * (0.5f * (ue4m3_value(c) + ue4m3_value(c + 1)));
    if (a > t || (a == t && ((c + 1) & 1u) == 0)) c += 1;
  }
  if (c > 0) {
    const float t = 6.0f * (0.5f * (ue4m3_value(c - 1) + ue4m3_value(c)));
    if (a < t || (a == t && (c & 1u))) c -= 1;
  }
  return c;
}

// E2M1 nibble of RNE_satfinite(x / s) from exact thresholds t_i = midpoint_i * s: the
// magnitude index counts the midpoints below |x|; at a midpoint the even index wins, i.e.
// midpoints 1, 3, 5 (0.75, 1.75, 3.5) count when equal as well.  `t` holds thresholds for a
// strict comparison: t_i itself for i = 0, 2, 4, 6 and the float just below t_i for i = 1, 3, 5
// (a >= t  <=>  a > prev(t) for positive floats).  Seven independent comparisons summed beat a
// three-step binary search here (its steps depend on each other).  The sign bit is the sign of
// x (a negative value that rounds to zero gives -0), as the E4M3 conversion does.
__device__ __forceinline__ uint32_t e2m1_nibble(float x, const float (&t)[7]) {
  const float a = fabsf(x);
  const uint32_t idx = (a > t[0]) + (a > t[1]) + (a > t[2]) + (a > t[3]) + (a > t[4]) + (a > t[5]) + (a > t[6]);
  return idx | ((__float_as_uint(x) >> 28) & 8u);
}

// The seven strict-comparison thresholds of e2m1_nibble for scale s > 0.
__device__ __forceinline__ void e2m1_thresholds(float s, float (&t)[7]) {
  const float m[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
#pragma unroll
  for (int i = 0; i < 7; ++i) {
    const float v = m[i] * s;  // exact: at most 3 + 4 significant bits
    t[i] = (i & 1) ? __uint_as_float(__float_as_uint(v) - 1u) : v;
  }
}

// Raw loads (streaming: each input is read once) and their exact widening to fp32.  A bf16
// warp keeps twice the units in flight (the same bytes as fp32) in the same registers.
__device__ __forceinline__ float4 bf16x4_to_float4(uint32_t lo, uint32_t hi) {  // element 2i: low half of word i
  return make_float4(__uint_as_float(lo << 16), __uint_as_float(lo & 0xffff0000u), __uint_as_float(hi << 16),
                     __uint_as_float(hi & 0xffff0000u));
}
// One lane's block of N inputs (N = 16 or 32): raw 16-byte loads kept in flight, widened to fp32
// when the block is processed.
template <typename TIn, int N>
struct BlockIn;
template <int N>
struct BlockIn<float, N> {
  float4 a[N / 4];
  __device__ __forceinline__ void load(const float* p, bool ok) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i)
      a[i] = ok ? __ldcs(reinterpret_cast<const float4*>(p) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __device__ __forceinline__ void widen(float (&v)[N]) const {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      v[4 * i] = a[i].x; v[4 * i + 1] = a[i].y; v[4 * i + 2] = a[i].z; v[4 * i + 3] = a[i].w;
    }
  }
};
template <int N>
struct BlockIn<__nv_bfloat16, N> {
  uint4 a[N / 8];
  __device__ __forceinline__ void load(const __nv_bfloat16* p, bool ok) {
#pragma unroll
    for (int i = 0; i < N / 8; ++i)
      a[i] = ok ? __ldcs(reinterpret_cast<const uint4*>(p) + i) : make_uint4(0u, 0u, 0u, 0u);
  }
  __device__ __forceinline__ void widen(float (&v)[N]) const {
#pragma unroll
    for (int i = 0; i < N / 8; ++i) {
      const float4 lo = bf16x4_to_float4(a[i].x, a[i].y), hi = bf16x4_to_float4(a[i].z, a[i].w);
      v[8 * i] = lo.x; v[8 * i + 1] = lo.y; v[8 * i + 2] = lo.z; v[8 * i + 3] = lo.w;
      v[8 * i + 4] = hi.x; v[8 * i + 5] = hi.y; v[8 * i + 6] = hi.z; v[8 * i + 7] = hi.w;
    }
  }
};

// fp32 MXFP8 loads: one float4 per lane per 128-value unit (fully coalesced), 8 units (4 KB) in
// flight per warp.
struct MxLoadsF32 {
  static constexpr int kUnits = 8;
  static __device__ __forceinline__ float4 load4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
};

// MXFP8 from fp32: a unit is 128 consecutive values (one float4 per lane, fully coalesced), four
// blocks of 32 held by 8 lanes each (block maxima reduced with shuffles), the codes leave as one
// 32-bit store per lane and lane 0 stores the unit's scale word.  (One block per lane, as the
// bf16 kernel below does, measured 15 % slower from fp32: its 128-byte lane stride spreads every
// load instruction over 32 lines.)
template <typename TIn>
__global__ void __launch_bounds__(kThreads) quantize_mxfp8_kernel(const TIn* __restrict__ x, int64_t rows, int k,
                                                                  uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                                  int64_t rows_padded, int units_per_row,
                                                                  int64_t total_rows, int64_t mt_n, int64_t kt_n) {
  static_assert(sizeof(TIn) == 4, "fp32 input");
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t num_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;

  // one (padded) row per warp iteration: the row's batch and index are computed once, then
  // the warp walks the row's units with 4 KB of loads in flight
  for (int64_t rg = warp_id; rg < total_rows; rg += num_warps) {
    const int64_t l = rg / rows_padded;
    const int64_t r = rg - l * rows_padded;
    const bool row_ok = r < rows;
    const int64_t row_g = l * rows + r;
    const TIn* xr = x + row_g * k;
    constexpr int U = MxLoadsF32::kUnits;
    for (int kc0 = 0; kc0 < units_per_row; kc0 += U) {
      float4 raw[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int kk = (kc0 + j) * 128 + lane * 4;
        raw[j] = (row_ok && kc0 + j < units_per_row && kk < k) ? MxLoadsF32::load4(xr + kk)
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int kc = kc0 + j;
        if (kc >= units_per_row) break;  // uniform across the warp
        const int kk = kc * 128 + lane * 4;
        const bool elem_ok = row_ok && kk < k;
        const float4 vj = raw[j];
        float a = fmaxf(fmaxf(fabsf(vj.x), fabsf(vj.y)), fmaxf(fabsf(vj.z), fabsf(vj.w)));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        const uint32_t code = e8m0_ceil_code(a);
        const float inv = e8m0_inv_scale(code);
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(vj.x, inv), __fmul_rn(vj.y, inv));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(vj.z, inv), __fmul_rn(vj.w, inv));
        if (elem_ok) *reinterpret_cast<uint32_t*>(q + row_g * k + kk) = lo | (hi << 16);
        const uint32_t c1 = __shfl_sync(0xffffffffu, code, 8);
        const uint32_t c2 = __shfl_sync(0xffffffffu, code, 16);
        const uint32_t c3 = __shfl_sync(0xffffffffu, code, 24);
        if (lane == 0) {
          const uint64_t off = sf_offset(r, kc * 4, l, mt_n, kt_n);
          *reinterpret_cast<uint32_t*>(sf + off) = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
        }
      }
    }
  }
}

// MXFP8 from bf16: a unit is 1024 consecutive values of one row and lane i owns its block i (32
// values: four 16-byte loads), so the block maximum and the scale
// decision are made once per block with no shuffle, and the lane's 32 codes leave as two 16-byte
// stores.  The 32 scale bytes of a unit are eight 32-bit words of the atom layout, gathered from
// lanes 4w .. 4w + 3 and stored by lane 4w.
template <typename TIn>
__global__ void __launch_bounds__(kThreads)
    quantize_mxfp8_bf16_kernel(const TIn* __restrict__ x, int64_t rows, int k, uint8_t* __restrict__ q,
                               uint8_t* __restrict__ sf, int64_t rows_padded, int units_per_row, int64_t total_rows,
                               int64_t mt_n, int64_t kt_n) {
  static_assert(sizeof(TIn) == 2, "bf16 input");
  constexpr int kU = 2;  // units in flight per warp: 4 KB of bf16 loads
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t num_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  // one (padded) row per warp iteration: the row's batch and index are computed once, then
  // the warp walks the row's units
  for (int64_t rg = warp_id; rg < total_rows; rg += num_warps) {
    const int64_t l = rg / rows_padded;
    const int64_t r = rg - l * rows_padded;
    const bool row_ok = r < rows;
    const int64_t row_g = l * rows + r;
    const TIn* xr = x + row_g * k;
    for (int kc0 = 0; kc0 < units_per_row; kc0 += kU) {
      BlockIn<TIn, 32> raw[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int kk = (kc0 + j) * 1024 + lane * 32;
        raw[j].load(xr + kk, row_ok && kc0 + j < units_per_row && kk < k);
      }
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int kc = kc0 + j;
        if (kc >= units_per_row) break;  // uniform across the warp
        const int kk = kc * 1024 + lane * 32;
        float xs[32];
        raw[j].widen(xs);
        float m[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) m[e] = fmaxf(fabsf(xs[2 * e]), fabsf(xs[2 * e + 1]));
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
          for (int e = 0; e < w; ++e) m[e] = fmaxf(m[e], m[e + w]);
        }
        const uint32_t code = e8m0_ceil_code(m[0]);
        const float inv = e8m0_inv_scale(code);
        uint32_t w8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          w8[e] = cvt_e4m3x2(__fmul_rn(xs[4 * e], inv), __fmul_rn(xs[4 * e + 1], inv)) |
                  (cvt_e4m3x2(__fmul_rn(xs[4 * e + 2], inv), __fmul_rn(xs[4 * e + 3], inv)) << 16);
        if (row_ok && kk < k) {
          uint4* dst = reinterpret_cast<uint4*>(q + row_g * k + kk);
          dst[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
          dst[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
        }
        // block 4w + i of the unit is held by lane 4w + i; scale word w gathers lanes 4w .. 4w + 3
        const uint32_t c1 = __shfl_down_sync(0xffffffffu, code, 1);
        const uint32_t c2 = __shfl_down_sync(0xffffffffu, code, 2);
        const uint32_t c3 = __shfl_down_sync(0xffffffffu, code, 3);
        if ((lane & 3) == 0) {
          const int64_t kb = static_cast<int64_t>(kc) * 32 + lane;
          if ((kb >> 2) < kt_n) {
            const uint64_t off = sf_offset(r, kb, l, mt_n, kt_n);
            *reinterpret_cast<uint32_t*>(sf + off) = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
          }
        }
      }
    }
  }
}

// NVFP4: a unit is 512 consecutive values of one row and lane i owns its block i (16 values:
// four float4 loads of fp32, or two 16-byte loads of bf16), so the block maximum and the scale
// decision are made once per block with no shuffle, and the lane's 16 codes leave as one 64-bit
// store.  The 32 scale bytes of a unit are eight 32-bit words of the atom layout, gathered from
// lanes 4w .. 4w + 3 and stored by lane 4w.
template <typename TIn>
// fp32 input: four blocks resident per SM (64 registers, 72 without the bound; measured 10 %
// faster: more loads in flight); bf16 input: two (its 4-unit items need the registers)
__global__ void __launch_bounds__(kThreads, sizeof(TIn) == 4 ? 4 : 2)
    quantize_nvfp4_kernel(const TIn* __restrict__ x, int64_t rows, int k, uint8_t* __restrict__ q,
                          uint8_t* __restrict__ sf, int64_t rows_padded, int units_per_row, int64_t total_rows,
                          int64_t mt_n, int64_t kt_n) {
  // units in flight per warp: 4 KB of fp32 loads (two units) or of bf16 loads (four)
  constexpr int kU = sizeof(TIn) == 4 ? 2 : 4;
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t num_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  for (int64_t rg = warp_id; rg < total_rows; rg += num_warps) {
    const int64_t l = rg / rows_padded;
    const int64_t r = rg - l * rows_padded;
    const bool row_ok = r < rows;
    const int64_t row_g = l * rows + r;
    const TIn* xr = x + row_g * k;
    for (int kc0 = 0; kc0 < units_per_row; kc0 += kU) {
      BlockIn<TIn, 16> raw[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int kk = (kc0 + j) * 512 + lane * 16;
        raw[j].load(xr + kk, row_ok && kc0 + j < units_per_row && kk < k);
      }
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int kc = kc0 + j;
        if (kc >= units_per_row) break;  // uniform across the warp
        const int kk = kc * 512 + lane * 16;
        float xs[16];
        raw[j].widen(xs);
        float m[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m[e] = fmaxf(fabsf(xs[2 * e]), fabsf(xs[2 * e + 1]));
        const float a = fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
        const uint32_t code = ue4m3_code_of_amax_over_6(a);
        const float s = ue4m3_value(code);
        // Codes from the hardware's RNE conversion, bracketing the exact quotient v = x / s:
        // y_up = x * RN(RN(1/s) (1 + 2^-20)) and y_dn = x * RN(RN(1/s) (1 - 2^-20)) lie on either
        // side of v (their rounding errors are below 2^-22 relative), and RNE rounding is
        // monotonic, so where both convert to the same code so does v.  Where they differ a
        // midpoint lies between them: fp32 inputs take the exact threshold path (rare); for bf16
        // inputs v is then exactly that midpoint (x has 8 significant bits, a midpoint times s
        // at most 7: x / s is a midpoint or at least 2^-9 away from one), and the tie goes to the
        // even code of the two.  The conversion keeps the sign of x, also where the magnitude
        // rounds to zero (-0, as on the exact path); s = 0 gives +0.
        const float inv = code != 0 ? __frcp_rn(s) : 0.0f;
        const float inv_up = inv * (1.0f + 0x1p-20f), inv_dn = inv * (1.0f - 0x1p-20f);
        uint32_t up[2] = {0u, 0u}, dn[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          up[e >> 3] |= cvt_e2m1x2(xs[e] * inv_up, xs[e + 1] * inv_up) << (4 * (e & 7));
          dn[e >> 3] |= cvt_e2m1x2(xs[e] * inv_dn, xs[e + 1] * inv_dn) << (4 * (e & 7));
        }
        uint32_t nib[2] = {up[0], up[1]};
        bool near = false;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          if (up[w] != dn[w]) {
            if constexpr (sizeof(TIn) == 2) {
              // nibble k differs -> bit 4k of `differs`; the two codes are neighbours, and the one
              // whose last bit (bit 4k) is clear is the even one
              const uint32_t diff = up[w] ^ dn[w];
              const uint32_t differs = (diff | (diff >> 1) | (diff >> 2) | (diff >> 3)) & 0x11111111u;
              const uint32_t take_dn = (differs & up[w]) * 0xFu;  // whole nibbles where dn is even
              nib[w] = (up[w] & ~take_dn) | (dn[w] & take_dn);
            } else {
              near = true;
            }
          }
        }
        if (!__any_sync(0xffffffffu, near)) {
          if (code == 0) nib[0] = nib[1] = 0u;
        } else {
          float t[7];
          e2m1_thresholds(s, t);
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            uint32_t n = 0u;
#pragma unroll
            for (int e = 0; e < 8; ++e) n |= e2m1_nibble(xs[8 * w + e], t) << (4 * e);
            nib[w] = code != 0 ? n : 0u;
          }
        }
        if (row_ok && kk < k)
          *reinterpret_cast<uint2*>(q + (row_g * k + kk) / 2) = make_uint2(nib[0], nib[1]);
        // block 4w + i of the unit is held by lane 4w + i; scale word w gathers lanes 4w .. 4w + 3
        const uint32_t c1 = __shfl_down_sync(0xffffffffu, code, 1);
        const uint32_t c2 = __shfl_down_sync(0xffffffffu, code, 2);
        const uint32_t c3 = __shfl_down_sync(0xffffffffu, code, 3);
        if ((lane & 3) == 0) {
          const int64_t kb = static_cast<int64_t>(kc) * 32 + lane;
          if ((kb >> 2) < kt_n) {
            const uint64_t off = sf_offset(r, kb, l, mt_n, kt_n);
            *reinterpret_cast<uint32_t*>(sf + off) = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_quantize(int fmt, const void* x, bool x_bf16, int64_t batch, int64_t rows, int64_t k, uint8_t* q,
                            uint8_t* sf, int num_sms, cudaStream_t stream) {
  const int v = fmt == kMXFP8 ? 32 : 16;
  const int64_t mt_n = (rows + 127) / 128;
  const int64_t kt_n = (k / v + 3) / 4;
  const int64_t rows_padded = mt_n * 128;
  const int units_per_row = static_cast<int>((k + 1023) / 1024);  // bf16 MXFP8 units
  const int64_t total_rows = batch * rows_padded;
  int64_t blocks = (total_rows + (kThreads / 32) - 1) / (kThreads / 32);
  // up to 16 blocks per SM (more than are resident): with fewer rows per warp the block scheduler
  // evens out the load (measured 3-4 % faster than 8 on 4 x 8192 rows; 32 gained no more)
  const int64_t max_blocks = static_cast<int64_t>(num_sms) * 16;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  const unsigned grid = static_cast<unsigned>(blocks);
  const int units_nvfp4 = static_cast<int>((k + 511) / 512);
  const float* xf = static_cast<const float*>(x);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (fmt == kMXFP8 && !x_bf16) {
    quantize_mxfp8_kernel<<<grid, kThreads, 0, stream>>>(xf, rows, static_cast<int>(k), q, sf, rows_padded,
                                                         static_cast<int>((k + 127) / 128), total_rows, mt_n, kt_n);
  } else if (fmt == kMXFP8) {
    quantize_mxfp8_bf16_kernel<<<grid, kThreads, 0, stream>>>(xb, rows, static_cast<int>(k), q, sf, rows_padded,
                                                              units_per_row, total_rows, mt_n, kt_n);
  } else if (!x_bf16) {
    quantize_nvfp4_kernel<<<grid, kThreads, 0, stream>>>(xf, rows, static_cast<int>(k), q, sf, rows_padded,
                                                         units_nvfp4, total_rows, mt_n, kt_n);
  } else {
    quantize_nvfp4_kernel<<<grid, kThreads, 0, stream>>>(xb, rows, static_cast<int>(k), q, sf, rows_padded,
                                                         units_nvfp4, total_rows, mt_n, kt_n);
  }
  return cudaGetLastError();
}

}  // namespace bsg
