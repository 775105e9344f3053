// quantize.cu -- fp32 -> MXFP8 / NVFP4 block quantiser (memory-bound).
//
// Each warp step handles one "unit": 128 consecutive fp32 values of one row (512 bytes,
// one float4 per lane, fully coalesced).  For MXFP8 a unit is 4 blocks of 32 (8 lanes per
// block), for NVFP4 8 blocks of 16 (4 lanes per block).  Block maxima are reduced with
// warp shuffles, the scale bytes of 4 consecutive blocks are adjacent in the atom layout
// and leave as one 32-bit store, the codes as one 32-bit (E4M3) or 16-bit (E2M1) store
// per lane.  Units of the padding rows of the last 128-row atom produce zero scale bytes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace bsg {
namespace {

constexpr int kUnroll = 4;
constexpr int kThreads = 256;

// RNE_UE4M3(a / 6) decided exactly: candidate from the rounded fp32 quotient, then moved
// by at most one code after comparing a with 6 * (neighbouring midpoints), products that
// are exact in fp32 (a midpoint has at most 5 significant bits).  Saturates at 448.
__device__ __forceinline__ uint32_t ue4m3_code_of_amax_over_6(float a) {
  if (!(a > 0.0f)) return 0;
  const float q = __fdiv_rn(a, 6.0f);
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

// E2M1 nibble of RNE_satfinite(x / s) from exact thresholds t[i] = midpoint_i * s: the
// magnitude index counts the midpoints below |x|; at a midpoint the even index wins, i.e.
// midpoints 1, 3, 5 (0.75, 1.75, 3.5) count when equal as well.  The sign bit is the sign
// of x (a negative value that rounds to zero gives -0), as the E4M3 conversion does.
__device__ __forceinline__ uint32_t e2m1_nibble(float x, const float (&t)[7]) {
  const float a = fabsf(x);
  uint32_t idx = (a > t[0]) + (a >= t[1]) + (a > t[2]) + (a >= t[3]) + (a > t[4]) + (a >= t[5]) + (a > t[6]);
  return idx | ((__float_as_uint(x) >> 28) & 8u);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const float* __restrict__ x, int64_t rows, int64_t k,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                            int64_t rows_padded, int64_t units_per_row,
                                                            int64_t total_units, int64_t mt_n, int64_t kt_n) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t num_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;

  for (int64_t u0 = warp_id * kUnroll; u0 < total_units; u0 += num_warps * kUnroll) {
    float4 v[kUnroll];
    int64_t row_g[kUnroll], r_[kUnroll], l_[kUnroll], kc_[kUnroll];
    bool row_ok[kUnroll], elem_ok[kUnroll], unit_ok[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int64_t u = u0 + j;
      unit_ok[j] = u < total_units;
      const int64_t kc = u % units_per_row;
      const int64_t rg = u / units_per_row;  // row index over batch * rows_padded
      const int64_t l = rg / rows_padded, r = rg % rows_padded;
      kc_[j] = kc;
      r_[j] = r;
      l_[j] = l;
      row_g[j] = l * rows + r;
      const int64_t kk = kc * 128 + lane * 4;
      row_ok[j] = unit_ok[j] && r < rows;
      elem_ok[j] = row_ok[j] && kk < k;
      v[j] = elem_ok[j] ? __ldcs(reinterpret_cast<const float4*>(x + row_g[j] * k + kk))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      if (!unit_ok[j]) continue;  // uniform across the warp
      const int64_t kk = kc_[j] * 128 + lane * 4;
      float a = fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w)));
      if (FMT == kMXFP8) {
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        const uint32_t code = e8m0_ceil_code(a);
        const float inv = e8m0_inv_scale(code);
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(v[j].x, inv), __fmul_rn(v[j].y, inv));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(v[j].z, inv), __fmul_rn(v[j].w, inv));
        if (elem_ok[j]) *reinterpret_cast<uint32_t*>(q + row_g[j] * k + kk) = lo | (hi << 16);
        const uint32_t c1 = __shfl_sync(0xffffffffu, code, 8);
        const uint32_t c2 = __shfl_sync(0xffffffffu, code, 16);
        const uint32_t c3 = __shfl_sync(0xffffffffu, code, 24);
        if (lane == 0) {
          const uint64_t off = sf_offset(r_[j], kc_[j] * 4, l_[j], mt_n, kt_n);
          *reinterpret_cast<uint32_t*>(sf + off) = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
        }
      } else {
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const uint32_t code = ue4m3_code_of_amax_over_6(a);
        const float s = ue4m3_value(code);
        const float t[7] = {0.25f * s, 0.75f * s, 1.25f * s, 1.75f * s, 2.5f * s, 3.5f * s, 5.0f * s};
        uint32_t nib = 0;
        if (code != 0) {
          nib = e2m1_nibble(v[j].x, t) | (e2m1_nibble(v[j].y, t) << 4) | (e2m1_nibble(v[j].z, t) << 8) |
                (e2m1_nibble(v[j].w, t) << 12);
        }
        if (elem_ok[j]) *reinterpret_cast<uint16_t*>(q + (row_g[j] * k + kk) / 2) = static_cast<uint16_t>(nib);
        // scale bytes: blocks 0-3 from lanes 0, 4, 8, 12 and blocks 4-7 from lanes 16, 20, 24, 28
        const uint32_t c1 = __shfl_down_sync(0xffffffffu, code, 4);
        const uint32_t c2 = __shfl_down_sync(0xffffffffu, code, 8);
        const uint32_t c3 = __shfl_down_sync(0xffffffffu, code, 12);
        if ((lane & 15) == 0) {
          const int64_t kb = kc_[j] * 8 + (lane >> 2);
          if ((kb >> 2) < kt_n) {
            const uint64_t off = sf_offset(r_[j], kb, l_[j], mt_n, kt_n);
            *reinterpret_cast<uint32_t*>(sf + off) = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
          }
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_quantize(int fmt, const float* x, int64_t batch, int64_t rows, int64_t k, uint8_t* q,
                            uint8_t* sf, int num_sms, cudaStream_t stream) {
  const int v = fmt == kMXFP8 ? 32 : 16;
  const int64_t mt_n = (rows + 127) / 128;
  const int64_t kt_n = (k / v + 3) / 4;
  const int64_t rows_padded = mt_n * 128;
  const int64_t units_per_row = (k + 127) / 128;
  const int64_t total_units = batch * rows_padded * units_per_row;
  const int64_t warps_needed = (total_units + kUnroll - 1) / kUnroll;
  int64_t blocks = (warps_needed + (kThreads / 32) - 1) / (kThreads / 32);
  const int64_t max_blocks = static_cast<int64_t>(num_sms) * 8;
  if (blocks > max_blocks) blocks = max_blocks;
  if (blocks < 1) blocks = 1;
  if (fmt == kMXFP8) {
    quantize_kernel<kMXFP8><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        x, rows, k, q, sf, rows_padded, units_per_row, total_units, mt_n, kt_n);
  } else {
    quantize_kernel<kNVFP4><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        x, rows, k, q, sf, rows_padded, units_per_row, total_units, mt_n, kt_n);
  }
  return cudaGetLastError();
}

}  // namespace bsg
