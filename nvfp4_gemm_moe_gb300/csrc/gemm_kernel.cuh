// gemm_kernel.cuh -- persistent, warp-specialised block-scaled GEMM for sm_103a.
//
// One CTA per SM walks a static list of 128 x BN output tiles (dense and RoPE projection:
// batch-major, then groups of 16 M-tiles swept along N; grouped: M-tile-major over the
// experts' padded row ranges).  Fourteen warps:
//   warp 0     TMA producer: per 128-byte K slice, A (128 rows) and B (BN rows) tiles with
//              128-byte swizzle via cp.async.bulk.tensor, and the scale-factor atoms via
//              cp.async.bulk, into a STAGES-deep shared-memory ring (full/empty mbarriers); with
//              per-expert weights, expert g's B tensor map is read from global memory;
//   warp 1     TMEM owner and MMA issuer: the warp issues the stage's four block-scaled
//              tcgen05.mma (kind::mxf8f6f4 scale_vec::1X for MXFP8, kind::mxf4nvf4 scale_vec::4X
//              for NVFP4) into an fp32 accumulator in TMEM, then tcgen05.commit frees the stage
//              (one lane per instruction, chosen by elect.sync, with no branch around the issue);
//   warps 2-9  epilogue: two warps per 32-lane quadrant of TMEM (= 32 rows of the tile), each
//              taking its share of the 32-column chunks, read with tcgen05.ld, and applying the
//              dense (C + amax), grouped sReLU (alpha, C, sReLU / tanh clamp, D, per-expert amax
//              or MXFP8 row and column re-quantisation), grouped dSwiGLU backward (C input,
//              ab / dswiglu, dprob) or RoPE projection (rotation, row and column MXFP8)
//              epilogue; rows leave (and the dSwiGLU C rows arrive) through a per-warp shared-
//              memory transpose block as coalesced whole-sector accesses;
//   warps 10-13 scale-factor stagers: each warp writes its 32-lane quadrant of the stage's
//              scale factors from shared memory into TMEM with tcgen05.st, in the layout a
//              tcgen05.cp 32x128b.warpx4 of each atom would produce.  tcgen05.cp runs in the
//              tensor pipe, serialised with the MMAs (about 40 cycles per 2 KB atom copy, i.e.
//              up to twelve copies per four MMAs for NVFP4); the stores run beside it.
// Tiles are 128 x BN with BN in {128, 192, 224, 256}; below 256 two accumulator buffers (ACC)
// let the epilogue of one tile overlap the MMAs of the next.
// Every wait is bounded: a wait longer than kWaitLimitNs records a device error, the CTA
// drains its own in-flight copies and MMAs, frees TMEM and exits.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace bsg {

constexpr int kThreadsGemm = 448;  // producer, MMA issuer, eight epilogue and four scale-factor warps
constexpr int kTileM = 128;
constexpr int kTileKBytes = 128;  // one 128-byte swizzle row of K per stage
constexpr int kXposeBlockBytes = 32 * 64;  // a warp's 32 rows x 64 bytes transpose block

template <int FMT, int BN, int EPI = kEpiDense>
struct GemmTraits {
  // elements per 128-byte K slice and per tcgen05.mma (32 bytes of K)
  static constexpr int kElemsPerKTile = FMT == kMXFP8 ? 128 : FMT == kNVFP4 ? 256 : 64;
  static constexpr int kMmaK = FMT == kMXFP8 ? 32 : FMT == kNVFP4 ? 64 : 16;
  static constexpr int kMmasPerStage = 4;
  // SF atoms (128 rows x 4 blocks) along K per stage; bf16 operands carry none
  static constexpr int kAtomsPerStage = FMT == kMXFP8 ? 1 : FMT == kNVFP4 ? 4 : 0;
  static_assert(BN % 32 == 0 && BN >= 128 && BN <= 256, "tile width");
  static_assert(BN % 128 == 0 || FMT != kNVFP4, "NVFP4 tiles are 128 or 256 wide");
  // A tile of B rows starting at a multiple of BN: aligned to the 128-row scale-factor atoms
  // when BN is a multiple of 128, else it may start inside an atom and touch three of them.
  static constexpr bool kSfbAligned = BN % 128 == 0;
  static constexpr int kBRowGroups = kSfbAligned ? BN / 128 : 3;  // SFB atom groups loaded per stage
  static constexpr int kBBlocks = BN / 32;                         // 32-row blocks of the tile
  static constexpr int kABytes = kTileM * kTileKBytes;
  static constexpr int kBBytes = BN * kTileKBytes;
  static constexpr int kSfaBytes = kAtomsPerStage * 512;
  static constexpr int kSfbBytes = kBRowGroups * kAtomsPerStage * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kAcc = (BN == 256) ? 1 : 2;
  static constexpr int kSfaCols = kAtomsPerStage * 4;
  // SFB columns per MMA: column n / 32 of a unit holds the scales of tile rows n (TMEM lane n % 32
  // of every quadrant), padded to whole four-column groups
  static constexpr int kSfbColsPerMma = ((kBBlocks + 3) / 4) * 4;
  static constexpr int kSfbCols = kSfbColsPerMma * kAtomsPerStage;
  static constexpr int kSfStride = kAtomsPerStage == 0 ? 0 : ((kSfaCols + kSfbCols + 15) / 16) * 16;
  static constexpr int kSfBase = kAcc * BN;
  // barrier / scalar area after the stages
  static constexpr int kBarBytes = 1024;
  // padded_offsets of up to 1024 experts (grouped only)
  static constexpr int kOffsetsBytes = epi_is_grouped(EPI) ? 4096 : 0;
  // per-expert amax staging (grouped), the dense amax, or the warps' 32-float scale exchange
  static constexpr int kAmaxBytes = epi_is_grouped(EPI) ? 4096 : 1024;
  // one transpose block per epilogue warp: 32 rows x 64 bytes (grouped), 32 x 32 bytes (RoPE)
  static constexpr int kXposeBlock = EPI == kEpiRope ? 1024 : kXposeBlockBytes;
  static constexpr int kXposeBytes = 8 * kXposeBlock;
  // shared-memory ring: as many stages as fit, at most six
  static constexpr int kStagesSmem =
      (232448 - 1024 - kBarBytes - kOffsetsBytes - kAmaxBytes - kXposeBytes) / kStageBytes;
  static constexpr int kStages = kStagesSmem < 6 ? kStagesSmem : 6;
  static_assert(kStages >= 3, "pipeline depth");
  // TMEM scale-factor slots: one per stage when TMEM has room, else fewer, recycled through the
  // sf_free barriers
  static constexpr int kSfSlotsTmem = kSfStride == 0 ? kStages : (512 - kSfBase) / kSfStride;
  static constexpr int kSfSlots = kSfSlotsTmem < kStages ? kSfSlotsTmem : kStages;
  static constexpr bool kSfRing = kSfSlots < kStages;
  static_assert(kSfSlots >= 3, "TMEM scale-factor slots");
  static constexpr int kTmemUsed = kSfBase + kSfSlots * kSfStride;
  static constexpr int kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                   : kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + kBarBytes +
                                    kOffsetsBytes + kAmaxBytes + kXposeBytes;
  static_assert(kSmemBytes <= 232448, "shared memory budget");

  // Instruction descriptor: A/B formats (bits 7-12), K-major A and B, N >> 3 (bits 17-22),
  // scale format (bit 23: 1 = UE8M0, 0 = UE4M3), M >> 4 (bits 24-28).  kind::f16 (bf16): fp32
  // accumulator (bits 4-5 = 1), A and B both bf16 (1 at bits 7 and 10), no scale field.
  static constexpr uint32_t kIdesc = (FMT == kMXFP8   ? ((0u << 7) | (0u << 10) | (1u << 23))
                                      : FMT == kNVFP4 ? ((1u << 7) | (1u << 10) | (0u << 23))
                                                      : ((1u << 4) | (1u << 7) | (1u << 10))) |
                                     (static_cast<uint32_t>(BN >> 3) << 17) |
                                     (static_cast<uint32_t>(kTileM >> 4) << 24);
};

struct TileCoord {
  int l;   // batch (dense) or expert (grouped)
  int mt;  // 128-row tile index
  int nt;  // BN-column tile index
};

__device__ __forceinline__ int find_expert(const int32_t* offs, int num_experts, int row) {
  int lo = 0, hi = num_experts - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (offs[mid] > row) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Tile t -> (batch or expert, M tile of TM rows, N tile).  Dense: batch-major, then groups of GM
// M tiles swept along N (neighbouring CTAs share A and B in L2); grouped: M-tile-major.
template <int EPI, int TM = kTileM, int GM = 16>
__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, int t, const int32_t* offs) {
  TileCoord tc;
  if (!epi_is_grouped(EPI)) {
    const int per_batch = p.m_tiles * p.n_tiles;
    tc.l = t / per_batch;
    const int idx = t - tc.l * per_batch;
    constexpr int kGroupM = GM;
    const int group = idx / (kGroupM * p.n_tiles);
    const int first_m = group * kGroupM;
    const int gm = min(kGroupM, p.m_tiles - first_m);
    const int loc = idx - group * kGroupM * p.n_tiles;
    tc.mt = first_m + loc % gm;
    tc.nt = loc / gm;
  } else {
    tc.mt = t / p.n_tiles;
    tc.nt = t - tc.mt * p.n_tiles;
    tc.l = find_expert(offs, p.l, tc.mt * TM);
  }
  return tc;
}

__device__ __forceinline__ void store16(void* dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(dst) = make_uint4(a, b, c, d);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Stores the 32 fp32 values v of one row chunk as `kind` at element `off` of `base` (row-major,
// N columns, chunk starting at column col0), in 16-byte granules; a granule is written when its
// first column is below N (N is a multiple of the granule width for every kind the host allows).
__device__ __forceinline__ void store_row32(void* base, uint64_t off, int kind, const float (&v)[32], int col0, int n) {
  if (kind == kOutF32) {
    float* dst = reinterpret_cast<float*>(base) + off;
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      if (col0 + j < n)
        store16(dst + j, __float_as_uint(v[j]), __float_as_uint(v[j + 1]), __float_as_uint(v[j + 2]),
                __float_as_uint(v[j + 3]));
  } else if (kind == kOutBF16 || kind == kOutF16) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(base) + off;
    const bool bf = kind == kOutBF16;
#pragma unroll
    for (int j = 0; j < 32; j += 8)
      if (col0 + j < n)
        store16(dst + j, bf ? pack_bf16x2(v[j], v[j + 1]) : pack_f16x2(v[j], v[j + 1]),
                bf ? pack_bf16x2(v[j + 2], v[j + 3]) : pack_f16x2(v[j + 2], v[j + 3]),
                bf ? pack_bf16x2(v[j + 4], v[j + 5]) : pack_f16x2(v[j + 4], v[j + 5]),
                bf ? pack_bf16x2(v[j + 6], v[j + 7]) : pack_f16x2(v[j + 6], v[j + 7]));
  } else if (kind == kOutE4M3) {
    uint8_t* dst = reinterpret_cast<uint8_t*>(base) + off;
    uint32_t q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      q[j] = cvt_e4m3x2(v[4 * j], v[4 * j + 1]) | (static_cast<uint32_t>(cvt_e4m3x2(v[4 * j + 2], v[4 * j + 3])) << 16);
    if (col0 < n) store16(dst, q[0], q[1], q[2], q[3]);
    if (col0 + 16 < n) store16(dst + 16, q[4], q[5], q[6], q[7]);
  } else if (kind == kOutE2M1) {
    uint8_t* dst = reinterpret_cast<uint8_t*>(base) + off / 2;
    uint32_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      q[j] = cvt_e2m1x2(v[8 * j], v[8 * j + 1]) | (cvt_e2m1x2(v[8 * j + 2], v[8 * j + 3]) << 8) |
             (cvt_e2m1x2(v[8 * j + 4], v[8 * j + 5]) << 16) | (cvt_e2m1x2(v[8 * j + 6], v[8 * j + 7]) << 24);
    if (col0 < n) store16(dst, q[0], q[1], q[2], q[3]);
  }
}

// Byte offset of 16-byte unit `unit` (0..3) of row `row` (0..31) in a warp's 32 x 64-byte
// transpose block.  The unit index is XORed with (row / 2) % 4, so that eight threads writing
// unit u of eight consecutive rows, and eight threads reading the four units of two consecutive
// rows, each touch eight distinct 16-byte bank groups (no bank conflicts either way).
__device__ __forceinline__ uint32_t xpose_off(int row, int unit) {
  return static_cast<uint32_t>(row * 64 + ((unit ^ ((row >> 1) & 3)) << 4));
}

// Stores 64 bytes per row for the warp's 32 rows row0 .. row0 + 31 (this thread's row holds the
// four 16-byte units u): row r goes to base + (row0 + r) * pitch + col_byte.  The rows pass
// through the warp's transpose block, so each global store instruction writes 8 rows x 64
// contiguous bytes (whole sectors) instead of 32 rows x 16 bytes.  Units at or past byte
// `limit_byte` of a row, and rows at or past row_end, are not written.
__device__ __forceinline__ void store_rows64(uint8_t* s_blk, void* base, uint64_t pitch, int row0, int col_byte,
                                             int limit_byte, const uint4 (&u)[4], int lane, int row_end = 1 << 30) {
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(s_blk + xpose_off(lane, j)) = u[j];
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2), j = lane & 3;
    const uint4 v = *reinterpret_cast<const uint4*>(s_blk + xpose_off(r, j));
    if (col_byte + j * 16 < limit_byte && row0 + r < row_end)
      *reinterpret_cast<uint4*>(static_cast<char*>(base) + static_cast<uint64_t>(row0 + r) * pitch + col_byte +
                                j * 16) = v;
  }
  __syncwarp();
}

// As store_rows64 for 32 bytes per row (two 16-byte units, E4M3 blocks): the unit index is
// XORed with (row / 4) % 2, and each global store instruction writes 16 rows x 32 bytes.
__device__ __forceinline__ uint32_t xpose32_off(int row, int unit) {
  return static_cast<uint32_t>(row * 32 + ((unit ^ ((row >> 2) & 1)) << 4));
}

__device__ __forceinline__ void store_rows32(uint8_t* s_blk, void* base, uint64_t pitch, int row0, int col_byte,
                                             const uint4& u0, const uint4& u1, int lane) {
  *reinterpret_cast<uint4*>(s_blk + xpose32_off(lane, 0)) = u0;
  *reinterpret_cast<uint4*>(s_blk + xpose32_off(lane, 1)) = u1;
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int r = it * 16 + (lane >> 1), j = lane & 1;
    const uint4 v = *reinterpret_cast<const uint4*>(s_blk + xpose32_off(r, j));
    *reinterpret_cast<uint4*>(static_cast<char*>(base) + static_cast<uint64_t>(row0 + r) * pitch + col_byte + j * 16) = v;
  }
  __syncwarp();
}

// The inverse, in two steps: fetch_rows64 loads 64 bytes per row of the warp's 32 rows
// (streaming loads, whole sectors per instruction) into v; xpose_rows64 passes them through the
// transpose block and returns this thread's row as four 16-byte units.  Several fetches may be
// in flight before their transposes.
__device__ __forceinline__ void fetch_rows64(const void* base, uint64_t pitch, int row0, int col_byte, uint4 (&v)[4],
                                             int lane) {
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2), j = lane & 3;
    v[it] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const char*>(base) +
                                                  static_cast<uint64_t>(row0 + r) * pitch + col_byte + j * 16));
  }
}

__device__ __forceinline__ void xpose_rows64(uint8_t* s_blk, const uint4 (&v)[4], uint4 (&u)[4], int lane) {
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = it * 8 + (lane >> 2), j = lane & 3;
    *reinterpret_cast<uint4*>(s_blk + xpose_off(r, j)) = v[it];
  }
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) u[j] = *reinterpret_cast<const uint4*>(s_blk + xpose_off(lane, j));
  __syncwarp();
}

// Stores this thread's 32 fp32 values v (one row chunk) as f32 / bf16 / f16 at element column
// col0 of the warp's rows row0 .. row0 + 31 of a row-major array of `ld` elements per row and
// `n` valid columns (rows at or past row_end are not written), through the transpose block (see
// store_rows64).
__device__ __forceinline__ void store_block_coalesced(uint8_t* s_blk, void* base, int kind, int ld, int n, int row0,
                                                      int col0, const float (&v)[32], int lane,
                                                      int row_end = 1 << 30) {
  if (kind == kOutF32) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 u[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        u[j] = make_uint4(__float_as_uint(v[16 * h + 4 * j]), __float_as_uint(v[16 * h + 4 * j + 1]),
                          __float_as_uint(v[16 * h + 4 * j + 2]), __float_as_uint(v[16 * h + 4 * j + 3]));
      store_rows64(s_blk, base, static_cast<uint64_t>(ld) * 4, row0, (col0 + 16 * h) * 4, n * 4, u, lane, row_end);
    }
  } else {
    const bool bf = kind == kOutBF16;
    uint4 u[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* w = v + 8 * j;
      u[j] = bf ? make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]),
                             pack_bf16x2(w[6], w[7]))
                : make_uint4(pack_f16x2(w[0], w[1]), pack_f16x2(w[2], w[3]), pack_f16x2(w[4], w[5]),
                             pack_f16x2(w[6], w[7]));
    }
    store_rows64(s_blk, base, static_cast<uint64_t>(ld) * 2, row0, col0 * 2, n * 2, u, lane, row_end);
  }
}

__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v) {
  atomicMax(reinterpret_cast<int*>(addr), __float_as_int(v));
}

// sReLU with optional tanh soft clamp: s * min(tanh(relu(c) / s), 1) (or relu(c)), squared, times
// prob.  relu(c) / s is taken as relu(c) * (1/s): within an ulp of the quotient (exact for a
// power-of-two s), far inside the output tolerances.
__device__ __forceinline__ float srelu_clamp(float c, float prob, float s, float inv_s, int tanh_approx) {
  float r = fmaxf(c, 0.0f);
  if (s > 0.0f) {
    const float u = r * inv_s;
    float t;
    if (tanh_approx) {
      asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(u));
    } else {
      t = tanhf(u);
    }
    r = s * fminf(t, 1.0f);
  }
  return prob * (r * r);
}

// Butterfly reduce-scatter of 32 values across the warp: afterwards v[0] of lane i holds the
// maximum over all 32 lanes of the original v[i].
__device__ __forceinline__ void warp_colmax_scatter(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int j = 0; j < w; ++j) {
      const float send = upper ? v[j] : v[j + w];
      const float keep = upper ? v[j + w] : v[j];
      const float recv = __shfl_xor_sync(0xffffffffu, send, w);
      v[j] = fmaxf(keep, recv);
    }
  }
}

// Dense epilogue with bf16 C that gives the accumulator back early: this warp's chunks
// (c_first, c_first + 2, ...) are read from TMEM, folded into the running |max| and packed to
// bf16 in registers; then `release` (the accumulator-empty arrival) runs, and only then are the
// packed rows stored, overlapping the next tile's MMAs.  With kXpose the rows are stored
// through the warp's transpose block s_blk (coalesced, whole sectors), else one row per thread.
template <int BN, bool kXpose, class Release>
__device__ __forceinline__ void epilogue_dense_bf16_early(const GemmParams& p, int l, int row, int col_base,
                                                          uint32_t tmem_acc, int c_first, float& run_max,
                                                          Release release, uint8_t* s_blk, int lane) {
  constexpr int kChunks = (BN / 32 + 1) / 2;  // this warp's chunks (alternate 32-column chunks)
  uint32_t pk[kChunks][16];
#pragma unroll
  for (int ci = 0; ci < kChunks; ++ci) {
    const int c = c_first + 2 * ci;
    if (c < BN / 32 && col_base + c * 32 < p.n) {  // warp-uniform
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem_acc + c * 32, r);
      tmem_ld_wait(r);
#pragma unroll
      for (int j = 0; j < 32; ++j) run_max = fmaxf(run_max, fabsf(__uint_as_float(r[j])));
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[ci][j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    }
  }
  release();
  if constexpr (kXpose) {
    __nv_bfloat16* batch = reinterpret_cast<__nv_bfloat16*>(p.c) + static_cast<uint64_t>(l) * p.m * p.n;
#pragma unroll
    for (int ci = 0; ci < kChunks; ++ci) {
      const int c = c_first + 2 * ci;
      const int col0 = col_base + c * 32;
      if (c < BN / 32 && col0 < p.n) {  // warp-uniform
        const uint4 u[4] = {make_uint4(pk[ci][0], pk[ci][1], pk[ci][2], pk[ci][3]),
                            make_uint4(pk[ci][4], pk[ci][5], pk[ci][6], pk[ci][7]),
                            make_uint4(pk[ci][8], pk[ci][9], pk[ci][10], pk[ci][11]),
                            make_uint4(pk[ci][12], pk[ci][13], pk[ci][14], pk[ci][15])};
        store_rows64(s_blk, batch, static_cast<uint64_t>(p.n) * 2, row - lane, col0 * 2, p.n * 2, u, lane, p.m);
      }
    }
  } else {
    if (row >= p.m) return;
    __nv_bfloat16* rowp = reinterpret_cast<__nv_bfloat16*>(p.c) + (static_cast<uint64_t>(l) * p.m + row) *
                                                                       static_cast<uint64_t>(p.n);
#pragma unroll
    for (int ci = 0; ci < kChunks; ++ci) {
      const int c = c_first + 2 * ci;
      const int col0 = col_base + c * 32;
      if (c < BN / 32 && col0 < p.n) {
#pragma unroll
        for (int j = 0; j < 32; j += 8)
          if (col0 + j < p.n)
            store16(rowp + col0 + j, pk[ci][j / 2], pk[ci][j / 2 + 1], pk[ci][j / 2 + 2], pk[ci][j / 2 + 3]);
      }
    }
  }
}

// Row- and column-quantised E4M3 store of one 32-column block of D: row `row`, D columns
// dcol0 .. dcol0 + 31 of a row-major D that is n_d wide (n_d a multiple of 32), values already
// multiplied by norm_const.  D_row takes one E8M0 scale per row and block (this thread's 32
// values), D_col one per column and 32-row block (the warp's 32 lanes are 32 consecutive rows).
// s_inv: 32 floats of shared memory owned by this warp; s_blk: the warp's transpose block (the
// code rows are stored coalesced through it).
// With kPlainScales the scales go to plain row-major arrays instead of the atom layout:
// sfd_row[row * (n_d / 32) + dcol0 / 32] and sfd_col[(row / 32) * n_d + dcol0 + lane].
template <bool kPlainScales = false>
__device__ __forceinline__ void store_e4m3_block(const GemmParams& p, int row, int dcol0, int n_d, const float (&d)[32],
                                                 int lane, float* s_inv, uint8_t* s_blk) {
  const int row0 = row - lane;
  float bmax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) bmax = fmaxf(bmax, fabsf(d[j]));
  const uint32_t code_r = e8m0_ceil_code(bmax);
  const float inv_r = e8m0_inv_scale(code_r);
  uint32_t q[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t lo = cvt_e4m3x2(__fmul_rn(d[4 * j], inv_r), __fmul_rn(d[4 * j + 1], inv_r));
    const uint32_t hi = cvt_e4m3x2(__fmul_rn(d[4 * j + 2], inv_r), __fmul_rn(d[4 * j + 3], inv_r));
    q[j] = lo | (hi << 16);
  }
  if (p.d_v8)  // this thread's 32 codes are one whole sector of its row
    st_global_v8(static_cast<uint8_t*>(p.d) + static_cast<uint64_t>(row) * n_d + dcol0, q);
  else
    store_rows32(s_blk, p.d, static_cast<uint64_t>(n_d), row0, dcol0, make_uint4(q[0], q[1], q[2], q[3]),
                 make_uint4(q[4], q[5], q[6], q[7]), lane);
  // one byte per block: a tile need not start on a four-block word of the SF layout; the row's
  // last block also zeroes the padding blocks of its word
  if constexpr (kPlainScales) {
    p.sfd_row[static_cast<uint64_t>(row) * (n_d >> 5) + (dcol0 >> 5)] = static_cast<uint8_t>(code_r);
  } else {
    const int nb = dcol0 >> 5;
    const int nb_end = dcol0 + 32 >= n_d ? (nb | 3) : nb;
    for (int b = nb; b <= nb_end; ++b)
      p.sfd_row[sf_offset(row, b, 0, (p.m + 127) / 128, p.sfd_row_kt)] = static_cast<uint8_t>(b == nb ? code_r : 0u);
  }
  float cm[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) cm[j] = fabsf(d[j]);
  warp_colmax_scatter(cm, lane);
  const uint32_t code_c = e8m0_ceil_code(cm[0]);
  const int mblk = row >> 5;  // same for the whole warp
  if constexpr (kPlainScales)
    p.sfd_col[static_cast<uint64_t>(mblk) * n_d + dcol0 + lane] = static_cast<uint8_t>(code_c);
  else
    p.sfd_col[sf_offset(dcol0 + lane, mblk, 0, p.sfd_col_mt, p.sfd_col_kt)] = static_cast<uint8_t>(code_c);
  // every lane needs the 32 column reciprocals: one shared-memory round trip (broadcast reads)
  // instead of 32 shuffles
  s_inv[lane] = e8m0_inv_scale(code_c);
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 iv = reinterpret_cast<const float4*>(s_inv)[j];
    const uint32_t lo = cvt_e4m3x2(__fmul_rn(d[4 * j], iv.x), __fmul_rn(d[4 * j + 1], iv.y));
    const uint32_t hi = cvt_e4m3x2(__fmul_rn(d[4 * j + 2], iv.z), __fmul_rn(d[4 * j + 3], iv.w));
    q[j] = lo | (hi << 16);
  }
  __syncwarp();  // the next block overwrites s_inv
  if (p.d_v8)
    st_global_v8(static_cast<uint8_t*>(p.d_col) + static_cast<uint64_t>(row) * n_d + dcol0, q);
  else
    store_rows32(s_blk, p.d_col, static_cast<uint64_t>(n_d), row0, dcol0, make_uint4(q[0], q[1], q[2], q[3]),
                 make_uint4(q[4], q[5], q[6], q[7]), lane);
}

// Decodes 16-byte units of `kind` (bf16, f16, f32 or E4M3 values) into fp32 v[first ..].
__device__ __forceinline__ void decode_units(int kind, const uint4 (&u)[4], float* v) {
  if (kind == kOutF32) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[4 * j] = __uint_as_float(u[j].x);
      v[4 * j + 1] = __uint_as_float(u[j].y);
      v[4 * j + 2] = __uint_as_float(u[j].z);
      v[4 * j + 3] = __uint_as_float(u[j].w);
    }
  } else if (kind == kOutE4M3) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 lo = e4m3x2_to_float2(static_cast<uint16_t>(w[i] & 0xffffu));
        const float2 hi = e4m3x2_to_float2(static_cast<uint16_t>(w[i] >> 16));
        v[16 * j + 4 * i] = lo.x;
        v[16 * j + 4 * i + 1] = lo.y;
        v[16 * j + 4 * i + 2] = hi.x;
        v[16 * j + 4 * i + 3] = hi.y;
      }
    }
  } else {
    const bool bf = kind == kOutBF16;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (bf) {
          v[8 * j + 2 * i] = __uint_as_float(w[i] << 16);
          v[8 * j + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        } else {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
          v[8 * j + 2 * i] = f.x;
          v[8 * j + 2 * i + 1] = f.y;
        }
      }
    }
  }
}

// Loads the input block x and the gate block g (32 values each, this thread's row) of ref
// columns col0 .. col0 + 31 from C (valid_m, 2N) for the warp's rows row0 .. row0 + 31: the
// 64 * element-size contiguous bytes of each row in 64-byte pieces, fetched coalesced and
// transposed through the warp's block (see fetch_rows64 / xpose_rows64).
__device__ __forceinline__ void load_dswiglu_c(uint8_t* s_blk, const GemmParams& p, int row0, int col0,
                                               float (&x)[32], float (&g)[32], int lane) {
  const int kind = p.c_in_kind;
  uint4 v0[4], v1[4], u[4];
  if (kind == kOutE4M3) {  // one piece: 32 input codes then 32 gate codes
    fetch_rows64(p.c_in, static_cast<uint64_t>(2 * p.n), row0, 2 * col0, v0, lane);
    xpose_rows64(s_blk, v0, u, lane);
    float t[64];
    decode_units(kind, u, t);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      x[j] = t[j];
      g[j] = t[32 + j];
    }
  } else if (kind == kOutF32) {  // four pieces of 16 values: x low, x high, g low, g high
    const uint64_t pitch = static_cast<uint64_t>(2 * p.n) * 4;
    const int b0 = 2 * col0 * 4;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float* dst = h == 0 ? x : g;
      fetch_rows64(p.c_in, pitch, row0, b0 + 128 * h, v0, lane);
      fetch_rows64(p.c_in, pitch, row0, b0 + 128 * h + 64, v1, lane);
      xpose_rows64(s_blk, v0, u, lane);
      decode_units(kind, u, dst);
      xpose_rows64(s_blk, v1, u, lane);
      decode_units(kind, u, dst + 16);
    }
  } else {  // 16-bit: two pieces, the input block and the gate block
    const uint64_t pitch = static_cast<uint64_t>(2 * p.n) * 2;
    fetch_rows64(p.c_in, pitch, row0, 4 * col0, v0, lane);
    fetch_rows64(p.c_in, pitch, row0, 4 * col0 + 64, v1, lane);
    xpose_rows64(s_blk, v0, u, lane);
    decode_units(kind, u, x);
    xpose_rows64(s_blk, v1, u, lane);
    decode_units(kind, u, g);
  }
}

// Prefetches into L2 the C lines the warp's chunks of a dSwiGLU tile will read (row `row`,
// ref columns col_base + 32 c for c = c_first, c_first + c_step, ...): issued before the wait for
// the tile's accumulator, so C streams in while the tile's MMAs run.
template <int BN>
__device__ __forceinline__ void prefetch_dswiglu_c(const GemmParams& p, int row, int col_base, int c_first,
                                                   int c_step) {
  const int es = p.c_in_kind == kOutF32 ? 4 : p.c_in_kind == kOutE4M3 ? 1 : 2;
  const char* base = static_cast<const char*>(p.c_in) + static_cast<uint64_t>(row) * (2 * p.n) * es;
  for (int c = c_first; c < BN / 32; c += c_step) {
    const int col0 = col_base + c * 32;
    if (col0 >= p.n) break;
    const char* line = base + static_cast<uint64_t>(2 * col0) * es;  // 64 elements: input + gate block
    for (int b = 0; b < 64 * es; b += 128) prefetch_l2(line + b);
  }
}

// dSwiGLU backward epilogue of one tile for the rows of one warp ("Grouped GEMM + dSwiGLU
// (SM100)", Step 2).  Accumulator chunk c (ref columns n0 .. n0 + 31, n0 = col_base + 32 c)
// pairs with the input block at C columns 2 n0 .. 2 n0 + 31 and the gate block right after it;
// with x = beta_g * input, g = beta_g * gate, s = sigmoid(g) and ref = alpha_g * acc:
//   ab = ref * prob * g * s,   dswiglu = ref * prob * x * s * (1 + g (1 - s)),
// stored at the same two D blocks; sum(g * s * x * ref) over the warp's chunks is added to
// dprob[row].  Float D folds |ab| and |dswiglu| into max_ab / max_dsw; E4M3 D quantises each
// block by rows and by columns.  N is a multiple of 32, so a chunk is wholly in or out.
template <int BN, bool kFP8>
__device__ __forceinline__ void epilogue_tile_dswiglu(const GemmParams& p, int row, int col_base, uint32_t tmem_acc,
                                                      int lane, float alpha_g, float beta_g, float prob_r, float nc,
                                                      float& max_ab, float& max_dsw, int c_first, int c_step,
                                                      float* s_inv, uint8_t* s_blk) {
  const int n_d = 2 * p.n;
  const int row0 = row - lane;
  float dprob_part = 0.0f;
#pragma unroll 1
  for (int c = c_first; c < BN / 32; c += c_step) {
    const int col0 = col_base + c * 32;
    if (col0 >= p.n) break;  // warp-uniform
    float x[32], g[32];
    load_dswiglu_c(s_blk, p, row0, col0, x, g, lane);
    uint32_t r[32];
    tmem_ld_32x32b_x32(tmem_acc + c * 32, r);
    tmem_ld_wait(r);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float ref = alpha_g * __uint_as_float(r[j]);
      const float xv = beta_g * x[j];
      const float gv = beta_g * g[j];
      // sigmoid from the fast exponential and division: a few ulp, and 0 / 1 at the tails
      const float sig = __fdividef(1.0f, 1.0f + __expf(-gv));
      const float sw = gv * sig;
      dprob_part = fmaf(sw * xv, ref, dprob_part);
      const float rp = ref * prob_r;
      x[j] = rp * sw;                                        // ab
      g[j] = rp * xv * sig * fmaf(gv, 1.0f - sig, 1.0f);     // dswiglu
    }
    if (!kFP8) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        max_ab = fmaxf(max_ab, fabsf(x[j]));
        max_dsw = fmaxf(max_dsw, fabsf(g[j]));
      }
      store_block_coalesced(s_blk, p.d, p.d_kind, n_d, n_d, row0, 2 * col0, x, lane);
      store_block_coalesced(s_blk, p.d, p.d_kind, n_d, n_d, row0, 2 * col0 + 32, g, lane);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        x[j] = __fmul_rn(x[j], nc);
        g[j] = __fmul_rn(g[j], nc);
      }
      store_e4m3_block(p, row, 2 * col0, n_d, x, lane, s_inv, s_blk);
      store_e4m3_block(p, row, 2 * col0 + 32, n_d, g, lane, s_inv, s_blk);
    }
  }
  if (dprob_part != 0.0f) atomicAdd(&p.dprob[row], dprob_part);
}

// bf16 bit pattern to fp32 (exact).
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits) { return __uint_as_float(bits << 16); }

// One 32-feature chunk of the RoPE projection that passes unchanged: read from TMEM at
// tmem_chunk, quantised by rows and columns at output column dcol0.
__device__ __forceinline__ void rope_plain_chunk(const GemmParams& p, int row, uint32_t tmem_chunk, int dcol0,
                                                 int lane, float* s_inv, uint8_t* s_blk) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(tmem_chunk, r);
  tmem_ld_wait(r);
  float d[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) d[j] = __uint_as_float(r[j]);
  store_e4m3_block<true>(p, row, dcol0, p.n, d, lane, s_inv, s_blk);
}

// The two rotary chunks of one head (TMEM tmem_chunk and tmem_chunk + 32, output columns dcol0
// and dcol0 + 32): 32 interleaved pairs (a_j, b_j) = (y[2j], y[2j+1]) leave as halves,
//   out[j] = a_j cos[t, j] - b_j sin[t, j],   out[32 + j] = b_j cos[t, 32 + j] + a_j sin[t, 32 + j],
// then both output blocks are quantised by rows and columns.
__device__ __forceinline__ void rope_rotary_pair(const GemmParams& p, int row, uint32_t tmem_chunk, int dcol0,
                                                 int lane, float* s_inv, uint8_t* s_blk) {
  uint32_t r0[32], r1[32];
  tmem_ld_32x32b_x32(tmem_chunk, r0);
  tmem_ld_32x32b_x32(tmem_chunk + 32, r1);
  tmem_ld_wait(r0);
  tmem_ld_wait(r1);
  const uint16_t* cs = p.rope_cos + static_cast<uint64_t>(row) * p.qk_rope;
  const uint16_t* sn = p.rope_sin + static_cast<uint64_t>(row) * p.qk_rope;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    uint32_t(&src)[32] = g == 0 ? r0 : r1;  // pairs j = 16 g .. 16 g + 15
    // cos / sin of j (first half) and 32 + j (second half): 32 bytes each
    uint4 c_lo[2], c_hi[2], s_lo[2], s_hi[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      c_lo[i] = __ldg(reinterpret_cast<const uint4*>(cs + 16 * g) + i);
      c_hi[i] = __ldg(reinterpret_cast<const uint4*>(cs + 32 + 16 * g) + i);
      s_lo[i] = __ldg(reinterpret_cast<const uint4*>(sn + 16 * g) + i);
      s_hi[i] = __ldg(reinterpret_cast<const uint4*>(sn + 32 + 16 * g) + i);
    }
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const uint4& cl = c_lo[jj >> 3];
      const uint4& ch = c_hi[jj >> 3];
      const uint4& sl = s_lo[jj >> 3];
      const uint4& sh = s_hi[jj >> 3];
      const int w = (jj >> 1) & 3, hw = jj & 1;  // 32-bit word and 16-bit half within the uint4
      const uint32_t wc = w == 0 ? cl.x : w == 1 ? cl.y : w == 2 ? cl.z : cl.w;
      const uint32_t wch = w == 0 ? ch.x : w == 1 ? ch.y : w == 2 ? ch.z : ch.w;
      const uint32_t ws = w == 0 ? sl.x : w == 1 ? sl.y : w == 2 ? sl.z : sl.w;
      const uint32_t wsh = w == 0 ? sh.x : w == 1 ? sh.y : w == 2 ? sh.z : sh.w;
      const float c1 = bf16_bits_to_float(hw ? wc >> 16 : wc & 0xffffu);
      const float c2 = bf16_bits_to_float(hw ? wch >> 16 : wch & 0xffffu);
      const float s1 = bf16_bits_to_float(hw ? ws >> 16 : ws & 0xffffu);
      const float s2 = bf16_bits_to_float(hw ? wsh >> 16 : wsh & 0xffffu);
      const float a = __uint_as_float(src[2 * jj]);
      const float b = __uint_as_float(src[2 * jj + 1]);
      src[2 * jj] = __float_as_uint(fmaf(a, c1, -b * s1));      // out[j]
      src[2 * jj + 1] = __float_as_uint(fmaf(b, c2, a * s2));   // out[32 + j]
    }
  }
  float lo[32], hi[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    lo[j] = __uint_as_float(r0[2 * j]);
    lo[16 + j] = __uint_as_float(r1[2 * j]);
    hi[j] = __uint_as_float(r0[2 * j + 1]);
    hi[16 + j] = __uint_as_float(r1[2 * j + 1]);
  }
  store_e4m3_block<true>(p, row, dcol0, p.n, lo, lane, s_inv, s_blk);
  store_e4m3_block<true>(p, row, dcol0 + 32, p.n, hi, lane, s_inv, s_blk);
}

// One output block of a head's rotary pair: out[j] (kHi = false, output columns dcol0 ..
// dcol0 + 31) or out[32 + j] (kHi, dcol0 + 32 .. dcol0 + 63) for the 32 interleaved pairs of both
// rotary chunks (formulas as in rope_rotary_pair, the same products), then the block is quantised
// by rows and columns.  The two halves of a quadrant's warps take one block each.
template <bool kHi>
__device__ __forceinline__ void rope_rotary_block(const GemmParams& p, int row, uint32_t tmem_chunk, int dcol0,
                                                  int lane, float* s_inv, uint8_t* s_blk) {
  uint32_t r0[32], r1[32];
  tmem_ld_32x32b_x32(tmem_chunk, r0);
  tmem_ld_32x32b_x32(tmem_chunk + 32, r1);
  tmem_ld_wait(r0);
  tmem_ld_wait(r1);
  const int t0 = kHi ? 32 : 0;  // the block's cos / sin columns
  const uint16_t* cs = p.rope_cos + static_cast<uint64_t>(row) * p.qk_rope + t0;
  const uint16_t* sn = p.rope_sin + static_cast<uint64_t>(row) * p.qk_rope + t0;
  float out[32];
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const uint32_t(&src)[32] = g == 0 ? r0 : r1;  // pairs j = 16 g .. 16 g + 15
    uint4 cv[2], sv[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      cv[i] = __ldg(reinterpret_cast<const uint4*>(cs + 16 * g) + i);
      sv[i] = __ldg(reinterpret_cast<const uint4*>(sn + 16 * g) + i);
    }
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const uint4& c4 = cv[jj >> 3];
      const uint4& s4 = sv[jj >> 3];
      const int w = (jj >> 1) & 3, hw = jj & 1;  // 32-bit word and 16-bit half within the uint4
      const uint32_t wc = w == 0 ? c4.x : w == 1 ? c4.y : w == 2 ? c4.z : c4.w;
      const uint32_t ws = w == 0 ? s4.x : w == 1 ? s4.y : w == 2 ? s4.z : s4.w;
      const float c = bf16_bits_to_float(hw ? wc >> 16 : wc & 0xffffu);
      const float sv1 = bf16_bits_to_float(hw ? ws >> 16 : ws & 0xffffu);
      const float a = __uint_as_float(src[2 * jj]);
      const float b = __uint_as_float(src[2 * jj + 1]);
      out[16 * g + jj] = kHi ? fmaf(b, c, a * sv1) : fmaf(a, c, -b * sv1);
    }
  }
  store_e4m3_block<true>(p, row, dcol0 + t0, p.n, out, lane, s_inv, s_blk);
}

// GEMM + RoPE + MXFP8 epilogue of one tile ("GEMM + RoPE + MXFP8 Projection (SM100)",
// Equations) for the rows (tokens) of one warp: output columns col_base .. col_base + BN - 1
// of the (tokens, heads x 192) projection.  Global 32-column chunk g is chunk g % 6 of head
// g / 6; chunks 4 and 5 of a head are rotary (RoPE, rope_rotary_pair), the rest pass unchanged.
// BN = 192 (one head per tile): half 0 of a quadrant's warps takes chunks 0-1 and the rotary
// pair's first output block, half 1 chunks 2-3 and its second block (equal work).  BN = 256:
// the tile's chunks go in pairs (0,1), (2,3), (4,5), (6,7), half 0 taking the first and third,
// half 1 the others; a pair starts at an even global chunk, so it is either two plain chunks or
// one head's rotary pair (g % 6 == 4), never split.
template <int BN>
__device__ __forceinline__ void epilogue_tile_rope(const GemmParams& p, int row, int col_base, uint32_t tmem_acc,
                                                   int lane, int half, float* s_inv, uint8_t* s_blk) {
  static_assert(BN == 192 || BN == 256, "RoPE tiles");
  if constexpr (BN == 192) {
    // col_base = head * 192: chunks 0-3 plain, 4-5 rotary
    const int c0 = 2 * half;
#pragma unroll 1
    for (int c = c0; c < c0 + 2; ++c)
      rope_plain_chunk(p, row, tmem_acc + c * 32, col_base + c * 32, lane, s_inv, s_blk);
    if (half == 0) rope_rotary_block<false>(p, row, tmem_acc + 4 * 32, col_base + 4 * 32, lane, s_inv, s_blk);
    else rope_rotary_block<true>(p, row, tmem_acc + 4 * 32, col_base + 4 * 32, lane, s_inv, s_blk);
  } else {
#pragma unroll 1
    for (int q = half; q < 4; q += 2) {
      const int c = 2 * q;  // first chunk of the pair within the tile
      const int g = (col_base >> 5) + c;
      if (g % 6 == 4) {
        rope_rotary_pair(p, row, tmem_acc + c * 32, col_base + c * 32, lane, s_inv, s_blk);
      } else {
        rope_plain_chunk(p, row, tmem_acc + c * 32, col_base + c * 32, lane, s_inv, s_blk);
        rope_plain_chunk(p, row, tmem_acc + (c + 1) * 32, col_base + (c + 1) * 32, lane, s_inv, s_blk);
      }
    }
  }
}

// Dense amax without a cleared output: every CTA (one thread) folds its maximum into the
// workspace record and counts itself finished with one 128-bit compare-and-swap (lo = epoch << 32
// | count, hi = maximum bits; non-negative floats order like their bit patterns).  A record with
// another epoch is a previous call's and is replaced.  The CTA whose swap completes the count
// holds the final maximum in its own result: it writes *p.amax and resets the record under this
// epoch (count and maximum zero), so a replay of the same call (a CUDA graph) starts from zero.
__device__ __forceinline__ void dense_amax_finalize(const GemmParams& p, float cta_max) {
  void* rec = reinterpret_cast<uint8_t*>(p.err) + kWsAmaxRecordByte;
  const uint64_t tag = static_cast<uint64_t>(p.epoch) << 32;
  const uint32_t v = cta_max > 0.0f ? __float_as_uint(cta_max) : 0u;
  const volatile uint64_t* rv = reinterpret_cast<const volatile uint64_t*>(rec);
  uint64_t lo = rv[0], hi = rv[1];  // a guess: a torn or stale read only costs one more round
  uint64_t new_lo, new_hi;
  for (;;) {
    const bool mine = (lo >> 32) == p.epoch;
    const uint32_t count = mine ? static_cast<uint32_t>(lo) : 0u;
    const uint32_t cur = mine ? static_cast<uint32_t>(hi) : 0u;
    new_lo = tag | (count + 1u);
    new_hi = v > cur ? v : cur;
    uint64_t old_lo, old_hi;
    atomic_cas_b128(rec, lo, hi, new_lo, new_hi, old_lo, old_hi);
    if (old_lo == lo && old_hi == hi) break;
    lo = old_lo;
    hi = old_hi;
  }
  if (static_cast<uint32_t>(new_lo) == gridDim.x) {
    p.amax[0] = __uint_as_float(static_cast<uint32_t>(new_hi));
    // every other CTA of this call has swapped already: a plain store resets the record
    volatile uint64_t* w = reinterpret_cast<volatile uint64_t*>(rec);
    w[1] = 0;
    w[0] = tag;
  }
}

// Folds one warp's running maxima of expert g into shared memory: the per-expert amax of the
// grouped sReLU float D, or the (|ab|, |dswiglu|) pair of the dSwiGLU float D.
template <int EPI>
__device__ __forceinline__ void fold_expert_max(float* s_amax, int g, float m1, float m2, int lane) {
  if constexpr (EPI == kEpiGroupedBF16 || EPI == kEpiDswigluF) {
    for (int o = 16; o >= 1; o >>= 1) {
      m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
      m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
    }
    if (lane == 0) {
      if (EPI == kEpiGroupedBF16) {
        atomic_max_nonneg(&s_amax[g], m1);
      } else {
        atomic_max_nonneg(&s_amax[2 * g], m1);
        atomic_max_nonneg(&s_amax[2 * g + 1], m2);
      }
    }
  }
}

// Epilogue of one tile for the rows of one warp: reads the fp32 accumulator chunk by chunk
// (32 columns of this thread's row per tcgen05.ld) from `tmem_acc` (this warp's lane
// quadrant, first accumulator column) and writes the outputs of row `row`, columns
// col_base .. col_base + BN - 1 (clipped at N).  `l` is the batch (dense) or expert (grouped).
// s_inv: 32 floats of shared memory owned by this warp (E4M3 D only: the column scales'
// reciprocals are exchanged through it).
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, int l, int row, int col_base, uint32_t tmem_acc,
                                              int lane, float alpha_g, float prob_r, float nc, float& run_max,
                                              int c_first, int c_step, float* s_inv, uint8_t* s_blk) {
  const bool row_ok = row < p.m;
  const float s_clamp = p.clamp_s;
  const float inv_s = s_clamp > 0.0f ? 1.0f / s_clamp : 0.0f;
#pragma unroll 1
  for (int c = c_first; c < BN / 32; c += c_step) {
    const int col0 = col_base + c * 32;
    if (col0 >= p.n) break;  // warp-uniform
    uint32_t r[32];
    tmem_ld_32x32b_x32(tmem_acc + c * 32, r);
    tmem_ld_wait(r);
    if (EPI == kEpiDense) {
#pragma unroll
      for (int j = 0; j < 32; ++j) run_max = fmaxf(run_max, fabsf(__uint_as_float(r[j])));
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
      if (p.c_kind == kOutF32 || p.c_kind == kOutBF16 || p.c_kind == kOutF16) {
        // whole rows of the warp's 32 x 32 block through the transpose block (coalesced)
        const int esz = p.c_kind == kOutF32 ? 4 : 2;
        void* batch = static_cast<uint8_t*>(p.c) + static_cast<uint64_t>(l) * p.m * p.n * esz;
        store_block_coalesced(s_blk, batch, p.c_kind, p.n, p.n, row - lane, col0, v, lane, p.m);
      } else if (row_ok) {
        store_row32(p.c, (static_cast<uint64_t>(l) * p.m + row) * static_cast<uint64_t>(p.n) + col0, p.c_kind, v,
                    col0, p.n);
      }
    } else {
      float d[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float cv = alpha_g * __uint_as_float(r[j]);
        r[j] = __float_as_uint(cv);
        d[j] = srelu_clamp(cv, prob_r, s_clamp, inv_s, p.tanh_approx);
      }
      // a chunk may run past N: 16-byte granules (N % 8 == 0 for 16-bit outputs, % 4 for fp32)
      // C and float D pass through the warp's transpose block (coalesced, whole-sector stores)
      if (p.c_kind != kOutNone) {
        if (p.c_v8 && col0 + 32 <= p.n) {
          // bf16 C: this thread's 32 values are two whole sectors of its row
          uint32_t w0[8], w1[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            w0[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            w1[j] = pack_bf16x2(__uint_as_float(r[16 + 2 * j]), __uint_as_float(r[16 + 2 * j + 1]));
          }
          uint16_t* crow = reinterpret_cast<uint16_t*>(p.c) + static_cast<uint64_t>(row) * p.n + col0;
          st_global_v8(crow, w0);
          st_global_v8(crow + 16, w1);
        } else {
          float cvals[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) cvals[j] = __uint_as_float(r[j]);
          store_block_coalesced(s_blk, p.c, p.c_kind, p.n, p.n, row - lane, col0, cvals, lane);
        }
      }
      if (EPI == kEpiGroupedBF16) {
        // columns past N hold zeros (zero-filled B rows), so they cannot raise the maximum
#pragma unroll
        for (int j = 0; j < 32; ++j) run_max = fmaxf(run_max, fabsf(d[j]));
        store_block_coalesced(s_blk, p.d, p.d_kind, p.n, p.n, row - lane, col0, d, lane);
      } else {
        // D * norm_const once (rounding is monotonic, so the block maxima of the products are
        // norm_const times the block maxima of D, rounded); scaling by 2^-e is exact
#pragma unroll
        for (int j = 0; j < 32; ++j) d[j] = __fmul_rn(d[j], nc);
        store_e4m3_block(p, row, col0, p.n, d, lane, s_inv, s_blk);
      }
    }
  }
}

// Grouped sReLU epilogue with bf16 D and bf16 or no C, stored by TMA: for each of this warp's
// 32-column chunks the fp32 accumulator is read from TMEM, C = alpha * acc and D are computed as
// in epilogue_tile, and this thread's row of each 32 x 32 bf16 block is written into the warp's
// staging blocks s_c / s_d (64 bytes per row, 16-byte granule g at granule g ^ ((row / 2) % 4):
// the 64-byte swizzle of the tensor maps); then one elected lane stores both blocks with
// cp.async.bulk.tensor (rows past M and columns past N are clipped by the maps).  The next chunk
// rewrites the blocks once those stores have read them.  `release` (the accumulator-empty
// arrival) runs as soon as the warp's last chunk has been read from TMEM, so the accumulator is
// held neither while the last chunk is staged nor while any block travels to global memory.
template <int BN, class Release>
__device__ __forceinline__ void epilogue_tile_grouped_tma(const GemmParams& p, int row, int col_base,
                                                          uint32_t tmem_acc, int lane, float alpha_g, float prob_r,
                                                          float& run_max, int c_first, int c_step, uint8_t* s_c,
                                                          uint8_t* s_d, const CUtensorMap* tmap_c,
                                                          const CUtensorMap* tmap_d, Release release) {
  const float s_clamp = p.clamp_s;
  const float inv_s = s_clamp > 0.0f ? 1.0f / s_clamp : 0.0f;
  const int row0 = row - lane;
  const bool with_c = p.c_kind != kOutNone;
  const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
  bool released = false;
#pragma unroll 1
  for (int c = c_first; c < BN / 32; c += c_step) {
    const int col0 = col_base + c * 32;
    if (col0 >= p.n) break;  // warp-uniform
    uint32_t r[32];
    tmem_ld_32x32b_x32(tmem_acc + c * 32, r);
    tmem_ld_wait(r);
    if (c + c_step >= BN / 32 || col0 + c_step * 32 >= p.n) {  // this warp's last chunk is in registers
      release();
      released = true;
    }
    uint32_t cw[16], dw[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float c0 = alpha_g * __uint_as_float(r[2 * j]);
      const float c1 = alpha_g * __uint_as_float(r[2 * j + 1]);
      const float d0 = srelu_clamp(c0, prob_r, s_clamp, inv_s, p.tanh_approx);
      const float d1 = srelu_clamp(c1, prob_r, s_clamp, inv_s, p.tanh_approx);
      // columns past N hold zeros (zero-filled B rows), so they cannot raise the maximum
      run_max = fmaxf(run_max, fmaxf(fabsf(d0), fabsf(d1)));
      cw[j] = pack_bf16x2(c0, c1);
      dw[j] = pack_bf16x2(d0, d1);
    }
    // the previous chunk's stores have read the staging blocks
    warp_bulk_wait_all<true>();
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t off = static_cast<uint32_t>(lane) * 64u + ((static_cast<uint32_t>(g) ^ sw) << 4);
      if (with_c)
        *reinterpret_cast<uint4*>(s_c + off) = make_uint4(cw[4 * g], cw[4 * g + 1], cw[4 * g + 2], cw[4 * g + 3]);
      *reinterpret_cast<uint4*>(s_d + off) = make_uint4(dw[4 * g], dw[4 * g + 1], dw[4 * g + 2], dw[4 * g + 3]);
    }
    fence_async_shared();
    __syncwarp();
    if (with_c) warp_tma_store_2d(tmap_c, s_c, col0, row0);
    warp_tma_store_2d(tmap_d, s_d, col0, row0);
    warp_bulk_commit();
  }
  if (!released) release();
}

// NM block-scaled MMAs of one stage into d_tmem, issued by the whole warp (one elected lane per
// instruction); the stage's scale factors are in TMEM at sfa_t / sfb_t.  MXFP8 stages hold one
// scale column per row (four K blocks, one per MMA, selected by the instruction descriptor's
// scale-factor id); NVFP4 stages hold one column of four UE4M3 scales per row and MMA.  The
// first MMA accumulates iff acc0.  idesc and b_step (the B descriptor's advance per MMA) are
// loop-invariant, computed once by the caller: for K-major B, T::kIdesc and 32 bytes (2 encoded);
// for N-major B (MXFP8 only), bit 16 of the instruction descriptor set and 32 rows of 128 bytes
// (four 1024-byte swizzle atoms, 256 encoded).
template <int FMT, class T, int NM>
__device__ __forceinline__ void issue_stage(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t sfa_t,
                                            uint32_t sfb_t, uint32_t acc0, uint32_t idesc, uint32_t b_step) {
#pragma unroll
  for (int j = 0; j < NM; ++j) {
    const uint32_t accumulate = j > 0 ? 1u : acc0;
    // advance the start address by 32 bytes of K per MMA (encoded >> 4)
    if (FMT == kBF16) {
      warp_mma_f16(d_tmem, adesc + 2 * j, bdesc + 2 * j, T::kIdesc, accumulate);
    } else if (FMT == kMXFP8) {
      warp_mma_mxf8f6f4(d_tmem, adesc + 2 * j, bdesc + b_step * j, idesc | (j << 29) | (j << 4), sfa_t, sfb_t,
                        accumulate);
    } else {
      warp_mma_mxf4nvf4(d_tmem, adesc + 2 * j, bdesc + 2 * j, T::kIdesc, sfa_t + j * 4,
                        sfb_t + j * T::kSfbColsPerMma, accumulate);
    }
  }
}

// One stager warp's share of a stage's scale factors: lane i of quadrant q (TMEM lanes 32q + i)
// receives row i of every 512-byte SFA atom (16 bytes: the scales of rows i, 32 + i, 64 + i and
// 96 + i of the 128-row group, four K blocks each) as four consecutive 32-bit columns, i.e. what
// tcgen05.cp 32x128b.warpx4 of the atom writes into every quadrant; SFA atom a goes to columns
// sfa_t + 4a.  For B, column sfb_t + kSfbColsPerMma * a + c holds, in lane i of every quadrant,
// the scales of tile row 32c + i: for tiles aligned to the atoms these are again whole atom rows
// (atom g of the unit fills columns 4g .. 4g + 3), otherwise single 32-bit words gathered from the
// (up to three) atoms the tile's rows fall in.  b_blk0 is the 32-row block index of the tile's
// first row within the first atom group loaded.
// kWideGather: for unaligned tiles, read whole 16-byte group rows and select words (fewer
// shared-memory wavefronts; measured faster in the one-CTA kernel, slower in the pair kernel's
// dSwiGLU variant) rather than single, four-way bank-conflicting words.
template <class T, bool kWideGather = false>
__device__ __forceinline__ void stage_scale_factors(const uint8_t* sfa_s, const uint8_t* sfb_s, uint32_t sfa_t,
                                                    uint32_t sfb_t, int lane, int b_blk0) {
  constexpr int A = T::kAtomsPerStage, G = T::kBRowGroups, C = T::kSfbColsPerMma;
  uint32_t ra[4 * A];
#pragma unroll
  for (int a = 0; a < A; ++a) {
    const uint4 v = *reinterpret_cast<const uint4*>(sfa_s + a * 512 + lane * 16);
    ra[4 * a] = v.x; ra[4 * a + 1] = v.y; ra[4 * a + 2] = v.z; ra[4 * a + 3] = v.w;
  }
  uint32_t rb[C * A];
  if constexpr (T::kSfbAligned) {
#pragma unroll
    for (int a = 0; a < A; ++a) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint4 v = *reinterpret_cast<const uint4*>(sfb_s + (g * A + a) * 512 + lane * 16);
        const int c = C * a + 4 * g;
        rb[c] = v.x; rb[c + 1] = v.y; rb[c + 2] = v.z; rb[c + 3] = v.w;
      }
    }
  } else if constexpr (kWideGather) {
    // Word w of the loaded groups (group w / 4, word w % 4 of this lane's 16 bytes) holds the
    // scales of 32-row block w; the tile's block c is word b_blk0 + c.  Each group's 16 bytes
    // are read whole (conflict-free, unlike four-way conflicting single words) and the words
    // picked with selects (b_blk0 <= 3, so word b_blk0 + c is one of words c .. c + 3).
    static_assert(T::kBBlocks + 3 <= 4 * G, "loaded groups cover the tile's blocks");
#pragma unroll
    for (int a = 0; a < A; ++a) {
      uint32_t w[4 * G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint4 v = *reinterpret_cast<const uint4*>(sfb_s + (g * A + a) * 512 + lane * 16);
        w[4 * g] = v.x; w[4 * g + 1] = v.y; w[4 * g + 2] = v.z; w[4 * g + 3] = v.w;
      }
#pragma unroll
      for (int c = 0; c < C; ++c) {
        uint32_t x = 0u;
        if (c < T::kBBlocks) {
          x = w[c];
          x = b_blk0 == 1 ? w[c + 1] : x;
          x = b_blk0 == 2 ? w[c + 2] : x;
          x = b_blk0 == 3 ? w[c + 3] : x;
        }
        rb[C * a + c] = x;
      }
    }
  } else {
#pragma unroll
    for (int a = 0; a < A; ++a) {
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const int blk = b_blk0 + c;  // 32-row block within the loaded atom groups
        rb[C * a + c] = c < T::kBBlocks
                            ? *reinterpret_cast<const uint32_t*>(sfb_s + ((blk >> 2) * A + a) * 512 + lane * 16 +
                                                                 (blk & 3) * 4)
                            : 0u;
      }
    }
  }
  tmem_st_32x32b<4 * A>(sfa_t, ra);
  tmem_st_32x32b<C * A>(sfb_t, rb);
}

template <int FMT, int BN, int EPI>
__global__ void __launch_bounds__(kThreadsGemm, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                const __grid_constant__ GemmParams p) {
  using T = GemmTraits<FMT, BN, EPI>;
  constexpr int S = T::kStages;
  constexpr int ACC = T::kAcc;

  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzled TMA tiles need 1024-byte aligned shared addresses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* s_a = smem;
  uint8_t* s_b = s_a + S * T::kABytes;
  uint8_t* s_sfa = s_b + S * T::kBBytes;
  uint8_t* s_sfb = s_sfa + S * T::kSfaBytes;
  uint8_t* s_bar = s_sfb + S * T::kSfbBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_bar);
  uint64_t* empty = full + S;
  uint64_t* tmem_full = empty + S;
  uint64_t* tmem_empty = tmem_full + ACC;
  uint64_t* drain = tmem_empty + ACC;
  uint64_t* sf_ready = drain + 1;  // the stage's scale factors are in TMEM (four stager arrivals)
  uint64_t* sf_free = sf_ready + S;  // TMEM scale slot free again (its MMAs completed)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_free + T::kSfSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bad_flag = const_cast<int*>(abort_flag) + 1;
  int32_t* s_offs = reinterpret_cast<int32_t*>(s_bar + T::kBarBytes);
  float* s_amax = reinterpret_cast<float*>(s_bar + T::kBarBytes + T::kOffsetsBytes);
  uint8_t* s_xpose = s_bar + T::kBarBytes + T::kOffsetsBytes + T::kAmaxBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(&tmem_full[a], 1);
      mbar_init(&tmem_empty[a], 8);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < S; ++s) mbar_init(&sf_ready[s], 4);
    for (int f = 0; f < T::kSfSlots; ++f) mbar_init(&sf_free[f], 1);
    *abort_flag = 0;
    *bad_flag = 0;
    fence_mbar_init();
  }
  if (epi_is_grouped(EPI)) {
    for (int i = threadIdx.x; i < 1024; i += kThreadsGemm) s_amax[i] = 0.0f;
  } else if (threadIdx.x == 0) {
    s_amax[0] = 0.0f;
  }
  __syncthreads();
  if (epi_is_grouped(EPI)) {
    // stage padded_offsets and check: multiples of 256, non-decreasing, last == valid_m
    for (int i = threadIdx.x; i < p.l; i += kThreadsGemm) {
      const int32_t o = p.offsets[i];
      const int32_t prev = i == 0 ? 0 : p.offsets[i - 1];
      s_offs[i] = o;
      if ((o & 255) != 0 || o < prev || o > p.m || (i == p.l - 1 && o != p.m)) atomicOr(bad_flag, 1);
    }
    // per-expert weights: the descriptor kernel before this one found an invalid weight pointer
    if (p.b_maps != nullptr && threadIdx.x == 0 &&
        reinterpret_cast<volatile uint32_t*>(p.err)[kWsBadPointersWord] == p.epoch)
      atomicOr(bad_flag, 2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, T::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool bad = *bad_flag != 0;
  const ErrSink es{p.err, p.epoch};
  if (threadIdx.x == 0) mark_call(es);
  if ((*bad_flag & 1) && blockIdx.x == 0 && threadIdx.x == 0) report_error(es, kErrBadOffsets);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop and executes every copy, which elect.sync predicates to one
    // lane (warp_* helpers); wait outcomes are made warp-uniform before they steer it.
    if (!bad) {
      uint32_t stage = 0, phase = 0;
      uint64_t issued = 0;
      bool ok = true;
      int fenced_l = -1;  // expert whose global tensor map the warp has acquired
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        const TileCoord tc = decode_tile<EPI>(p, t, s_offs);
        const int a_batch = epi_is_grouped(EPI) ? 0 : tc.l;
        // per-expert weights: the expert's own tensor map and scale array, else batch tc.l of one
        const CUtensorMap* bmap = p.b_maps ? p.b_maps + tc.l : &tmap_b;
        if (p.b_maps && tc.l != fenced_l) { tmap_acquire(bmap); fenced_l = tc.l; }
        const int b_batch = p.b_maps ? 0 : tc.l;
        const uint8_t* sfb_base =
            p.sfb_ptrs ? reinterpret_cast<const uint8_t*>(p.sfb_ptrs[tc.l])
                       : p.sfb + static_cast<uint64_t>(tc.l) * p.sfb_mt * p.sf_kt * 512;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!__all_sync(0xffffffffu, wait_bounded(&empty[stage], phase ^ 1u, abort_flag, es))) {
            ok = false;
            break;
          }
          const int k_left = p.k - kt * T::kElemsPerKTile;
          const int n_mma = min(T::kMmasPerStage, (k_left + T::kMmaK - 1) / T::kMmaK);
          const int atoms = FMT == kMXFP8 ? 1 : FMT == kNVFP4 ? n_mma : 0;
          const uint32_t sf_bytes = static_cast<uint32_t>(atoms * 512 * (1 + T::kBRowGroups));
          warp_arrive_expect_tx(&full[stage], T::kABytes + T::kBBytes + sf_bytes);
          warp_tma_load_3d(s_a + stage * T::kABytes, &tmap_a, &full[stage], kt * kTileKBytes, tc.mt * kTileM, a_batch);
          if (FMT == kMXFP8 && BN == 128 && p.b_mn_major)  // N-major B: 128 bytes of N x 128 rows of K
            warp_tma_load_3d(s_b + stage * T::kBBytes, bmap, &full[stage], tc.nt * BN, kt * T::kElemsPerKTile,
                             b_batch);
          else
            warp_tma_load_3d(s_b + stage * T::kBBytes, bmap, &full[stage], kt * kTileKBytes, tc.nt * BN, b_batch);
          if constexpr (FMT != kBF16) {
            const uint8_t* sfa_src =
                p.sfa + ((static_cast<uint64_t>(a_batch) * p.sfa_mt + tc.mt) * p.sf_kt +
                         static_cast<uint64_t>(kt) * T::kAtomsPerStage) * 512;
            warp_bulk_load(s_sfa + stage * T::kSfaBytes, sfa_src, atoms * 512, &full[stage]);
#pragma unroll
            for (int i = 0; i < T::kBRowGroups; ++i) {
              // a 128-row group past N reuses the last group's (finite) scales: its B rows are zero
              const int rb = min((tc.nt * BN) / 128 + i, p.sfb_mt - 1);
              const uint8_t* sfb_src = sfb_base + (static_cast<uint64_t>(rb) * p.sf_kt +
                                                   static_cast<uint64_t>(kt) * T::kAtomsPerStage) * 512;
              warp_bulk_load(s_sfb + stage * T::kSfbBytes + i * T::kAtomsPerStage * 512, sfb_src, atoms * 512,
                             &full[stage]);
            }
          }
          ++issued;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // drain: every load issued must land before the CTA leaves
        for (int s = 0; s < S; ++s) {
          if (issued > static_cast<uint64_t>(s)) {
            const uint32_t ph = (s < static_cast<int>(stage)) ? phase : (phase ^ 1u);
            wait_bounded_plain(&full[s], ph);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (!bad) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, fslot = 0;
      bool ok = true;
      const uint32_t a_base = smem_u32(s_a), b_base = smem_u32(s_b);
      const uint32_t b_mn = (FMT == kMXFP8 && BN == 128 && p.b_mn_major) ? 1u : 0u;
      const uint32_t idesc = T::kIdesc | (b_mn << 16);
      const uint32_t b_step = b_mn ? 256u : 2u;
      // MMAs in the last K stage (fewer than a stage's when K is not a multiple of its depth)
      const int last_mmas =
          min(T::kMmasPerStage, (p.k - (p.k_tiles - 1) * T::kElemsPerKTile + T::kMmaK - 1) / T::kMmaK);
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        // outcomes of waits are made warp-uniform before they steer the warp-collective issue
        if (!__all_sync(0xffffffffu, wait_bounded(&tmem_empty[acc], acc_phase ^ 1u, abort_flag, es))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          // Control flow and every tcgen05 operand stay warp-uniform: the whole warp computes
          // the operands and executes each MMA and commit, which elect.sync predicates to one
          // lane (no branch around the issue), and a failed wait (timeout or abort) is recorded
          // rather than acted on until the tile ends, so the k-loop has no data-dependent exit.
          // Issued from inside a one-lane branch, each MMA costs the issuing thread about as long
          // as the MMA itself runs and the per-stage bookkeeping leaves the tensor pipe idle.
          // Issuing after a failed wait reads stale shared memory, which is harmless: the
          // results are discarded with the error.
          // the stagers arrive after the stage's data landed and its scale factors are in TMEM
          // bf16 stages carry no scale factors: their data landing (full) is all the MMAs need
          ok &= wait_bounded(FMT == kBF16 ? &full[stage] : &sf_ready[stage], phase, abort_flag, es);
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + T::kSfBase + fslot * T::kSfStride;
          const uint32_t sfb_t = sfa_t + T::kSfaCols;
          const uint64_t adesc = smem_desc(a_base + stage * T::kABytes, 16, 1024, kSwizzle128B);
          // K-major B: rows of 128 bytes of K, 8-row groups 1024 bytes apart; N-major B (one
          // 128-byte swizzle row of N per K row): 8-K-row atoms 1024 bytes apart
          const uint64_t bdesc = smem_desc(b_base + stage * T::kBBytes, 16, 1024, kSwizzle128B);
          const uint32_t acc0 = kt > 0 ? 1u : 0u;  // the first MMA of a tile overwrites the accumulator
          const int n_mma = kt == p.k_tiles - 1 ? last_mmas : T::kMmasPerStage;
          // (elect.sync waits for the whole warp: no separate reconvergence is needed)
          if (n_mma == T::kMmasPerStage) {
            issue_stage<FMT, T, T::kMmasPerStage>(d_tmem, adesc, bdesc, sfa_t, sfb_t, acc0, idesc, b_step);
          } else {
            // the last, partial K stage (K not a multiple of the stage depth)
            if (n_mma == 1) issue_stage<FMT, T, 1>(d_tmem, adesc, bdesc, sfa_t, sfb_t, acc0, idesc, b_step);
            if (n_mma == 2) issue_stage<FMT, T, 2>(d_tmem, adesc, bdesc, sfa_t, sfb_t, acc0, idesc, b_step);
            if (n_mma == 3) issue_stage<FMT, T, 3>(d_tmem, adesc, bdesc, sfa_t, sfb_t, acc0, idesc, b_step);
          }
          warp_commit(&empty[stage]);
          if (T::kSfRing) warp_commit(&sf_free[fslot]);
          if (++stage == S) { stage = 0; phase ^= 1u; }
          if (++fslot == T::kSfSlots) fslot = 0;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        warp_commit(&tmem_full[acc]);
        if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        // drain: wait for every MMA issued so far before TMEM is released
        __syncwarp();
        warp_commit(drain);
        if (lane == 0) wait_bounded_plain(drain, 0);
        __syncwarp();
      }
    }
  } else if (warp >= 10) {
    // ------------------------------------------------------------ scale-factor stagers 10..13
    // With one TMEM scale slot per stage, a slot is free once its smem stage has been refilled
    // (the refill waited for the commit of the MMAs that read it); with fewer slots, the MMA
    // thread commits each slot's release to sf_free.
    const uint32_t quad_lanes = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t stage = 0, phase = 0, fslot = 0, fphase = 0;
    bool ok = FMT != kBF16;  // bf16 operands have no scale factors to stage
    for (int t = blockIdx.x; !bad && ok && t < p.num_tiles; t += gridDim.x) {
      const TileCoord tc = decode_tile<EPI>(p, t, s_offs);
      const int b_blk0 = ((tc.nt * BN) >> 5) & 3;  // the tile's first 32-row block within its first atom
      for (int kt = 0; kt < p.k_tiles; ++kt) {
        ok &= wait_bounded(&full[stage], phase, abort_flag, es);
        // with fewer TMEM slots than stages, the slot's previous MMAs must have completed
        if (T::kSfRing) ok &= wait_bounded(&sf_free[fslot], fphase ^ 1u, abort_flag, es);
        tc_fence_after();
        const uint32_t sfa_t = tmem_base + quad_lanes + T::kSfBase + fslot * T::kSfStride;
        if constexpr (FMT != kBF16)
          stage_scale_factors<T, true>(s_sfa + stage * T::kSfaBytes, s_sfb + stage * T::kSfbBytes, sfa_t,
                                       sfa_t + T::kSfaCols, lane, b_blk0);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[stage]);
        if (++stage == S) { stage = 0; phase ^= 1u; }
        if (++fslot == T::kSfSlots) { fslot = 0; fphase ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 2..9
    const int quad = warp & 3;          // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;   // two warps per quadrant take alternate 32-column chunks
    float run_max = 0.0f;       // dense amax, or grouped per-expert segment max (dSwiGLU: of |ab|)
    float run_max2 = 0.0f;      // dSwiGLU: per-expert segment max of |dswiglu|
    int run_expert = -1;
    uint32_t acc = 0, acc_phase = 0;
    const float nc = epi_has_fp8_d(EPI) ? *p.norm_const : 1.0f;
    for (int t = blockIdx.x; !bad && t < p.num_tiles; t += gridDim.x) {
      const TileCoord tc = decode_tile<EPI>(p, t, s_offs);
      const int row = tc.mt * kTileM + quad * 32 + lane;
      if constexpr (epi_is_dswiglu(EPI)) prefetch_dswiglu_c<BN>(p, row, tc.nt * BN, half, 2);
      // warp-uniform outcome: the epilogues use whole-warp shuffles and syncs
      if (!__all_sync(0xffffffffu, wait_bounded(&tmem_full[acc], acc_phase, abort_flag, es))) break;
      tc_fence_after();
      float alpha_g = 1.0f, prob_r = 0.0f;
      if (epi_is_grouped(EPI)) {
        alpha_g = p.alpha[tc.l];
        prob_r = p.prob[row];
        if (tc.l != run_expert) {
          if (run_expert >= 0) fold_expert_max<EPI>(s_amax, run_expert, run_max, run_max2, lane);
          run_expert = tc.l;
          run_max = 0.0f;
          run_max2 = 0.0f;
        }
      }
      const uint32_t tmem_acc = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tmem_empty[acc]);
      };
      if constexpr (EPI == kEpiRope) {
        epilogue_tile_rope<BN>(p, row, tc.nt * BN, tmem_acc, lane, half, s_amax + (warp - 2) * 32,
                               s_xpose + (warp - 2) * T::kXposeBlock);
        release();
      } else if constexpr (epi_is_dswiglu(EPI)) {
        epilogue_tile_dswiglu<BN, EPI == kEpiDswigluFP8>(p, row, tc.nt * BN, tmem_acc, lane, alpha_g, p.beta[tc.l],
                                                         prob_r, nc, run_max, run_max2, half, 2,
                                                         s_amax + (warp - 2) * 32,
                                                         s_xpose + (warp - 2) * T::kXposeBlock);
        release();
      } else if (EPI == kEpiDense && p.c_kind == kOutBF16) {
        epilogue_dense_bf16_early<BN, true>(p, tc.l, row, tc.nt * BN, tmem_acc, half, run_max, release,
                                            s_xpose + (warp - 2) * T::kXposeBlock, lane);
      } else {
        epilogue_tile<BN, EPI>(p, tc.l, row, tc.nt * BN, tmem_acc, lane, alpha_g, prob_r, nc, run_max, half, 2,
                               s_amax + (warp - 2) * 32, s_xpose + (warp - 2) * T::kXposeBlock);
        release();
      }
      if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
    }
    // fold this warp's running maxima into shared memory
    if (EPI == kEpiDense) {
      float v = run_max;
      for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (lane == 0) atomic_max_nonneg(&s_amax[0], v);
    } else if (epi_is_grouped(EPI) && run_expert >= 0) {
      fold_expert_max<EPI>(s_amax, run_expert, run_max, run_max2, lane);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (EPI == kEpiDense) {
    // every CTA folds its maximum into the workspace; the last one to finish writes the amax
    if (threadIdx.x == 0) dense_amax_finalize(p, (!bad && *abort_flag == 0) ? s_amax[0] : 0.0f);
  }
  if (!bad && *abort_flag == 0) {
    // one global atomicMax per CTA and expert touched (grouped float D)
    if (EPI == kEpiGroupedBF16) {
      for (int g = threadIdx.x; g < p.l; g += kThreadsGemm)
        if (s_amax[g] > 0.0f) atomic_max_nonneg(&p.amax[g], s_amax[g]);
    } else if (EPI == kEpiDswigluF) {
      // (|ab|, |dswiglu|) per expert: 2 * num_experts <= 1024 values
      for (int i = threadIdx.x; i < 2 * p.l; i += kThreadsGemm)
        if (s_amax[i] > 0.0f) atomic_max_nonneg(&p.amax[i], s_amax[i]);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, T::kTmemCols);
  }
}

// The fewest CTAs (or CTA pairs) that still take `tiles` tiles in as many rounds as `grid` does.
// With static round-robin tiles the launch takes ceil(tiles / grid) tile times either way; the
// SMs left out are those that would have idled through a partial last round (measured: the
// grouped 1152-tile launch on 72 pairs instead of 76 runs 1.5 % faster).
inline int balanced_grid(int64_t tiles, int grid) {
  if (tiles < 1 || grid < 1) return grid < 1 ? 1 : grid;
  const int64_t rounds = (tiles + grid - 1) / grid;
  return static_cast<int>((tiles + rounds - 1) / rounds);
}

template <int FMT, int BN, int EPI>
cudaError_t launch_gemm_t(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const GemmParams& p, int grid,
                          cudaStream_t stream) {
  using T = GemmTraits<FMT, BN, EPI>;
  auto kern = gemm_kernel<FMT, BN, EPI>;
  // per instantiation and device; calls from several host threads may set the (idempotent)
  // attribute more than once, never read a torn flag
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  grid = balanced_grid(p.num_tiles, grid);
  kern<<<grid, kThreadsGemm, T::kSmemBytes, stream>>>(tmap_a, tmap_b, p);
  return cudaGetLastError();
}

}  // namespace bsg
