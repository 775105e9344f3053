// gemm_pair_kernel.cuh -- the block-scaled GEMM on CTA pairs (tcgen05 cta_group::2), 256 x 256 tiles.
//
// A cluster of two CTAs on the two SMs of a TPC computes one 256 x 256 output tile: each CTA
// holds 128 rows of A and 128 rows (one half) of B in its shared memory, and one thread of the
// even CTA issues tcgen05.mma.cta_group::2 with M = 256, N = 256, so each B tile is fetched from
// L2 once for 256 rows of A.  Each CTA's TMEM holds the fp32 accumulator of its own 128 rows and
// the scale factors of all 256 B rows (its tensor core scales every column of its rows).
//   warp 0     TMA producer in each CTA: its A / B halves and scale-factor atoms.  The loads of
//              both CTAs complete bytes on the even CTA's stage barrier (cta_group::2 loads); only
//              the even CTA arrives on that barrier, expecting the bytes of both CTAs, with a
//              CTA-scope arrive (a cluster-scope release per stage costs about a microsecond);
//   warp 1     TMEM allocation in both CTAs (collective); in the even CTA one thread copies the
//              scale factors into both CTAs' TMEM, issues the MMAs, and commits to the stage and
//              accumulator barriers of both CTAs (multicast);
//   warps 2-5  epilogue in each CTA on its own rows, then a relaxed arrival on the even CTA's
//              accumulator-empty barrier.
// Stages: 6 (MXFP8) or 5 (NVFP4) of 128 bytes of K.  Waits are bounded as in the 1-CTA kernel.
#pragma once

#include "gemm_kernel.cuh"

namespace bsg {

constexpr int kThreadsPair = 192;  // producer, MMA issuer, four epilogue warps

template <int FMT>
struct PairTraits {
  static constexpr int kTileMPair = 256;
  static constexpr int kTileN = 256;
  static constexpr int kElemsPerKTile = FMT == kMXFP8 ? 128 : 256;
  static constexpr int kMmaK = FMT == kMXFP8 ? 32 : 64;
  static constexpr int kMmasPerStage = 4;
  static constexpr int kAtomsPerStage = FMT == kMXFP8 ? 1 : 4;
  static constexpr int kSfbGroups = 2;  // scale factors of both 128-row halves of the B tile
  static constexpr int kABytes = 128 * kTileKBytes;
  static constexpr int kBBytes = 128 * kTileKBytes;
  static constexpr int kSfaBytes = kAtomsPerStage * 512;
  static constexpr int kSfbBytes = kSfbGroups * kAtomsPerStage * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kStages = FMT == kMXFP8 ? 6 : 5;
  static constexpr int kSfaCols = kAtomsPerStage * 4;
  static constexpr int kSfbCols = kSfbGroups * kAtomsPerStage * 4;
  static constexpr int kSfStride = ((kSfaCols + kSfbCols + 15) / 16) * 16;
  static constexpr int kSfBase = kTileN;  // one accumulator of 256 columns
  static constexpr int kTmemCols = 512;
  static_assert(kSfBase + kStages * kSfStride <= 512, "TMEM budget");
  static constexpr int kBarBytes = 1024;
  static constexpr int kOffsetsBytes = 4096;
  static constexpr int kAmaxBytes = 4096;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes + kOffsetsBytes + kAmaxBytes;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // M = 256 across the pair (M >> 4 at bit 24), N = 256 (N >> 3 at bit 17)
  static constexpr uint32_t kIdesc = (FMT == kMXFP8 ? ((0u << 7) | (0u << 10) | (1u << 23))
                                                    : ((1u << 7) | (1u << 10) | (0u << 23))) |
                                     (static_cast<uint32_t>(kTileN >> 3) << 17) |
                                     (static_cast<uint32_t>(kTileMPair >> 4) << 24);
};

// One stage's scale-factor copies into both CTAs' TMEM and NM pair MMAs (M = 256), issued by one
// thread of the even CTA (layout as in issue_stage; each CTA holds the scales of all B rows).
template <int FMT, class T, int NM>
__device__ __forceinline__ void issue_stage_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t sfa_t,
                                                 uint32_t sfb_t, uint32_t sfa_s, uint32_t sfb_s, uint32_t acc0) {
  constexpr int kAtoms = FMT == kMXFP8 ? 1 : NM;
#pragma unroll
  for (int a = 0; a < kAtoms; ++a) {
    tc_cp_32x128b_warpx4_pair(sfa_t + a * 4, smem_desc(sfa_s + a * 512, 0, 128, kSwizzleNone));
#pragma unroll
    for (int g = 0; g < T::kSfbGroups; ++g)
      tc_cp_32x128b_warpx4_pair(sfb_t + (a * T::kSfbGroups + g) * 4,
                                smem_desc(sfb_s + (g * T::kAtomsPerStage + a) * 512, 0, 128, kSwizzleNone));
  }
#pragma unroll
  for (int j = 0; j < NM; ++j) {
    const uint32_t accumulate = j > 0 ? 1u : acc0;
    if (FMT == kMXFP8) {
      tc_mma_mxf8f6f4_pair(d_tmem, adesc + 2 * j, bdesc + 2 * j, T::kIdesc | (j << 29) | (j << 4), sfa_t, sfb_t,
                           accumulate);
    } else {
      tc_mma_mxf4nvf4_pair(d_tmem, adesc + 2 * j, bdesc + 2 * j, T::kIdesc, sfa_t + j * 4,
                           sfb_t + j * T::kSfbGroups * 4, accumulate);
    }
  }
}

template <int FMT, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsPair, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                     const __grid_constant__ GemmParams p) {
  using T = PairTraits<FMT>;
  constexpr int S = T::kStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* s_a = smem;
  uint8_t* s_b = s_a + S * T::kABytes;
  uint8_t* s_sfa = s_b + S * T::kBBytes;
  uint8_t* s_sfb = s_sfa + S * T::kSfaBytes;
  uint8_t* s_bar = s_sfb + S * T::kSfbBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_bar);
  uint64_t* empty = full + S;
  uint64_t* tmem_full = empty + S;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* drain = tmem_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bad_flag = const_cast<int*>(abort_flag) + 1;
  int32_t* s_offs = reinterpret_cast<int32_t*>(s_bar + T::kBarBytes);
  float* s_amax = reinterpret_cast<float*>(s_bar + T::kBarBytes + T::kOffsetsBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);  // the even CTA's expect_tx arrival; both CTAs' loads complete bytes on it
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 8);  // four epilogue warps in each CTA (used in the even CTA)
    mbar_init(drain, 1);
    *abort_flag = 0;
    *bad_flag = 0;
    fence_mbar_init();
  }
  if (EPI != kEpiDense) {
    for (int i = threadIdx.x; i < 1024; i += kThreadsPair) s_amax[i] = 0.0f;
  } else if (threadIdx.x == 0) {
    s_amax[0] = 0.0f;
  }
  __syncthreads();
  if (EPI != kEpiDense) {
    for (int i = threadIdx.x; i < p.l; i += kThreadsPair) {
      const int32_t o = p.offsets[i];
      const int32_t prev = i == 0 ? 0 : p.offsets[i - 1];
      s_offs[i] = o;
      if ((o & 255) != 0 || o < prev || o > p.m || (i == p.l - 1 && o != p.m)) atomicOr(bad_flag, 1);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, T::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    prefetch_tmap(&tmap_sfa);
    prefetch_tmap(&tmap_sfb);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool bad = *bad_flag != 0;
  if (bad && blockIdx.x == 0 && threadIdx.x == 0) report_error(p.err, kErrBadOffsets);
  const int pair_id = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0 && !bad) {
      uint32_t stage = 0, phase = 0;
      uint64_t issued = 0;
      bool ok = true;
      const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);
      for (int t = pair_id; ok && t < p.num_tiles; t += num_pairs) {
        const TileCoord tc = decode_tile<EPI, 256>(p, t, s_offs);
        const int a_batch = EPI == kEpiDense ? tc.l : 0;
        const int a_row = tc.mt * 256 + static_cast<int>(rank) * 128;
        const int b_row = tc.nt * 256 + static_cast<int>(rank) * 128;
        const int sfa_group = min(tc.mt * 2 + static_cast<int>(rank), p.sfa_mt - 1);
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.err)) { ok = false; break; }
          const uint32_t fbar = full0 + stage * 8;
          // The odd CTA cannot load stage s of the next round before this round's phase has
          // completed (its empty barrier is released after the MMAs that needed that phase), so
          // its bytes always land in the phase the even CTA's arrival belongs to.
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * T::kStageBytes);
          tma_load_3d_pair(s_a + stage * T::kABytes, &tmap_a, fbar, kt * kTileKBytes, a_row, a_batch);
          tma_load_3d_pair(s_b + stage * T::kBBytes, &tmap_b, fbar, kt * kTileKBytes, b_row, tc.l);
          tma_load_2d_pair(s_sfa + stage * T::kSfaBytes, &tmap_sfa, fbar, 0,
                           (a_batch * p.sfa_mt + sfa_group) * p.sf_kt + kt * T::kAtomsPerStage);
#pragma unroll
          for (int g = 0; g < T::kSfbGroups; ++g) {
            // a 128-row group past N reuses the last group's (finite) scales: its B rows are zero
            const int grp = min(tc.nt * 2 + g, p.sfb_mt - 1);
            tma_load_2d_pair(s_sfb + stage * T::kSfbBytes + g * T::kAtomsPerStage * 512, &tmap_sfb, fbar, 0,
                             (tc.l * p.sfb_mt + grp) * p.sf_kt + kt * T::kAtomsPerStage);
          }
          ++issued;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok && leader) {
        // the even CTA's stage barriers count both CTAs' loads: wait for every stage issued
        for (int s = 0; s < S; ++s) {
          if (issued > static_cast<uint64_t>(s)) {
            const uint32_t ph = (s < static_cast<int>(stage)) ? phase : (phase ^ 1u);
            wait_bounded_plain(&full[s], ph);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && !bad) {
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t a_base = smem_u32(s_a), b_base = smem_u32(s_b);
      const uint32_t sfa_base = smem_u32(s_sfa), sfb_base = smem_u32(s_sfb);
      for (int t = pair_id; ok && t < p.num_tiles; t += num_pairs) {
        if (!wait_bounded(tmem_empty, acc_phase ^ 1u, abort_flag, p.err)) { ok = false; break; }
        tc_fence_after();
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          // warp-uniform control flow and operands, failures acted on per tile (as in the 1-CTA
          // kernel)
          ok &= wait_bounded(&full[stage], phase, abort_flag, p.err);
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + T::kSfBase + stage * T::kSfStride;
          const uint32_t sfb_t = sfa_t + T::kSfaCols;
          const uint32_t sfa_s = sfa_base + stage * T::kSfaBytes;
          const uint32_t sfb_s = sfb_base + stage * T::kSfbBytes;
          const uint64_t adesc = smem_desc(a_base + stage * T::kABytes, 16, 1024, kSwizzle128B);
          const uint64_t bdesc = smem_desc(b_base + stage * T::kBBytes, 16, 1024, kSwizzle128B);
          const uint32_t acc0 = kt > 0 ? 1u : 0u;
          const int n_mma = min(T::kMmasPerStage, (p.k - kt * T::kElemsPerKTile + T::kMmaK - 1) / T::kMmaK);
          if (lane == 0) {
            if (n_mma == T::kMmasPerStage) {
              issue_stage_pair<FMT, T, T::kMmasPerStage>(tmem_base, adesc, bdesc, sfa_t, sfb_t, sfa_s, sfb_s, acc0);
            } else {
              if (n_mma == 1) issue_stage_pair<FMT, T, 1>(tmem_base, adesc, bdesc, sfa_t, sfb_t, sfa_s, sfb_s, acc0);
              if (n_mma == 2) issue_stage_pair<FMT, T, 2>(tmem_base, adesc, bdesc, sfa_t, sfb_t, sfa_s, sfb_s, acc0);
              if (n_mma == 3) issue_stage_pair<FMT, T, 3>(tmem_base, adesc, bdesc, sfa_t, sfb_t, sfa_s, sfb_s, acc0);
            }
            tc_commit_pair_multicast(&empty[stage], 0x3);
          }
          __syncwarp();
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) tc_commit_pair_multicast(tmem_full, 0x3);
        __syncwarp();
        acc_phase ^= 1u;
      }
      if (!ok) {
        if (lane == 0) {
          tc_commit_pair(drain);
          wait_bounded_plain(drain, 0);
        }
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 2..5 (both CTAs)
    const int quad = warp & 3;
    float run_max = 0.0f;
    int run_expert = -1;
    uint32_t acc_phase = 0;
    const float nc = (EPI == kEpiGroupedFP8) ? *p.norm_const : 1.0f;
    const uint32_t empty_leader = mapa_shared(smem_u32(tmem_empty), 0);
    for (int t = pair_id; !bad && t < p.num_tiles; t += num_pairs) {
      const TileCoord tc = decode_tile<EPI, 256>(p, t, s_offs);
      if (!wait_bounded(tmem_full, acc_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const int row = tc.mt * 256 + static_cast<int>(rank) * 128 + quad * 32 + lane;
      float alpha_g = 1.0f, prob_r = 0.0f;
      if (EPI != kEpiDense) {
        alpha_g = p.alpha[tc.l];
        prob_r = p.prob[row];
        if (tc.l != run_expert) {
          if (run_expert >= 0) {
            float v = run_max;
            for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0 && EPI == kEpiGroupedBF16) atomic_max_nonneg(&s_amax[run_expert], v);
          }
          run_expert = tc.l;
          run_max = 0.0f;
        }
      }
      epilogue_tile<256, EPI>(p, tc.l, row, tc.nt * 256, tmem_base + (static_cast<uint32_t>(quad * 32) << 16), lane,
                              alpha_g, prob_r, nc, run_max, 0, 1, s_amax + (warp - 2) * 32);
      tc_fence_before();
      __syncwarp();
      // the arrival publishes no memory the even CTA reads, so it needs no release
      if (lane == 0) mbar_arrive_cluster_relaxed(empty_leader);
      acc_phase ^= 1u;
    }
    float v = run_max;
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) {
      if (EPI == kEpiDense) atomic_max_nonneg(&s_amax[0], v);
      else if (EPI == kEpiGroupedBF16 && run_expert >= 0) atomic_max_nonneg(&s_amax[run_expert], v);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrival or MMA into this CTA's TMEM is still pending
  if (!bad && *abort_flag == 0) {
    if (EPI == kEpiDense) {
      if (threadIdx.x == 0 && s_amax[0] > 0.0f) atomic_max_nonneg(p.amax, s_amax[0]);
    } else if (EPI == kEpiGroupedBF16) {
      for (int g = threadIdx.x; g < p.l; g += kThreadsPair)
        if (s_amax[g] > 0.0f) atomic_max_nonneg(&p.amax[g], s_amax[g]);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, T::kTmemCols);
  }
}

// Launches at most as many CTA pairs as can be resident at once (a cluster must fit in one GPC,
// so fewer than #SMs / 2 pairs may fit); `max_pairs` is the caller's upper bound.
template <int FMT, int EPI>
cudaError_t launch_gemm_pair_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsfa,
                               const CUtensorMap& tsfb, const GemmParams& p, int max_pairs, cudaStream_t stream) {
  using T = PairTraits<FMT>;
  auto kern = gemm_pair_kernel<FMT, EPI>;
  static int resident_pairs[64] = {};  // per device; 0 = not queried yet
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (resident_pairs[dev] == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreadsPair, 1, 1);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    resident_pairs[dev] = clusters > 0 ? clusters : 1;
  }
  int pairs = max_pairs < resident_pairs[dev] ? max_pairs : resident_pairs[dev];
  if (pairs < 1) pairs = 1;
  kern<<<2 * pairs, kThreadsPair, T::kSmemBytes, stream>>>(ta, tb, tsfa, tsfb, p);
  return cudaGetLastError();
}

}  // namespace bsg
