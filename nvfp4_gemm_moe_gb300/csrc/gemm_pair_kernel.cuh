// gemm_pair_kernel.cuh -- the block-scaled GEMM on CTA pairs (tcgen05 cta_group::2), 256 x BN tiles.
//
// A cluster of two CTAs (two SMs) computes one 256 x BN output tile (BN = 256, or 224 / 192 with
// two TMEM accumulators so that the epilogue overlaps the next tile's MMAs; 192 for the RoPE
// projection, one head per CTA, with MXFP8 or bf16 operands), with any of the one-CTA kernel's
// epilogues: each CTA holds 128 rows of A and one BN/2-row half of B in shared memory, and the
// even CTA's MMA warp issues tcgen05.mma.cta_group::2 with M = 256, N = BN (one elected lane per
// instruction), so each SM fetches its own A rows and half of the B tile per K slice instead of
// all of B.  Each CTA's TMEM holds the fp32 accumulator of its
// 128 rows and the scale factors of its A rows and of all BN B rows (its tensor core scales
// every column of its rows).  Roles in each CTA (448 threads, as in the one-CTA kernel):
//   warp 0      TMA producer: its A rows and B half with cta_group::2 tensor loads, which
//               complete bytes on the even CTA's stage barrier (only the even CTA arrives on it,
//               expecting the A/B bytes of both CTAs and its own scale atoms); its scale atoms
//               with bulk copies on its own CTA's barrier (the even CTA's stage barrier, or the
//               odd CTA's own sf_full barrier);
//   warp 1      TMEM allocation in both CTAs; in the even CTA the warp waits until both CTAs'
//               scale factors are in TMEM, issues the pair MMAs and commits to the stage barriers
//               of both CTAs (multicast) and, per tile, to both accumulator barriers;
//   warps 2-9   epilogue on the CTA's own 128 rows (as in the one-CTA kernel), then an arrival
//               on the even CTA's accumulator-empty barrier;
//   warps 10-13 scale-factor stagers: the CTA's atoms from shared memory into its own TMEM with
//               tcgen05.st, then an arrival on the even CTA's sf_ready barrier.
// Arrivals of the odd CTA on the even CTA's barriers are relaxed: they publish nothing the even
// CTA reads through the generic proxy (TMEM stores are complete after tcgen05.wait::st and
// ordered before the arrival by tcgen05.fence::before_thread_sync), and a cluster-scope release
// per arrival costs about a microsecond.  Waits are bounded as in the one-CTA kernel.
#pragma once

#include "gemm_kernel.cuh"

namespace bsg {

template <int FMT, int BN, int EPI = kEpiDense>
struct PairTraits {
  static_assert(BN == 256 || (BN == 224 && FMT == kMXFP8) || (BN == 192 && EPI == kEpiRope && FMT != kNVFP4),
                "pair tile widths");
  static_assert(FMT != kBF16 || EPI == kEpiRope, "bf16 operands: the RoPE projection only");
  static constexpr int kTileMPair = 256;
  static constexpr int kTileN = BN;
  static constexpr int kBHalf = BN / 2;  // B rows each CTA holds
  static constexpr int kElemsPerKTile = FMT == kMXFP8 ? 128 : FMT == kNVFP4 ? 256 : 64;
  static constexpr int kMmaK = FMT == kMXFP8 ? 32 : FMT == kNVFP4 ? 64 : 16;
  static constexpr int kMmasPerStage = 4;
  static constexpr int kAtomsPerStage = FMT == kMXFP8 ? 1 : FMT == kNVFP4 ? 4 : 0;  // bf16: no scales
  // the scale-factor layout fields stage_scale_factors reads: the scales of all BN B rows, from
  // two atom groups, or three when a 224-wide tile starts inside one
  static constexpr bool kSfbAligned = BN % 128 == 0;
  static constexpr int kBRowGroups = kSfbAligned ? BN / 128 : 3;
  static constexpr int kBBlocks = BN / 32;
  static constexpr int kSfbColsPerMma = ((kBBlocks + 3) / 4) * 4;
  static constexpr int kABytes = 128 * kTileKBytes;
  static constexpr int kBBytes = kBHalf * kTileKBytes;
  static constexpr int kSfaBytes = kAtomsPerStage * 512;
  static constexpr int kSfbBytes = kBRowGroups * kAtomsPerStage * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kAcc = BN == 256 ? 1 : 2;  // 224, 192: two accumulators, epilogue overlapped
  // dense raster: groups of M tiles swept along N (measured best: 16 for MXFP8 8192-square
  // batches, 32 for the NVFP4 16384-square GEMM, whose B panels are then read half as often)
  static constexpr int kRasterM = FMT == kNVFP4 ? 32 : 16;
  static constexpr int kSfaCols = kAtomsPerStage * 4;
  static constexpr int kSfbCols = kSfbColsPerMma * kAtomsPerStage;
  static constexpr int kSfStride = kAtomsPerStage == 0 ? 0 : ((kSfaCols + kSfbCols + 15) / 16) * 16;
  static constexpr int kSfBase = kAcc * BN;
  static constexpr int kTmemCols = 512;
  static constexpr int kBarBytes = 1024;
  static constexpr int kOffsetsBytes = 4096;
  static constexpr int kAmaxBytes = 4096;
  // one transpose block per epilogue warp; the grouped bf16-D epilogue on 256-wide tiles stages
  // a C and a D block per warp for its TMA stores
  static constexpr bool kOutTma = EPI == kEpiGroupedBF16 && BN == 256;
  static constexpr int kXposeBlock = kOutTma ? 2 * kXposeBlockBytes : kXposeBlockBytes;
  static constexpr int kXposeBytes = 8 * kXposeBlock;
  // shared-memory ring: as many stages as fit, at most six (five for RoPE tiles)
  static constexpr int kStagesSmem =
      (232448 - 1024 - kBarBytes - kOffsetsBytes - kAmaxBytes - kXposeBytes) / kStageBytes;
  // the RoPE tiles stop at five (measured faster: their epilogue reads the cos / sin rows through
  // L1, which gets the shared memory a sixth stage would take)
  static constexpr int kMaxStages = EPI == kEpiRope ? 5 : 6;
  static constexpr int kStages = kStagesSmem < kMaxStages ? kStagesSmem : kMaxStages;
  static_assert(kStages >= 3, "pipeline depth");
  // TMEM scale-factor slots: one per stage when TMEM has room, else fewer, recycled through the
  // sf_free barriers (the two-accumulator tiles leave room for only four)
  static constexpr int kSfSlotsTmem = kSfStride == 0 ? kStages : (512 - kSfBase) / kSfStride;
  static constexpr int kSfSlots = kSfSlotsTmem < kStages ? kSfSlotsTmem : kStages;
  static constexpr bool kSfRing = kSfSlots < kStages;
  static_assert(kSfSlots >= 3 && kSfBase + kSfSlots * kSfStride <= 512, "TMEM scale-factor slots");
  static constexpr int kSmemBytes =
      1024 + kStages * kStageBytes + kBarBytes + kOffsetsBytes + kAmaxBytes + kXposeBytes;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // M = 256 across the pair (M >> 4 at bit 24), N = BN (N >> 3 at bit 17)
  // kind::f16 (bf16 A and B): fp32 accumulator at bits 4-5, bf16 = 1 at bits 7 and 10
  static constexpr uint32_t kIdesc = (FMT == kMXFP8   ? ((0u << 7) | (0u << 10) | (1u << 23))
                                      : FMT == kNVFP4 ? ((1u << 7) | (1u << 10) | (0u << 23))
                                                      : ((1u << 4) | (1u << 7) | (1u << 10))) |
                                     (static_cast<uint32_t>(kTileN >> 3) << 17) |
                                     (static_cast<uint32_t>(kTileMPair >> 4) << 24);
};

// NM pair MMAs (M = 256) of one stage, issued by the even CTA's MMA warp (all lanes; one elected
// lane issues each instruction); the scale factors
// are in both CTAs' TMEM at sfa_t / sfb_t (layout as in issue_stage).
// idesc and b_step as in issue_stage (N-major B: MXFP8, 256-wide tiles, 128 N per CTA).
template <int FMT, class T, int NM>
__device__ __forceinline__ void issue_stage_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t sfa_t,
                                                 uint32_t sfb_t, uint32_t acc0, uint32_t idesc, uint32_t b_step) {
#pragma unroll
  for (int j = 0; j < NM; ++j) {
    const uint32_t accumulate = j > 0 ? 1u : acc0;
    if (FMT == kBF16) {
      warp_mma_f16_pair(d_tmem, adesc + 2 * j, bdesc + 2 * j, T::kIdesc, accumulate);
    } else if (FMT == kMXFP8) {
      warp_mma_mxf8f6f4_pair(d_tmem, adesc + 2 * j, bdesc + b_step * j, idesc | (j << 29) | (j << 4), sfa_t,
                             sfb_t, accumulate);
    } else {
      warp_mma_mxf4nvf4_pair(d_tmem, adesc + 2 * j, bdesc + 2 * j, T::kIdesc, sfa_t + j * 4,
                             sfb_t + j * T::kSfbColsPerMma, accumulate);
    }
  }
}

template <int FMT, int BN, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsGemm, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_d,
                     const __grid_constant__ GemmParams p) {
  using T = PairTraits<FMT, BN, EPI>;
  constexpr int S = T::kStages;
  constexpr int ACC = T::kAcc;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* s_a = smem;
  uint8_t* s_b = s_a + S * T::kABytes;
  uint8_t* s_sfa = s_b + S * T::kBBytes;
  uint8_t* s_sfb = s_sfa + S * T::kSfaBytes;
  uint8_t* s_bar = s_sfb + S * T::kSfbBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_bar);  // even CTA: A/B of both CTAs + its scales
  uint64_t* empty = full + S;
  uint64_t* sf_full = empty + S;                        // odd CTA: its own scale atoms
  uint64_t* sf_ready = sf_full + S;                     // even CTA: both CTAs' scales in TMEM
  uint64_t* tmem_full = sf_ready + S;
  uint64_t* tmem_empty = tmem_full + ACC;
  uint64_t* drain = tmem_empty + ACC;
  uint64_t* sf_free = drain + 1;                        // TMEM scale slot free again (MMAs done)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sf_free + T::kSfSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* bad_flag = const_cast<int*>(abort_flag) + 1;
  int32_t* s_offs = reinterpret_cast<int32_t*>(s_bar + T::kBarBytes);
  float* s_amax = reinterpret_cast<float*>(s_bar + T::kBarBytes + T::kOffsetsBytes);
  uint8_t* s_xpose = s_bar + T::kBarBytes + T::kOffsetsBytes + T::kAmaxBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);  // the even CTA's expect_tx arrival; both CTAs' A/B loads complete bytes on it
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 1);
      mbar_init(&sf_ready[s], 8);  // four stagers in each CTA
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(&tmem_full[a], 1);
      mbar_init(&tmem_empty[a], 16);  // eight epilogue warps in each CTA (used in the even CTA)
    }
    mbar_init(drain, 1);
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
    tmem_alloc_pair(tmem_slot, T::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    if (T::kOutTma && p.out_tma) {
      prefetch_tmap(&tmap_c);
      prefetch_tmap(&tmap_d);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool bad = *bad_flag != 0;
  const ErrSink es{p.err, p.epoch};
  if (threadIdx.x == 0) mark_call(es);
  if ((*bad_flag & 1) && blockIdx.x == 0 && threadIdx.x == 0) report_error(es, kErrBadOffsets);
  const int pair_id = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    // warp-collective, as in the one-CTA kernel
    if (!bad) {
      uint32_t stage = 0, phase = 0;
      uint64_t issued = 0;
      bool ok = true;
      int fenced_l = -1;  // expert whose global tensor map the warp has acquired
      const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);
      for (int t = pair_id; ok && t < p.num_tiles; t += num_pairs) {
        const TileCoord tc = decode_tile<EPI, 256, T::kRasterM>(p, t, s_offs);
        const int a_batch = epi_is_grouped(EPI) ? 0 : tc.l;
        const int a_row = tc.mt * 256 + static_cast<int>(rank) * 128;
        const int b_row = tc.nt * BN + static_cast<int>(rank) * T::kBHalf;
        const int sfa_group = min(tc.mt * 2 + static_cast<int>(rank), p.sfa_mt - 1);
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
          // The odd CTA cannot load stage s of the next round before this round's phase has
          // completed (its empty barrier is released after the MMAs that needed that phase), so
          // its A/B bytes always land in the phase the even CTA's arrival belongs to.
          uint64_t* sf_bar = leader ? &full[stage] : &sf_full[stage];
          if (leader) warp_arrive_expect_tx(&full[stage], 2 * (T::kABytes + T::kBBytes) + sf_bytes);
          else warp_arrive_expect_tx(&sf_full[stage], sf_bytes);
          const uint32_t fbar = full0 + stage * 8;
          warp_tma_load_3d_pair(s_a + stage * T::kABytes, &tmap_a, fbar, kt * kTileKBytes, a_row, a_batch);
          if (FMT == kMXFP8 && BN == 256 && p.b_mn_major)  // N-major B: 128 bytes of N x 128 rows of K
            warp_tma_load_3d_pair(s_b + stage * T::kBBytes, bmap, fbar, b_row, kt * T::kElemsPerKTile,
                                  b_batch);
          else
            warp_tma_load_3d_pair(s_b + stage * T::kBBytes, bmap, fbar, kt * kTileKBytes, b_row, b_batch);
          if constexpr (FMT != kBF16) {
            const uint8_t* sfa_src =
                p.sfa + ((static_cast<uint64_t>(a_batch) * p.sfa_mt + sfa_group) * p.sf_kt +
                         static_cast<uint64_t>(kt) * T::kAtomsPerStage) * 512;
            warp_bulk_load(s_sfa + stage * T::kSfaBytes, sfa_src, atoms * 512, sf_bar);
#pragma unroll
            for (int g = 0; g < T::kBRowGroups; ++g) {
              // a 128-row group past N reuses the last group's (finite) scales: its B rows are zero
              const int rb = min((tc.nt * BN) / 128 + g, p.sfb_mt - 1);
              const uint8_t* sfb_src = sfb_base + (static_cast<uint64_t>(rb) * p.sf_kt +
                                                   static_cast<uint64_t>(kt) * T::kAtomsPerStage) * 512;
              warp_bulk_load(s_sfb + stage * T::kSfbBytes + g * T::kAtomsPerStage * 512, sfb_src, atoms * 512,
                             sf_bar);
            }
          }
          ++issued;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // drain: every stage barrier this CTA's copies complete on must see them land (the even
        // CTA's stage barriers count both CTAs' A/B loads)
        uint64_t* bars = leader ? full : sf_full;
        for (int s = 0; s < S; ++s) {
          if (issued > static_cast<uint64_t>(s)) {
            const uint32_t ph = (s < static_cast<int>(stage)) ? phase : (phase ^ 1u);
            wait_bounded_plain(&bars[s], ph);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && !bad) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, fslot = 0;
      bool ok = true;
      const uint32_t a_base = smem_u32(s_a), b_base = smem_u32(s_b);
      const uint32_t b_mn = (FMT == kMXFP8 && BN == 256 && p.b_mn_major) ? 1u : 0u;
      const uint32_t idesc = T::kIdesc | (b_mn << 16);
      const uint32_t b_step = b_mn ? 256u : 2u;
      const int last_mmas =
          min(T::kMmasPerStage, (p.k - (p.k_tiles - 1) * T::kElemsPerKTile + T::kMmaK - 1) / T::kMmaK);
      for (int t = pair_id; ok && t < p.num_tiles; t += num_pairs) {
        // outcomes of waits are made warp-uniform before they steer the warp-collective issue
        if (!__all_sync(0xffffffffu, wait_bounded(&tmem_empty[acc], acc_phase ^ 1u, abort_flag, es))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          // warp-uniform control flow and operands, failures acted on per tile (as in the
          // one-CTA kernel); sf_ready implies the stage's A/B data landed (the even CTA's
          // stagers waited for it)
          // bf16 operands carry no scales: the even CTA's stage barrier (both CTAs' A/B bytes) is
          // all the MMAs need
          ok &= wait_bounded(FMT == kBF16 ? &full[stage] : &sf_ready[stage], phase, abort_flag, es);
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + T::kSfBase + fslot * T::kSfStride;
          const uint32_t sfb_t = sfa_t + T::kSfaCols;
          const uint64_t adesc = smem_desc(a_base + stage * T::kABytes, 16, 1024, kSwizzle128B);
          const uint64_t bdesc = smem_desc(b_base + stage * T::kBBytes, 16, 1024, kSwizzle128B);
          const uint32_t acc0 = kt > 0 ? 1u : 0u;
          const int n_mma = kt == p.k_tiles - 1 ? last_mmas : T::kMmasPerStage;
          // the whole warp issues; elect.sync picks the lane (warp-uniform branches only)
          if (n_mma == T::kMmasPerStage) {
            issue_stage_pair<FMT, T, T::kMmasPerStage>(d_tmem, adesc, bdesc, sfa_t, sfb_t, acc0, idesc, b_step);
          } else {
            if (n_mma == 1) issue_stage_pair<FMT, T, 1>(d_tmem, adesc, bdesc, sfa_t, sfb_t, acc0, idesc, b_step);
            if (n_mma == 2) issue_stage_pair<FMT, T, 2>(d_tmem, adesc, bdesc, sfa_t, sfb_t, acc0, idesc, b_step);
            if (n_mma == 3) issue_stage_pair<FMT, T, 3>(d_tmem, adesc, bdesc, sfa_t, sfb_t, acc0, idesc, b_step);
          }
          warp_commit_pair_multicast(&empty[stage], 0x3);
          if (T::kSfRing) warp_commit_pair_multicast(&sf_free[fslot], 0x3);
          if (++stage == S) { stage = 0; phase ^= 1u; }
          if (++fslot == T::kSfSlots) fslot = 0;
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        warp_commit_pair_multicast(&tmem_full[acc], 0x3);
        if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) {
        __syncwarp();
        warp_commit_pair(drain);
        if (lane == 0) wait_bounded_plain(drain, 0);
        __syncwarp();
      }
    }
  } else if (warp >= 10) {
    // ------------------------------------------------------------ scale-factor stagers (both CTAs)
    const uint32_t quad_lanes = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ready0 = mapa_shared(smem_u32(&sf_ready[0]), 0);
    uint64_t* landed = leader ? full : sf_full;
    uint32_t stage = 0, phase = 0, fslot = 0, fphase = 0;
    bool ok = FMT != kBF16;  // bf16 operands have no scale factors to stage
    for (int t = pair_id; !bad && ok && t < p.num_tiles; t += num_pairs) {
      const TileCoord tc = decode_tile<EPI, 256, T::kRasterM>(p, t, s_offs);
      const int b_blk0 = ((tc.nt * BN) >> 5) & 3;  // the tile's first 32-row block within its first atom
      for (int kt = 0; kt < p.k_tiles; ++kt) {
        ok &= wait_bounded(&landed[stage], phase, abort_flag, es);
        // with fewer TMEM slots than stages, the slot's previous MMAs must have completed (with one
        // slot per stage the refill of the stage already waited for them)
        if (T::kSfRing) ok &= wait_bounded(&sf_free[fslot], fphase ^ 1u, abort_flag, es);
        tc_fence_after();
        const uint32_t sfa_t = tmem_base + quad_lanes + T::kSfBase + fslot * T::kSfStride;
        // the wide B-scale gather measured faster for the RoPE tiles, slower for the dSwiGLU ones
        if constexpr (FMT != kBF16)
          stage_scale_factors<T, EPI == kEpiRope>(s_sfa + stage * T::kSfaBytes, s_sfb + stage * T::kSfbBytes, sfa_t,
                                                  sfa_t + T::kSfaCols, lane, b_blk0);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&sf_ready[stage]);
          else mbar_arrive_cluster_relaxed(ready0 + stage * 8);
        }
        if (++stage == S) { stage = 0; phase ^= 1u; }
        if (++fslot == T::kSfSlots) { fslot = 0; fphase ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 2..9 (both CTAs)
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    float run_max = 0.0f, run_max2 = 0.0f;
    int run_expert = -1;
    uint32_t acc = 0, acc_phase = 0;
    const float nc = epi_has_fp8_d(EPI) ? *p.norm_const : 1.0f;
    const uint32_t empty_leader = mapa_shared(smem_u32(&tmem_empty[0]), 0);
    for (int t = pair_id; !bad && t < p.num_tiles; t += num_pairs) {
      const TileCoord tc = decode_tile<EPI, 256, T::kRasterM>(p, t, s_offs);
      const int row = tc.mt * 256 + static_cast<int>(rank) * 128 + quad * 32 + lane;
      if constexpr (epi_is_dswiglu(EPI)) prefetch_dswiglu_c<BN>(p, row, tc.nt * BN, half, 2);
      // warp-uniform outcome: the epilogues use whole-warp shuffles, syncs and elected copies
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
      // the arrival publishes no memory the even CTA reads, so it needs no release
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(empty_leader + acc * 8);
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
      } else if (T::kOutTma && p.out_tma) {
        uint8_t* blk = s_xpose + (warp - 2) * T::kXposeBlock;
        epilogue_tile_grouped_tma<BN>(p, row, tc.nt * BN, tmem_acc, lane, alpha_g, prob_r, run_max, half, 2, blk,
                                      blk + kXposeBlockBytes, &tmap_c, &tmap_d, release);
      } else {
        epilogue_tile<BN, EPI>(p, tc.l, row, tc.nt * BN, tmem_acc, lane, alpha_g, prob_r, nc, run_max, half, 2,
                               s_amax + (warp - 2) * 32, s_xpose + (warp - 2) * T::kXposeBlock);
        release();
      }
      if (++acc == ACC) { acc = 0; acc_phase ^= 1u; }
    }
    // the TMA stores have completed (their staging blocks are freed with the CTA)
    if (T::kOutTma && p.out_tma) warp_bulk_wait_all<false>();
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
  cluster_sync();  // no remote arrival or MMA into this CTA's TMEM is still pending
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
    tmem_dealloc_pair(tmem_base, T::kTmemCols);
  }
}

// Launches at most as many CTA pairs as can be resident at once (a cluster must fit in one GPC,
// so fewer than #SMs / 2 pairs may fit); `max_pairs` is the caller's upper bound.
template <int FMT, int BN, int EPI>
cudaError_t launch_gemm_pair_t(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int max_pairs,
                               cudaStream_t stream, const CUtensorMap* tc = nullptr,
                               const CUtensorMap* td = nullptr) {
  using T = PairTraits<FMT, BN, EPI>;
  auto kern = gemm_pair_kernel<FMT, BN, EPI>;
  static std::atomic<int> resident_pairs[64];  // per device; 0 = not queried yet
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int resident = resident_pairs[dev].load(std::memory_order_acquire);
  if (resident == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreadsGemm, 1, 1);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    resident = clusters > 0 ? clusters : 1;
    resident_pairs[dev].store(resident, std::memory_order_release);
  }
  int pairs = max_pairs < resident ? max_pairs : resident;
  if (pairs < 1) pairs = 1;
  // as few pairs as take the tiles in the same number of rounds
  pairs = balanced_grid(p.num_tiles, pairs);
  // output maps only for the TMA-store epilogue; otherwise the kernel never reads them
  kern<<<2 * pairs, kThreadsGemm, T::kSmemBytes, stream>>>(ta, tb, tc ? *tc : ta, td ? *td : ta, p);
  return cudaGetLastError();
}

}  // namespace bsg
