// gemm_kernels_pair.cuh -- the persistent GEMM on CTA pairs (tcgen05
// cta_group::2): a cluster of two CTAs on the two SMs of a TPC computes one
// 256 x BN output tile.
//
//   * Each CTA stages its own 128 rows of A and its own half (BN/2 rows) of
//     B per k-block, so each SM streams half the B traffic of a 128 x BN
//     single-CTA tile for the same MMA work, and a stage is 16 KB + BN*64 B
//     (6 stages fit beside the epilogue staging).
//   * The even CTA's MMA thread issues tcgen05.mma.cta_group::2 (M = 256);
//     the hardware reads A and B from both CTAs' shared memory at the same
//     offsets and writes D rows 0..127 to the even CTA's TMEM and rows
//     128..255 to the odd CTA's TMEM.
//   * Both producers count their TMA bytes on the even CTA's `full` barrier
//     (which expects the pair's total); the MMA completion is multicast to
//     both CTAs' `empty` and `acc_full` barriers; both CTAs' epilogue warps
//     arrive on the even CTA's `acc_empty` (8 arrivals).
//   * Gate/up: the even CTA stages the Wg tile and the odd CTA the Wu tile,
//     so one MMA of N = 256 yields gate (columns 0..127) and up (128..255)
//     for all 256 rows.
//
// The epilogue, the bounded waits and the tile order are those of the
// single-CTA kernel (gemm_kernels.cuh).
#pragma once

#include "gemm_kernels.cuh"
#include "rms_norm.cuh"

namespace gb3 {

constexpr int kPairBM = 256;  // tile rows of a CTA pair

// The normalisation of the activation that the gate/up kernel runs before its
// GEMM when instantiated with NORM != 0 ("Tiles and shared memory", section
// "A complete kernel"): Xn = rms_norm(X, G, eps) in BF16, written to the
// buffer its A operand map reads.  NORM selects the row geometry the
// standalone normalisation would use for this row length (1: one warp and 4
// cached vectors per lane; 2: two warps of 8), so Xn has the same bits.
struct NormParams {
  const void* X;
  long long ldx;
  const float* G;
  float eps;
  void* Xn;
  long long ldxn;
  int rows, D;
  unsigned int* sync;  // grid barrier counters [arrivals, departures], zero between launches
};

// Grid-wide barrier of a cooperative launch, run by thread 0 of every CTA:
// arrive (release: the CTA's writes, fenced before, are visible first), wait
// (acquire, bounded) until all gridDim.x CTAs have arrived, then count the
// departure; the last CTA to leave resets both counters for the next launch.
// On timeout the CTA's abort flag and the device status word are set and
// false is returned (the counters are then cleared by the host when it reads
// the status).
__device__ __noinline__ bool grid_sync_bounded(unsigned int* sync, volatile int* abort_flag) {
  __threadfence();
  atomicAdd(&sync[0], 1u);
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    unsigned int arrived;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(arrived) : "l"(sync) : "memory");
    if (arrived >= gridDim.x) break;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      record_timeout(SITE_GRID_SYNC);
      return false;
    }
    __nanosleep(64);
  }
  if (atomicAdd(&sync[1], 1u) == gridDim.x - 1) {
    sync[0] = 0;
    sync[1] = 0;
  }
  return true;
}

// RING: the epilogue reads C through a ring of kRingSlots staging slots per
// warp (epilogue_tile_ring), each slot with its own barrier.
template <int BN, int STAGES, int EPI, bool RING = false>
struct PairCfg {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "tile width");
  static constexpr int kABytes = 128 * kBK * 2;       // this CTA's 128 rows of A
  static constexpr int kBBytes = (BN / 2) * kBK * 2;  // this CTA's half of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static_assert(kStageBytes % 1024 == 0, "stages must keep the 1024-byte swizzle phase");
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kSlots = RING ? kRingSlots : kStagingPerWarp;  // staging slots per warp
  static constexpr int kStagingBytes = kEpiWarps * kSlots * kStageBox;
  static constexpr int kBarOffset = kRingBytes + kStagingBytes;
  // full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain, then with
  // RING one barrier per staging slot of each epilogue warp
  static constexpr int kNumBars = 2 * STAGES + 5 + (RING ? kEpiWarps * kRingSlots : 0);
  static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
  static constexpr int kOutCols = (EPI == EPI_GATE_UP) ? BN / 2 : BN;
  static_assert(!RING || EPI != EPI_GATE_UP, "the gate/up epilogue reads no C");
  static constexpr int kAccStride = 256;
  static constexpr int kTmemCols = 512;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int BN, int STAGES, int EPI, bool STATS = false, bool RING = false, int NORM = 0>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmB2,
                     const __grid_constant__ CUtensorMap tmOut, const TileParams p,
                     const RowStatsParams rs, const NormParams nrm) {
  using Cfg = PairCfg<BN, STAGES, EPI, RING>;
  static_assert(NORM == 0 || EPI == EPI_GATE_UP, "the normalised activation feeds gate/up");
  // Strip units (TileParams::strip_tiles) exist only for plain GEMMs of 256-column
  // tiles; each CTA then loads kPairStripN / 2 rows of B through tmB2.
  constexpr bool kStrips = BN == 256 && EPI != EPI_GATE_UP && !STATS;
  constexpr int kStripBBytes = (kPairStripN / 2) * kBK * 2;
  if (!launch_smem_ok(Cfg::kSmemBytes)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOffset);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

  if constexpr (NORM != 0) {
    // Phase 1: this CTA's contiguous share of the rows of X, normalised into
    // Xn.  The rows (and the gains) come into the still unused pipeline
    // shared memory by bulk copies, as many rows per batch as fit, so that a
    // whole batch is in flight at once; the row groups (1 or 2 warps, the
    // standalone normalisation's geometry, two rows at a time) normalise each
    // row over its copy and send it to Xn with one bulk copy.  Those copies
    // have completed before the grid barrier below, after which every CTA's
    // TMA loads read Xn.
    constexpr int kRW = NORM == 2 ? 2 : 1;
    constexpr int kGroups = (kThreads / 32) / kRW;
    constexpr int kSlots = 3;  // chunks of rows in flight
    __shared__ float norm_partial[2][2][kThreads / 32];
    __shared__ __align__(8) uint64_t chunk_bar[kSlots];
    const uint32_t row_bytes = (static_cast<uint32_t>(nrm.D) * 2 + 15u) & ~15u;
    const uint32_t g_bytes = static_cast<uint32_t>(nrm.D) * 4;  // the gains, first
    const int per_cta = (nrm.rows + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
    const int r0 = min(nrm.rows, static_cast<int>(blockIdx.x) * per_cta);
    const int r1 = min(nrm.rows, r0 + per_cta);
    // Rows per chunk: kSlots chunks fit in the pipeline region beside the
    // gains (the host takes this path only for rows of whole 16-byte vectors
    // of which kSlots fit there with the gains).
    const uint32_t room = static_cast<uint32_t>(Cfg::kBarOffset);
    const int chunk = room > g_bytes ? static_cast<int>((room - g_bytes) / row_bytes) / kSlots : 0;
    const int nchunks = chunk > 0 ? (r1 - r0 + chunk - 1) / chunk : 0;
    auto slot_addr = [&](int c) {
      return sbase + g_bytes + static_cast<uint32_t>((c % kSlots) * chunk) * row_bytes;
    };
    auto load_chunk = [&](int c) {  // thread 0: chunk c's rows (and, first, the gains)
      const int first = r0 + c * chunk, n = min(chunk, r1 - first);
      const uint32_t bar = smem_u32(&chunk_bar[c % kSlots]);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * row_bytes + (c == 0 ? g_bytes : 0u));
      if (c == 0) bulk_load(sbase, nrm.G, g_bytes, bar);
      for (int r = 0; r < n; ++r)
        bulk_load(slot_addr(c) + static_cast<uint32_t>(r) * row_bytes,
                  static_cast<const uint8_t*>(nrm.X) + static_cast<long long>(first + r) * nrm.ldx * 2,
                  row_bytes, bar);
    };
    if (threadIdx.x == 0) {
      for (int i = 0; i < kSlots; ++i) mbar_init(smem_u32(&chunk_bar[i]), 1);
      fence_barrier_init();
      for (int c = 0; c < min(kSlots, nchunks); ++c) load_chunk(c);
    }
    __syncthreads();
    for (int c = 0; c < nchunks; ++c) {
      const int first = r0 + c * chunk, n = min(chunk, r1 - first);
      const uint32_t bar = smem_u32(&chunk_bar[c % kSlots]);
      const bool landed =
          wait_bounded(bar, static_cast<uint32_t>(c / kSlots) & 1u, nullptr, SITE_GRID_SYNC);
      // One decision for the whole CTA (the row groups meet at named barriers).
      if (__syncthreads_and(landed))
        rms_norm_rows<NORM_BF16, NORM_BF16, NORM == 2 ? 8 : 4, kRW, kThreads / 32, true, 2, true>(
            smem + (slot_addr(c) - sbase), row_bytes / 2, reinterpret_cast<const float*>(smem),
            nrm.eps, nrm.Xn, nrm.ldxn, first + n, nrm.D,
            first + static_cast<int>(threadIdx.x >> 5) / kRW, kGroups, norm_partial, 1, first,
            row_bytes);
      if (c + kSlots < nchunks) {
        // The chunk's copies to Xn have read its slot before the slot is refilled.
        bulk_wait_group_read<0>();
        __syncthreads();
        if (threadIdx.x == 0) load_chunk(c + kSlots);
      }
    }
    // Every copy to Xn has completed before the grid barrier below.
    bulk_wait_group<0>();
    __syncthreads();
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs, 1: its peer
  const int cluster = static_cast<int>(cluster_id_x());
  const int nclusters = static_cast<int>(num_clusters_x());
  const int nunits = cluster_unit_count(p, cluster, nclusters);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 2 * kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    if constexpr (RING)
      for (int i = 0; i < kEpiWarps * kRingSlots; ++i) mbar_init(drain_bar + 8u * (1 + i), 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if constexpr (EPI == EPI_GATE_UP) prefetch_tensormap(&tmB2);
    prefetch_tensormap(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish_alloc_permit_pair();
  }
  tc_fence_before_sync();
  cluster_sync();  // both CTAs' barriers exist and TMEM is allocated in both
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  if constexpr (NORM != 0) {
    // Every CTA's rows of Xn are written before any CTA loads a tile of it.
    // A barrier that gives up sets the abort flag: every role then leaves
    // through its bounded waits.
    if (threadIdx.x == 0) grid_sync_bounded(nrm.sync, abort_flag);
    __syncthreads();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Xn was written by other CTAs through the generic proxy (NORM).
      if constexpr (NORM != 0) asm volatile("fence.proxy.async.global;" ::: "memory");
      const uint32_t full0_even = mapa_shared(full_bar(0), 0);
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      bool ok = *abort_flag == 0;
      for (int i = 0; ok && i < nunits; ++i) {
        const WorkUnit un = cluster_unit(p, cluster, nclusters, i);
        int bt, mb, nb;
        tile_coords(un.tile, p, bt, mb, nb);
        const int a_row = mb * kPairBM + static_cast<int>(rank) * 128;
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + s * Cfg::kStageBytes;
          const uint32_t b_dst = a_dst + Cfg::kABytes;
          const uint32_t fbar = full0_even + 8u * s;
          const bool strip = kStrips && un.strip >= 0;
          if (rank == 0)
            mbar_arrive_expect_tx(full_bar(s), strip ? 2 * (Cfg::kABytes + kStripBBytes)
                                                     : 2 * Cfg::kStageBytes);
          tma_load_3d_pair(a_dst, &tmA, fbar, kb * kBK, a_row, bt);
          if constexpr (EPI == EPI_GATE_UP) {
            tma_load_3d_pair(b_dst, rank == 0 ? &tmB : &tmB2, fbar, kb * kBK, nb * (BN / 2), bt);
          } else {
            if (strip)
              tma_load_3d_pair(b_dst, &tmB2, fbar, kb * kBK,
                               nb * BN + un.strip * kPairStripN +
                                   static_cast<int>(rank) * (kPairStripN / 2),
                               bt);
            else
              tma_load_3d_pair(b_dst, &tmB, fbar, kb * kBK,
                               nb * BN + static_cast<int>(rank) * (BN / 2), bt);
          }
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (rank == 0) {
        // The even CTA's full barriers count both CTAs' copies: wait (bounded)
        // until the last STAGES rounds have landed before shared memory goes.
        const long long first = issued > STAGES ? issued - STAGES : 0;
        for (long long i = first; i < issued; ++i)
          wait_bounded(full_bar(static_cast<int>(i % STAGES)),
                       static_cast<uint32_t>((i / STAGES) & 1), nullptr, SITE_DRAIN);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      bool ok = true;
      for (int i = 0; ok && i < nunits; ++i, ++local) {
        const WorkUnit un = cluster_unit(p, cluster, nclusters, i);
        const int buf = local & 1;
        const uint32_t aph = static_cast<uint32_t>(local >> 1) & 1u;
        if (!wait_bounded_cluster(acce_bar(buf), aph ^ 1u, abort_flag, SITE_MMA_ACC_EMPTY)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * Cfg::kAccStride);
        const uint32_t idesc = (kStrips && un.strip >= 0) ? p.idesc_strip : p.idesc;
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          if (!wait_bounded(full_bar(s), ph, abort_flag, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = sbase + s * Cfg::kStageBytes;
          const uint64_t adesc = smem_desc_sw128(a_addr);
          const uint64_t bdesc = smem_desc_sw128(a_addr + Cfg::kABytes);
#pragma unroll
          for (int j = 0; j < kBK / kUmmaK; ++j)
            umma_bf16_pair(d_tmem, adesc + 2u * j, bdesc + 2u * j, idesc,
                           (kb != un.kb0 || j != 0) ? 1u : 0u);
          umma_commit_pair_multicast(empty_bar(s), 0x3);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_multicast(accf_bar(buf), 0x3);
      }
      umma_commit_pair_multicast(drain_bar, 0x1);
      wait_bounded(drain_bar, 0, nullptr, SITE_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 2;
    const int band = (warp & 3) * 32;
    const uint32_t staging = sbase + Cfg::kRingBytes + ew * Cfg::kSlots * kStageBox;
    const uint32_t acce0_even = mapa_shared(acce_bar(0), 0);
    const int band_id = static_cast<int>(rank) * 4 + (warp & 3);  // 32-row band of the pair tile
    int local = 0;
    int sc = 0;
    // C ring (RING kernels run only with beta != 0): the load cursor walks
    // this warp's boxes of whole tiles in the order the epilogue computes
    // them, starting at the first whole tile.  Split pieces come first in
    // every cluster's unit order; the last piece of a split tile loads its
    // boxes on demand.
    bool cursor_started = false;
    const uint32_t cbar0 = drain_bar + 8u * (1 + ew * kRingSlots);
    long long r_done = 0, r_issued = 0;
    int cu = nunits, cc0 = 0, cb = 0, cm0 = 0, cn0 = 0, cw = Cfg::kOutCols;
    auto cursor_at = [&](int i) {  // onto this cluster's unit i
      cu = i;
      cc0 = 0;
      if (i < nunits) {
        const WorkUnit cun = cluster_unit(p, cluster, nclusters, i);
        int mb_, nb_;
        tile_coords(cun.tile, p, cb, mb_, nb_);
        cm0 = mb_ * kPairBM + static_cast<int>(rank) * 128 + band;
        const bool strip = kStrips && cun.strip >= 0;
        cn0 = strip ? nb_ * BN + cun.strip * kPairStripN : nb_ * Cfg::kOutCols;
        cw = strip ? kPairStripN : Cfg::kOutCols;
      }
    };
    auto cursor_settle = [&]() {  // onto the next box inside C, or past the last unit
      while (cu < nunits) {
        if (cc0 < cw && cm0 < p.M && cn0 + cc0 < p.N) return;
        cursor_at(cu + 1);
      }
    };
    auto topup = [&](long long r_now) {
      using Box = EpiBox<EPI == EPI_GATE_UP ? EPI_BF16 : EPI, Cfg::kOutCols>;
      while (cu < nunits && r_issued <= r_now + kRingAhead) {
        const int slot = static_cast<int>(r_issued % kRingSlots);
        if (lane == 0) {
          // The slot's previous box was stored kRingSlots boxes ago.
          bulk_wait_group_read<kRingSlots - 1 - kRingAhead>();
          mbar_arrive_expect_tx(cbar0 + 8u * slot, 32 * Box::kRowBytes);
          tma_load_3d(staging + slot * kStageBox, &tmOut, cbar0 + 8u * slot, cn0 + cc0, cm0, cb);
        }
        ++r_issued;
        cc0 += Box::kCols;
        cursor_settle();
      }
    };
    for (int i = 0; i < nunits; ++i, ++local) {
      const WorkUnit un = cluster_unit(p, cluster, nclusters, i);
      int bt, mb, nb;
      tile_coords(un.tile, p, bt, mb, nb);
      if (RING && un.pieces == 1 && !cursor_started) {
        // First whole tile: start its C loads before waiting for its accumulator.
        cursor_started = true;
        r_issued = r_done;
        cursor_at(i);
        cursor_settle();
        topup(r_done);
      }
      const int buf = local & 1;
      const uint32_t aph = static_cast<uint32_t>(local >> 1) & 1u;
      const bool got = wait_bounded(accf_bar(buf), aph, abort_flag, SITE_EPI_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const uint32_t tacc = tmem_addr(tmem_base, static_cast<uint32_t>(band),
                                      static_cast<uint32_t>(buf * Cfg::kAccStride));
      const int m0 = mb * kPairBM + static_cast<int>(rank) * 128 + band;
      const bool strip = kStrips && un.strip >= 0;
      const int n0 = strip ? nb * BN + un.strip * kPairStripN : nb * Cfg::kOutCols;
      SplitCtx split{1, 0, nullptr, nullptr, 0};
      bool store = true;
      if (un.pieces > 1) {
        // One K piece of a split tile: publish the partial; the band's last
        // piece adds them all up and writes C.  A piece's partial is 8 bands
        // of 32 x BN floats.  Tail split: [tail tile][piece][band]; balanced
        // division: [slot][band] with the slots of balanced_slot; arrival
        // counters per (tail tile or tile, band).
        const long long band_f4 = 32LL * BN / 4;
        const long long piece_f4 = 8 * band_f4;
        const float4* ws = reinterpret_cast<const float4*>(p.ws) + band_id * band_f4;
        int* counter;
        split.pieces = un.pieces;
        split.piece = un.piece;
        if (p.balanced) {
          const int bt_ = un.tile - p.dp_tiles;   // tile index within the balanced ranges
          split.ws0 = ws + balanced_slot(p.work_per_cluster, p.work_extra, p.k_blocks, bt_, 0) *
                               piece_f4;
          split.ws1 = ws + balanced_slot(p.work_per_cluster, p.work_extra, p.k_blocks, bt_, 1) *
                               piece_f4;
          split.rest_stride = 2 * piece_f4;
          counter = p.counters +
                    balanced_counter(p.work_per_cluster, p.work_extra, p.k_blocks, bt_) * 8 +
                    band_id;
        } else {
          const int tail = un.tile - p.num_full;
          split.ws0 = ws + static_cast<long long>(tail) * p.tail_split * piece_f4;
          split.ws1 = split.ws0 + piece_f4;
          split.rest_stride = piece_f4;
          counter = p.counters + tail * 8 + band_id;
        }
        store = publish_partial(tacc, BN, lane, split, counter, un.pieces);
        if (store) {
          // Last piece: the sum goes into this accumulator; from here on the
          // tile is finished like a whole one.
          combine_into_tmem<BN>(tacc, lane, split);
          split = SplitCtx{1, 0, nullptr, nullptr, 0};
        }
      }
      // A strip computes the first kPairStripN columns of its accumulator.
      const int cols = strip ? kPairStripN : Cfg::kOutCols;
      if constexpr (RING) {
        bool ok = true;
        if (un.pieces == 1)
          ok = epilogue_tile_ring<BN, EPI, STATS, false>(p, &tmOut, tacc, bt, m0, n0, staging,
                                                         cbar0, lane, r_done, r_issued, sc, split,
                                                         rs, abort_flag, topup, cols);
        else if (store)
          ok = epilogue_tile_ring<BN, EPI, STATS, true>(p, &tmOut, tacc, bt, m0, n0, staging,
                                                        cbar0, lane, r_done, r_issued, sc, split,
                                                        rs, abort_flag, topup);
        if (!ok) break;
      } else {
        if (store)
          epilogue_tile<BN, EPI, STATS>(p, &tmOut, tacc, bt, m0, n0, staging, lane, sc,
                                        un.kb1 > un.kb0, split, rs, cols);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acce0_even + 8u * buf);
    }
    if (lane == 0) {
      // C loads still in flight (only after a wait gave up) land before exit.
      for (long long g = r_done; g < r_issued; ++g)
        wait_bounded(cbar0 + 8u * static_cast<uint32_t>(g % kRingSlots),
                     static_cast<uint32_t>((g / kRingSlots) & 1), nullptr, SITE_DRAIN);
      bulk_wait_group<0>();
    }
    __syncwarp();
  }

  tc_fence_before_sync();
  cluster_sync();  // neither CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace gb3
