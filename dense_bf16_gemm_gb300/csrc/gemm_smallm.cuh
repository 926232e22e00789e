// gemm_smallm.cuh -- small-M GEMM (M <= 128) without split-K, bound by the
// HBM stream of B.
//
// As in the swapped-operand decode kernel, C^T = B(N,K) . A(M,K)^T: the weight
// rows fill the MMA's M side and the activation rows its N side.  Here the
// weight tile is 64 rows (tcgen05.mma cta_group::1 with M = 64), so a weight
// splits into twice as many units as 128-row tiles would give, and each unit
// streams its 64 rows through the whole of K into one TMEM accumulator.  No
// workspace, no second pass, no arrival counters: every output is written once
// by the unit that owns it, so the call allocates nothing and is
// deterministic by construction.
//
// Where it pays (measured on GB300): a CTA's TMA stream of B from HBM runs at
// about 32-37 GB/s whatever the number of busy SMs, so a weight is read at full
// speed only when every SM streams.  64-row units spread a moderate weight over
// more SMs than 128- or 256-row tiles do without cutting K; for weights of many
// waves the other kernels are as fast and this one is not chosen.
//
// Accumulator placement of an M = 64 MMA (measured on GB300): D row i sits in
// TMEM lane 32*(i/16) + i%16, its columns unchanged.  So epilogue warp w (which
// may access lanes 32*(w%4)..+31) finds weight rows 16*(w%4)..+15 in its lanes
// 0..15; lanes 16..31 carry nothing and store nothing.
//
// Roles: warp 0 TMA producer, warp 1 MMA issuer and TMEM owner, warps 2-5
// epilogue.  Two accumulators (2*NX TMEM columns) let the epilogue of one unit
// overlap the main loop of the next.
#pragma once

#include "gemm_kernels.cuh"

namespace gb3 {

constexpr int kSmallRows = 64;   // weight rows per unit (the MMA's M)

struct SmallMParams {
  int M, N, K;                // sizes of each matrix of the batch
  int n_blocks, k_blocks;     // ceil(N / 64), ceil(K / 64)
  int batch;
  int num_units;              // batch * n_blocks
  float alpha, beta;
  void* C;
  long long ldc;
  long long c_stride;         // elements between consecutive matrices of C
  int out_kind;               // 0 FP32, 1 BF16, 2 FP16
  uint32_t idesc;             // tcgen05 instruction descriptor (M = 64, N = NX)
};

// NX: activation rows per MMA (the MMA's N), 16, 32, 64 or 128.
template <int NX>
struct SmallMCfg {
  static_assert(NX == 16 || NX == 32 || NX == 64 || NX == 128, "activation tile");
  static constexpr int kWBytes = kSmallRows * kBK * 2;  // 8 KB
  static constexpr int kXBytes = NX * kBK * 2;          // 2..16 KB
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  // As many stages as fit in about 200 KB.
  static constexpr int kStages = (200 * 1024) / kStageBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kBarOffset = kRingBytes;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
  static constexpr int kAccStride = NX;
  static constexpr int kTmemCols = (2 * NX < 32) ? 32 : 2 * NX;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// alpha * acc + beta * c for activation rows m0..m0+kCols-1 of output column n.
template <int kCols>
__device__ __forceinline__ void smallm_store(const SmallMParams& p, int b, int n, int m0,
                                             const float* acc) {
  if (n >= p.N) return;
#pragma unroll
  for (int i = 0; i < kCols; ++i) {
    const int m = m0 + i;
    if (m < p.M) {
      const long long off = b * p.c_stride + static_cast<long long>(m) * p.ldc + n;
      float v = __fmul_rn(p.alpha, acc[i]);
      if (p.out_kind != 0) {
        const bool f16 = p.out_kind == 2;
        uint16_t* c = static_cast<uint16_t*>(p.C);
        if (p.beta != 0.0f) v = __fmaf_rn(p.beta, half16_to_float(c[off], f16), v);
        c[off] = static_cast<uint16_t>(pack_half16x2(v, 0.0f, f16) & 0xFFFFu);
      } else {
        float* c = static_cast<float*>(p.C);
        if (p.beta != 0.0f) v = __fmaf_rn(p.beta, c[off], v);
        c[off] = v;
      }
    }
  }
}

template <int NX>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_smallm_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmX, const SmallMParams p) {
  using Cfg = SmallMCfg<NX>;
  constexpr int STAGES = Cfg::kStages;
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

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), Cfg::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t stream_policy = l2_policy_evict_first();  // B is read once
      const uint64_t keep_policy = l2_policy_evict_last();     // A is re-read by every unit
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
        const int bt = u / p.n_blocks, nb = u - bt * p.n_blocks;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t w_dst = sbase + s * Cfg::kStageBytes;
          mbar_arrive_expect_tx(full_bar(s), Cfg::kStageBytes);
          tma_load_3d_hint(w_dst, &tmW, full_bar(s), kb * kBK, nb * kSmallRows, bt, stream_policy);
          tma_load_3d_hint(w_dst + Cfg::kWBytes, &tmX, full_bar(s), kb * kBK, 0, bt, keep_policy);
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // Leave only when every issued copy has landed (bounded).
      const long long first = issued > STAGES ? issued - STAGES : 0;
      for (long long i = first; i < issued; ++i)
        wait_bounded(full_bar(static_cast<int>(i % STAGES)),
                     static_cast<uint32_t>((i / STAGES) & 1), nullptr, SITE_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t aph = static_cast<uint32_t>(local >> 1) & 1u;
        if (!wait_bounded(acce_bar(buf), aph ^ 1u, abort_flag, SITE_MMA_ACC_EMPTY)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * Cfg::kAccStride);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_bounded(full_bar(s), ph, abort_flag, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t w_addr = sbase + s * Cfg::kStageBytes;
          const uint64_t wdesc = smem_desc_sw128(w_addr);
          const uint64_t xdesc = smem_desc_sw128(w_addr + Cfg::kWBytes);
#pragma unroll
          for (int j = 0; j < kBK / kUmmaK; ++j)
            umma_bf16(d_tmem, wdesc + 2u * j, xdesc + 2u * j, p.idesc,
                      (kb != 0 || j != 0) ? 1u : 0u);
          umma_commit(empty_bar(s));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(accf_bar(buf));
      }
      // Leave only when every issued MMA has completed (bounded).
      umma_commit(drain_bar);
      wait_bounded(drain_bar, 0, nullptr, SITE_DRAIN);
    }
  } else {
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    constexpr int kGroup = NX < 64 ? NX : 64;  // columns held in registers at once
    int local = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++local) {
      const int bt = u / p.n_blocks, nb = u - bt * p.n_blocks;
      const int buf = local & 1;
      const uint32_t aph = static_cast<uint32_t>(local >> 1) & 1u;
      const bool got = wait_bounded(accf_bar(buf), aph, abort_flag, SITE_EPI_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const int n = nb * kSmallRows + 16 * quarter + lane;
      const uint32_t tacc = tmem_base + lane_base + static_cast<uint32_t>(buf * Cfg::kAccStride);
#pragma unroll 1
      for (int g0 = 0; g0 < NX; g0 += kGroup) {
        float acc[kGroup];
#pragma unroll
        for (int c = 0; c < kGroup; c += 16) {
          float t[16];
          tmem_load_32x32b_x16(tacc + g0 + c, t);
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[c + i] = t[i];
        }
        if (g0 + kGroup >= NX) {
          // Every column of this accumulator is in registers: hand it back.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce_bar(buf));
        }
        if (lane < 16 && g0 < p.M) smallm_store<kGroup>(p, bt, n, g0, acc);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace gb3
