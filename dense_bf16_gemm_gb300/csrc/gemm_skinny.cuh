// gemm_skinny.cuh -- decode-shaped GEMM (M <= 16) on the tensor cores, bound by
// the HBM stream of B.
//
// The operands are swapped: C^T = B^T-stored-as-(N,K) times A^T, so the long
// weight dimension N fills the 128-row M side of tcgen05.mma and the M <= 16
// activation rows become its N = 16 side.  Both operands are K-contiguous, so
// the swap needs no data movement.
//
// Work units are (128-row block of B, slice of K).  Each unit's FP32 partial
// (16 x 128) goes to a workspace; the last unit to finish a block (counted
// per 32-row band with an atomic) adds the partials in split order 0..S-1,
// applies alpha/beta and writes C, so the result does not depend on which
// unit finishes last.  No CTA waits for another.
//
// Roles as in the tiled kernel: warp 0 TMA producer, warp 1 MMA issuer and
// TMEM owner, warps 2-5 epilogue (warp w reads TMEM lanes 32*(w%4)..+31, i.e.
// rows n of B; lane i holds the 16 activation rows of output column n).
//
// GATE: the fused gate/up projection Y = silu(X Wg^T) * (X Wu^T) at decode
// sizes ("TMA and Hopper WGMMA", section "Worked consumers and current
// validation": the fused gate/up consumer).  A stage holds the same 128 rows
// of Wg and of Wu; two MMAs per K step accumulate gate and up side by side in
// TMEM; split partials keep gate and up apart, and silu(g) * u is formed only
// on the summed values.
#pragma once

#include "gemm_kernels.cuh"

namespace gb3 {

constexpr int kSkinnyRows = 128;  // rows of B per unit (the MMA's M)
constexpr int kSkinnyNX = 16;     // activation rows per MMA (the MMA's N)

struct SkinnyParams {
  int M, N, K;                // sizes of each matrix of the batch
  int n_blocks, k_blocks;
  int splits, kb_per_split;
  int batch;
  int num_units;              // batch * splits * n_blocks
  float alpha, beta;
  void* C;
  long long ldc;
  long long c_stride;         // elements between consecutive matrices of C
  int out_kind;               // 0 FP32, 1 BF16, 2 FP16
  uint32_t idesc;             // tcgen05 instruction descriptor (BF16 or FP16 operands)
  float* ws;      // [batch][splits][M][N] FP32 partial sums (splits > 1)
  int* counters;  // [batch][n_blocks][4] arrival counters, zero between calls
  int issue_group;  // k-blocks the producer issues back to back (1 .. STAGES)
  // -1, except in the failure-path self-test: the producer issues only this
  // many k-blocks and then stops, as if the next copy never landed, so the
  // MMA thread's wait for it runs out and the CTA takes its abort path.
  int stall_after;
};

template <int STAGES, bool GATE = false>
struct SkinnyCfg {
  static constexpr int kWeights = GATE ? 2 : 1;           // Wg and Wu, or B
  static constexpr int kWBytes = kSkinnyRows * kBK * 2;  // 16 KB per weight
  static constexpr int kXBytes = kSkinnyNX * kBK * 2;    // 2 KB
  static constexpr int kXOffset = kWeights * kWBytes;
  static constexpr int kStageBytes = kXOffset + kXBytes;  // keeps 1024-byte alignment
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kBarOffset = kRingBytes;
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
  static constexpr int kAccStride = kWeights * kSkinnyNX;  // gate in columns 0..15, up in 16..31
  static constexpr int kTmemCols = 2 * kAccStride < 32 ? 32 : 2 * kAccStride;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

__device__ __forceinline__ void skinny_unit(int u, const SkinnyParams& p, int& b, int& nb, int& sp,
                                            int& kb0, int& kb1) {
  nb = u % p.n_blocks;
  const int r = u / p.n_blocks;
  sp = r % p.splits;
  b = r / p.splits;
  kb0 = sp * p.kb_per_split;
  kb1 = min(p.k_blocks, kb0 + p.kb_per_split);
}

// Writes alpha * acc + beta * c for the M rows of output column n of matrix b.
__device__ __forceinline__ void skinny_store(const SkinnyParams& p, int b, int n,
                                             const float (&acc)[16]) {
  if (n >= p.N) return;
#pragma unroll
  for (int m = 0; m < kSkinnyNX; ++m) {
    if (m < p.M) {
      const long long off = b * p.c_stride + static_cast<long long>(m) * p.ldc + n;
      float v = __fmul_rn(p.alpha, acc[m]);
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

// Writes silu(g) * u (BF16, nearest even) for the M rows of output column n.
__device__ __forceinline__ void skinny_store_gate_up(const SkinnyParams& p, int n,
                                                     const float (&g)[16], const float (&u)[16]) {
  if (n >= p.N) return;
  uint16_t* y = static_cast<uint16_t*>(p.C);
#pragma unroll
  for (int m = 0; m < kSkinnyNX; ++m)
    if (m < p.M)
      y[static_cast<long long>(m) * p.ldc + n] =
          static_cast<uint16_t>(pack_bf16x2(silu_f32(g[m]) * u[m], 0.0f) & 0xFFFFu);
}

// tmW2: Wu (GATE only; tmW is then Wg).
template <int STAGES, bool GATE = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmW2,
                       const __grid_constant__ CUtensorMap tmX, const SkinnyParams p) {
  using Cfg = SkinnyCfg<STAGES, GATE>;
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
    if constexpr (GATE) prefetch_tensormap(&tmW2);
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
        int bt, nb, sp, kb0, kb1;
        skinny_unit(u, p, bt, nb, sp, kb0, kb1);
        // k-blocks are issued p.issue_group at a time, back to back, once
        // that many stages are free: each row of B is then read as one
        // longer run of consecutive bytes.
        const int group = max(1, min(p.issue_group, STAGES));
        for (int g0 = kb0; ok && g0 < kb1; g0 += group) {
          const int gn = min(group, kb1 - g0);
          int s_free = s;
          uint32_t ph_free = ph;
          for (int j = 0; j < gn; ++j) {
            if (!wait_bounded(empty_bar(s_free), ph_free ^ 1u, abort_flag, SITE_PRODUCER_EMPTY)) {
              ok = false;
              break;
            }
            if (++s_free == STAGES) {
              s_free = 0;
              ph_free ^= 1u;
            }
          }
          for (int j = 0; ok && j < gn; ++j) {
            if (issued == p.stall_after) {
              ok = false;
              break;
            }
            const int kb = g0 + j;
            const uint32_t w_dst = sbase + s * Cfg::kStageBytes;
            mbar_arrive_expect_tx(full_bar(s), Cfg::kStageBytes);
            tma_load_3d_hint(w_dst, &tmW, full_bar(s), kb * kBK, nb * kSkinnyRows, bt,
                             stream_policy);
            if constexpr (GATE)
              tma_load_3d_hint(w_dst + Cfg::kWBytes, &tmW2, full_bar(s), kb * kBK,
                               nb * kSkinnyRows, bt, stream_policy);
            tma_load_3d_hint(w_dst + Cfg::kXOffset, &tmX, full_bar(s), kb * kBK, 0, bt,
                             keep_policy);
            ++issued;
            if (++s == STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
      }
      {
        const long long first = issued > STAGES ? issued - STAGES : 0;
        for (long long i = first; i < issued; ++i)
          wait_bounded(full_bar(static_cast<int>(i % STAGES)),
                       static_cast<uint32_t>((i / STAGES) & 1), nullptr, SITE_DRAIN);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++local) {
        int bt, nb, sp, kb0, kb1;
        skinny_unit(u, p, bt, nb, sp, kb0, kb1);
        const int buf = local & 1;
        const uint32_t aph = static_cast<uint32_t>(local >> 1) & 1u;
        if (!wait_bounded(acce_bar(buf), aph ^ 1u, abort_flag, SITE_MMA_ACC_EMPTY)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * Cfg::kAccStride);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_bounded(full_bar(s), ph, abort_flag, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t w_addr = sbase + s * Cfg::kStageBytes;
          const uint64_t wdesc = smem_desc_sw128(w_addr);
          const uint64_t xdesc = smem_desc_sw128(w_addr + Cfg::kXOffset);
#pragma unroll
          for (int j = 0; j < kBK / kUmmaK; ++j) {
            umma_bf16(d_tmem, wdesc + 2u * j, xdesc + 2u * j, p.idesc,
                      (kb != kb0 || j != 0) ? 1u : 0u);
            if constexpr (GATE)
              umma_bf16(d_tmem + kSkinnyNX, smem_desc_sw128(w_addr + Cfg::kWBytes) + 2u * j,
                        xdesc + 2u * j, p.idesc, (kb != kb0 || j != 0) ? 1u : 0u);
          }
          umma_commit(empty_bar(s));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(accf_bar(buf));
      }
      umma_commit(drain_bar);
      wait_bounded(drain_bar, 0, nullptr, SITE_DRAIN);
    }
  } else {
    const int band = (warp & 3) * 32;
    int local = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++local) {
      int bt, nb, sp, kb0, kb1;
      skinny_unit(u, p, bt, nb, sp, kb0, kb1);
      const int buf = local & 1;
      const uint32_t aph = static_cast<uint32_t>(local >> 1) & 1u;
      const bool got = wait_bounded(accf_bar(buf), aph, abort_flag, SITE_EPI_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      // acc[w][m]: weight w (0: B or Wg, 1: Wu) for activation row m
      float acc[Cfg::kWeights][16];
      const uint32_t tacc = tmem_addr(tmem_base, static_cast<uint32_t>(band),
                                      static_cast<uint32_t>(buf * Cfg::kAccStride));
#pragma unroll
      for (int w = 0; w < Cfg::kWeights; ++w) {
        if (kb1 > kb0) {
          tmem_load_32x32b_x16(tacc + w * kSkinnyNX, acc[w]);
        } else {
#pragma unroll
          for (int m = 0; m < 16; ++m) acc[w][m] = 0.0f;
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));

      const int n = nb * kSkinnyRows + band + lane;
      auto store = [&](const float (&v)[Cfg::kWeights][16]) {
        if constexpr (GATE)
          skinny_store_gate_up(p, n, v[0], v[1]);
        else
          skinny_store(p, bt, n, v[0]);
      };
      if (p.splits == 1) {
        store(acc);
        continue;
      }
      // Partials [batch][split][weight][M][N].
      float* ws_b = p.ws + static_cast<long long>(bt) * p.splits * Cfg::kWeights * p.M * p.N;
      auto ws_at = [&](int sp_, int w, int m) {
        return ws_b + ((static_cast<long long>(sp_) * Cfg::kWeights + w) * p.M + m) * p.N + n;
      };
      // Publish this unit's partial, then count arrivals for this band.
      if (n < p.N) {
#pragma unroll
        for (int w = 0; w < Cfg::kWeights; ++w)
#pragma unroll
          for (int m = 0; m < kSkinnyNX; ++m)
            if (m < p.M) *ws_at(sp, w, m) = acc[w][m];
      }
      __threadfence();
      __syncwarp();
      int prev = 0;
      int* counter = p.counters + (static_cast<long long>(bt) * p.n_blocks + nb) * 4 + (warp & 3);
      if (lane == 0) prev = atomicAdd(counter, 1);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == p.splits - 1) {
        __threadfence();
        float sum[Cfg::kWeights][16];
#pragma unroll
        for (int w = 0; w < Cfg::kWeights; ++w)
#pragma unroll
          for (int m = 0; m < kSkinnyNX; ++m) sum[w][m] = 0.0f;
        if (n < p.N) {
          for (int s = 0; s < p.splits; ++s) {
#pragma unroll
            for (int w = 0; w < Cfg::kWeights; ++w) {
#pragma unroll
              for (int m = 0; m < kSkinnyNX; ++m) {
                if (m < p.M) sum[w][m] += (s == sp) ? acc[w][m] : __ldcg(ws_at(s, w, m));
              }
            }
          }
        }
        store(sum);
        if (lane == 0) *counter = 0;  // ready for the next call
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
