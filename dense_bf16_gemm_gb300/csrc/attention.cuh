// attention.cuh -- softmax attention O = softmax(scale * Q.K^T) . V on the
// tcgen05 tensor cores, as the flash-attention loop ("Tiles and shared
// memory", section "How long a tile lives": a query tile, a running maximum m
// and a running sum l kept across the key loop, s = dot_t(q, k) per key tile,
// acc / l at the end).
//
// One CTA per (head, 128-row query block).  Per key block j of 128 keys:
//
//   S_j = Q . K_j^T                tcgen05.mma M = 128, N = 128 over D, into one of two
//                                  TMEM score buffers (K_j is K-major: D contiguous)
//   m_j = max(m_{j-1}, rowmax S_j)  softmax warps: a query row is one TMEM lane, so the
//   P_j = exp(S_j - m_j)            reduction is local to the threads of that lane (two
//   l_j = l_{j-1} a_j + rowsum P_j  warps, half of the keys each); a_j = exp(m_{j-1} - m_j)
//   O_j = P_j . V_j                tcgen05.mma M = 128, N = D over the 128 keys, with P_j
//                                  written as BF16 back into Tensor Memory (the A
//                                  operand read from TMEM) and V_j the MN-major operand
//                                  (D contiguous, as TMA loads it)
//   acc = acc a_j + O_j            FP32 in the softmax threads' registers
//
// and finally O = acc / l.  Scores are handled in base-2 units (exp2 of
// s * scale * log2 e), which is the same function.  Keys past Nk score -inf.
//
// Tensor Memory: two 128-column buffers, each holding S_j as FP32 and then,
// in the first 32 columns of each half's 64, that half's P_j as packed BF16
// (its scores are in registers by then); two D-column output buffers.  A
// buffer is reused for S_{j+2} once O_j = P_j . V_j has completed.
//
// Warp roles: warp 0 TMA (Q once, K_j and V_j through a ring), warp 1 MMA
// issue and TMEM owner, warps 2-9 softmax and output (two warps per TMEM lane
// quarter, each taking half of the keys of a block and half of the output
// columns, so that two softmax warps share each SM sub-partition).  The MMA
// warp issues S_{j+1} before O_j, so the tensor core works on the next scores
// while the softmax threads finish the current block.
//
// Every wait is bounded as in the GEMM kernels (status word, abort flag,
// drained copies and MMAs, TMEM freed).
#pragma once

#include "gemm_kernels.cuh"

namespace gb3 {

constexpr int kAttnBR = 128;   // query rows per CTA (the MMA's M)
constexpr int kAttnBC = 128;   // keys per block
constexpr int kAttnSoftWarps = 8;                          // two per TMEM lane quarter
constexpr int kAttnThreads = 32 * (2 + kAttnSoftWarps);    // TMA, MMA, softmax

struct AttnParams {
  int heads, Nq, Nk;
  int q_blocks, k_blocks;     // ceil(Nq / 128), ceil(Nk / 128)
  float scale_log2;           // scale * log2(e)
  void* O;
  long long ldo, o_stride;    // elements
  int out_kind;               // 0 FP32, 1 BF16
  uint32_t idesc_s;           // M = 128, N = 128, A and B K-major
  uint32_t idesc_o;           // M = 128, N = D, B MN-major
};

template <int D>
struct AttnCfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int kChunks = D / 64;                 // 64-element swizzle rows per row
  static constexpr int kTileBytes = 128 * D * 2;         // Q, K_j or V_j (128 rows)
  static constexpr int kStages = D == 128 ? 2 : 4;       // K/V ring depth
  static constexpr int kStageBytes = 2 * kTileBytes;     // K_j and V_j
  static constexpr int kQOffset = 0;
  static constexpr int kRingOffset = kTileBytes;
  static constexpr int kRedOffset = kRingOffset + kStages * kStageBytes;  // [2][2][128] floats
  static constexpr int kBarOffset = kRedOffset + 2 * 2 * kAttnBR * 4;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2], o_empty[2],
  // drain, xchg[4]
  static constexpr int kNumBars = 1 + 2 * kStages + 8 + 1 + 4;
  static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
  static constexpr int kTmemCols = 512;                  // S/P: 2 x 128, O: 2 x D
  static constexpr int kSCol = 0;
  static constexpr int kOCol = 256;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// UMMA shared-memory descriptor of an MN-major operand in 128-byte swizzled
// tiles as TMA writes a [rows = K][64 contiguous MN elements] box: eight-row
// (K) groups 1024 bytes apart (SBO), consecutive 64-element MN chunks
// `mn_chunk_bytes` apart (LBO).  Checked on GB300 against known products.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t mn_chunk_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((mn_chunk_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// 2^x by the hardware's approximate exp2 (relative error about 2^-22;
// results below the normal range flush to zero, exp2(-inf) = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using Cfg = AttnCfg<D>;
  constexpr int S = Cfg::kStages;
  constexpr int kChunkBytes = 128 * 128;  // one 64-element-wide swizzled chunk of 128 rows
  constexpr int kHalfKeys = kAttnBC / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOffset);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0;
  auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (1 + S + s); };
  auto s_full = [&](int b) { return bar0 + 8u * (1 + 2 * S + b); };   // S_j in buffer b
  auto p_full = [&](int b) { return bar0 + 8u * (3 + 2 * S + b); };   // P_j written over it
  auto o_full = [&](int b) { return bar0 + 8u * (5 + 2 * S + b); };   // O_j done (buffer b free)
  auto o_empty = [&](int b) { return bar0 + 8u * (7 + 2 * S + b); };  // O_j taken
  const uint32_t drain_bar = bar0 + 8u * (9 + 2 * S);
  auto xchg_bar = [&](int qtr) { return bar0 + 8u * (10 + 2 * S + qtr); };

  const uint32_t q_smem = sb + Cfg::kQOffset;
  auto k_smem = [&](int s) { return sb + Cfg::kRingOffset + static_cast<uint32_t>(s * Cfg::kStageBytes); };
  auto v_smem = [&](int s) { return k_smem(s) + Cfg::kTileBytes; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x / p.q_blocks;
  const int qb = blockIdx.x - h * p.q_blocks;
  const int n = p.k_blocks;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_full(b), kAttnSoftWarps);
      mbar_init(o_full(b), 1);
      mbar_init(o_empty(b), kAttnSoftWarps);
    }
    mbar_init(drain_bar, 1);
    for (int qtr = 0; qtr < 4; ++qtr) mbar_init(xchg_bar(qtr), 2);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
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
      mbar_arrive_expect_tx(q_full, Cfg::kTileBytes);
      for (int c = 0; c < Cfg::kChunks; ++c)
        tma_load_3d(q_smem + c * kChunkBytes, &tmQ, q_full, c * 64, qb * kAttnBR, h);
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int s = j % S;
        const uint32_t ph = static_cast<uint32_t>(j / S) & 1u;
        if (!wait_bounded(kv_empty(s), ph ^ 1u, abort_flag, SITE_PRODUCER_EMPTY)) break;
        mbar_arrive_expect_tx(kv_full(s), Cfg::kStageBytes);
        for (int c = 0; c < Cfg::kChunks; ++c) {
          tma_load_3d(k_smem(s) + c * kChunkBytes, &tmK, kv_full(s), c * 64, j * kAttnBC, h);
          tma_load_3d(v_smem(s) + c * kChunkBytes, &tmV, kv_full(s), c * 64, j * kAttnBC, h);
        }
        ++issued;
      }
      // Leave only when every issued copy has landed (bounded).
      wait_bounded(q_full, 0, nullptr, SITE_DRAIN);
      for (int j = issued > S ? issued - S : 0; j < issued; ++j)
        wait_bounded(kv_full(j % S), static_cast<uint32_t>(j / S) & 1u, nullptr, SITE_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // S_j = Q . K_j^T into buffer j % 2, once O_{j-2} (which read P_{j-2}
      // from that buffer) has completed.
      auto issue_s = [&](int j) -> bool {
        const int s = j % S, b = j & 1;
        if (j >= 2 && !wait_bounded(o_full(b), static_cast<uint32_t>((j - 2) >> 1) & 1u, abort_flag,
                                    SITE_MMA_ACC_EMPTY))
          return false;
        if (!wait_bounded(kv_full(s), static_cast<uint32_t>(j / S) & 1u, abort_flag, SITE_MMA_FULL))
          return false;
        tc_fence_after_sync();
        const uint32_t d = tmem_base + Cfg::kSCol + static_cast<uint32_t>(b * kAttnBC);
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c) {
          const uint64_t qd = smem_desc_sw128(q_smem + c * kChunkBytes);
          const uint64_t kd = smem_desc_sw128(k_smem(s) + c * kChunkBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d, qd + 2u * kk, kd + 2u * kk, p.idesc_s, (c | kk) != 0 ? 1u : 0u);
        }
        umma_commit(s_full(b));
        return true;
      };
      bool ok = wait_bounded(q_full, 0, abort_flag, SITE_MMA_FULL) && n > 0 && issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) break;
        // O_j = P_j . V_j into output buffer j % 2; P_j is read from TMEM.
        const int s = j % S, b = j & 1;
        if (!wait_bounded(p_full(b), static_cast<uint32_t>(j >> 1) & 1u, abort_flag, SITE_MMA_FULL))
          break;
        if (!wait_bounded(o_empty(b), (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u, abort_flag,
                          SITE_MMA_ACC_EMPTY))
          break;
        tc_fence_after_sync();
        const uint32_t d = tmem_base + Cfg::kOCol + static_cast<uint32_t>(b * D);
        const uint32_t pa = tmem_base + Cfg::kSCol + static_cast<uint32_t>(b * kAttnBC);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t key_row = static_cast<uint32_t>(half * kHalfKeys + kk * 16);
            umma_bf16_tmem_a(d, pa + static_cast<uint32_t>(half * kHalfKeys + kk * 8),
                             smem_desc_mn_sw128(v_smem(s) + key_row * 128u, kChunkBytes), p.idesc_o,
                             (half | kk) != 0 ? 1u : 0u);
          }
        }
        umma_commit(o_full(b));
        umma_commit(kv_empty(s));
      }
      // Leave only when every issued MMA has completed (bounded).
      umma_commit(drain_bar);
      wait_bounded(drain_bar, 0, nullptr, SITE_DRAIN);
    }
  } else {
    // Softmax warps 2..9: warp w serves query rows 32*(w%4)..+31 (its TMEM
    // lane quarter) and one half of the keys of each block and of the output
    // columns; the two warps of a quarter exchange their partial row maxima
    // through shared memory each block (a bounded mbarrier, values double
    // buffered) and their partial row sums once at the end.
    constexpr int kHalfD = D / 2;
    const int half = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;             // query row of this thread in the block
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    float* xval = reinterpret_cast<float*>(smem + Cfg::kRedOffset);
    const uint32_t xbar = xchg_bar(quarter);
    // Publishes `mine` for the partner warp in exchange round r and returns
    // the partner's value (false if a wait gave up).
    auto exchange = [&](int r, float mine, float& other) -> bool {
      const int buf = r & 1;
      xval[(buf * 2 + half) * kAttnBR + row] = mine;
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      const bool got = wait_bounded(xbar, static_cast<uint32_t>(r) & 1u, abort_flag,
                                    SITE_EPI_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) return false;
      other = xval[(buf * 2 + (half ^ 1)) * kAttnBR + row];
      return true;
    };
    float acc[kHalfD];
#pragma unroll
    for (int i = 0; i < kHalfD; ++i) acc[i] = 0.0f;
    float m = -INFINITY, l = 0.0f, alpha_prev = 0.0f;
    bool ok = true;
    // acc = acc * alpha + this half of O_j (read from TMEM), then hand it back.
    auto take_o = [&](int j, float alpha) -> bool {
      const int b = j & 1;
      const bool got = wait_bounded(o_full(b), static_cast<uint32_t>(j >> 1) & 1u, abort_flag,
                                    SITE_EPI_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) return false;
      tc_fence_after_sync();
      const uint32_t to = tmem_base + lane_base + Cfg::kOCol + static_cast<uint32_t>(b * D + half * kHalfD);
      if constexpr (kHalfD == 64) {
        float o[64];
        tmem_load_32x32b_x64(to, o);
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = fmaf(acc[i], alpha, o[i]);
      } else {
        float o[32];
        tmem_load_32x32b_x32(to, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = fmaf(acc[i], alpha, o[i]);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty(b));
      return true;
    };
    const float c = p.scale_log2;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      const bool got = wait_bounded(s_full(b), static_cast<uint32_t>(j >> 1) & 1u, abort_flag,
                                    SITE_EPI_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t ts = tmem_base + lane_base + Cfg::kSCol +
                          static_cast<uint32_t>(b * kAttnBC + half * kHalfKeys);
      const int col0 = j * kAttnBC + half * kHalfKeys;
      const bool full = j * kAttnBC + kAttnBC <= p.Nk;   // the same for both halves
      // This half of the row of S, once, into registers (64 scores).
      float v[kHalfKeys];
      tmem_load_32x32b_x64(ts, v);
      // Pass 1: this half's maximum of the scaled scores (a full block needs no
      // key mask, and scaling by c is monotonic: c times the largest raw score,
      // the smallest for c < 0), four partial maxima.
      float mine;
      if (full) {
        const bool up = c >= 0.0f;
        float r0 = up ? -INFINITY : INFINITY, r1 = r0, r2 = r0, r3 = r0;
        if (up) {
#pragma unroll
          for (int i = 0; i < kHalfKeys; i += 4) {
            r0 = fmaxf(r0, v[i]);
            r1 = fmaxf(r1, v[i + 1]);
            r2 = fmaxf(r2, v[i + 2]);
            r3 = fmaxf(r3, v[i + 3]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kHalfKeys; i += 4) {
            r0 = fminf(r0, v[i]);
            r1 = fminf(r1, v[i + 1]);
            r2 = fminf(r2, v[i + 2]);
            r3 = fminf(r3, v[i + 3]);
          }
        }
        mine = (up ? fmaxf(fmaxf(r0, r1), fmaxf(r2, r3)) : fminf(fminf(r0, r1), fminf(r2, r3))) * c;
      } else {
        mine = -INFINITY;
#pragma unroll
        for (int i = 0; i < kHalfKeys; ++i)
          if (col0 + i < p.Nk) mine = fmaxf(mine, v[i] * c);
      }
      float other;
      if (!exchange(j, mine, other)) {
        ok = false;
        break;
      }
      const float m_new = fmaxf(m, fmaxf(mine, other));
      const float alpha = fast_exp2(m - m_new);   // 0 on the first block (m = -inf)
      // Pass 2: P = exp2(s * c - m_new), packed as BF16 pairs (even key in
      // the low half) into the first 32 columns of this half's scores, and
      // this half's row sum (four partial sums).
      float ps0 = 0.0f, ps1 = 0.0f, ps2 = 0.0f, ps3 = 0.0f;
      uint32_t w[kHalfKeys / 2];
#pragma unroll
      for (int i = 0; i < kHalfKeys; i += 4) {
        float q0 = fast_exp2(fmaf(v[i], c, -m_new));
        float q1 = fast_exp2(fmaf(v[i + 1], c, -m_new));
        float q2 = fast_exp2(fmaf(v[i + 2], c, -m_new));
        float q3 = fast_exp2(fmaf(v[i + 3], c, -m_new));
        if (!full) {
          const int k = col0 + i;
          q0 = k < p.Nk ? q0 : 0.0f;
          q1 = k + 1 < p.Nk ? q1 : 0.0f;
          q2 = k + 2 < p.Nk ? q2 : 0.0f;
          q3 = k + 3 < p.Nk ? q3 : 0.0f;
        }
        ps0 += q0;
        ps1 += q1;
        ps2 += q2;
        ps3 += q3;
        w[i / 2] = pack_bf16x2(q0, q1);
        w[i / 2 + 1] = pack_bf16x2(q2, q3);
      }
      tmem_store_32x32b_x32(ts, w);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(b));
      l = fmaf(l, alpha, (ps0 + ps1) + (ps2 + ps3));
      if (j > 0 && !take_o(j - 1, alpha_prev)) {
        ok = false;
        break;
      }
      alpha_prev = alpha;
      m = m_new;
    }
    if (ok && n > 0) ok = take_o(n - 1, alpha_prev);
    // The row sum is the two halves' sums (both at the final maximum).
    float l_other = 0.0f;
    if (ok) ok = exchange(n, l, l_other);
    const int qrow = qb * kAttnBR + row;
    if (ok && qrow < p.Nq) {
      const float inv = 1.0f / (l + l_other);
      if (p.out_kind == 0) {
        float* dst = static_cast<float*>(p.O) + h * p.o_stride + static_cast<long long>(qrow) * p.ldo +
                     half * kHalfD;
#pragma unroll
        for (int d = 0; d < kHalfD; d += 4)
          *reinterpret_cast<float4*>(dst + d) =
              make_float4(acc[d] * inv, acc[d + 1] * inv, acc[d + 2] * inv, acc[d + 3] * inv);
      } else {
        uint16_t* dst = static_cast<uint16_t*>(p.O) + h * p.o_stride +
                        static_cast<long long>(qrow) * p.ldo + half * kHalfD;
#pragma unroll
        for (int d = 0; d < kHalfD; d += 8)
          *reinterpret_cast<uint4*>(dst + d) =
              make_uint4(pack_bf16x2(acc[d] * inv, acc[d + 1] * inv),
                         pack_bf16x2(acc[d + 2] * inv, acc[d + 3] * inv),
                         pack_bf16x2(acc[d + 4] * inv, acc[d + 5] * inv),
                         pack_bf16x2(acc[d + 6] * inv, acc[d + 7] * inv));
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
