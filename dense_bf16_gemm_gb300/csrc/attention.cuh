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
//   O += P_j . V_j                 tcgen05.mma M = 128, N = D over the 128 keys into one
//                                  FP32 accumulator in Tensor Memory, with P_j written as
//                                  BF16 back into Tensor Memory (the A operand read from
//                                  TMEM) and V_j the MN-major operand (D contiguous, as
//                                  TMA loads it)
//
// and finally O / l.  Scores are handled in base-2 units (exp2 of
// s * scale * log2 e), which is the same function.  Keys past Nk score -inf.
//
// The running maximum is updated lazily: the m a row's probabilities are
// taken against moves only when a block's maximum exceeds it by more than
// kAttnRescaleLog2 (so probabilities stay below 2^8 and l, O keep their
// ratio), and only then is that row of O (and l) multiplied by a_j, in
// Tensor Memory, after O += P_{j-1} . V_{j-1} has completed.  The result
// O / l does not depend on which m was used.
//
// Tensor Memory: three 128-column buffers, each holding S_j as FP32 and then,
// in the first 32 columns of each half's 64, that half's P_j as packed BF16
// (its scores are in registers by then); one D-column output accumulator.
// A buffer is reused for S_{j+3} once O += P_j . V_j has completed (an MMA
// is not ordered after an earlier one into another accumulator, so the
// wait is needed; with three buffers it is almost never on the critical
// path, and the tensor core runs S and P.V products back to back).
//
// Warp roles: warp 0 TMA (Q once, K_j and V_j through a ring), warp 1 MMA
// issue and TMEM owner, warps 2-9 softmax and output (two warps per TMEM lane
// quarter, each taking half of the keys of a block and half of the output
// columns, so that two softmax warps share each SM sub-partition).  The MMA
// warp issues S_{j+1} before P_j . V_j, so the tensor core works on the next
// scores while the softmax threads finish the current block.
//
// Every wait is bounded as in the GEMM kernels (status word, abort flag,
// drained copies and MMAs, TMEM freed).
#pragma once

#include "gemm_kernels.cuh"

namespace gb3 {

constexpr int kAttnBR = 128;   // query rows per CTA (the MMA's M)
constexpr int kAttnBC = 128;   // keys per block
constexpr int kAttnSoftWarps = 8;                          // two per TMEM lane quarter
constexpr int kAttnSBufs = 3;                              // S/P buffers in Tensor Memory
constexpr int kAttnThreads = 32 * (2 + kAttnSoftWarps);    // TMA, MMA, softmax
constexpr float kAttnRescaleLog2 = 8.0f;  // lazy rescaling: probabilities stay below 2^8

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
  // Separate rings: a K slot frees when S_j has completed, a V slot when
  // O += P_j . V_j has, so K can be fetched further ahead than V.
  static constexpr int kKStages = D == 128 ? 3 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kQOffset = 0;
  static constexpr int kKOffset = kTileBytes;
  static constexpr int kVOffset = kKOffset + kKStages * kTileBytes;
  static constexpr int kRedOffset = kVOffset + kVStages * kTileBytes;  // [2][2][128] floats
  static constexpr int kBarOffset = kRedOffset + 2 * 2 * kAttnBR * 4;
  // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[3], p_full[3],
  // o_done[3], drain, xchg[4]
  static constexpr int kNumBars =
      1 + 2 * kKStages + 2 * kVStages + 3 * kAttnSBufs + 1 + 4;
  static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
  static constexpr int kTmemCols = 512;                  // S/P: 3 x 128, O: D
  static constexpr int kSCol = 0;
  static constexpr int kOCol = kAttnSBufs * kAttnBC;
  static_assert(kOCol + D <= kTmemCols, "Tensor Memory columns");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

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
  constexpr int KS = Cfg::kKStages;
  constexpr int VS = Cfg::kVStages;
  constexpr int kChunkBytes = 128 * 128;  // one 64-element-wide swizzled chunk of 128 rows
  constexpr int kHalfKeys = kAttnBC / 2;
  if (!launch_smem_ok(Cfg::kSmemBytes)) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOffset);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cfg::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0;
  // Ring and buffer barriers complete once per use; block j's use of a ring
  // of R slots is j / R, so its phase parity is (j / R) & 1.
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (1 + KS + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * KS + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (1 + 2 * KS + VS + s); };
  constexpr int R0 = 1 + 2 * KS + 2 * VS;
  constexpr int NB = kAttnSBufs;
  auto s_full = [&](int b) { return bar0 + 8u * (R0 + b); };        // S_j in buffer b = j % NB
  auto p_full = [&](int b) { return bar0 + 8u * (R0 + NB + b); };   // P_j written over it
  // O += P_j . V_j done (buffer b's P read, O holds block j)
  auto o_done = [&](int b) { return bar0 + 8u * (R0 + 2 * NB + b); };
  const uint32_t drain_bar = bar0 + 8u * (R0 + 3 * NB);
  auto xchg_bar = [&](int qtr) { return bar0 + 8u * (R0 + 3 * NB + 1 + qtr); };
  auto parity = [](int j, int r) { return static_cast<uint32_t>(j / r) & 1u; };
  auto use_parity = [&](int j) { return parity(j, NB); };

  const uint32_t q_smem = sb + Cfg::kQOffset;
  auto k_smem = [&](int s) { return sb + Cfg::kKOffset + static_cast<uint32_t>(s * Cfg::kTileBytes); };
  auto v_smem = [&](int s) { return sb + Cfg::kVOffset + static_cast<uint32_t>(s * Cfg::kTileBytes); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x / p.q_blocks;
  const int qb = blockIdx.x - h * p.q_blocks;
  const int n = p.k_blocks;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_full(b), kAttnSoftWarps);
      mbar_init(o_done(b), 1);
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
      // Loads in the order the MMAs consume them: K_0, then K_{j+1} before V_j.
      auto load_k = [&](int j) -> bool {
        const int s = j % KS;
        if (!wait_bounded(k_empty(s), parity(j, KS) ^ 1u, abort_flag, SITE_PRODUCER_EMPTY))
          return false;
        mbar_arrive_expect_tx(k_full(s), Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(k_smem(s) + c * kChunkBytes, &tmK, k_full(s), c * 64, j * kAttnBC, h);
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j % VS;
        if (!wait_bounded(v_empty(s), parity(j, VS) ^ 1u, abort_flag, SITE_PRODUCER_EMPTY))
          return false;
        mbar_arrive_expect_tx(v_full(s), Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(v_smem(s) + c * kChunkBytes, &tmV, v_full(s), c * 64, j * kAttnBC, h);
        return true;
      };
      int k_issued = 0, v_issued = 0;
      if (n > 0 && load_k(0)) k_issued = 1;
      for (int j = 0; j < n && k_issued == j + 1; ++j) {
        if (j + 1 < n) {
          if (!load_k(j + 1)) break;
          ++k_issued;
        }
        if (!load_v(j)) break;
        ++v_issued;
      }
      // Leave only when every issued copy has landed (bounded).
      wait_bounded(q_full, 0, nullptr, SITE_DRAIN);
      for (int j = k_issued > KS ? k_issued - KS : 0; j < k_issued; ++j)
        wait_bounded(k_full(j % KS), parity(j, KS), nullptr, SITE_DRAIN);
      for (int j = v_issued > VS ? v_issued - VS : 0; j < v_issued; ++j)
        wait_bounded(v_full(j % VS), parity(j, VS), nullptr, SITE_DRAIN);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // S_j = Q . K_j^T into buffer j % NB, once O += P_{j-NB} . V_{j-NB}
      // (which read P_{j-NB} from that buffer) has completed.
      auto issue_s = [&](int j) -> bool {
        const int s = j % KS, b = j % NB;
        if (j >= NB && !wait_bounded(o_done(b), use_parity(j - NB), abort_flag, SITE_MMA_ACC_EMPTY))
          return false;
        if (!wait_bounded(k_full(s), parity(j, KS), abort_flag, SITE_MMA_FULL)) return false;
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
        umma_commit(k_empty(s));
        return true;
      };
      bool ok = wait_bounded(q_full, 0, abort_flag, SITE_MMA_FULL) && n > 0 && issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) break;
        // O += P_j . V_j (O = P_0 . V_0 first); P_j is read from TMEM.  The
        // softmax threads arrive on p_full only after any rescaling of O.
        const int s = j % VS, b = j % NB;
        if (!wait_bounded(p_full(b), use_parity(j), abort_flag, SITE_MMA_FULL)) break;
        if (!wait_bounded(v_full(s), parity(j, VS), abort_flag, SITE_MMA_FULL)) break;
        tc_fence_after_sync();
        const uint32_t d = tmem_base + Cfg::kOCol;
        const uint32_t pa = tmem_base + Cfg::kSCol + static_cast<uint32_t>(b * kAttnBC);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t key_row = static_cast<uint32_t>(half * kHalfKeys + kk * 16);
            umma_bf16_tmem_a(d, pa + static_cast<uint32_t>(half * kHalfKeys + kk * 8),
                             smem_desc_mn_sw128(v_smem(s) + key_row * 128u, kChunkBytes), p.idesc_o,
                             (j | half | kk) != 0 ? 1u : 0u);
          }
        }
        umma_commit(o_done(b));
        umma_commit(v_empty(s));
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
    const uint32_t lane_base = tmem_addr(0, 32 * quarter, 0);
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
    // This thread's row of O: this warp's half of the D columns.
    const uint32_t t_o = tmem_base + lane_base + Cfg::kOCol + static_cast<uint32_t>(half * kHalfD);
    // Waits until O += P_j . V_j has completed (block j's products are in O).
    auto wait_o = [&](int j) -> bool {
      const bool got = wait_bounded(o_done(j % NB), use_parity(j), abort_flag, SITE_EPI_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) return false;
      tc_fence_after_sync();
      return true;
    };
    // This warp's half of O, 32 columns at a time, multiplied by f (per row).
    auto scale_o = [&](float f) {
#pragma unroll
      for (int c0 = 0; c0 < kHalfD; c0 += 32) {
        float o[32];
        tmem_load_32x32b_x32(t_o + c0, o);
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(o[i] * f);
        tmem_store_32x32b_x32(t_o + c0, w);
      }
    };
    float m = -INFINITY, l = 0.0f;   // m: the maximum this row's probabilities are taken against
    bool ok = true;
    const float c = p.scale_log2;
    for (int j = 0; j < n; ++j) {
      const int b = j % NB;
      const bool got = wait_bounded(s_full(b), use_parity(j), abort_flag, SITE_EPI_ACC_FULL);
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
      // Lazy rescaling: both warps of the row see the same block maximum and
      // the same m, so they take the same decision.  On the first block m is
      // -inf, so m moves and alpha = 0 (O and l hold nothing yet).
      const float m_blk = fmaxf(mine, other);
      float alpha = 1.0f;
      bool moved = false;
      if (m_blk > m + kAttnRescaleLog2) {
        alpha = fast_exp2(m - m_blk);
        m = m_blk;
        moved = j > 0;
      }
      if (__any_sync(0xffffffffu, moved)) {
        // O += P_{j-1} . V_{j-1} must be complete before its rows are scaled;
        // P_j . V_j is issued only after this warp arrives on p_full below.
        if (!wait_o(j - 1)) {
          ok = false;
          break;
        }
        scale_o(alpha);
      }
      // Pass 2: P = exp2(s * c - m) (at most 2^8), packed as BF16 pairs (even
      // key in the low half) into the first 32 columns of this half's scores,
      // and this half's row sum (four partial sums).
      float ps0 = 0.0f, ps1 = 0.0f, ps2 = 0.0f, ps3 = 0.0f;
      uint32_t w[kHalfKeys / 2];
#pragma unroll
      for (int i = 0; i < kHalfKeys; i += 4) {
        float q0 = fast_exp2(fmaf(v[i], c, -m));
        float q1 = fast_exp2(fmaf(v[i + 1], c, -m));
        float q2 = fast_exp2(fmaf(v[i + 2], c, -m));
        float q3 = fast_exp2(fmaf(v[i + 3], c, -m));
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
    }
    if (ok && n > 0) ok = wait_o(n - 1);
    // The row sum is the two halves' sums (both against the same m).
    float l_other = 0.0f;
    if (ok) ok = exchange(n, l, l_other);
    const int qrow = qb * kAttnBR + row;
    if (ok && n > 0) {
      const float inv = 1.0f / (l + l_other);
#pragma unroll
      for (int c0 = 0; c0 < kHalfD; c0 += 32) {
        float o[32];
        tmem_load_32x32b_x32(t_o + c0, o);
        if (qrow < p.Nq) {
          if (p.out_kind == 0) {
            float* dst = static_cast<float*>(p.O) + h * p.o_stride +
                         static_cast<long long>(qrow) * p.ldo + half * kHalfD + c0;
#pragma unroll
            for (int d = 0; d < 32; d += 4)
              *reinterpret_cast<float4*>(dst + d) =
                  make_float4(o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
          } else {
            uint16_t* dst = static_cast<uint16_t*>(p.O) + h * p.o_stride +
                            static_cast<long long>(qrow) * p.ldo + half * kHalfD + c0;
#pragma unroll
            for (int d = 0; d < 32; d += 8)
              *reinterpret_cast<uint4*>(dst + d) =
                  make_uint4(pack_bf16x2(o[d] * inv, o[d + 1] * inv),
                             pack_bf16x2(o[d + 2] * inv, o[d + 3] * inv),
                             pack_bf16x2(o[d + 4] * inv, o[d + 5] * inv),
                             pack_bf16x2(o[d + 6] * inv, o[d + 7] * inv));
          }
        }
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
