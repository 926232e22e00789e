// attention.cuh -- softmax attention O = softmax(scale * Q.K^T) . V on the
// tcgen05 tensor cores, as the flash-attention loop ("Tiles and shared
// memory", section "How long a tile lives": a query tile, a running maximum m
// and a running sum l kept across the key loop, s = dot_t(q, k) per key tile,
// acc / l at the end).
//
// One CTA per (head, 128-row query block).  The key blocks of 128 keys are
// dealt to two independent flash loops ("chains"): the even blocks to chain
// 0, the odd ones to chain 1.  Chain c owns a probability buffer P_c and an
// output accumulator O_c in Tensor Memory and keeps its own m_c and l_c.  Per
// key block j of chain c = j % 2:
//
//   S = Q . K_j^T                  tcgen05.mma M = 128, N = 128 over D (K_j is K-major:
//                                  D contiguous), into score buffer j % NS (at D = 64
//                                  blocks j and j + 1 as one set of N = 256 MMAs into
//                                  the two adjacent buffers)
//   m_c = max(m_c, rowmax S)       softmax warps of chain c: a query row is one TMEM lane
//   P_j = exp(S - m_c)             and one thread, which holds all 128 scores of its row
//   l_c = l_c a + rowsum P_j       (a = exp(m_old - m_new))
//   O_c += P_j . V_j               tcgen05.mma M = 128, N = D over the 128 keys, P_j stored
//                                  as BF16 in P_c and read from Tensor Memory as the A
//                                  operand, V_j the MN-major operand (D contiguous, as TMA
//                                  loads it)
//
// and at the end, with m = max(m_0, m_1),
//   O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)):
// the softmax sums over two disjoint key sets, each taken against its own
// maximum, merged exactly up to rounding.  Scores are handled in base-2
// units (exp2 of s * scale * log2 e), which is the same function.  Keys past
// Nk score -inf.
//
// Why two chains: a chain is serial -- P_j can be stored only once
// O_c += P_{j-2} . V_{j-2} has read P_c -- but the chains are independent,
// so the tensor core works on one chain's products while the other chain's
// softmax threads run, and every SM sub-partition has a warp of each chain
// to issue from.  No value is exchanged between warps inside the loop.  A
// score buffer is freed as soon as the softmax has loaded its scores into
// registers, so the next scores are computed while the softmax runs.
//
// The running maximum is updated lazily: the m a chain's probabilities are
// taken against moves only when a block's maximum exceeds it by more than
// kAttnRescaleLog2 (so probabilities stay below 2^8 and l_c, O_c keep their
// ratio), and only then is that row of O_c (and l_c) multiplied by a, in
// Tensor Memory, after O_c += P_{j-2} . V_{j-2} has completed and before
// P_j is stored.
//
// Tensor Memory (512 columns): NS score buffers of 128 FP32 columns (NS = 2,
// one per chain, at D = 64; NS = 1, shared by the chains, at D = 128), then
// P_0 and P_1 (64 columns of packed BF16 each), then O_0 and O_1 (D columns
// each).
//
// Warp roles: warp 0 TMA (Q once; K_j and V_j through separate rings, each
// refilled as soon as a slot frees), warp 1 MMA issue and TMEM owner, warps
// 2-5 the softmax of chain 0 and warps 6-9 that of chain 1 (warp w serves
// TMEM lane quarter w % 4).  The MMA thread issues the scores of block
// j + NS as soon as the softmax has read block j's scores out of the same
// buffer, and the P.V of block j once P_j is stored: in a fixed order with a
// buffer per chain, polling both conditions with one shared buffer.
//
// Every wait is bounded as in the GEMM kernels (status word, abort flag,
// drained copies and MMAs, TMEM freed).
#pragma once

#include "gemm_kernels.cuh"

namespace gb3 {

constexpr int kAttnBR = 128;   // query rows per CTA (the MMA's M)
constexpr int kAttnBC = 128;   // keys per block
constexpr int kAttnChains = 2;                             // key blocks dealt even / odd
constexpr int kAttnSoftWarps = 4 * kAttnChains;            // one per TMEM lane quarter and chain
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
  // Separate rings, each refilled as soon as a slot frees: a K slot when
  // S_j has completed, a V slot when O_c += P_j . V_j has.
  static constexpr int kKStages = D == 128 ? 3 : 6;
  static constexpr int kVStages = D == 128 ? 3 : 6;
  static constexpr int kQOffset = 0;
  static constexpr int kKOffset = kTileBytes;
  static constexpr int kVOffset = kKOffset + kKStages * kTileBytes;
  // [2 values (m, l)][2 chains][128 rows] floats, exchanged once at the end,
  // over Q (every MMA has completed by then)
  static constexpr int kRedOffset = kQOffset;
  static_assert(2 * kAttnChains * kAttnBR * 4 <= kTileBytes, "exchange area");
  static constexpr int kBarOffset = kVOffset + kVStages * kTileBytes;
  // Score buffers in Tensor Memory: block j's scores go to buffer j % kSBufs.
  static constexpr int kSBufs = D == 128 ? 1 : 2;
  // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_free[NS],
  // s_full[2], p_full[2], o_done[2], drain, xchg[4]
  static constexpr int kNumBars =
      1 + 2 * kKStages + 2 * kVStages + kSBufs + 3 * kAttnChains + 1 + 4;
  static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
  // Tensor Memory columns: S_b (128 FP32 scores) at kSCol + 128 b; P_c (128
  // BF16 probabilities, packed in pairs) at kPCol + 64 c; O_c at kOCol + D c.
  static constexpr int kTmemCols = 512;
  static constexpr int kSCol = 0;
  static constexpr int kPCol = kSBufs * kAttnBC;
  static constexpr int kOCol = kPCol + kAttnChains * (kAttnBC / 2);
  static_assert(kOCol + kAttnChains * D <= kTmemCols, "Tensor Memory columns");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Three-input maximum and minimum (one instruction each).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// (d0, d1) = (fma(a0, b, c), fma(a1, b, c)) as one paired FP32 instruction,
// each lane rounded exactly as fmaf rounds it.
__device__ __forceinline__ void fma2_bc(float& d0, float& d1, float a0, float a1, float b,
                                        float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %5};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (s0, s1) += (a0, a1) as one paired FP32 add.
__device__ __forceinline__ void add2(float& s0, float& s1, float a0, float a1) {
  asm("{\n\t.reg .b64 rs, ra;\n\t"
      "mov.b64 rs, {%0, %1};\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "add.rn.f32x2 rs, rs, ra;\n\t"
      "mov.b64 {%0, %1}, rs;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}

// 2^x by the hardware's approximate exp2 (relative error about 2^-22;
// results below the normal range flush to zero, exp2(-inf) = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One block's probabilities for one query row: p_i = exp2(s_i c - m), zero
// for keys at or past Nk when MASKED, rounded to BF16 pairs (to nearest
// even; even key in the low half) into w, and the row sum as four partial
// sums (lane-wise paired adds: partial k takes keys i with i % 4 == k).
template <bool MASKED>
__device__ __forceinline__ void attn_probabilities(const float (&v)[kAttnBC], float c, float m,
                                                   int col0, int Nk, uint32_t (&w)[kAttnBC / 2],
                                                   float& ps0, float& ps1, float& ps2,
                                                   float& ps3) {
#pragma unroll
  for (int i = 0; i < kAttnBC; i += 4) {
    float q0, q1, q2, q3;
    fma2_bc(q0, q1, v[i], v[i + 1], c, -m);
    fma2_bc(q2, q3, v[i + 2], v[i + 3], c, -m);
    q0 = fast_exp2(q0);
    q1 = fast_exp2(q1);
    q2 = fast_exp2(q2);
    q3 = fast_exp2(q3);
    if constexpr (MASKED) {
      const int k = col0 + i;
      q0 = k < Nk ? q0 : 0.0f;
      q1 = k + 1 < Nk ? q1 : 0.0f;
      q2 = k + 2 < Nk ? q2 : 0.0f;
      q3 = k + 3 < Nk ? q3 : 0.0f;
    }
    add2(ps0, ps1, q0, q1);
    add2(ps2, ps3, q2, q3);
    w[i / 2] = pack_bf16x2(q0, q1);
    w[i / 2 + 1] = pack_bf16x2(q2, q3);
  }
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using Cfg = AttnCfg<D>;
  constexpr int KS = Cfg::kKStages;
  constexpr int VS = Cfg::kVStages;
  constexpr int NS = Cfg::kSBufs;
  constexpr int NC = kAttnChains;
  constexpr int kChunkBytes = 128 * 128;  // one 64-element-wide swizzled chunk of 128 rows
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
  // A barrier that completes once per use of a set of R slots (a ring, the
  // score buffers, a chain) completes for block j's use in phase j / R, of
  // parity (j / R) & 1 (block j is use j / 2 of chain j % 2).  Each barrier
  // has one waiting role, which waits for every one of its phases in turn,
  // so a parity names one phase: the chain's own s_full, p_full and o_done
  // (not the shared score buffer's) are what the softmax warps and the MMA
  // thread wait on.
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (1 + KS + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * KS + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (1 + 2 * KS + VS + s); };
  constexpr int R0 = 1 + 2 * KS + 2 * VS;
  auto s_free = [&](int b) { return bar0 + 8u * (R0 + b); };            // S_b read by the softmax
  constexpr int R1 = R0 + NS;
  auto s_full = [&](int c) { return bar0 + 8u * (R1 + c); };            // chain c's scores ready
  auto p_full = [&](int c) { return bar0 + 8u * (R1 + NC + c); };       // P_j stored in P_c
  auto o_done = [&](int c) { return bar0 + 8u * (R1 + 2 * NC + c); };   // O_c += P_j . V_j done
  const uint32_t drain_bar = bar0 + 8u * (R1 + 3 * NC);                 // every MMA done
  auto xchg_bar = [&](int qtr) { return bar0 + 8u * (R1 + 3 * NC + 1 + qtr); };
  auto parity = [](int j, int r) { return static_cast<uint32_t>(j / r) & 1u; };

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
    for (int b = 0; b < NS; ++b) mbar_init(s_free(b), 4);   // the block's chain's four warps
    for (int c = 0; c < NC; ++c) {
      mbar_init(s_full(c), 1);
      mbar_init(p_full(c), 4);
      mbar_init(o_done(c), 1);
    }
    mbar_init(drain_bar, 1);
    for (int qtr = 0; qtr < 4; ++qtr) mbar_init(xchg_bar(qtr), NC);
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
      // K_j and V_j stream through their own rings, each refilled as soon
      // as a slot frees, so a late V does not hold back the next K.
      auto load_k = [&](int j) {
        const int s = j % KS;
        mbar_arrive_expect_tx(k_full(s), Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(k_smem(s) + c * kChunkBytes, &tmK, k_full(s), c * 64, j * kAttnBC, h);
      };
      auto load_v = [&](int j) {
        const int s = j % VS;
        mbar_arrive_expect_tx(v_full(s), Cfg::kTileBytes);
        for (int c = 0; c < Cfg::kChunks; ++c)
          tma_load_3d(v_smem(s) + c * kChunkBytes, &tmV, v_full(s), c * 64, j * kAttnBC, h);
      };
      int k_issued = 0, v_issued = 0;
      IdleBound bound;
      while (k_issued < n || v_issued < n) {
        bool issued = false;
        if (k_issued < n && mbar_test_wait(k_empty(k_issued % KS), parity(k_issued, KS) ^ 1u)) {
          load_k(k_issued++);
          issued = true;
        }
        if (v_issued < k_issued &&
            mbar_test_wait(v_empty(v_issued % VS), parity(v_issued, VS) ^ 1u)) {
          load_v(v_issued++);
          issued = true;
        }
        if (issued) {
          bound.progress();
          continue;
        }
        if (bound.expired(abort_flag, SITE_PRODUCER_EMPTY)) break;
        __nanosleep(20);
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
      // S_b = Q . K_j^T for block j into score buffer b = j % NS; chain
      // j % 2 is told on its own barrier.
      // Descriptors step through an operand by adding to their start-address
      // field (16-byte units): 2 per K = 16 step of a 128-byte row, 1024 per
      // 64-element chunk of 128 rows, 128 per 16 rows.
      const uint64_t qd0 = smem_desc_sw128(q_smem);
      auto issue_s = [&](int j) {
        const int s = j % KS, b = j % NS;
        const uint32_t d = tmem_base + Cfg::kSCol + static_cast<uint32_t>(b * kAttnBC);
        const uint64_t kd0 = smem_desc_sw128(k_smem(s));
#pragma unroll
        for (int ch = 0; ch < Cfg::kChunks; ++ch) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t step = static_cast<uint64_t>(ch * (kChunkBytes >> 4) + 2 * kk);
            umma_bf16(d, qd0 + step, kd0 + step, p.idesc_s, (ch | kk) != 0 ? 1u : 0u);
          }
        }
        umma_commit(s_full(j % NC));
        umma_commit(k_empty(s));
      };
      // O_c += P_j . V_j for chain c = j % 2 (O_c = P_j . V_j for the chain's
      // first block); P_j is read from P_c, 16 keys per 8 columns.
      auto issue_pv = [&](int j) {
        const int s = j % VS, c = j % NC;
        const uint32_t d = tmem_base + Cfg::kOCol + static_cast<uint32_t>(c * D);
        const uint32_t pa = tmem_base + Cfg::kPCol + static_cast<uint32_t>(c * (kAttnBC / 2));
        const uint64_t vd0 = smem_desc_mn_sw128(v_smem(s), kChunkBytes);
#pragma unroll
        for (int kk = 0; kk < kAttnBC / 16; ++kk)
          umma_bf16_tmem_a(d, pa + static_cast<uint32_t>(kk * 8),
                           vd0 + static_cast<uint64_t>(kk * (16 * 128 >> 4)), p.idesc_o,
                           (j >= NC || kk != 0) ? 1u : 0u);
        umma_commit(o_done(c));
        umma_commit(v_empty(s));
      };
      bool ok = wait_bounded(q_full, 0, abort_flag, SITE_MMA_FULL);
      if constexpr (NS >= 2) {
        // With a score buffer per chain, a fixed order: the scores of blocks
        // 0 and 1, then for each block j: at even j the scores of blocks j + 2
        // and j + 3 (once the softmax has read blocks j and j + 1 out of the
        // same buffers and the K blocks have landed), and the P.V of block j
        // (once P_j is stored and V_j has landed).  The softmax of block j
        // frees its score buffer before it stores P_j.  (Issuing the P.V one
        // block later instead measured slower; issuing the two blocks' scores
        // as one set of N = 256 MMAs saves an instruction per pair.)
        // The scores of blocks j and j + 1 (one per chain, buffers 0 and 1,
        // adjacent in Tensor Memory; K_j and K_{j+1} in adjacent ring slots)
        // as one set of N = 256 MMAs.
        constexpr uint32_t kIdescS2 = idesc_f32_acc(kAttnBR, 2 * kAttnBC, false);
        static_assert(KS % 2 == 0, "pairs of K slots must be adjacent");
        auto issue_s2 = [&](int j) {
          const int s = j % KS;
          const uint32_t d = tmem_base + Cfg::kSCol;
          const uint64_t kd0 = smem_desc_sw128(k_smem(s));
#pragma unroll
          for (int ch = 0; ch < Cfg::kChunks; ++ch) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t step = static_cast<uint64_t>(ch * (kChunkBytes >> 4) + 2 * kk);
              umma_bf16(d, qd0 + step, kd0 + step, kIdescS2, (ch | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit(s_full(0));
          umma_commit(s_full(1));
          umma_commit(k_empty(s));
          umma_commit(k_empty(s + 1));
        };
        auto scores_from = [&](int js) -> bool {   // the scores of js (even) and js + 1
          if (js + 1 < n) {
            if (!wait_bounded(k_full(js % KS), parity(js, KS), abort_flag, SITE_MMA_FULL) ||
                !wait_bounded(k_full((js + 1) % KS), parity(js + 1, KS), abort_flag, SITE_MMA_FULL))
              return false;
            tc_fence_after_sync();
            issue_s2(js);
          } else {
            if (!wait_bounded(k_full(js % KS), parity(js, KS), abort_flag, SITE_MMA_FULL))
              return false;
            tc_fence_after_sync();
            issue_s(js);
          }
          return true;
        };
        if (n > 0) ok = scores_from(0);
        for (int j = 0; ok && j < n; ++j) {
          const int js = j + 2;
          if (j % 2 == 0 && js < n) {
            if (!wait_bounded(s_free(0), parity(j, NS), abort_flag, SITE_MMA_ACC_EMPTY) ||
                (js + 1 < n &&
                 !wait_bounded(s_free(1), parity(j + 1, NS), abort_flag, SITE_MMA_ACC_EMPTY)) ||
                !scores_from(js))
              break;
          }
          if (!wait_bounded(p_full(j % NC), parity(j, NC), abort_flag, SITE_MMA_FULL) ||
              !wait_bounded(v_full(j % VS), parity(j, VS), abort_flag, SITE_MMA_FULL))
            break;
          tc_fence_after_sync();
          issue_pv(j);
        }
      } else {
        // With one score buffer shared by the chains, the scores of block j + 1
        // can be issued as soon as the other chain has read block j's, which
        // comes before or after P_{j-1} depending on the two softmaxes' pace:
        // poll both conditions and issue whichever product is ready (each
        // kind in block order; a ready P.V first, which measured ~1 % faster).
        int ns = 0, npv = 0;
        IdleBound bound;
        while (ok && npv < n) {
          bool issued = false;
          if (npv < ns) {
            const int j = npv;
            if (mbar_test_wait(p_full(j % NC), parity(j, NC)) &&
                mbar_test_wait(v_full(j % VS), parity(j, VS))) {
              tc_fence_after_sync();
              issue_pv(j);
              ++npv;
              issued = true;
            }
          }
          if (ns < n) {
            const int j = ns;
            if ((j < NS || mbar_test_wait(s_free(j % NS), parity(j - NS, NS))) &&
                mbar_test_wait(k_full(j % KS), parity(j, KS))) {
              tc_fence_after_sync();
              issue_s(j);
              ++ns;
              issued = true;
            }
          }
          if (issued) {
            bound.progress();
            continue;
          }
          if (bound.expired(abort_flag, SITE_MMA_FULL)) break;
          __nanosleep(20);
        }
      }
      // Every issued MMA completes before drain_bar does (bounded); the
      // softmax warps read O_0 and O_1 only after it.
      umma_commit(drain_bar);
      wait_bounded(drain_bar, 0, nullptr, SITE_DRAIN);
    }
  } else {
    // Softmax warps 2..9: warp w runs chain (w - 2) / 4 for query rows
    // 32*(w%4)..+31 (its TMEM lane quarter), one row per thread.
    const int chain = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = 32 * quarter + lane;             // query row of this thread in the block
    const uint32_t lane_base = tmem_base + tmem_addr(0, 32 * quarter, 0);
    const uint32_t t_p = lane_base + Cfg::kPCol + static_cast<uint32_t>(chain * (kAttnBC / 2));
    auto t_o = [&](int c) { return lane_base + Cfg::kOCol + static_cast<uint32_t>(c * D); };
    // This thread's row of O_chain, multiplied by f.
    auto scale_o = [&](float f) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float o[32];
        tmem_load_32x32b_x32(t_o(chain) + c0, o);
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(o[i] * f);
        tmem_store_32x32b_x32(t_o(chain) + c0, w);
      }
    };
    float m = -INFINITY, l = 0.0f;   // m: the maximum this chain's probabilities are taken against
    bool ok = true;
    const float c = p.scale_log2;
    for (int j = chain; j < n; j += NC) {
      const int b = j % NS;
      const bool got = wait_bounded(s_full(chain), parity(j, NC), abort_flag, SITE_EPI_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int col0 = j * kAttnBC;
      const bool full = col0 + kAttnBC <= p.Nk;
      // The row of S, once, into registers (128 scores); the buffer is then
      // free for the scores of block j + NS.
      float v[kAttnBC];
      tmem_load_32x32b_x128(lane_base + Cfg::kSCol + static_cast<uint32_t>(b * kAttnBC), v);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(b));
      // The block's maximum of the scaled scores (a full block needs no key
      // mask, and scaling by c is monotonic: c times the largest raw score,
      // the smallest for c < 0), four partial maxima.
      float m_blk;
      if (full) {
        const bool up = c >= 0.0f;
        float r0 = up ? -INFINITY : INFINITY, r1 = r0, r2 = r0, r3 = r0;
        if (up) {
#pragma unroll
          for (int i = 0; i < kAttnBC; i += 8) {
            r0 = max3f(r0, v[i], v[i + 1]);
            r1 = max3f(r1, v[i + 2], v[i + 3]);
            r2 = max3f(r2, v[i + 4], v[i + 5]);
            r3 = max3f(r3, v[i + 6], v[i + 7]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kAttnBC; i += 8) {
            r0 = min3f(r0, v[i], v[i + 1]);
            r1 = min3f(r1, v[i + 2], v[i + 3]);
            r2 = min3f(r2, v[i + 4], v[i + 5]);
            r3 = min3f(r3, v[i + 6], v[i + 7]);
          }
        }
        m_blk = (up ? fmaxf(fmaxf(r0, r1), fmaxf(r2, r3)) : fminf(fminf(r0, r1), fminf(r2, r3))) * c;
      } else {
        m_blk = -INFINITY;
#pragma unroll
        for (int i = 0; i < kAttnBC; ++i)
          if (col0 + i < p.Nk) m_blk = fmaxf(m_blk, v[i] * c);
      }
      // Lazy rescaling.  On the chain's first block m is -inf, so m moves
      // and alpha = 0 (O_chain and l hold nothing yet).
      float alpha = 1.0f;
      bool moved = false;
      if (m_blk > m + kAttnRescaleLog2) {
        alpha = fast_exp2(m - m_blk);
        m = m_blk;
        moved = j >= NC;
      }
      // P = exp2(s * c - m) (at most 2^8) rounded to BF16 pairs (to nearest
      // even; even key in the low half), and the row sum (four partial sums).
      float ps0 = 0.0f, ps1 = 0.0f, ps2 = 0.0f, ps3 = 0.0f;
      uint32_t w[kAttnBC / 2];
      // Two copies of the loop, so that a full block runs with no key test.
      if (full)
        attn_probabilities<false>(v, c, m, col0, p.Nk, w, ps0, ps1, ps2, ps3);
      else
        attn_probabilities<true>(v, c, m, col0, p.Nk, w, ps0, ps1, ps2, ps3);
      // O_chain += P_{j-2} . V_{j-2} must have completed: it reads P_chain,
      // and a rescaling of O_chain comes after it.
      if (j >= NC) {
        const bool done = wait_bounded(o_done(chain), parity(j - NC, NC), abort_flag,
                                       SITE_EPI_ACC_FULL);
        if (!__all_sync(0xffffffffu, done)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
      }
      if (__any_sync(0xffffffffu, moved)) scale_o(alpha);
      tmem_store_32x32b_x64(t_p, w);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(chain));
      l = fmaf(l, alpha, (ps0 + ps1) + (ps2 + ps3));
    }
    // Every MMA has completed once drain_bar has (O_0 and O_1 final).
    if (ok && n > 0) {
      const bool got = wait_bounded(drain_bar, 0, abort_flag, SITE_EPI_ACC_FULL);
      ok = __all_sync(0xffffffffu, got) && *abort_flag == 0;
      if (ok) tc_fence_after_sync();
    }
    // Exchange (m, l) with the other chain's warp of this lane quarter.
    float* xval = reinterpret_cast<float*>(smem + Cfg::kRedOffset);
    float m_x = -INFINITY, l_x = 0.0f;
    if (ok) {
      xval[(0 * NC + chain) * kAttnBR + row] = m;
      xval[(1 * NC + chain) * kAttnBR + row] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(xchg_bar(quarter));
      const bool got = wait_bounded(xchg_bar(quarter), 0, abort_flag, SITE_EPI_ACC_FULL);
      ok = __all_sync(0xffffffffu, got);
      if (ok) {
        m_x = xval[(0 * NC + (chain ^ 1)) * kAttnBR + row];
        l_x = xval[(1 * NC + (chain ^ 1)) * kAttnBR + row];
      }
    }
    const int qrow = qb * kAttnBR + row;
    if (ok && n > 0) {
      // Chain 1 has no blocks when n == 1: its O is never read.
      const bool two = n > 1;
      const float m0 = chain == 0 ? m : m_x, m1 = chain == 0 ? m_x : m;
      const float l0 = chain == 0 ? l : l_x, l1 = chain == 0 ? l_x : l;
      const float mm = fmaxf(m0, m1);
      const float f0 = fast_exp2(m0 - mm);
      const float f1 = two ? fast_exp2(m1 - mm) : 0.0f;
      const float inv = 1.0f / fmaf(l0, f0, l1 * f1);
      const float g0 = f0 * inv, g1 = f1 * inv;
      // This warp writes half of the D output columns of its rows.
      constexpr int kHalfD = D / 2;
#pragma unroll
      for (int c0 = 0; c0 < kHalfD; c0 += 32) {
        const int col = chain * kHalfD + c0;
        float o[32], o1[32];
        tmem_load_32x32b_x32(t_o(0) + col, o);
        if (two) {
          tmem_load_32x32b_x32(t_o(1) + col, o1);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = fmaf(o[i], g0, o1[i] * g1);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= g0;
        }
        if (qrow < p.Nq) {
          if (p.out_kind == 0) {
            float* dst = static_cast<float*>(p.O) + h * p.o_stride +
                         static_cast<long long>(qrow) * p.ldo + col;
#pragma unroll
            for (int d = 0; d < 32; d += 4)
              *reinterpret_cast<float4*>(dst + d) = make_float4(o[d], o[d + 1], o[d + 2], o[d + 3]);
          } else {
            uint16_t* dst = static_cast<uint16_t*>(p.O) + h * p.o_stride +
                            static_cast<long long>(qrow) * p.ldo + col;
#pragma unroll
            for (int d = 0; d < 32; d += 8)
              *reinterpret_cast<uint4*>(dst + d) =
                  make_uint4(pack_bf16x2(o[d], o[d + 1]), pack_bf16x2(o[d + 2], o[d + 3]),
                             pack_bf16x2(o[d + 4], o[d + 5]), pack_bf16x2(o[d + 6], o[d + 7]));
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
