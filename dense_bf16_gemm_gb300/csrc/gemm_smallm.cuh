// gemm_smallm.cuh -- small-M GEMM (M <= 128), bound by the HBM stream of B.
//
// As in the swapped-operand decode kernel, C^T = B(N,K) . A(M,K)^T: 128 weight
// rows fill the MMA's M side and the activation rows its N side (NX = 16, 32,
// 64 or 128).
//
// Work division (stream-K): the k-blocks of all tiles, tile after tile, form
// one sequence that is cut into gridDim.x contiguous ranges whose lengths
// differ by at most one.  A CTA walks its range as segments, one per tile it
// touches, each accumulated in one TMEM accumulator.  A segment that covers a
// whole tile is written straight to C.  A tile shared by several CTAs (its
// "pieces", numbered in K order) has each piece's FP32 partial written to a
// workspace slot (CTA index + tile index: both only grow along the sequence
// and every new segment advances one of them, so no two pieces share a slot);
// the last piece to arrive (an atomic counter per tile) adds the
// partials in piece order 0..P-1, applies alpha/beta and writes C, so the
// result does not depend on which CTA finishes last and no CTA waits for
// another.
//
// Why this shape (measured on GB300): one thread issues at most one
// tcgen05.mma of K = 16 per ~65 cycles when N (the activation rows) is small,
// and an M = 64 instruction takes as long as an M = 128 one, so a 128-row
// weight tile gives each instruction twice the bytes of B of a 64-row tile;
// each k-block also pays a barrier wait and a commit.  A 64-row kernel
// streamed B at about 32 GB/s per CTA, the 128-row one at about 60 GB/s, and
// HBM needs about 45 GB/s from each of the 152 SMs: so the tiles are 128
// rows and K is cut wherever the tiles alone would leave SMs idle (a 64 x
// 8192 x 8192 problem has 64 tiles for 152 SMs).
//
// Accumulator: D row i (weight row i of the tile) in TMEM lane i, activation
// row m in column m, so epilogue warp w (lanes 32*(w%4)..+31) holds weight
// rows 32*(w%4)..+31, one per lane.
//
// Roles: warp 0 TMA producer, warp 1 MMA issuer and TMEM owner, warps 2-5
// epilogue.  Two accumulators (2*NX TMEM columns) let the epilogue of one
// segment overlap the main loop of the next.
#pragma once

#include "gemm_kernels.cuh"

namespace gb3 {

constexpr int kSmallRows = 128;  // weight rows per tile (the MMA's M)

struct SmallMParams {
  int M, N, K;                // sizes of each matrix of the batch
  int n_blocks, k_blocks;     // ceil(N / 128), ceil(K / 64)
  int batch;
  int num_tiles;              // batch * n_blocks
  long long work;             // num_tiles * k_blocks: the k-block sequence
  long long work_per_cta;     // floor(work / gridDim.x) (>= 1)
  int work_extra;             // work % gridDim.x: CTAs 0..work_extra-1 take one more
  int max_pieces;             // most CTAs sharing one tile (reported by the plan)
  float alpha, beta;
  void* C;
  long long ldc;
  long long c_stride;         // elements between consecutive matrices of C
  int out_kind;               // 0 FP32, 1 BF16, 2 FP16
  uint32_t idesc;             // tcgen05 instruction descriptor (M = 128, N = NX)
  float* ws;      // [gridDim.x + num_tiles - 1][M][128] FP32 partials (max_pieces > 1)
  int* counters;  // [num_tiles] arrival counters (pieces of a tile), zero between calls
};

// First position of CTA c's range in the k-block sequence.
__host__ __device__ __forceinline__ long long smallm_range_start(const SmallMParams& p, int c) {
  return static_cast<long long>(c) * p.work_per_cta + (c < p.work_extra ? c : p.work_extra);
}

// The CTA whose range holds position x of the k-block sequence.
__host__ __device__ __forceinline__ int smallm_cta_of(const SmallMParams& p, long long x) {
  const long long big = static_cast<long long>(p.work_extra) * (p.work_per_cta + 1);
  if (x < big) return static_cast<int>(x / (p.work_per_cta + 1));
  return p.work_extra + static_cast<int>((x - big) / p.work_per_cta);
}

// One tile's share of a CTA's range: k-blocks kb0..kb1-1 of tile `tile`.
struct SmallMSeg {
  int tile, kb0, kb1;
};

// Walks CTA c's range: seg is the segment at `pos`; returns false past the end.
__device__ __forceinline__ bool smallm_segment(const SmallMParams& p, long long pos,
                                               long long end, SmallMSeg& seg) {
  if (pos >= end) return false;
  seg.tile = static_cast<int>(pos / p.k_blocks);
  const long long base = static_cast<long long>(seg.tile) * p.k_blocks;
  seg.kb0 = static_cast<int>(pos - base);
  seg.kb1 = static_cast<int>(end - base < p.k_blocks ? end - base : p.k_blocks);
  return true;
}

__device__ __forceinline__ long long smallm_next(const SmallMParams& p, const SmallMSeg& seg) {
  return static_cast<long long>(seg.tile) * p.k_blocks + seg.kb1;
}

// NX: activation rows per MMA (the MMA's N), 16, 32, 64 or 128.
template <int NX>
struct SmallMCfg {
  static_assert(NX == 16 || NX == 32 || NX == 64 || NX == 128, "activation tile");
  static constexpr int kWBytes = kSmallRows * kBK * 2;  // 16 KB
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

// C[m][n] of matrix b = alpha * acc + beta * C[m][n] (one rounding to a 16-bit
// output, from the FP32 value).
__device__ __forceinline__ void smallm_store_one(const SmallMParams& p, int b, int m, int n,
                                                 float acc) {
  const long long off = b * p.c_stride + static_cast<long long>(m) * p.ldc + n;
  float v = __fmul_rn(p.alpha, acc);
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

// Activation rows m0..m0+kCols-1 of output column n.
template <int kCols>
__device__ __forceinline__ void smallm_store(const SmallMParams& p, int b, int n, int m0,
                                             const float* acc) {
  if (n >= p.N) return;
#pragma unroll
  for (int i = 0; i < kCols; ++i)
    if (m0 + i < p.M) smallm_store_one(p, b, m0 + i, n, acc[i]);
}

// Reads tile nb's rows of C (matrix b) once, by the 128 epilogue threads, so
// that they sit in L2 when the combine writes them at the end of the call:
// measured on GB300 after an L2 flush, 64 x 4096 x 4096 22.6 us with this
// against 24.6 without.  Only whole 16-byte pieces inside the row are read;
// the values are not used.
__device__ __forceinline__ void smallm_touch_c(const SmallMParams& p, int b, int nb, int tid) {
  const int es = p.out_kind != 0 ? 2 : 4;
  const int per_row = kSmallRows * es / 16;  // 16-byte pieces per tile row
  const char* base = static_cast<const char*>(p.C);
  for (int idx = tid; idx < p.M * per_row; idx += 128) {
    const int m = idx / per_row, piece = idx - m * per_row;
    const long long n = static_cast<long long>(nb) * kSmallRows + piece * (16 / es);
    if (n + 16 / es > p.N) continue;
    const char* a = base + (b * p.c_stride + static_cast<long long>(m) * p.ldc + n) * es;
    uint32_t x, y, z, w;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(x), "=r"(y), "=r"(z), "=r"(w)
                 : "l"(a));
    asm volatile("" ::"r"(x), "r"(y), "r"(z), "r"(w));  // the values are not needed
  }
}

// C[m][n0..n0+CPT-1] of matrix b from the FP32 sums v (alpha, beta as in
// smallm_store_one), written by one 16-byte store when all CPT columns exist
// and the address is aligned: CPT = 8 for a 16-bit C, 4 for FP32 C.
template <int CPT>
__device__ __forceinline__ void smallm_store_run(const SmallMParams& p, int b, int m, int n0,
                                                 const float (&v)[CPT]) {
  const long long off = b * p.c_stride + static_cast<long long>(m) * p.ldc + n0;
  if (n0 + CPT - 1 < p.N) {
    const int es = p.out_kind != 0 ? 2 : 4;
    void* c = static_cast<char*>(p.C) + off * es;
    if ((reinterpret_cast<uintptr_t>(c) & 15u) == 0 && CPT * es == 16) {
      float y[CPT];
#pragma unroll
      for (int i = 0; i < CPT; ++i) y[i] = __fmul_rn(p.alpha, v[i]);
      if constexpr (CPT == 8) {
        const bool f16 = p.out_kind == 2;
        if (p.beta != 0.0f) {
          const uint4 old = *static_cast<const uint4*>(c);
          const uint32_t w[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            y[2 * j] = __fmaf_rn(p.beta, half16_to_float(w[j] & 0xFFFFu, f16), y[2 * j]);
            y[2 * j + 1] = __fmaf_rn(p.beta, half16_to_float(w[j] >> 16, f16), y[2 * j + 1]);
          }
        }
        *static_cast<uint4*>(c) =
            make_uint4(pack_half16x2(y[0], y[1], f16), pack_half16x2(y[2], y[3], f16),
                       pack_half16x2(y[4], y[5], f16), pack_half16x2(y[6], y[7], f16));
      } else {
        if (p.beta != 0.0f) {
          const float4 old = *static_cast<const float4*>(c);
          y[0] = __fmaf_rn(p.beta, old.x, y[0]);
          y[1] = __fmaf_rn(p.beta, old.y, y[1]);
          y[2] = __fmaf_rn(p.beta, old.z, y[2]);
          y[3] = __fmaf_rn(p.beta, old.w, y[3]);
        }
        *static_cast<float4*>(c) = make_float4(y[0], y[1], y[2], y[3]);
      }
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < CPT; ++i)
    if (n0 + i < p.N) smallm_store_one(p, b, m, n0 + i, v[i]);
}

// The combine of a shared tile by the 128 epilogue threads (tid 0..127): the
// partials of pieces 0..pieces-1 (slot first + pc + tile, laid out [M][128])
// are added in piece order and written to C.  128 / CPT threads cover one row
// of the tile (CPT consecutive outputs each: 16 bytes of C), so every warp
// store writes whole 32-byte sectors of C rows, and every C row segment is
// written at once: per-warp 32-column slices written at different times were
// measured to make the final stores of the call several times slower.  Each
// thread issues the loads of 4 rows of a piece before adding them.
template <int CPT>
__device__ __forceinline__ void smallm_combine_rows(const SmallMParams& p, int bt, int tile,
                                                    int nb, int first, int pieces, int tid) {
  constexpr int kTpr = kSmallRows / CPT;  // threads per row
  constexpr int kRpp = 128 / kTpr;        // rows per pass of the 128 threads
  constexpr int kV = CPT / 4;             // float4 per thread and row
  const int cn = (tid % kTpr) * CPT;      // first weight row within the tile
  const int n0 = nb * kSmallRows + cn;
#pragma unroll 1
  for (int m0 = tid / kTpr; m0 < p.M; m0 += 4 * kRpp) {
    float4 sum[4][kV];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int h = 0; h < kV; ++h) sum[k][h] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
    for (int pc = 0; pc < pieces; ++pc) {
      const float* base =
          p.ws + (static_cast<long long>(first + pc) + tile) * p.M * kSmallRows + cn;
      float4 v[4][kV];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int m = m0 + kRpp * k;
        const float4* src = reinterpret_cast<const float4*>(base + static_cast<long long>(m) * kSmallRows);
        const bool in = m < p.M;
#pragma unroll
        for (int h = 0; h < kV; ++h)
          v[k][h] = in ? __ldcg(src + h) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int h = 0; h < kV; ++h) {
          sum[k][h].x += v[k][h].x;
          sum[k][h].y += v[k][h].y;
          sum[k][h].z += v[k][h].z;
          sum[k][h].w += v[k][h].w;
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int m = m0 + kRpp * k;
      if (m < p.M) {
        float out[CPT];
#pragma unroll
        for (int h = 0; h < kV; ++h) {
          out[4 * h + 0] = sum[k][h].x;
          out[4 * h + 1] = sum[k][h].y;
          out[4 * h + 2] = sum[k][h].z;
          out[4 * h + 3] = sum[k][h].w;
        }
        smallm_store_run<CPT>(p, bt, m, n0, out);
      }
    }
  }
}

__device__ __forceinline__ void smallm_combine_tile(const SmallMParams& p, int bt, int tile,
                                                    int nb, int first, int pieces, int tid) {
  if (p.out_kind != 0)
    smallm_combine_rows<8>(p, bt, tile, nb, first, pieces, tid);
  else
    smallm_combine_rows<4>(p, bt, tile, nb, first, pieces, tid);
}

template <int NX>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_smallm_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmX, const SmallMParams p) {
  using Cfg = SmallMCfg<NX>;
  constexpr int STAGES = Cfg::kStages;
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
  // This CTA's range of the k-block sequence (every segment is non-empty).
  const long long range0 = smallm_range_start(p, blockIdx.x);
  const long long range1 = smallm_range_start(p, blockIdx.x + 1);

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t stream_policy = l2_policy_evict_first();  // B is read once
      const uint64_t keep_policy = l2_policy_evict_last();     // A is re-read by every unit
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      bool ok = true;
      SmallMSeg seg;
      for (long long pos = range0; ok && smallm_segment(p, pos, range1, seg);
           pos = smallm_next(p, seg)) {
        const int bt = seg.tile / p.n_blocks, nb = seg.tile - bt * p.n_blocks;
        for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
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
      SmallMSeg seg;
      for (long long pos = range0; ok && smallm_segment(p, pos, range1, seg);
           pos = smallm_next(p, seg), ++local) {
        const int buf = local & 1;
        const uint32_t aph = static_cast<uint32_t>(local >> 1) & 1u;
        if (!wait_bounded(acce_bar(buf), aph ^ 1u, abort_flag, SITE_MMA_ACC_EMPTY)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * Cfg::kAccStride);
        for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
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
                      (kb != seg.kb0 || j != 0) ? 1u : 0u);
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
    const int quarter = warp & 3;  // TMEM lanes (weight rows) 32*quarter..+31
    const uint32_t lane_base = tmem_addr(0, 32 * quarter, 0);
    constexpr int kGroup = NX < 64 ? NX : 64;  // columns held in registers at once
    const int col = 32 * quarter + lane;  // weight row within the tile
    const int tid = static_cast<int>(threadIdx.x) - 64;  // 0..127 over the epilogue warps
    __shared__ int arrivals_before;  // pieces of the current tile that arrived before this one
    int local = 0;
    SmallMSeg seg;
    for (long long pos = range0; smallm_segment(p, pos, range1, seg);
         pos = smallm_next(p, seg), ++local) {
      const int bt = seg.tile / p.n_blocks, nb = seg.tile - bt * p.n_blocks;
      const int buf = local & 1;
      const uint32_t aph = static_cast<uint32_t>(local >> 1) & 1u;
      // The last segment of a range is a tile's first piece, which almost
      // always arrives last and combines: fetch that tile's C while it runs.
      if (!(seg.kb0 == 0 && seg.kb1 == p.k_blocks) && smallm_next(p, seg) >= range1)
        smallm_touch_c(p, bt, nb, tid);
      const bool got = wait_bounded(accf_bar(buf), aph, abort_flag, SITE_EPI_ACC_FULL);
      // All four epilogue warps leave together (they meet at named barriers below).
      if (!named_barrier_and(1, 128, got)) break;
      tc_fence_after_sync();
      const int n = nb * kSmallRows + col;
      // A tile shared by several CTAs: its pieces are the CTAs whose ranges
      // hold its first to its last k-block, in K order.
      const bool whole = seg.kb0 == 0 && seg.kb1 == p.k_blocks;
      int first = static_cast<int>(blockIdx.x), pieces = 1;
      if (!whole) {
        const long long tile_pos = static_cast<long long>(seg.tile) * p.k_blocks;
        first = smallm_cta_of(p, tile_pos);
        pieces = smallm_cta_of(p, tile_pos + p.k_blocks - 1) - first + 1;
      }
      const int piece = static_cast<int>(blockIdx.x) - first;
      // Piece pc of this tile in slot first + pc + tile.
      auto ws_at = [&](int pc, int m) {
        return p.ws + ((static_cast<long long>(first + pc) + seg.tile) * p.M + m) * kSmallRows +
               col;
      };
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
        if (g0 < p.M) {
          if (whole) {
            smallm_store<kGroup>(p, bt, n, g0, acc);
          } else if (n < p.N) {
#pragma unroll
            for (int i = 0; i < kGroup; ++i)
              if (g0 + i < p.M) *ws_at(piece, g0 + i) = acc[i];
          }
        }
      }
      if (whole) continue;
      // Publish this piece (all four bands), then count it once for the tile.
      int* counter = p.counters + seg.tile;
      named_barrier_sync(1, 128);
      if (tid == 0) {
        __threadfence();
        arrivals_before = atomicAdd(counter, 1);
      }
      named_barrier_sync(1, 128);
      if (arrivals_before != pieces - 1) continue;
      __threadfence();
      smallm_combine_tile(p, bt, seg.tile, nb, first, pieces, tid);
      if (tid == 0) *counter = 0;  // ready for the next call
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
