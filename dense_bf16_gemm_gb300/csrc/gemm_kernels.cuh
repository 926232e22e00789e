// gemm_kernels.cuh -- persistent, warp-specialised tcgen05 GEMM kernels for
// sm_103a.
//
//   warp 0      TMA producer: one thread streams A and B k-blocks into a
//               STAGES-deep shared-memory ring (full/empty mbarriers with
//               transaction counts).
//   warp 1      MMA issuer: one thread issues tcgen05.mma (BF16 x BF16 -> FP32)
//               into one of two TMEM accumulators and commits completion to
//               the ring's empty barriers and to the accumulator's full
//               barrier.  The same warp allocates and frees TMEM.
//   warps 2-5   epilogue: warp w reads TMEM lanes 32*(w%4)..+31 (the row band
//               it may access) with tcgen05.ld, applies alpha/beta or
//               silu(gate)*up in FP32, packs, stages the tile in 128-byte
//               swizzled shared memory and writes it with TMA stores.
//
// Two accumulators let the epilogue of one tile overlap the main loop of the
// next.  Tiles are visited by a static persistent schedule (tile = blockIdx.x
// + i*gridDim.x) in grouped row order for L2 reuse.
//
// Every pipeline wait is bounded: past kWaitLimitNs the waiting thread sets a
// CTA abort flag and the device status word, every role leaves its loop, the
// in-flight copies and MMAs are drained (again with a bound), TMEM is freed
// and the kernel returns.
#pragma once

#include "ptx.cuh"

namespace gb3 {

constexpr int kBM = 128;          // tile rows = tcgen05 M (cta_group::1)
constexpr int kBK = 64;           // K per stage: one 128-byte swizzle row of BF16
constexpr int kUmmaK = 16;        // K of one tcgen05.mma kind::f16
constexpr int kThreads = 192;     // 6 warps
constexpr int kEpiWarps = 4;
constexpr int kStageBox = 4096;   // one epilogue store box: 32 rows x 128 bytes
constexpr int kStagingPerWarp = 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

enum EpiMode : int { EPI_F32 = 0, EPI_BF16 = 1, EPI_GATE_UP = 2 };

enum WaitSite : int {
  SITE_PRODUCER_EMPTY = 1,
  SITE_MMA_FULL = 2,
  SITE_MMA_ACC_EMPTY = 3,
  SITE_EPI_ACC_FULL = 4,
  SITE_DRAIN = 5,
  SITE_SKINNY = 6,
  SITE_SELFTEST = 7,
  SITE_EPI_C_FULL = 8,
  SITE_LAUNCH_SMEM = 9,
  SITE_GRID_SYNC = 10
};

// [0] status code, [1] wait site, [2] block index of the first failure.
__device__ int g_gemm_status[4];

__device__ __noinline__ void record_timeout(int site) {
  if (atomicCAS(&g_gemm_status[0], 0, 5) == 0) {
    g_gemm_status[1] = site;
    g_gemm_status[2] = static_cast<int>(blockIdx.x);
  }
}

// Entry check of every kernel with a dynamic shared-memory layout: a launch
// that gave less dynamic shared memory than the layout needs records status
// 4 (GEMM_ERR_CUDA) at site SITE_LAUNCH_SMEM, and every thread of the grid
// returns before touching shared memory, instead of running past the end of
// its allocation.  Uniform over the grid, so no CTA of a cluster is left
// waiting for a peer.
__device__ __forceinline__ bool launch_smem_ok(uint32_t need) {
  uint32_t have;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(have));
  if (have >= need) return true;
  if (threadIdx.x == 0 && atomicCAS(&g_gemm_status[0], 0, 4) == 0) {
    g_gemm_status[1] = SITE_LAUNCH_SMEM;
    g_gemm_status[2] = static_cast<int>(blockIdx.x);
  }
  return false;
}

template <bool kClusterScope = false>
__device__ __forceinline__ bool try_wait_scoped(uint32_t bar, uint32_t parity) {
  if constexpr (kClusterScope)
    return mbar_try_wait_cluster(bar, parity);
  else
    return mbar_try_wait(bar, parity);
}

// The global timer is read only every 256 failed attempts, starting from the
// first such check (a timer read costs the waiting thread far more than a
// try_wait), so a wait that completes soon pays nothing for its bound.
template <bool kClusterScope>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       int site, uint64_t limit_ns) {
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (try_wait_scoped<kClusterScope>(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      const uint64_t now = global_timer_ns();
      if (i == 256u) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        if (abort_flag != nullptr) *abort_flag = 1;
        record_timeout(site);
        return false;
      }
    }
  }
}

// Bound of a polling loop that serves several barriers (mbar_test_wait on
// each, no thread suspended): the clock starts at the 32nd pass in a row
// that made no progress and is read every 32 such passes, so progress never
// waits for a timer read.  expired() also reports an abort of the CTA.
struct IdleBound {
  uint64_t t0 = 0;
  uint32_t idle = 0;
  __device__ __forceinline__ void progress() { idle = 0; }
  __device__ __forceinline__ bool expired(volatile int* abort_flag, int site) {
    if ((++idle & 31u) != 0) return false;
    if (*abort_flag) return true;
    const uint64_t now = global_timer_ns();
    if (idle == 32u) {
      t0 = now;
      return false;
    }
    if (now - t0 <= kWaitLimitNs) return false;
    *abort_flag = 1;
    record_timeout(site);
    return true;
  }
};

// Waits for the phase of parity `parity` of `bar` to complete.  Returns false
// if the CTA aborted or the wait exceeded its limit.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, int site,
                                             uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow<false>(bar, parity, abort_flag, site, limit_ns);
}

// Same for a barrier that threads of the other CTA of a cluster arrive on
// (acquires at cluster scope).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                     volatile int* abort_flag, int site) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return wait_slow<true>(bar, parity, abort_flag, site, kWaitLimitNs);
}

// Self-test of the failure path: one thread waits on a barrier nothing
// arrives on, so the wait runs out after limit_ns and records
// GEMM_ERR_TIMEOUT with site SITE_SELFTEST.  Uses no TMA and no TMEM.
__global__ void wait_timeout_probe_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
    wait_bounded(smem_u32(&bar), 0, &abort_flag, SITE_SELFTEST, limit_ns);
  }
}

struct TileParams {
  int M, N, K;                // sizes of each matrix of the batch
  int m_blocks, n_blocks, k_blocks;
  int batch;                  // matrices (the third TMA coordinate)
  int tiles_per_matrix;       // m_blocks * n_blocks
  int num_tiles;              // batch * tiles_per_matrix
  int group_m;
  uint32_t idesc;             // tcgen05 instruction descriptor (BF16 or FP16 operands)
  int out_f16;                // a 16-bit output is FP16 (else BF16)
  long long c_stride;         // elements between consecutive matrices of C
  float alpha, beta;
  const void* C;      // read when beta != 0 (same storage as the output)
  long long ldc;      // elements
  // Work units: first the pieces of the "tail" tiles num_full .. num_tiles-1,
  // each cut into tail_split pieces of kb_per_piece k-blocks (the last piece
  // may be shorter), then tiles 0 .. num_full-1 whole.  The pieces come first
  // so that their partial-sum epilogues overlap later main loops.
  // num_units = (num_tiles - num_full) * tail_split + num_full.
  int num_full;
  int tail_split;
  int kb_per_piece;
  int num_units;
  // Balanced division (CTA-pair kernels, balanced != 0): the k-blocks of all
  // tiles, tile after tile, form one sequence of num_tiles * k_blocks
  // positions cut into one contiguous range per cluster, the ranges differing
  // in length by at most one (cluster c starts at c * work_per_cluster +
  // min(c, work_extra)).  A tile whose k-blocks fall in several ranges is
  // summed from its pieces (one per range, numbered in K order) by the
  // piece that arrives last.  The tail-split fields above are then unused.
  int balanced;
  long long work_per_cluster;
  int work_extra;
  // With the balanced division: its first dp_tiles tiles (a multiple of the
  // clusters) run whole, dp_tiles / clusters per cluster in round-robin order,
  // before each cluster's balanced range over the remaining tiles' k-blocks
  // (whose tile indices the ranges count from dp_tiles).
  int dp_tiles;
  // Strips (CTA-pair kernels of 256-column tiles, strip_tiles > 0): the last
  // strip_tiles tiles run as kPairStripN-column strips of the whole K, one
  // unit each, after every whole tile; num_full = num_tiles - strip_tiles and
  // tail_split = 1.  A strip needs no partial sums.
  int strip_tiles;
  uint32_t idesc_strip;       // tcgen05 instruction descriptor of a strip (N = kPairStripN)
  float* ws;          // FP32 partial tiles of split pieces
  int* counters;      // arrivals per (split tile, 32-row band), zero between calls
};

// One unit of a cluster's work: k-blocks kb0..kb1-1 of tile `tile`, piece
// `piece` of `pieces` (pieces == 1: the whole tile, piece 0); strip >= 0: the
// unit is that kPairStripN-column strip of the tile (all of K).
struct WorkUnit {
  int tile, kb0, kb1, piece, pieces, strip;
};

constexpr int kPairStripN = 64;   // columns of a strip of a 256-column pair tile

// Reductions along each row of the result (kernels instantiated with STATS):
// the sum, maximum and minimum over n of the FP32 values alpha*acc + beta*c,
// before any output rounding.  Every warp band of every tile stores the
// partials of its 32 rows over the tile's columns, and the band's last
// arrival over the n_blocks column tiles combines them in column-tile order.
// A separate kernel parameter, so that the plain kernels' parameters (and
// code) do not change.
struct RowStatsParams {
  float* row_sum;       // [batch][M]; each may be nullptr (not wanted)
  float* row_max;
  float* row_min;
  float* ws;            // partials [3][batch][n_blocks][M]
  int* counters;        // arrivals per (matrix, 32-row band), zero between calls
};

// Tile, k-block range and piece (-1: whole tile) of work unit u.
__device__ __forceinline__ void unit_of(int u, const TileParams& p, int& tile, int& kb0, int& kb1,
                                        int& piece) {
  const int split_units = (p.num_tiles - p.num_full) * p.tail_split;
  if (u >= split_units) {
    tile = u - split_units;
    kb0 = 0;
    kb1 = p.k_blocks;
    piece = -1;
  } else {
    tile = p.num_full + u / p.tail_split;
    piece = u % p.tail_split;
    kb0 = piece * p.kb_per_piece;
    kb1 = min(p.k_blocks, kb0 + p.kb_per_piece);
  }
}

// First position of cluster c's range in the balanced division.
__host__ __device__ __forceinline__ long long balanced_start(long long per, int extra, int c) {
  return static_cast<long long>(c) * per + (c < extra ? c : extra);
}

// The cluster whose balanced range holds position x.
__host__ __device__ __forceinline__ int balanced_owner(long long per, int extra, long long x) {
  const long long big = static_cast<long long>(extra) * (per + 1);
  if (x < big) return static_cast<int>(x / (per + 1));
  return extra + static_cast<int>((x - big) / per);
}

// The tiles a balanced range [r0, r1) touches: first and last tile, and
// whether the range holds only part of each.
struct BalancedRange {
  int t_first, t_last;
  bool first_part, last_part;  // last_part is false when t_last == t_first
};

__host__ __device__ __forceinline__ BalancedRange balanced_range(long long r0, long long r1,
                                                                 int k_blocks) {
  BalancedRange b;
  b.t_first = static_cast<int>(r0 / k_blocks);
  b.t_last = static_cast<int>((r1 - 1) / k_blocks);
  const long long f0 = static_cast<long long>(b.t_first) * k_blocks;
  b.first_part = r0 != f0 || r1 < f0 + k_blocks;
  b.last_part = b.t_last != b.t_first && r1 != static_cast<long long>(b.t_last + 1) * k_blocks;
  return b;
}

// Units of cluster c under the balanced division: the partial tiles of its
// range first, the shorter one first (so that their partial-sum epilogues
// overlap later main loops, and the first one's epilogue the longer second
// main loop), then its whole tiles in order.
__host__ __device__ __forceinline__ int balanced_units(long long per, int extra, int k_blocks,
                                                       int c) {
  const long long r0 = balanced_start(per, extra, c), r1 = balanced_start(per, extra, c + 1);
  if (r1 <= r0) return 0;
  const BalancedRange b = balanced_range(r0, r1, k_blocks);
  return b.t_last - b.t_first + 1;
}

__host__ __device__ __forceinline__ WorkUnit balanced_unit(long long per, int extra, int k_blocks,
                                                           int c, int i) {
  const long long r0 = balanced_start(per, extra, c), r1 = balanced_start(per, extra, c + 1);
  const BalancedRange b = balanced_range(r0, r1, k_blocks);
  const int parts = (b.first_part ? 1 : 0) + (b.last_part ? 1 : 0);
  int t;
  if (parts == 2) {
    // k-blocks of the first tile's piece and of the last tile's piece
    const long long len_first = static_cast<long long>(b.t_first + 1) * k_blocks - r0;
    const long long len_last = r1 - static_cast<long long>(b.t_last) * k_blocks;
    const bool last_first = len_last < len_first;
    if (i == 0) t = last_first ? b.t_last : b.t_first;
    else if (i == 1) t = last_first ? b.t_first : b.t_last;
    else t = b.t_first + 1 + (i - 2);
  } else if (i < parts)
    t = b.first_part ? b.t_first : b.t_last;
  else
    t = b.t_first + (b.first_part ? 1 : 0) + (i - parts);
  const long long f0 = static_cast<long long>(t) * k_blocks;
  WorkUnit u;
  u.tile = t;
  u.strip = -1;
  u.kb0 = static_cast<int>((r0 > f0 ? r0 : f0) - f0);
  u.kb1 = static_cast<int>((r1 < f0 + k_blocks ? r1 : f0 + k_blocks) - f0);
  const int c0 = balanced_owner(per, extra, f0);
  u.piece = c - c0;
  u.pieces = balanced_owner(per, extra, f0 + k_blocks - 1) - c0 + 1;
  return u;
}

// Partial-sum slot of piece q of tile t under the balanced division: every
// cluster has at most two partial tiles, the one its range starts in (slot
// 2c) and the one it ends in (slot 2c + 1).  Pieces q >= 1 start their
// cluster's range; piece 0 does only when the tile starts its range.
__host__ __device__ __forceinline__ long long balanced_slot(long long per, int extra, int k_blocks,
                                                            int t, int q) {
  const long long f0 = static_cast<long long>(t) * k_blocks;
  const int c0 = balanced_owner(per, extra, f0);
  if (q > 0) return 2LL * (c0 + q);
  return 2LL * c0 + (balanced_start(per, extra, c0) == f0 ? 0 : 1);
}

// Arrival counters (eight, one per 32-row band) of split tile t under the
// balanced division: those of the cluster holding its piece 1, whose range
// starts inside t (every range starts in one tile).
__host__ __device__ __forceinline__ int balanced_counter(long long per, int extra, int k_blocks,
                                                         int t) {
  return balanced_owner(per, extra, static_cast<long long>(t) * k_blocks) + 1;
}

// Units of cluster `cluster` (of `nclusters`) and the i-th of them: the
// balanced division, or the round-robin order of the tail-split units.
__device__ __forceinline__ int cluster_unit_count(const TileParams& p, int cluster, int nclusters) {
  if (p.balanced)
    return p.dp_tiles / nclusters +
           balanced_units(p.work_per_cluster, p.work_extra, p.k_blocks, cluster);
  return cluster < p.num_units ? (p.num_units - 1 - cluster) / nclusters + 1 : 0;
}

__device__ __forceinline__ WorkUnit cluster_unit(const TileParams& p, int cluster, int nclusters,
                                                 int i) {
  if (p.balanced) {
    const int dp = p.dp_tiles / nclusters;
    if (i < dp) {
      WorkUnit w;
      w.tile = cluster + i * nclusters;
      w.kb0 = 0;
      w.kb1 = p.k_blocks;
      w.piece = 0;
      w.pieces = 1;
      w.strip = -1;
      return w;
    }
    WorkUnit w = balanced_unit(p.work_per_cluster, p.work_extra, p.k_blocks, cluster, i - dp);
    w.tile += p.dp_tiles;
    return w;
  }
  WorkUnit u;
  u.strip = -1;
  if (p.strip_tiles > 0) {
    // whole tiles first, then the strips of the last strip_tiles tiles
    const int v = cluster + i * nclusters;
    const int whole = p.num_tiles - p.strip_tiles;
    u.kb0 = 0;
    u.kb1 = p.k_blocks;
    u.piece = 0;
    u.pieces = 1;
    if (v < whole) {
      u.tile = v;
    } else {
      constexpr int kStrips = 256 / kPairStripN;
      u.tile = whole + (v - whole) / kStrips;
      u.strip = (v - whole) % kStrips;
    }
    return u;
  }
  unit_of(cluster + i * nclusters, p, u.tile, u.kb0, u.kb1, u.piece);
  u.pieces = u.piece < 0 ? 1 : p.tail_split;
  if (u.piece < 0) u.piece = 0;
  return u;
}

// Where one warp band (32 rows) of a split tile keeps its partial sums.  The
// layout is private to the kernel and chosen for coalescing: 32-column slice
// c of the band is stored as 8 runs of 32 float4, run q holding lane i's
// q-th float4 at position i, so every warp-wide store or load of a run moves
// 512 contiguous bytes.  A band's partial is 32 * width floats.  Piece 0's
// partial is at ws0, piece q >= 1's at ws1 + (q - 1) * rest_stride.
struct SplitCtx {
  int pieces;              // 1: the unit is a whole tile
  int piece;               // this unit's piece
  const float4* ws0;       // band partial of piece 0
  const float4* ws1;       // band partial of piece 1
  long long rest_stride;   // float4s between the partials of pieces q and q + 1 (q >= 1)
};

__device__ __forceinline__ const float4* piece_partial(const SplitCtx& sp, int q) {
  return q == 0 ? sp.ws0 : sp.ws1 + (q - 1) * sp.rest_stride;
}

__device__ __forceinline__ long long split_index(int col, int q, int lane) {
  return (static_cast<long long>(col >> 5) * 8 + q) * 32 + lane;
}

// Matrix b of the batch, then a grouped raster inside it: group_m
// consecutive row blocks share each column block.
__device__ __forceinline__ void tile_coords(int tile, const TileParams& p, int& b, int& mb,
                                            int& nb) {
  b = tile / p.tiles_per_matrix;
  const int t = tile - b * p.tiles_per_matrix;
  const int span = p.group_m * p.n_blocks;
  const int g = t / span;
  const int first = g * p.group_m;
  const int rows = min(p.m_blocks - first, p.group_m);
  const int r = t - g * span;
  mb = first + r % rows;
  nb = r / rows;
}

template <int BN, int STAGES, int EPI>
struct GemmCfg {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "tile width");
  static constexpr int kABytes = kBM * kBK * 2;  // 16 KB
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kStagingBytes = kEpiWarps * kStagingPerWarp * kStageBox;
  static constexpr int kBarOffset = kRingBytes + kStagingBytes;
  // full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain
  static constexpr int kNumBars = 2 * STAGES + 5;
  static constexpr int kSmemBytes = 1024 + kBarOffset + kNumBars * 8 + 16;
  static constexpr int kOutCols = (EPI == EPI_GATE_UP) ? BN / 2 : BN;
  static constexpr int kAccStride = 256;  // TMEM columns between the two accumulators
  static constexpr int kTmemCols = 512;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// The 32 values of C at (row, col0..col0+31) in FP32, zero outside C.  The
// loads are plain (C is written later by this same CTA's TMA stores).
template <int EPI>
__device__ __forceinline__ void load_c_slice(float (&c)[32], const TileParams& p, int b, int row,
                                             int col0) {
#pragma unroll
  for (int i = 0; i < 32; ++i) c[i] = 0.0f;
  if (row >= p.M || col0 >= p.N) return;
  if constexpr (EPI == EPI_F32) {
    const float* src = static_cast<const float*>(p.C) + b * p.c_stride +
                       static_cast<long long>(row) * p.ldc + col0;
    if (col0 + 32 <= p.N) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = reinterpret_cast<const float4*>(src)[q];
        c[4 * q + 0] = x.x;
        c[4 * q + 1] = x.y;
        c[4 * q + 2] = x.z;
        c[4 * q + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i < p.N) c[i] = src[i];
    }
  } else {
    const uint16_t* src = static_cast<const uint16_t*>(p.C) + b * p.c_stride +
                          static_cast<long long>(row) * p.ldc + col0;
    const bool f16 = p.out_f16 != 0;
    if (col0 + 32 <= p.N) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 x = reinterpret_cast<const uint4*>(src)[q];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          c[8 * q + 2 * j + 0] = half16_to_float(w[j] & 0xFFFFu, f16);
          c[8 * q + 2 * j + 1] = half16_to_float(w[j] >> 16, f16);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i < p.N) c[i] = half16_to_float(src[i], f16);
    }
  }
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + __expf(-g)); }

// The raw FP32 accumulator slice (32 columns from `col`) of this lane's row:
// from TMEM for a whole tile; for the last piece of a split tile, the sum of
// every piece's partial in piece order 0, 1, ..., with this piece's own
// partial taken from TMEM (bit-identical to the copy it wrote), so the result
// does not depend on which piece finished last.
__device__ __forceinline__ void acc_slice(float (&v)[32], uint32_t tacc, int col, int lane,
                                          const SplitCtx& sp) {
  if (sp.pieces <= 1) {
    tmem_load_32x32b_x32(tacc + col, v);
    return;
  }
  float sum[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) sum[i] = 0.0f;
  // Pieces are visited two at a time so that the workspace loads of both are
  // in flight together; the addition order stays 0, 1, 2, ...
  for (int q0 = 0; q0 < sp.pieces; q0 += 2) {
    float4 x[2][8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = q0 + h;
      if (q < sp.pieces && q != sp.piece) {
        const float4* src = piece_partial(sp, q);
#pragma unroll
        for (int j = 0; j < 8; ++j) x[h][j] = __ldcg(src + split_index(col, j, lane));
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = q0 + h;
      if (q >= sp.pieces) break;
      if (q == sp.piece) {
        tmem_load_32x32b_x32(tacc + col, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) sum[i] += v[i];
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          sum[4 * j + 0] += x[h][j].x;
          sum[4 * j + 1] += x[h][j].y;
          sum[4 * j + 2] += x[h][j].z;
          sum[4 * j + 3] += x[h][j].w;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = sum[i];
}

// Writes this warp band's raw accumulator (acc_cols columns) to its piece's
// partial in the workspace, then counts the band's arrival.  Returns true on
// the band's last arrival (the caller then runs the epilogue on the sum).
__device__ __forceinline__ bool publish_partial(uint32_t tacc, int acc_cols, int lane,
                                                const SplitCtx& sp, int* counter, int pieces) {
  float4* dst = const_cast<float4*>(piece_partial(sp, sp.piece));
#pragma unroll 1
  for (int c = 0; c < acc_cols; c += 32) {
    float v[32];
    tmem_load_32x32b_x32(tacc + c, v);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      __stcg(dst + split_index(c, j, lane), make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
  }
  __threadfence();
  __syncwarp();
  int prev = 0;
  if (lane == 0) prev = atomicAdd(counter, 1);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  const bool last = prev == pieces - 1;
  if (last) {
    __threadfence();
    if (lane == 0) *counter = 0;  // ready for the next call
  }
  return last;
}

// The last piece of a split tile (publish_partial returned true) adds the
// other pieces' partials into its own accumulator in TMEM, in piece order
// 0, 1, ... with its own partial taken from TMEM -- the same FP32 additions,
// in the same order, as acc_slice -- so that the tile's epilogue then runs
// as for a whole tile.  With two pieces the workspace loads run kAhead
// 32-column slices ahead of the additions, so that several L2 round trips
// overlap instead of one per slice.
template <int ACC_COLS>
__device__ __forceinline__ void combine_into_tmem(uint32_t tacc, int lane, const SplitCtx& sp) {
  static_assert(ACC_COLS % 32 == 0, "whole slices");
  constexpr int kSlices = ACC_COLS / 32;
  if (sp.pieces == 2) {
    constexpr int kAhead = 2;
    const float4* src = piece_partial(sp, 1 - sp.piece);
    float4 buf[kAhead][8];
#pragma unroll
    for (int s = 0; s < kAhead && s < kSlices; ++s)
#pragma unroll
      for (int j = 0; j < 8; ++j) buf[s][j] = __ldcg(src + split_index(32 * s, j, lane));
#pragma unroll
    for (int s = 0; s < kSlices; ++s) {
      float4 cur[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) cur[j] = buf[s % kAhead][j];
      if (s + kAhead < kSlices) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          buf[s % kAhead][j] = __ldcg(src + split_index(32 * (s + kAhead), j, lane));
      }
      float v[32];
      tmem_load_32x32b_x32(tacc + 32 * s, v);
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float o[4] = {cur[j].x, cur[j].y, cur[j].z, cur[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mine = v[4 * j + e];
          // 0 + p0 + p1, as acc_slice adds them
          const float sum = sp.piece == 0 ? (0.0f + mine) + o[e] : (0.0f + o[e]) + mine;
          r[4 * j + e] = __float_as_uint(sum);
        }
      }
      tmem_store_32x32b_x32(tacc + 32 * s, r);
    }
  } else {
#pragma unroll 1
    for (int s = 0; s < kSlices; ++s) {
      float v[32];
      acc_slice(v, tacc, 32 * s, lane, sp);
      uint32_t r[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
      tmem_store_32x32b_x32(tacc + 32 * s, r);
    }
  }
}

// Running reductions of one lane's row over the columns an epilogue visits.
struct RowAcc {
  float sum, max, min;
};

__device__ __forceinline__ void row_acc_init(RowAcc& r) {
  r.sum = 0.0f;
  r.max = -INFINITY;
  r.min = INFINITY;
}

// Adds the 32 values of a slice at columns col0.. (those below N) in order.
__device__ __forceinline__ void row_acc_slice(RowAcc& r, const float (&v)[32], int col0, int N) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (col0 + i < N) {
      r.sum += v[i];
      r.max = fmaxf(r.max, v[i]);
      r.min = fminf(r.min, v[i]);
    }
  }
}

// Stores this warp band's partial reductions (rows m0..m0+31 of matrix b over
// column tile nb) and counts the band's arrival; the last of the n_blocks
// arrivals adds the partials in column-tile order 0, 1, ... and writes the
// row results, so they do not depend on which tile finished last.
__device__ __forceinline__ void publish_row_stats(const TileParams& p, const RowStatsParams& rs,
                                                  int b, int nb, int m0, int lane,
                                                  const RowAcc& r) {
  const int row = m0 + lane;
  const bool live = row < p.M;
  const long long plane = static_cast<long long>(p.batch) * p.n_blocks * p.M;
  const long long base = static_cast<long long>(b) * p.n_blocks * p.M + row;
  if (live) {
    const long long idx = base + static_cast<long long>(nb) * p.M;
    __stcg(rs.ws + idx, r.sum);
    __stcg(rs.ws + plane + idx, r.max);
    __stcg(rs.ws + 2 * plane + idx, r.min);
  }
  __threadfence();
  __syncwarp();
  int* counter = rs.counters + static_cast<long long>(b) * ((p.M + 31) >> 5) + (m0 >> 5);
  int prev = 0;
  if (lane == 0) prev = atomicAdd(counter, 1);
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != p.n_blocks - 1) return;
  __threadfence();
  if (live) {
    float sum = 0.0f, mx = -INFINITY, mn = INFINITY;
#pragma unroll 4
    for (int j = 0; j < p.n_blocks; ++j) {
      const long long idx = base + static_cast<long long>(j) * p.M;
      sum += __ldcg(rs.ws + idx);
      mx = fmaxf(mx, __ldcg(rs.ws + plane + idx));
      mn = fminf(mn, __ldcg(rs.ws + 2 * plane + idx));
    }
    const long long out = static_cast<long long>(b) * p.M + row;
    if (rs.row_sum != nullptr) rs.row_sum[out] = sum;
    if (rs.row_max != nullptr) rs.row_max[out] = mx;
    if (rs.row_min != nullptr) rs.row_min[out] = mn;
  }
  __syncwarp();
  if (lane == 0) *counter = 0;  // ready for the next call
}

template <int EPI, int OUT_COLS>
struct EpiBox {
  static constexpr int kCols = (EPI == EPI_F32) ? 32 : (OUT_COLS % 64 == 0 ? 64 : 32);
  static constexpr int kRowBytes = (EPI == EPI_F32) ? 128 : kCols * 2;
  static constexpr bool kSwizzle128 = kRowBytes == 128;
  static_assert(OUT_COLS % kCols == 0, "tile width must be a whole number of boxes");
  static_assert(32 * kRowBytes <= kStageBox, "staging slot");
};

// Shared-memory byte offset of 16-byte chunk `chunk` of staging row `row`, as
// the TMA swizzle lays the box out: 128-byte rows XOR the chunk with row % 8,
// 64-byte rows XOR it with (row / 2) % 4 (both are the address bits 7.. folded
// into bits 4..).  Consecutive rows then hit different banks.
template <bool kSw128>
__host__ __device__ __forceinline__ uint32_t staging_offset(int row, uint32_t chunk) {
  if constexpr (kSw128)
    return static_cast<uint32_t>(row) * 128u + ((chunk ^ static_cast<uint32_t>(row & 7)) << 4);
  else
    return static_cast<uint32_t>(row) * 64u +
           ((chunk ^ static_cast<uint32_t>((row >> 1) & 3)) << 4);
}

// One warp's share of a tile epilogue: rows m0..m0+31 (this warp's TMEM lane
// band, accumulator at TMEM address `tacc`) and the tile's output columns
// from n0.  Each box is loaded from TMEM 32 columns at a time, transformed in
// FP32, written to a staging slot in the swizzled layout and stored with TMA.
// `sc` counts the boxes this warp staged (two slots alternate); every staged
// box is committed as its own bulk group.  The value before output rounding
// is fma(beta, c, RN(alpha * acc)) in FP32, written out with intrinsics so
// that no contraction choice of the compiler differs between the epilogues
// of the different kernels.
// STATS: also reduce each row (sum, max, min) into p's row-statistics outputs.
// cols: the output columns computed, a multiple of the box width up to the
// tile's (a strip of a pair tile: its first cols accumulator columns).
template <int BN, int EPI, bool STATS = false>
__device__ __forceinline__ void epilogue_tile(const TileParams& p, const CUtensorMap* tmOut,
                                              uint32_t tacc, int b, int m0, int n0,
                                              uint32_t staging, int lane, int& sc, bool have_acc,
                                              const SplitCtx& split, const RowStatsParams& rs,
                                              int cols = (EPI == EPI_GATE_UP) ? BN / 2 : BN) {
  constexpr int OUT = (EPI == EPI_GATE_UP) ? BN / 2 : BN;
  using Box = EpiBox<EPI, OUT>;
  constexpr int kSub = Box::kCols / 32;  // 32-column slices per box
  const int row = m0 + lane;
  const bool read_c = (EPI != EPI_GATE_UP) && p.beta != 0.0f;
  constexpr bool stats = STATS && (EPI != EPI_GATE_UP);
  RowAcc racc;
  row_acc_init(racc);
  // C of the next slice is loaded one slice ahead so its latency overlaps the
  // TMEM load and conversion of the current one.
  float c_next[32];
  if (read_c) load_c_slice<EPI>(c_next, p, b, row, n0);
#pragma unroll 1
  for (int c0 = 0; c0 < cols; c0 += Box::kCols) {
    // Boxes wholly outside C are neither computed nor stored (warp-uniform).
    if (m0 >= p.M || n0 + c0 >= p.N) continue;
    const uint32_t stg = staging + (sc & 1) * kStageBox;
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
#pragma unroll
    for (int h = 0; h < kSub; ++h) {
      float v[32];
      if constexpr (EPI == EPI_GATE_UP) {
        float u[32];
        if (have_acc) {
          acc_slice(v, tacc, c0 + 32 * h, lane, split);
          acc_slice(u, tacc, OUT + c0 + 32 * h, lane, split);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = u[i] = 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = silu_f32(v[i]) * u[i];
      } else {
        float c_cur[32];
        if (read_c) {
#pragma unroll
          for (int i = 0; i < 32; ++i) c_cur[i] = c_next[i];
          const int next = c0 + 32 * (h + 1);
          if (next < cols) load_c_slice<EPI>(c_next, p, b, row, n0 + next);
        }
        if (have_acc) {
          acc_slice(v, tacc, c0 + 32 * h, lane, split);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        }
        const float alpha = p.alpha;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(alpha, v[i]);
        if (read_c) {
          const float beta = p.beta;
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __fmaf_rn(beta, c_cur[i], v[i]);
        }
        if constexpr (stats) row_acc_slice(racc, v, n0 + c0 + 32 * h, p.N);
      }
      if constexpr (EPI == EPI_F32) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_shared_v4(stg + staging_offset<true>(lane, static_cast<uint32_t>(q)),
                       __float_as_uint(v[4 * q + 0]), __float_as_uint(v[4 * q + 1]),
                       __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
      } else {
        const bool f16 = p.out_f16 != 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(stg + staging_offset<Box::kSwizzle128>(lane, static_cast<uint32_t>(4 * h + q)),
                       pack_half16x2(v[8 * q + 0], v[8 * q + 1], f16),
                       pack_half16x2(v[8 * q + 2], v[8 * q + 3], f16),
                       pack_half16x2(v[8 * q + 4], v[8 * q + 5], f16),
                       pack_half16x2(v[8 * q + 6], v[8 * q + 7], f16));
      }
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmOut, stg, n0 + c0, m0, b);
      bulk_commit_group();
    }
    ++sc;
  }
  if constexpr (stats) {
    if (m0 < p.M) publish_row_stats(p, rs, b, n0 / OUT, m0, lane, racc);
  }
}

// C through a staging ring (beta != 0, whole tiles).  Each epilogue warp owns
// kRingSlots staging slots.  Its lane 0 loads the boxes of C with TMA into
// the slots kRingAhead boxes ahead of the box being computed; a box is then
// computed in place (C read from the slot, the result written over it) and
// stored from the same slot.  The look-ahead runs across tile boundaries, so
// the first boxes of a tile load while the previous tile's last ones are
// computed: one L2 round trip per tile band instead of one per 32-column
// slice, with no registers held for C.
constexpr int kRingSlots = 4;
constexpr int kRingAhead = 2;  // boxes loaded beyond the one being computed
static_assert(kRingAhead < kRingSlots, "a slot must be free before its next load");

// The ring boxes of one warp are numbered r = 0, 1, ... in the order they are
// computed: box r lives in slot r % kRingSlots, whose barrier completes phase
// (r / kRingSlots) & 1 when the box has landed; `issued` counts the boxes
// whose loads were issued.  Whole tiles (ON_DEMAND false): topup(r) issues
// the loads of every box up to r + kRingAhead that exists.  The last piece
// of a split tile (ON_DEMAND true, `split` its pieces), whose turn to write C
// is known only when it arrives, loads each box just before computing it
// (these come before every whole tile of the warp, so the two never
// interleave).  Returns false when a wait gave up (the abort flag is then set).
template <int BN, int EPI, bool STATS, bool ON_DEMAND, typename TopUp>
__device__ __forceinline__ bool epilogue_tile_ring(const TileParams& p, const CUtensorMap* tmOut,
                                                   uint32_t tacc, int b, int m0, int n0,
                                                   uint32_t ring, uint32_t cbar0, int lane,
                                                   long long& r, long long& issued, int& sc,
                                                   const SplitCtx& split,
                                                   const RowStatsParams& rs,
                                                   volatile int* abort_flag, TopUp&& topup,
                                                   int cols = BN) {
  static_assert(EPI != EPI_GATE_UP, "the gate/up epilogue reads no C");
  using Box = EpiBox<EPI, BN>;
  constexpr int kSub = Box::kCols / 32;
  RowAcc racc;
  row_acc_init(racc);
  // ON_DEMAND: the tile's boxes inside C (a prefix of its columns) take ring
  // positions r0, r0 + 1, ...; their loads run kRingAhead boxes ahead of the
  // one computed, starting once every earlier store has read its slot.
  const long long r0 = r;
  const int nbox = (m0 < p.M && n0 < p.N)
                       ? (min(cols, p.N - n0) + Box::kCols - 1) / Box::kCols
                       : 0;
  auto load_box = [&](int j) {  // lane 0: box j of this tile into its slot
    const int sl = static_cast<int>((r0 + j) % kRingSlots);
    mbar_arrive_expect_tx(cbar0 + 8u * sl, 32 * Box::kRowBytes);
    tma_load_3d(ring + sl * kStageBox, tmOut, cbar0 + 8u * sl, n0 + j * Box::kCols, m0, b);
  };
  if constexpr (ON_DEMAND) {
    const int first = min(nbox, kRingAhead + 1);
    if (lane == 0 && first > 0) {
      bulk_wait_group_read<0>();
      for (int j = 0; j < first; ++j) load_box(j);
    }
    issued = r0 + first;
  }
#pragma unroll 1
  for (int c0 = 0; c0 < cols; c0 += Box::kCols) {
    if (m0 >= p.M || n0 + c0 >= p.N) continue;
    const int slot = static_cast<int>(r % kRingSlots);
    const uint32_t stg = ring + slot * kStageBox;
    if constexpr (!ON_DEMAND) topup(r);
    const bool got = wait_bounded(cbar0 + 8u * slot, static_cast<uint32_t>((r / kRingSlots) & 1),
                                  abort_flag, SITE_EPI_C_FULL);
    if (!__all_sync(0xffffffffu, got)) return false;
#pragma unroll 1
    for (int h = 0; h < kSub; ++h) {
      float v[32], c[32];
      acc_slice(v, tacc, c0 + 32 * h, lane, split);
      if constexpr (EPI == EPI_F32) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 x = ld_shared_v4(stg + staging_offset<true>(lane, static_cast<uint32_t>(q)));
          c[4 * q + 0] = __uint_as_float(x.x);
          c[4 * q + 1] = __uint_as_float(x.y);
          c[4 * q + 2] = __uint_as_float(x.z);
          c[4 * q + 3] = __uint_as_float(x.w);
        }
      } else {
        const bool f16 = p.out_f16 != 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 x = ld_shared_v4(
              stg + staging_offset<Box::kSwizzle128>(lane, static_cast<uint32_t>(4 * h + q)));
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            c[8 * q + 2 * j + 0] = half16_to_float(w[j] & 0xFFFFu, f16);
            c[8 * q + 2 * j + 1] = half16_to_float(w[j] >> 16, f16);
          }
        }
      }
      const float alpha = p.alpha, beta = p.beta;
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __fmaf_rn(beta, c[i], __fmul_rn(alpha, v[i]));
      if constexpr (STATS) row_acc_slice(racc, v, n0 + c0 + 32 * h, p.N);
      if constexpr (EPI == EPI_F32) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_shared_v4(stg + staging_offset<true>(lane, static_cast<uint32_t>(q)),
                       __float_as_uint(v[4 * q + 0]), __float_as_uint(v[4 * q + 1]),
                       __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
      } else {
        const bool f16 = p.out_f16 != 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(stg + staging_offset<Box::kSwizzle128>(lane, static_cast<uint32_t>(4 * h + q)),
                       pack_half16x2(v[8 * q + 0], v[8 * q + 1], f16),
                       pack_half16x2(v[8 * q + 2], v[8 * q + 3], f16),
                       pack_half16x2(v[8 * q + 4], v[8 * q + 5], f16),
                       pack_half16x2(v[8 * q + 6], v[8 * q + 7], f16));
      }
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmOut, stg, n0 + c0, m0, b);
      bulk_commit_group();
    }
    if constexpr (ON_DEMAND) {
      // The next box's slot was last stored from kRingSlots - kRingAhead - 1
      // boxes before this one's store.
      const int next = static_cast<int>(r - r0) + kRingAhead + 1;
      if (next < nbox) {
        if (lane == 0) {
          bulk_wait_group_read<kRingSlots - 1 - kRingAhead>();
          load_box(next);
        }
        issued = r0 + next + 1;
      }
    }
    ++r;
    ++sc;
  }
  if constexpr (STATS) {
    if (m0 < p.M) publish_row_stats(p, rs, b, n0 / BN, m0, lane, racc);
  }
  return true;
}

// When C is read (beta != 0): ask L2 for this warp's band of C of a coming
// tile (rows m0..m0+31, the tile's columns from n0), box by box.
template <int BN, int EPI>
__device__ __forceinline__ void prefetch_c_band(const TileParams& p, const CUtensorMap* tmOut,
                                                int b, int m0, int n0) {
  if constexpr (EPI == EPI_GATE_UP) {
    return;
  } else {
    if (p.beta == 0.0f || m0 >= p.M) return;
    using Box = EpiBox<EPI, BN>;
    for (int c0 = 0; c0 < BN && n0 + c0 < p.N; c0 += Box::kCols)
      tma_prefetch_l2_3d(tmOut, n0 + c0, m0, b);
  }
}

template <int BN, int STAGES, int EPI, bool STATS = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmOut, const TileParams p,
                   const RowStatsParams rs) {
  using Cfg = GemmCfg<BN, STAGES, EPI>;
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
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if constexpr (EPI == EPI_GATE_UP) prefetch_tensormap(&tmB2);
    prefetch_tensormap(&tmOut);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        int bt, mb, nb;
        tile_coords(tile, p, bt, mb, nb);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + s * Cfg::kStageBytes;
          const uint32_t b_dst = a_dst + Cfg::kABytes;
          mbar_arrive_expect_tx(full_bar(s), Cfg::kStageBytes);
          tma_load_3d(a_dst, &tmA, full_bar(s), kb * kBK, mb * kBM, bt);
          if constexpr (EPI == EPI_GATE_UP) {
            tma_load_3d(b_dst, &tmB, full_bar(s), kb * kBK, nb * (BN / 2), bt);
            tma_load_3d(b_dst + Cfg::kBBytes / 2, &tmB2, full_bar(s), kb * kBK, nb * (BN / 2), bt);
          } else {
            tma_load_3d(b_dst, &tmB, full_bar(s), kb * kBK, nb * BN, bt);
          }
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      {
        // Let the copies already issued land before shared memory goes away
        // (they have, unless a wait gave up; then this waits, bounded, for
        // the last STAGES of them).
        const long long first = issued > STAGES ? issued - STAGES : 0;
        for (long long i = first; i < issued; ++i)
          wait_bounded(full_bar(static_cast<int>(i % STAGES)),
                       static_cast<uint32_t>((i / STAGES) & 1), nullptr, SITE_DRAIN);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++local) {
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
          const uint32_t a_addr = sbase + s * Cfg::kStageBytes;
          const uint64_t adesc = smem_desc_sw128(a_addr);
          const uint64_t bdesc = smem_desc_sw128(a_addr + Cfg::kABytes);
#pragma unroll
          for (int j = 0; j < kBK / kUmmaK; ++j) {
            // +32 bytes along K inside the swizzled row = +2 in the address field.
            umma_bf16(d_tmem, adesc + 2u * j, bdesc + 2u * j, p.idesc, (kb | j) != 0 ? 1u : 0u);
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
      // Every MMA issued by this thread has completed once this arrives.
      umma_commit(drain_bar);
      wait_bounded(drain_bar, 0, nullptr, SITE_DRAIN);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                 // staging slot owner
    const int band = (warp & 3) * 32;        // TMEM lanes this warp may access
    const uint32_t staging = sbase + Cfg::kRingBytes + ew * kStagingPerWarp * kStageBox;
    int local = 0;
    int sc = 0;
    if (lane == 0 && blockIdx.x < p.num_tiles) {
      int b_, mb_, nb_;
      tile_coords(blockIdx.x, p, b_, mb_, nb_);
      prefetch_c_band<BN, EPI>(p, &tmOut, b_, mb_ * kBM + band, nb_ * Cfg::kOutCols);
    }
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++local) {
      int bt, mb, nb;
      tile_coords(tile, p, bt, mb, nb);
      // C of the next tile of this CTA travels to L2 during this tile's
      // epilogue and the next tile's main loop.
      if (lane == 0 && tile + gridDim.x < p.num_tiles) {
        int b_, mb_, nb_;
        tile_coords(tile + gridDim.x, p, b_, mb_, nb_);
        prefetch_c_band<BN, EPI>(p, &tmOut, b_, mb_ * kBM + band, nb_ * Cfg::kOutCols);
      }
      const int buf = local & 1;
      const uint32_t aph = static_cast<uint32_t>(local >> 1) & 1u;
      const bool got = wait_bounded(accf_bar(buf), aph, abort_flag, SITE_EPI_ACC_FULL);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const uint32_t tacc = tmem_addr(tmem_base, static_cast<uint32_t>(band),
                                      static_cast<uint32_t>(buf * Cfg::kAccStride));
      const int m0 = mb * kBM + band;
      const int n0 = nb * Cfg::kOutCols;
      const SplitCtx whole{1, 0, nullptr, nullptr, 0};
      epilogue_tile<BN, EPI, STATS>(p, &tmOut, tacc, bt, m0, n0, staging, lane, sc,
                                    p.k_blocks > 0, whole, rs);
      // The accumulator may be overwritten once every lane's TMEM reads are done.
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(buf));
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

}  // namespace gb3
