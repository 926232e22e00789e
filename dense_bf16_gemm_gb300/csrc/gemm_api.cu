// gemm_api.cu -- host side of the library: argument validation, tile
// planning, TMA descriptor encoding (cuTensorMapEncodeTiled, 128-byte
// swizzle) with a descriptor cache, kernel launch and the C ABI declared in
// include/gemm_bf16.h.
//
// Descriptor contract ("TMA and Hopper WGMMA", section "The same storage
// contract on both sides"): a descriptor names the element type, the tile
// (box) shape, the inner axis and a 128-byte swizzle row; the box's inner
// extent is one swizzle row (64 16-bit or 32 FP32 elements) and its outer
// extent is at most 256.  The same section states that a descriptor stays
// valid while values change and must be re-encoded for a new address or new
// dimensions: the cache key is therefore (address, element type, dimensions,
// pitches, box, swizzle).  Every descriptor is three-dimensional, the third
// coordinate selecting one matrix of a batch, bounded on its own (the same
// section's three-dimensional binding); a single matrix is a batch of one.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/gemm_bf16.h"
#include "gemm_kernels.cuh"
#include "gemm_kernels_pair.cuh"
#include "gemm_skinny.cuh"
#include "attention.cuh"
#include "gemm_smallm.cuh"
#include "norm_api.h"

namespace {

using namespace gb3;

// ----------------------------------------------------------------------------
// Kernel configurations
// ----------------------------------------------------------------------------
constexpr int kTileN = 256;        // output columns per tile of the single-CTA GEMM
constexpr int kStages = 4;         // its ring depth (48 KB per stage)
constexpr int kGateUpStages = 4;   // single-CTA gate/up: 16 KB X + 16 KB Wg + 16 KB Wu per stage
constexpr int kSkinnyStages = 12;  // 18 KB per stage
constexpr int kSkinnyGateUpStages = 6;  // 34 KB per stage (Wg, Wu and X rows)
constexpr int kSkinnyMaxM = 16;
constexpr int kGroupM = 16;

constexpr int kPairStages = 6;     // CTA-pair kernels: 16 KB A + BN*64 B per stage and CTA
constexpr int kPairMinM = 129;     // pair tiles (256 rows) from this M on

using CfgF32 = GemmCfg<kTileN, kStages, EPI_F32>;
using CfgBF16 = GemmCfg<kTileN, kStages, EPI_BF16>;
using CfgGU = GemmCfg<256, kGateUpStages, EPI_GATE_UP>;
using CfgSkinny = SkinnyCfg<kSkinnyStages>;
using CfgSkinnyGU = SkinnyCfg<kSkinnyGateUpStages, true>;
using CfgPairGU = PairCfg<256, kPairStages, EPI_GATE_UP>;

// Tile widths compiled for the CTA-pair GEMM.
constexpr int kPairWidths[] = {256, 224};

constexpr int64_t kMaxDim = 0x7FFFFFFF;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : fallback;
}

// ----------------------------------------------------------------------------
// The problem a call describes
// ----------------------------------------------------------------------------
struct Problem {
  int64_t batch, M, N, K;
  float alpha, beta;
  const void* A;
  int64_t lda, sa;   // row pitch and matrix stride, elements
  const void* B;
  int64_t ldb, sb;
  void* C;
  int64_t ldc, sc;
  int in_dtype;      // gemm_in_dtype
  int out_dtype;     // gemm_out_dtype
  // Reductions along each row of the result ([batch][M] FP32 each; nullptr:
  // not wanted).  Any non-null one asks for all three to be computed.
  float* row_sum = nullptr;
  float* row_max = nullptr;
  float* row_min = nullptr;
  bool stats() const { return row_sum != nullptr || row_max != nullptr || row_min != nullptr; }
};

int out_elem_bytes(int out_dtype) { return out_dtype == GEMM_OUT_F32 ? 4 : 2; }

CUtensorMapDataType in_tma_type(int in_dtype) {
  return in_dtype == GEMM_IN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// ----------------------------------------------------------------------------
// Planning (pure host logic)
// ----------------------------------------------------------------------------
enum KernelKind {
  K_NONE = 0,
  K_TILED = 1,
  K_SKINNY = 2,
  K_SCALE = 3,
  K_GATE_UP = 4,
  K_PAIR = 5,
  K_PAIR_GATE_UP = 6,
  K_SMALL_M = 7,
  K_SKINNY_GATE_UP = 8
};

constexpr int kSmallMMaxM = 128;   // the small-M kernel's widest activation tile

// Activation tile (the MMA's N) of the small-M kernel for M rows.
int smallm_nx(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

int smallm_smem(int nx) {
  switch (nx) {
    case 16: return SmallMCfg<16>::kSmemBytes;
    case 32: return SmallMCfg<32>::kSmemBytes;
    case 64: return SmallMCfg<64>::kSmemBytes;
    default: return SmallMCfg<128>::kSmemBytes;
  }
}

int smallm_stages(int nx) {
  switch (nx) {
    case 16: return SmallMCfg<16>::kStages;
    case 32: return SmallMCfg<32>::kStages;
    case 64: return SmallMCfg<64>::kStages;
    default: return SmallMCfg<128>::kStages;
  }
}

// Shortest share of the k-block sequence worth giving a CTA of the small-M
// kernel when the tiles alone leave SMs idle (512 of K: below that the
// partial sums cost about what the extra streaming SMs save).
constexpr int64_t kSmallMinShareKb = 8;

// CTAs the small-M kernel runs.  Tiles that fill at most half the SMs are
// divided over every SM (stream-K); between half and all of the SMs each CTA
// takes one whole tile, because the combine of shared tiles (the last piece
// writes C after the others' partial sums) costs more there than the idle SMs
// (measured on GB300: 64 x 14336 x 4096, 112 tiles, 28.7 us whole against 38.7
// divided; 64 x 8192 x 8192, 64 tiles, 43.1 against 41.0).  More tiles than
// SMs are divided over every SM.  GB3_SMALL_M_STREAM_K = 1 or 0 forces the
// division or whole tiles (one CTA per tile, up to one per SM).
int smallm_grid(int64_t tiles, int64_t k_blocks, int sms) {
  const int64_t work = tiles * k_blocks;
  const int mode = env_int("GB3_SMALL_M_STREAM_K", -1);
  if (mode == 0 || (mode != 1 && tiles > sms / 2 && tiles <= sms))
    return static_cast<int>(std::min<int64_t>(tiles, sms));
  const int64_t g = std::max<int64_t>(tiles, work / kSmallMinShareKb);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(g, sms)));
}

// The stream-K division of a small-M problem on `grid` CTAs: each CTA's share
// of the k-block sequence and the most CTAs any one tile is shared by.
void smallm_divide(int64_t tiles, int64_t k_blocks, int grid, SmallMParams* p) {
  p->work = tiles * k_blocks;
  p->work_per_cta = p->work / grid;
  p->work_extra = static_cast<int>(p->work % grid);
  int most = 1;
  for (int64_t t = 0; t < tiles; ++t) {
    const int first = smallm_cta_of(*p, t * k_blocks);
    const int last = smallm_cta_of(*p, t * k_blocks + k_blocks - 1);
    most = std::max(most, last - first + 1);
  }
  p->max_pieces = most;
}

// Partial-sum slots of the small-M kernel: one per (CTA, tile) it touches,
// numbered CTA + tile, so at most grid + tiles - 1 of them.
size_t smallm_workspace_bytes(int64_t grid, int64_t tiles, int64_t M) {
  return static_cast<size_t>(grid + tiles - 1) * M * kSmallRows * sizeof(float);
}

// Whether an M <= 128 problem runs on the small-M kernel (128-row weight
// tiles, see smallm_grid for how the work is divided).  Measured on GB300
// against the kernel each problem would otherwise take: with tiles for at
// most every SM it beat the single-CTA tiled kernel on every 16 < M <= 128
// shape measured (64 x 8192 x 8192 41.0 us against 59.0, 64 x 14336 x 4096
// 28.7 against 36.2); for M <= 16 it beat the split-K kernel while its tiles
// fill at most half the SMs (16 x 8192 x 8192 32.8 against 37.6, 8 x 4096 x
// 4096 18.5 against 20.5) and matched it above.  With more tiles than SMs the
// tiled kernel (M > 16) or the split-K kernel is as fast or faster.
// GB3_GEMM_SMALL_M = 0 or 1 forces the choice.
bool use_small_m(int64_t batch, int64_t M, int64_t N, int64_t K, int sms) {
  (void)K;
  if (M > kSmallMMaxM) return false;
  const int force = env_int("GB3_GEMM_SMALL_M", -1);
  if (force == 0 || force == 1) return force == 1;
  const int64_t tiles = batch * ceil_div(N, kSmallRows);
  if (M <= kSkinnyMaxM) return tiles <= sms / 2;
  return tiles <= sms;
}

template <int BN>
constexpr int pair_smem_bytes() {
  return PairCfg<BN, kPairStages, EPI_BF16>::kSmemBytes;
}

int pair_smem_for(int bn) {
  switch (bn) {
    case 256: return pair_smem_bytes<256>();
    case 224: return pair_smem_bytes<224>();
    default: return 0;
  }
}

// The CTA-pair epilogue reads C (beta != 0) through the staging ring unless
// GB3_GEMM_C_RING = 0 (for comparisons and tests).
bool pair_reads_c_ring(float beta) {
  return beta != 0.0f && env_int("GB3_GEMM_C_RING", 1) != 0;
}

int pair_ring_smem_for(int bn) {
  switch (bn) {
    case 256: return PairCfg<256, kPairStages - 1, EPI_BF16, true>::kSmemBytes;
    case 224: return PairCfg<224, kPairStages - 1, EPI_BF16, true>::kSmemBytes;
    default: return 0;
  }
}

int pair_stage_bytes(int bn) { return 128 * kBK * 2 + (bn / 2) * kBK * 2; }

// Split of K for the skinny path, from a time model fit to same-box
// measurements of nine decode shapes at 1..8 splits (it picks the fastest
// measured split for each).  Every wave of units streams each unit's weight
// rows at min(60 GB/s per SM, 7.1 TB/s shared by the busy SMs) -- 60 GB/s is
// the measured rate of one SM streaming 128-row units through its MMAs and
// barriers -- and every split beyond the first costs about 4 us per wave
// (partial sums, arrival counters and the combine).  GB3_SKINNY_SPLITS forces
// a split (tuning).
// weights: weight matrices a unit streams (2 for gate/up).
void choose_split(int64_t n_blocks, int64_t k_blocks, int sms, int* splits, int* kb_per,
                  int weights = 1) {
  const int forced = env_int("GB3_SKINNY_SPLITS", 0);
  if (forced > 0) {   // at most 32 splits, as the model below
    const int64_t kbp = ceil_div(k_blocks, std::min<int64_t>({forced, k_blocks, 32}));
    *kb_per = static_cast<int>(kbp);
    *splits = static_cast<int>(ceil_div(k_blocks, kbp));
    return;
  }
  constexpr double kSmGBs = 60.0, kTotalGBs = 7100.0, kSplitNs = 4000.0;
  int best_s = 1;
  double best = 1e300;
  for (int s = 1; s <= 32; ++s) {
    const int64_t kbp = ceil_div(k_blocks, s);
    if (s > 1 && kbp < 4) break;
    const int64_t real_s = ceil_div(k_blocks, kbp);  // splits that get work
    if (real_s != s) continue;
    const int64_t units = n_blocks * s;
    const double waves = static_cast<double>(ceil_div(units, sms));
    const double active = static_cast<double>(std::min<int64_t>(units, sms));
    const double gbs = std::min(kSmGBs, kTotalGBs / active);        // bytes per ns per SM
    const double unit_bytes = static_cast<double>(kSkinnyRows) * kbp * kBK * 2 * weights;
    const double cost = waves * (unit_bytes / gbs + kSplitNs * (s - 1));  // ns
    if (cost < best) {
      best = cost;
      best_s = s;
    }
  }
  *splits = best_s;
  *kb_per = static_cast<int>(ceil_div(k_blocks, best_s));
}

constexpr int kMinPieceKb = 24;        // shortest K piece of a split tail tile (1536 of K)
constexpr int kMaxTailSplit = 2;       // more pieces cost more partial-sum traffic than they save
constexpr double kSplitCharge = 0.1;   // partial-sum traffic of a split tail, in waves
constexpr int kWidthCostOffset = 320;  // per-wave time model of a pair tile: width + 320

struct PairChoice {
  int bn = 256;
  int64_t tiles = 0;
  int64_t full = 0;      // tiles run whole
  int split = 1;         // K pieces per tail tile
  int kb_per_piece = 0;
  // Balanced division (see TileParams): every cluster takes one contiguous
  // range of the tiles' k-blocks; `units` counts the (tile, range) units and
  // `max_pieces` the most ranges any tile falls in.
  bool balanced = false;
  int64_t per = 0;       // k-blocks per cluster (floor)
  int extra = 0;         // clusters 0..extra-1 take one more
  int64_t units = 0;
  int max_pieces = 1;
  int64_t dp_tiles = 0;  // balanced: whole tiles run first, data-parallel
  // Strips: the last strip_tiles tiles run as 256 / kPairStripN strips each.
  int64_t strip_tiles = 0;
  int64_t unit_count() const {
    if (balanced) return units;
    if (strip_tiles > 0) return tiles - strip_tiles + strip_tiles * (256 / kPairStripN);
    return full + (tiles - full) * split;
  }
};

// Time of a wave of kPairStripN-column strips of 256-column pair tiles, in
// waves of whole tiles of the same K.  A strip streams all of A's k-blocks
// but a quarter of B's (20 of 32 KB per CTA and k-block).  Measured on GB300
// at 3000 x 5000 x 2000 (32 k-blocks, 12 tail tiles as 48 strips): 55.6 us
// against 57.9 us for four waves of 224-wide tiles, i.e. (3 + 0.63) x 576
// against 4 x 544 in the width-weighted wave model.
constexpr double kStripWave = 0.63;

// The balanced division of `tiles` pair tiles of `k_blocks` k-blocks over
// `slots` clusters, after dp_waves waves of whole tiles (dp_waves * slots
// tiles run data-parallel first; the ranges cover the rest).
void plan_balanced(int64_t tiles, int64_t k_blocks, int slots, PairChoice* c,
                   int64_t dp_waves = 0) {
  c->tiles = tiles;
  c->full = tiles;
  c->split = 1;
  c->kb_per_piece = static_cast<int>(k_blocks);
  c->balanced = true;
  c->dp_tiles = dp_waves * slots;
  const int64_t work = (tiles - c->dp_tiles) * k_blocks;
  c->per = work / slots;
  c->extra = static_cast<int>(work % slots);
  c->units = c->dp_tiles;
  c->max_pieces = 1;
  for (int k = 0; k < slots; ++k) {
    const int n = balanced_units(c->per, c->extra, static_cast<int>(k_blocks), k);
    c->units += n;
    for (int i = 0; i < std::min(n, 2); ++i)
      c->max_pieces = std::max(
          c->max_pieces, balanced_unit(c->per, c->extra, static_cast<int>(k_blocks), k, i).pieces);
  }
}

// Whether the balanced division is used: only when GB3_GEMM_BALANCED = 1
// (then wherever it applies: every cluster gets at least one tile's worth of
// k-blocks); the tests' forced split of every tile (GB3_GEMM_SPLIT_ALL)
// turns it off.  It is not chosen by default because it measured slower on
// GB300 than the tail split: 4096^3 1519 against 1667 TFLOP/s, 3000 x 5000 x
// 2000 66.3 against 56.9 us, gate/up 4096 x 14336 x 4096 718 against 509 us.
// The last piece of a cut tile sums the partials while the next main loop
// streams its operands, and its loads from L2 queue behind that stream: a
// combining epilogue took 13-22 us against 3-6 us for a whole tile, and with
// up to two cut tiles per cluster, placed first, both accumulators wait.
int balanced_mode() {
  if (env_int("GB3_GEMM_SPLIT_ALL", 0) > 1) return 0;
  const int m = env_int("GB3_GEMM_BALANCED", 0);
  return m == 1 || m == 2 ? m : 0;
}

// Tail split of `tiles` pair tiles on `slots` resident pairs: the last,
// partial wave's tiles are cut along K so that their pieces fill the pairs.
void plan_tail(int64_t tiles, int64_t k_blocks, int slots, bool allow_split, PairChoice* c) {
  c->tiles = tiles;
  c->full = tiles;
  c->split = 1;
  c->kb_per_piece = static_cast<int>(k_blocks);
  const int64_t tail = tiles % slots;
  const int split_all = env_int("GB3_GEMM_SPLIT_ALL", 0);
  if (allow_split && split_all > 1) {  // tests: every tile split into split_all pieces
    const int64_t kbp = ceil_div(k_blocks, std::min<int64_t>(split_all, k_blocks));
    c->full = 0;
    c->kb_per_piece = static_cast<int>(kbp);
    c->split = static_cast<int>(ceil_div(k_blocks, kbp));
    return;
  }
  if (!allow_split || tail == 0 || env_int("GB3_GEMM_TAIL_SPLIT", 1) == 0) return;
  const int64_t s = std::min<int64_t>(
      {static_cast<int64_t>(kMaxTailSplit), slots / tail, k_blocks / kMinPieceKb});
  if (s < 2) return;
  const int64_t kbp = ceil_div(k_blocks, s);
  c->full = tiles - tail;
  c->kb_per_piece = static_cast<int>(kbp);
  c->split = static_cast<int>(ceil_div(k_blocks, kbp));
}

// Waves of pair tiles a division takes on `slots` pairs: a split tail wave
// counts 1/split of a wave, the balanced division its longest range in
// tiles; either adds a charge for its partial sums.
double pair_waves(const PairChoice& c, int64_t k_blocks, int slots) {
  if (c.strip_tiles > 0) return static_cast<double>((c.tiles - c.strip_tiles) / slots) + kStripWave;
  if (c.balanced) {
    const double w = static_cast<double>(c.dp_tiles / slots) +
                     static_cast<double>(ceil_div((c.tiles - c.dp_tiles) * k_blocks, slots)) /
                         k_blocks;
    return w + (c.max_pieces > 1 ? kSplitCharge : 0.0);
  }
  double waves = static_cast<double>(c.full / slots);
  const int64_t left = c.tiles - (c.full / slots) * slots;
  if (left > 0) waves += c.split > 1 ? 1.0 / c.split + kSplitCharge : 1.0;
  return waves;
}

// The division of `tiles` pair tiles of one width: the tail split; for
// 256-column tiles whose partial last wave cannot be split along K (pieces
// would be shorter than kMinPieceKb), strips of that wave's tiles along N
// when they fit on the resident pairs (GB3_GEMM_STRIPS = 0 turns them off,
// 1 takes them wherever they apply); or the balanced division where it is
// enabled and applies.
PairChoice choose_pair_division(int64_t tiles, int64_t k_blocks, int slots, bool allow_split,
                                int bn, bool allow_strips = false, bool allow_dp_prefix = true) {
  PairChoice c;
  c.bn = bn;
  plan_tail(tiles, k_blocks, slots, allow_split, &c);
  const int64_t tail = tiles % slots;
  const int strips_env = env_int("GB3_GEMM_STRIPS", -1);
  if (allow_strips && allow_split && bn == 256 && strips_env != 0 && tail > 0 &&
      tail * (256 / kPairStripN) <= slots && env_int("GB3_GEMM_SPLIT_ALL", 0) <= 1 &&
      (c.split == 1 || strips_env == 1)) {
    PairChoice st;
    st.bn = bn;
    st.tiles = tiles;
    st.full = tiles;
    st.split = 1;
    st.kb_per_piece = static_cast<int>(k_blocks);
    st.strip_tiles = tail;
    if (strips_env == 1 || pair_waves(st, k_blocks, slots) < pair_waves(c, k_blocks, slots)) c = st;
  }
  const int mode = balanced_mode();
  if (!allow_split || mode == 0 || tiles < slots || (mode == 2 && !allow_dp_prefix)) return c;
  PairChoice b;
  b.bn = bn;
  // mode 2: all whole waves but the last run data-parallel, the last whole
  // wave and the partial one are divided
  plan_balanced(tiles, k_blocks, slots, &b, mode == 2 ? tiles / slots - 1 : 0);
  return b;
}

// Tile width of the CTA-pair GEMM and its division: the fewest waves of pair
// tiles weighted by the time a wave of that width takes.
PairChoice choose_pair(int64_t batch, int64_t M, int64_t N, int64_t K, int slots,
                       bool allow_split, bool allow_strips = false, bool allow_dp_prefix = true) {
  PairChoice best;
  double best_cost = 1e300;
  const int64_t mb = ceil_div(M, kPairBM);
  const int64_t kb = ceil_div(K, kBK);
  // GB3_GEMM_PAIR_TILE_N=<width> restricts the choice to one compiled width
  // (tuning and tests); other values are ignored.
  const int forced = env_int("GB3_GEMM_PAIR_TILE_N", 0);
  bool forced_valid = false;
  for (int bn : kPairWidths) forced_valid |= (bn == forced);
  for (int bn : kPairWidths) {
    if (forced_valid && bn != forced) continue;
    PairChoice c =
        choose_pair_division(batch * mb * ceil_div(N, bn), kb, slots, allow_split, bn, allow_strips,
                             allow_dp_prefix);
    // Measured on GB300 (8192^3): a wave of 256-wide pair tiles takes 1.057x
    // the time of 224-wide ones for 1.143x the work, i.e. time ~ width + 320.
    const double cost = pair_waves(c, kb, slots) * static_cast<double>(bn + kWidthCostOffset);
    if (cost < best_cost) {
      best_cost = cost;
      best = c;
    }
  }
  return best;
}

// Partial sums of a division: one 256 x bn FP32 tile per piece of a split
// tail tile, or per slot of the balanced division (two per cluster).
int64_t pair_workspace_bytes(const PairChoice& c, int slots) {
  if (c.balanced) return c.max_pieces > 1 ? 2LL * slots * kPairBM * c.bn * 4 : 0;
  if (c.split <= 1) return 0;
  return (c.tiles - c.full) * c.split * static_cast<int64_t>(kPairBM) * c.bn * 4;
}

// Arrival counters of a division (8 bands of 32 rows per split tile): per
// tail tile, or per cluster of the balanced division (a split tile's counter
// belongs to the cluster holding its second piece).
int64_t pair_counter_count(const PairChoice& c, int slots) {
  if (c.balanced) return c.max_pieces > 1 ? 8LL * (slots + 1) : 0;
  if (c.split <= 1) return 0;
  return 8 * (c.tiles - c.full);
}

// pair_slots: CTA pairs that fit on the device at once (0: assume sms / 2,
// negative: pair kernels unavailable).
// The split-K kernel's plan for an M <= 16, K > 0 problem (also the plan of
// the allocation-free entry point, which runs that kernel whatever plan_gemm
// would choose).
int plan_skinny(int64_t batch, int64_t M, int64_t N, int64_t K, int sms, gemm_plan* pl) {
  (void)M;
  const int64_t nb = ceil_div(N, kSkinnyRows), kb = ceil_div(K, kBK);
  int s, kbp;
  choose_split(batch * nb, kb, sms, &s, &kbp);
  pl->kernel = K_SKINNY;
  pl->tile_m = kSkinnyRows;
  pl->tile_n = kSkinnyNX;
  pl->tile_k = kBK;
  pl->stages = kSkinnyStages;
  pl->split_k = s;
  pl->tiles = batch * nb * s;
  pl->grid = static_cast<int>(std::min<int64_t>(pl->tiles, sms));
  pl->smem_bytes = CfgSkinny::kSmemBytes;
  pl->launches = 1;
  pl->stage_tx_bytes = CfgSkinny::kStageBytes;
  return GEMM_OK;
}

int plan_gemm(int64_t batch, int64_t M, int64_t N, int64_t K, int sms, gemm_plan* pl,
              int pair_slots = 0, bool allow_split = true, bool row_stats = false) {
  std::memset(pl, 0, sizeof(*pl));
  pl->split_k = 1;
  if (batch == 0 || M == 0 || N == 0) return GEMM_OK;
  if (K == 0) {
    pl->kernel = K_SCALE;
    pl->tiles = 1;
    pl->grid = static_cast<int>(std::min<int64_t>(ceil_div(batch * M * N, 256), 4 * sms));
    pl->launches = row_stats ? 2 : 1;
    return GEMM_OK;
  }
  pl->tile_k = kBK;
  // Row reductions run in the tile epilogues; the swapped-operand kernels hold
  // rows across threads, so those problems take the tiled path.
  if (!row_stats && use_small_m(batch, M, N, K, sms)) {
    const int nx = smallm_nx(M);
    pl->kernel = K_SMALL_M;
    pl->tile_m = kSmallRows;
    pl->tile_n = nx;
    pl->tiles = batch * ceil_div(N, kSmallRows);
    pl->grid = smallm_grid(pl->tiles, ceil_div(K, kBK), sms);
    SmallMParams d;
    smallm_divide(pl->tiles, ceil_div(K, kBK), pl->grid, &d);
    pl->split_k = d.max_pieces;
    pl->stages = smallm_stages(nx);
    pl->smem_bytes = smallm_smem(nx);
    pl->launches = 1;
    pl->stage_tx_bytes = kSmallRows * kBK * 2 + static_cast<int64_t>(nx) * kBK * 2;
    return GEMM_OK;
  }
  if (M <= kSkinnyMaxM && !row_stats) return plan_skinny(batch, M, N, K, sms, pl);
  if (M >= kPairMinM && pair_slots >= 0) {
    const int slots = pair_slots > 0 ? pair_slots : std::max(1, sms / 2);
    const PairChoice c = choose_pair(batch, M, N, K, slots, allow_split, !row_stats);
    const int64_t units = c.unit_count();
    pl->kernel = K_PAIR;
    pl->tile_m = kPairBM;
    pl->tile_n = c.bn;
    pl->stages = kPairStages;
    pl->split_k = c.balanced ? c.max_pieces : c.split;
    pl->tiles = units;
    pl->grid = 2 * static_cast<int>(std::min<int64_t>(units, slots));
    pl->smem_bytes = pair_smem_for(c.bn);
    pl->launches = 1;
    pl->stage_tx_bytes = 2 * pair_stage_bytes(c.bn);
    return GEMM_OK;
  }
  pl->kernel = K_TILED;
  pl->tile_m = kBM;
  pl->tile_n = kTileN;
  pl->stages = kStages;
  pl->tiles = batch * ceil_div(M, kBM) * ceil_div(N, kTileN);
  pl->grid = static_cast<int>(std::min<int64_t>(pl->tiles, sms));
  pl->smem_bytes = CfgBF16::kSmemBytes;
  pl->launches = 1;
  pl->stage_tx_bytes = CfgBF16::kStageBytes;
  return GEMM_OK;
}

int plan_gate_up(int64_t M, int64_t N, int64_t K, int sms, gemm_plan* pl, int pair_slots = 0,
                 bool allow_split = true) {
  std::memset(pl, 0, sizeof(*pl));
  pl->split_k = 1;
  if (M == 0 || N == 0) return GEMM_OK;
  if (K == 0) {
    pl->kernel = K_SCALE;
    pl->tiles = 1;
    pl->grid = static_cast<int>(std::min<int64_t>(ceil_div(M * N, 256), 4 * sms));
    pl->launches = 1;
    return GEMM_OK;
  }
  if (M >= kPairMinM && pair_slots >= 0) {
    const int slots = pair_slots > 0 ? pair_slots : std::max(1, sms / 2);
    const PairChoice c =
        choose_pair_division(ceil_div(M, kPairBM) * ceil_div(N, CfgPairGU::kOutCols),
                             ceil_div(K, kBK), slots, allow_split, 256);
    const int64_t units = c.unit_count();
    pl->kernel = K_PAIR_GATE_UP;
    pl->tile_m = kPairBM;
    pl->tile_n = CfgPairGU::kOutCols;
    pl->tile_k = kBK;
    pl->stages = kPairStages;
    pl->split_k = c.balanced ? c.max_pieces : c.split;
    pl->tiles = units;
    pl->grid = 2 * static_cast<int>(std::min<int64_t>(units, slots));
    pl->smem_bytes = CfgPairGU::kSmemBytes;
    pl->launches = 1;
    pl->stage_tx_bytes = 2 * CfgPairGU::kStageBytes;
    return GEMM_OK;
  }
  if (M <= kSkinnyMaxM && env_int("GB3_GATE_UP_SKINNY", 1) != 0) {
    // Decode sizes: Wg and Wu stream through the split-K kernel together.
    const int64_t nb = ceil_div(N, kSkinnyRows), kb = ceil_div(K, kBK);
    int s, kbp;
    choose_split(nb, kb, sms, &s, &kbp, 2);
    pl->kernel = K_SKINNY_GATE_UP;
    pl->tile_m = kSkinnyRows;
    pl->tile_n = kSkinnyNX;
    pl->tile_k = kBK;
    pl->stages = kSkinnyGateUpStages;
    pl->split_k = s;
    pl->tiles = nb * s;
    pl->grid = static_cast<int>(std::min<int64_t>(pl->tiles, sms));
    pl->smem_bytes = CfgSkinnyGU::kSmemBytes;
    pl->launches = 1;
    pl->stage_tx_bytes = CfgSkinnyGU::kStageBytes;
    return GEMM_OK;
  }
  pl->kernel = K_GATE_UP;
  pl->tile_m = kBM;
  pl->tile_n = CfgGU::kOutCols;
  pl->tile_k = kBK;
  pl->stages = kGateUpStages;
  pl->tiles = ceil_div(M, kBM) * ceil_div(N, CfgGU::kOutCols);
  pl->grid = static_cast<int>(std::min<int64_t>(pl->tiles, sms));
  pl->smem_bytes = CfgGU::kSmemBytes;
  pl->launches = 1;
  pl->stage_tx_bytes = CfgGU::kStageBytes;
  return GEMM_OK;
}

// ----------------------------------------------------------------------------
// Validation (no CUDA calls)
// ----------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The kernels count work units (output tiles, split pieces, strips) in 32-bit
// integers, and a plan has at most 32 units per block of 128 x 128 outputs
// (split K), so a call may hold at most 2^25 such blocks: at least 5.5 * 10^11
// output elements (1.1 TB in BF16), more than any GPU memory holds, so no
// problem whose operands fit is refused.
constexpr int64_t kMaxOutputBlocks = int64_t{1} << 25;

bool bad_dims(int64_t batch, int64_t M, int64_t N, int64_t K) {
  if (batch < 0 || M < 0 || N < 0 || K < 0 || batch > kMaxDim || M > kMaxDim || N > kMaxDim ||
      K > kMaxDim)
    return true;
  if (batch == 0 || M == 0 || N == 0) return false;
  const int64_t mb = ceil_div(M, 128), nb = ceil_div(N, 128);   // each at most 2^24
  return mb * nb > kMaxOutputBlocks || batch > kMaxOutputBlocks / (mb * nb);
}

int validate_problem(const Problem& p) {
  if (bad_dims(p.batch, p.M, p.N, p.K)) return GEMM_ERR_INVALID_ARG;
  if (p.in_dtype != GEMM_IN_BF16 && p.in_dtype != GEMM_IN_F16) return GEMM_ERR_INVALID_ARG;
  if (p.out_dtype != GEMM_OUT_F32 && p.out_dtype != GEMM_OUT_BF16 && p.out_dtype != GEMM_OUT_F16)
    return GEMM_ERR_INVALID_ARG;
  if (p.batch == 0 || p.M == 0 || p.N == 0) return GEMM_OK;
  const int64_t esize = out_elem_bytes(p.out_dtype);
  if (p.C == nullptr || p.ldc < p.N) return GEMM_ERR_INVALID_ARG;
  if (p.batch > 1 && p.sc < p.M * p.ldc) return GEMM_ERR_INVALID_ARG;
  if (p.K > 0) {
    if (p.A == nullptr || p.B == nullptr || p.lda < p.K || p.ldb < p.K)
      return GEMM_ERR_INVALID_ARG;
    if (p.batch > 1 && (p.sa < p.M * p.lda || p.sb < p.N * p.ldb)) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(p.A) || !aligned16(p.B) || (p.lda * 2) % 16 != 0 || (p.ldb * 2) % 16 != 0)
      return GEMM_ERR_ALIGNMENT;
    if (p.batch > 1 && ((p.sa * 2) % 16 != 0 || (p.sb * 2) % 16 != 0)) return GEMM_ERR_ALIGNMENT;
  }
  if (!aligned16(p.C) || (p.ldc * esize) % 16 != 0) return GEMM_ERR_ALIGNMENT;
  if (p.batch > 1 && (p.sc * esize) % 16 != 0) return GEMM_ERR_ALIGNMENT;
  return GEMM_OK;
}

int validate_gate_up(int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx, const void* Wg,
                     const void* Wu, int64_t ldw, const void* Y, int64_t ldy) {
  if (bad_dims(1, M, N, K)) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (Y == nullptr || ldy < N) return GEMM_ERR_INVALID_ARG;
  if (K > 0) {
    if (X == nullptr || Wg == nullptr || Wu == nullptr || ldx < K || ldw < K)
      return GEMM_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Wg) || !aligned16(Wu) || (ldx * 2) % 16 != 0 ||
        (ldw * 2) % 16 != 0)
      return GEMM_ERR_ALIGNMENT;
  }
  if (!aligned16(Y) || (ldy * 2) % 16 != 0) return GEMM_ERR_ALIGNMENT;
  return GEMM_OK;
}

// ----------------------------------------------------------------------------
// Device state
// ----------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

struct DeviceState {
  bool probed = false;
  bool supported = false;
  int sms = 0;
  // CTA pairs that fit on the device at once (0: not queried yet, -1: none)
  int pair_slots = 0;
  // kernels whose shared-memory limit has been raised on this device
  std::vector<const void*> configured;
  // split-K workspace (skinny path and split tail tiles)
  float* ws = nullptr;
  size_t ws_bytes = 0;
  int* counters = nullptr;
  size_t counter_count = 0;
  // row-reduction partials and arrival counters
  float* stats_ws = nullptr;
  size_t stats_ws_bytes = 0;
  int* stats_counters = nullptr;
  size_t stats_counter_count = 0;
  // device address of the grid-barrier counters (a library array, not allocated)
  unsigned int* grid_sync = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (*dev < 0 || *dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
  return GEMM_OK;
}

// Caller holds g_mu.
int probe_device(int dev) {
  DeviceState& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    d.probed = true;
    d.supported = (major == 10 && minor == 3);
    d.sms = sms;
  }
  return d.supported ? GEMM_OK : GEMM_ERR_UNSUPPORTED;
}

// Caller holds g_mu.
int ensure_smem_attr(int dev, const void* fn, int smem) {
  DeviceState& d = g_dev[dev];
  if (std::find(d.configured.begin(), d.configured.end(), fn) != d.configured.end())
    return GEMM_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  d.configured.push_back(fn);
  return GEMM_OK;
}

// Caller holds g_mu.  Grows the split-K workspace; refuses to allocate while
// the stream is being captured.
int ensure_workspace(int dev, size_t ws_bytes, size_t counters, cudaStream_t stream) {
  DeviceState& d = g_dev[dev];
  if (d.ws_bytes >= ws_bytes && d.counter_count >= counters) return GEMM_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return GEMM_ERR_CUDA;
  // Work already queued may still use the old buffers.
  if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
  if (d.ws_bytes < ws_bytes) {
    if (d.ws) cudaFree(d.ws);
    d.ws = nullptr;
    d.ws_bytes = 0;
    if (cudaMalloc(&d.ws, ws_bytes) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    d.ws_bytes = ws_bytes;
  }
  if (d.counter_count < counters) {
    if (d.counters) cudaFree(d.counters);
    d.counters = nullptr;
    d.counter_count = 0;
    if (cudaMalloc(&d.counters, counters * sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    if (cudaMemset(d.counters, 0, counters * sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    d.counter_count = counters;
  }
  return GEMM_OK;
}

// Caller holds g_mu.  Grows one (buffer, counters) pair; refuses to allocate
// while the stream is being captured.
int grow_buffers(float** buf, size_t* buf_bytes, int** cnt, size_t* cnt_count, size_t need_bytes,
                 size_t need_counters, cudaStream_t stream) {
  if (*buf_bytes >= need_bytes && *cnt_count >= need_counters) return GEMM_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return GEMM_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
  if (*buf_bytes < need_bytes) {
    if (*buf) cudaFree(*buf);
    *buf = nullptr;
    *buf_bytes = 0;
    if (cudaMalloc(buf, need_bytes) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    *buf_bytes = need_bytes;
  }
  if (*cnt_count < need_counters) {
    if (*cnt) cudaFree(*cnt);
    *cnt = nullptr;
    *cnt_count = 0;
    if (cudaMalloc(cnt, need_counters * sizeof(int)) != cudaSuccess ||
        cudaMemset(*cnt, 0, need_counters * sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    *cnt_count = need_counters;
  }
  return GEMM_OK;
}

// Fills rs with q's row-reduction outputs and the device's partials buffer,
// grown for n_blocks column tiles.  Leaves rs empty when q wants none.
int attach_row_stats(int dev, const Problem& q, int n_blocks, RowStatsParams* rs,
                     cudaStream_t stream) {
  *rs = RowStatsParams{nullptr, nullptr, nullptr, nullptr, nullptr};
  if (!q.stats()) return GEMM_OK;
  const size_t bytes = 3 * static_cast<size_t>(q.batch) * n_blocks * q.M * sizeof(float);
  const size_t counters = static_cast<size_t>(q.batch) * ceil_div(q.M, 32);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  const int st = grow_buffers(&d.stats_ws, &d.stats_ws_bytes, &d.stats_counters,
                              &d.stats_counter_count, bytes, counters, stream);
  if (st != GEMM_OK) return st;
  *rs = RowStatsParams{q.row_sum, q.row_max, q.row_min, d.stats_ws, d.stats_counters};
  return GEMM_OK;
}

// ----------------------------------------------------------------------------
// Tensor-map descriptors
// ----------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  int dtype;
  uint64_t inner, outer, batch, pitch, bstride;
  uint32_t box_inner, box_outer;
  int swizzle;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && dtype == o.dtype && inner == o.inner && outer == o.outer &&
           batch == o.batch && pitch == o.pitch && bstride == o.bstride &&
           box_inner == o.box_inner && box_outer == o.box_outer && swizzle == o.swizzle;
  }
};

struct MapEntry {
  MapKey key;
  CUtensorMap map;
  uint64_t used;
};

constexpr size_t kMapCacheSize = 64;
std::mutex g_map_mu;
std::vector<MapEntry> g_maps;
uint64_t g_map_clock = 0;

// Encodes a 3-D map: `batch` matrices `bstride` bytes apart, each of `outer`
// rows of `inner` elements with a row pitch of `pitch` bytes; box of
// box_inner x box_outer elements of one matrix; out-of-bounds elements read
// as zero.  No cache, no allocation.
int encode_map_3d(CUtensorMap* out, const void* ptr, CUtensorMapDataType dtype, uint64_t inner,
                  uint64_t outer, uint64_t batch, uint64_t pitch, uint64_t bstride,
                  uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr) return GEMM_ERR_CUDA;
  const cuuint64_t dims[3] = {inner, outer, batch};
  const cuuint64_t strides[2] = {pitch, bstride};
  const cuuint32_t box[3] = {box_inner, box_outer, 1};
  const cuuint32_t estrides[3] = {1, 1, 1};
  const CUresult r = fn(out, dtype, 3, const_cast<void*>(ptr), dims, strides, box, estrides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// encode_map_3d through the descriptor cache.  A single matrix passes
// batch = 1 and bstride = pitch * outer.
int tensor_map_3d(CUtensorMap* out, const void* ptr, CUtensorMapDataType dtype, uint64_t inner,
                  uint64_t outer, uint64_t batch, uint64_t pitch, uint64_t bstride,
                  uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const MapKey key{ptr,     static_cast<int>(dtype), inner,     outer, batch,
                   pitch,   bstride,                 box_inner, box_outer,
                   static_cast<int>(swizzle)};
  std::lock_guard<std::mutex> lk(g_map_mu);
  for (MapEntry& e : g_maps) {
    if (e.key == key) {
      e.used = ++g_map_clock;
      *out = e.map;
      return GEMM_OK;
    }
  }
  CUtensorMap map;
  const int st = encode_map_3d(&map, ptr, dtype, inner, outer, batch, pitch, bstride, box_inner,
                               box_outer, swizzle);
  if (st != GEMM_OK) return st;
  if (g_maps.size() < kMapCacheSize) {
    g_maps.push_back(MapEntry{key, map, ++g_map_clock});
  } else {
    auto victim = std::min_element(g_maps.begin(), g_maps.end(),
                                   [](const MapEntry& a, const MapEntry& b) { return a.used < b.used; });
    *victim = MapEntry{key, map, ++g_map_clock};
  }
  *out = map;
  return GEMM_OK;
}

// Operand map of A (rows = M) or B (rows = N): box of 64 K-elements by `rows_box` rows.
int operand_map(CUtensorMap* out, const void* ptr, int in_dtype, int64_t K, int64_t rows,
                int64_t batch, int64_t ld, int64_t stride, uint32_t rows_box) {
  const uint64_t pitch = static_cast<uint64_t>(ld) * 2;
  const uint64_t bstride = batch > 1 ? static_cast<uint64_t>(stride) * 2 : pitch * rows;
  return tensor_map_3d(out, ptr, in_tma_type(in_dtype), K, rows, batch, pitch, bstride, kBK,
                       rows_box);
}

// Output descriptor of an epilogue box: FP32 32 x 32 (128-byte swizzle);
// 16-bit 64 x 32 (128-byte swizzle) or, for tile widths not a multiple of 64,
// 32 x 32 (64-byte swizzle).  Must match EpiBox in gemm_kernels.cuh.
int output_map(CUtensorMap* out, void* C, int64_t batch, int64_t M, int64_t N, int64_t ldc,
               int64_t sc, int out_dtype, int tile_out_cols) {
  const int es = out_elem_bytes(out_dtype);
  const uint64_t pitch = static_cast<uint64_t>(ldc) * es;
  const uint64_t bstride = batch > 1 ? static_cast<uint64_t>(sc) * es : pitch * M;
  if (out_dtype == GEMM_OUT_F32)
    return tensor_map_3d(out, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, N, M, batch, pitch, bstride, 32,
                         32);
  const CUtensorMapDataType t = out_dtype == GEMM_OUT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (tile_out_cols % 64 == 0)
    return tensor_map_3d(out, C, t, N, M, batch, pitch, bstride, 64, 32);
  return tensor_map_3d(out, C, t, N, M, batch, pitch, bstride, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// ----------------------------------------------------------------------------
// Launch
// ----------------------------------------------------------------------------
template <typename... ExpT, typename... ActT>
int launch(void (*kernel)(ExpT...), int grid, int block, int smem, cudaStream_t stream,
           ActT&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(block), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  if (cudaLaunchKernelEx(&cfg, kernel, std::forward<ActT>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}

// cooperative: every CTA of the grid is resident at once (the kernel's CTAs
// wait on one another at a grid-wide barrier); the launch fails otherwise.
template <typename... ExpT, typename... ActT>
int launch_pair(void (*kernel)(ExpT...), int grid, int smem, cudaStream_t stream, bool cooperative,
                ActT&&... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(kThreads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, kernel, std::forward<ActT>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}

// Caller holds g_mu.  Number of CTA pairs of the pair kernels (about 226 KB of
// shared memory each, one CTA per SM) that can be resident at once.
int query_pair_slots(int dev) {
  DeviceState& d = g_dev[dev];
  if (d.pair_slots != 0) return d.pair_slots;
  auto kern = gemm_pair_kernel<256, kPairStages, EPI_BF16>;
  const int smem = pair_smem_bytes<256>();
  if (ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), smem) != GEMM_OK) {
    d.pair_slots = -1;
    return d.pair_slots;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * std::max(1, d.sms / 2)), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(kern), &cfg) !=
          cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    d.pair_slots = -1;
  } else {
    d.pair_slots = n;
  }
  return d.pair_slots;
}

// Row geometry of the normalisation the gate/up kernel runs before its GEMM,
// the one the standalone normalisation takes for BF16 rows of D elements (so
// that Xn has the same bits): 1 for rows of at most 4 vectors of 16 bytes per
// lane (one warp, 4 cached), 2 above (two warps of 8 cached each); 0 when the
// standalone normalisation is forced onto one warp per long row
// (GB3_NORM_ROW_WARPS = 1), which the two-launch path then runs.
int fused_norm_geometry(int64_t D) {
  const int64_t vecs_per_lane = (D * 2 + 32 * 16 - 1) / (32 * 16);
  if (vecs_per_lane <= 4) return 1;
  return env_int("GB3_NORM_ROW_WARPS", 2) == 1 ? 0 : 2;
}

// The device address of the grid-barrier counters (a fixed array of the
// library, zero at load, reset by the last CTA of every launch).
__device__ unsigned int g_grid_sync[2];

// Caller holds g_mu.
int grid_sync_counters(int dev, unsigned int** out) {
  DeviceState& d = g_dev[dev];
  if (d.grid_sync == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_grid_sync) != cudaSuccess || addr == nullptr) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    d.grid_sync = static_cast<unsigned int*>(addr);
  }
  *out = d.grid_sync;
  return GEMM_OK;
}

// C = beta * C for every matrix of the batch (K == 0); C is not read when
// beta == 0.  out_kind: 0 FP32, 1 BF16, 2 FP16.
__global__ void scale_kernel(void* C, long long ldc, long long sc, int batch, int M, int N,
                             float beta, int out_kind) {
  const long long per = static_cast<long long>(M) * N;
  const long long total = per * batch;
  const bool f16 = out_kind == 2;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long b = i / per, r = i % per;
    const long long m = r / N, n = r % N;
    const long long off = b * sc + m * ldc + n;
    if (out_kind != 0) {
      uint16_t* c = static_cast<uint16_t*>(C);
      const float v = beta == 0.0f ? 0.0f : beta * half16_to_float(c[off], f16);
      c[off] = static_cast<uint16_t>(pack_half16x2(v, 0.0f, f16) & 0xFFFFu);
    } else {
      float* c = static_cast<float*>(C);
      c[off] = beta == 0.0f ? 0.0f : beta * c[off];
    }
  }
}

// Row reductions of beta * C when K == 0 (C not read when beta == 0): one
// warp per row, lanes over the columns, then a shuffle butterfly.
__global__ void row_stats_k0_kernel(const void* C, long long ldc, long long sc, int batch, int M,
                                    int N, float beta, int out_kind, float* rsum, float* rmax,
                                    float* rmin) {
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(batch) * M;
  const bool f16 = out_kind == 2;
  for (long long r = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
       r < rows; r += (static_cast<long long>(gridDim.x) * blockDim.x) >> 5) {
    const long long b = r / M, m = r % M;
    const long long off = b * sc + m * ldc;
    float sum = 0.0f, mx = -INFINITY, mn = INFINITY;
    for (int n = lane; n < N; n += 32) {
      float v = 0.0f;
      if (beta != 0.0f) {
        const float c = out_kind == 0 ? static_cast<const float*>(C)[off + n]
                                      : half16_to_float(static_cast<const uint16_t*>(C)[off + n], f16);
        v = beta * c;
      }
      sum += v;
      mx = fmaxf(mx, v);
      mn = fminf(mn, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
      if (rsum) rsum[r] = sum;
      if (rmax) rmax[r] = mx;
      if (rmin) rmin[r] = mn;
    }
  }
}

int run_scale(const gemm_plan& pl, void* C, int64_t ldc, int64_t sc, int64_t batch, int64_t M,
              int64_t N, float beta, int out_dtype, cudaStream_t stream) {
  return launch(scale_kernel, pl.grid, 256, 0, stream, C, static_cast<long long>(ldc),
                static_cast<long long>(sc), static_cast<int>(batch), static_cast<int>(M),
                static_cast<int>(N), beta, out_dtype);
}

TileParams tile_params(const Problem& q, int tile_m, int tile_n_out, uint32_t idesc) {
  TileParams p;
  p.M = static_cast<int>(q.M);
  p.N = static_cast<int>(q.N);
  p.K = static_cast<int>(q.K);
  p.m_blocks = static_cast<int>(ceil_div(q.M, tile_m));
  p.n_blocks = static_cast<int>(ceil_div(q.N, tile_n_out));
  p.k_blocks = static_cast<int>(ceil_div(q.K, kBK));
  p.batch = static_cast<int>(q.batch);
  p.tiles_per_matrix = p.m_blocks * p.n_blocks;
  p.num_tiles = static_cast<int>(q.batch * p.tiles_per_matrix);
  p.group_m = kGroupM;
  p.idesc = idesc;
  p.out_f16 = q.out_dtype == GEMM_OUT_F16 ? 1 : 0;
  p.c_stride = q.batch > 1 ? q.sc : 0;
  p.alpha = q.alpha;
  p.beta = q.beta;
  p.C = q.C;
  p.ldc = q.ldc;
  p.num_full = p.num_tiles;
  p.tail_split = 1;
  p.kb_per_piece = p.k_blocks;
  p.num_units = p.num_tiles;
  p.balanced = 0;
  p.work_per_cluster = 0;
  p.work_extra = 0;
  p.dp_tiles = 0;
  p.strip_tiles = 0;
  p.idesc_strip = idesc_f32_acc(kPairBM, kPairStripN, q.in_dtype == GEMM_IN_F16);
  p.ws = nullptr;
  p.counters = nullptr;
  return p;
}

// Work units of a pair plan (split tail pieces, then whole tiles) and the
// workspace they need.  A plan that needs a workspace the device cannot get
// (the stream is being captured) runs its tiles whole instead.
void pair_units(int dev, gemm_plan* pl, const Problem& q, int out_cols, TileParams* p,
                cudaStream_t stream, bool gate_up, int slots) {
  PairChoice c;
  if (gate_up) {
    c = choose_pair_division(p->num_tiles, p->k_blocks, slots, true, 256);
  } else {
    // The C ring's look-ahead assumes a cluster's split pieces come before its
    // whole tiles, which whole waves ahead of the divided ranges break.
    c = choose_pair(q.batch, q.M, q.N, q.K, slots, true, !q.stats(), !pair_reads_c_ring(q.beta));
  }
  (void)out_cols;
  if (pair_workspace_bytes(c, slots) > 0) {
    const size_t ws = static_cast<size_t>(pair_workspace_bytes(c, slots));
    const size_t counters = static_cast<size_t>(pair_counter_count(c, slots));
    int st;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      st = ensure_workspace(dev, ws, counters, stream);
      if (st == GEMM_OK) {
        p->ws = g_dev[dev].ws;
        p->counters = g_dev[dev].counters;
      }
    }
    if (st != GEMM_OK) {
      c.balanced = false;
      c.dp_tiles = 0;
      c.full = c.tiles;
      c.split = 1;
      c.kb_per_piece = p->k_blocks;
      pl->split_k = 1;
      pl->tiles = c.tiles;
      pl->grid = 2 * static_cast<int>(std::min<int64_t>(c.tiles, slots));
    }
  }
  p->num_full = static_cast<int>(c.full);
  p->tail_split = c.split;
  p->kb_per_piece = c.kb_per_piece;
  p->num_units = static_cast<int>(c.unit_count());
  p->balanced = c.balanced ? 1 : 0;
  p->work_per_cluster = c.per;
  p->work_extra = c.extra;
  p->dp_tiles = static_cast<int>(c.dp_tiles);
  p->strip_tiles = static_cast<int>(c.strip_tiles);
}

// RING: C is read through the deeper staging ring (beta != 0), which takes
// the shared memory of one pipeline stage.
// NORM != 0: the gate/up kernel that normalises its activation first (one
// cooperative launch, see NormParams).
template <int BN, int EPI, bool STATS = false, bool RING = false, int NORM = 0>
int launch_pair_gemm(const gemm_plan& pl, int dev, const CUtensorMap& tmA, const CUtensorMap& tmB,
                     const CUtensorMap& tmB2, const CUtensorMap& tmOut, const TileParams& p,
                     cudaStream_t stream, const RowStatsParams& rs = RowStatsParams{},
                     const NormParams& nrm = NormParams{}) {
  constexpr int kStagesHere = RING ? kPairStages - 1 : kPairStages;
  using Cfg = PairCfg<BN, kStagesHere, EPI, RING>;
  auto kern = gemm_pair_kernel<BN, kStagesHere, EPI, STATS, RING, NORM>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const int st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), Cfg::kSmemBytes);
    if (st != GEMM_OK) return st;
  }
  return launch_pair(kern, pl.grid, Cfg::kSmemBytes, stream, NORM != 0, tmA, tmB, tmB2, tmOut, p,
                     rs, nrm);
}

template <int BN, int STAGES, int EPI, bool STATS = false>
int launch_single_gemm(const gemm_plan& pl, int dev, const CUtensorMap& tmA,
                       const CUtensorMap& tmB, const CUtensorMap& tmB2, const CUtensorMap& tmOut,
                       const TileParams& p, cudaStream_t stream,
                       const RowStatsParams& rs = RowStatsParams{}) {
  using Cfg = GemmCfg<BN, STAGES, EPI>;
  auto kern = gemm_tc_kernel<BN, STAGES, EPI, STATS>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const int st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), Cfg::kSmemBytes);
    if (st != GEMM_OK) return st;
  }
  return launch(kern, pl.grid, kThreads, Cfg::kSmemBytes, stream, tmA, tmB, tmB2, tmOut, p, rs);
}

int run_pair(gemm_plan& pl, int dev, int slots, const Problem& q, cudaStream_t stream) {
  const int bn = pl.tile_n;
  const bool f16in = q.in_dtype == GEMM_IN_F16;
  CUtensorMap tmA, tmB, tmOut;
  int st;
  if ((st = operand_map(&tmA, q.A, q.in_dtype, q.K, q.M, q.batch, q.lda, q.sa, 128)) != GEMM_OK)
    return st;
  if ((st = operand_map(&tmB, q.B, q.in_dtype, q.K, q.N, q.batch, q.ldb, q.sb, bn / 2)) !=
      GEMM_OK)
    return st;
  if ((st = output_map(&tmOut, q.C, q.batch, q.M, q.N, q.ldc, q.sc, q.out_dtype, bn)) != GEMM_OK)
    return st;
  TileParams p = tile_params(q, kPairBM, bn, idesc_f32_acc(kPairBM, bn, f16in));
  RowStatsParams rs;
  if ((st = attach_row_stats(dev, q, p.n_blocks, &rs, stream)) != GEMM_OK) return st;
  pair_units(dev, &pl, q, bn, &p, stream, false, slots);
  if (bn != 256 && bn != 224) return GEMM_ERR_UNSUPPORTED;
  // Strip units load kPairStripN / 2 rows of B per CTA.
  CUtensorMap tmBs = tmB;
  if (p.strip_tiles > 0 &&
      (st = operand_map(&tmBs, q.B, q.in_dtype, q.K, q.N, q.batch, q.ldb, q.sb,
                        kPairStripN / 2)) != GEMM_OK)
    return st;
  // The ring kernels always read C.
  const bool ring = pair_reads_c_ring(q.beta);
  if (ring) {
    pl.stages = kPairStages - 1;
    pl.smem_bytes = pair_ring_smem_for(bn);
  }
  const int sel = (q.out_dtype == GEMM_OUT_F32 ? 1 : 0) | (q.stats() ? 2 : 0) | (ring ? 4 : 0) |
                  (bn == 224 ? 8 : 0);
#define GB3_PAIR_CASE(S, BN_, EPI_, STATS_, RING_)                                              \
  case S:                                                                                       \
    return launch_pair_gemm<BN_, EPI_, STATS_, RING_>(pl, dev, tmA, tmB, tmBs, tmOut, p,      \
                                                      stream, rs);
  switch (sel) {
    GB3_PAIR_CASE(0, 256, EPI_BF16, false, false)
    GB3_PAIR_CASE(1, 256, EPI_F32, false, false)
    GB3_PAIR_CASE(2, 256, EPI_BF16, true, false)
    GB3_PAIR_CASE(3, 256, EPI_F32, true, false)
    GB3_PAIR_CASE(4, 256, EPI_BF16, false, true)
    GB3_PAIR_CASE(5, 256, EPI_F32, false, true)
    GB3_PAIR_CASE(6, 256, EPI_BF16, true, true)
    GB3_PAIR_CASE(7, 256, EPI_F32, true, true)
    GB3_PAIR_CASE(8, 224, EPI_BF16, false, false)
    GB3_PAIR_CASE(9, 224, EPI_F32, false, false)
    GB3_PAIR_CASE(10, 224, EPI_BF16, true, false)
    GB3_PAIR_CASE(11, 224, EPI_F32, true, false)
    GB3_PAIR_CASE(12, 224, EPI_BF16, false, true)
    GB3_PAIR_CASE(13, 224, EPI_F32, false, true)
    GB3_PAIR_CASE(14, 224, EPI_BF16, true, true)
    GB3_PAIR_CASE(15, 224, EPI_F32, true, true)
    default:
      return GEMM_ERR_UNSUPPORTED;
  }
#undef GB3_PAIR_CASE
}

int run_single(const gemm_plan& pl, int dev, const Problem& q, cudaStream_t stream) {
  const bool f16in = q.in_dtype == GEMM_IN_F16;
  CUtensorMap tmA, tmB, tmOut;
  int st;
  if ((st = operand_map(&tmA, q.A, q.in_dtype, q.K, q.M, q.batch, q.lda, q.sa, kBM)) != GEMM_OK)
    return st;
  if ((st = operand_map(&tmB, q.B, q.in_dtype, q.K, q.N, q.batch, q.ldb, q.sb, kTileN)) !=
      GEMM_OK)
    return st;
  if ((st = output_map(&tmOut, q.C, q.batch, q.M, q.N, q.ldc, q.sc, q.out_dtype, kTileN)) !=
      GEMM_OK)
    return st;
  const TileParams p = tile_params(q, kBM, kTileN, idesc_f32_acc(kBM, kTileN, f16in));
  RowStatsParams rs;
  if ((st = attach_row_stats(dev, q, p.n_blocks, &rs, stream)) != GEMM_OK) return st;
  const bool f32 = q.out_dtype == GEMM_OUT_F32;
  if (q.stats())
    return f32 ? launch_single_gemm<kTileN, kStages, EPI_F32, true>(pl, dev, tmA, tmB, tmB, tmOut,
                                                                     p, stream, rs)
               : launch_single_gemm<kTileN, kStages, EPI_BF16, true>(pl, dev, tmA, tmB, tmB, tmOut,
                                                                      p, stream, rs);
  return f32 ? launch_single_gemm<kTileN, kStages, EPI_F32>(pl, dev, tmA, tmB, tmB, tmOut, p, stream)
             : launch_single_gemm<kTileN, kStages, EPI_BF16>(pl, dev, tmA, tmB, tmB, tmOut, p,
                                                             stream);
}

// k-blocks of the weight the split-K producer issues back to back (see the
// kernel); GB3_SKINNY_ISSUE_GROUP overrides it for tuning.
int skinny_issue_group(int kb_per_split) {
  (void)kb_per_split;
  const int forced = env_int("GB3_SKINNY_ISSUE_GROUP", 0);
  if (forced > 0) return std::min(forced, kSkinnyStages);
  return 4;
}

SkinnyParams skinny_params(const gemm_plan& pl, const Problem& q) {
  SkinnyParams p;
  p.M = static_cast<int>(q.M);
  p.N = static_cast<int>(q.N);
  p.K = static_cast<int>(q.K);
  p.n_blocks = static_cast<int>(ceil_div(q.N, kSkinnyRows));
  p.k_blocks = static_cast<int>(ceil_div(q.K, kBK));
  p.splits = pl.split_k;
  p.kb_per_split = static_cast<int>(ceil_div(p.k_blocks, p.splits));
  p.batch = static_cast<int>(q.batch);
  p.num_units = static_cast<int>(pl.tiles);
  p.alpha = q.alpha;
  p.beta = q.beta;
  p.C = q.C;
  p.ldc = q.ldc;
  p.c_stride = q.batch > 1 ? q.sc : 0;
  p.out_kind = q.out_dtype;
  p.idesc = idesc_f32_acc(kSkinnyRows, kSkinnyNX, q.in_dtype == GEMM_IN_F16);
  p.ws = nullptr;
  p.counters = nullptr;
  p.issue_group = skinny_issue_group(p.kb_per_split);
  p.stall_after = -1;
  return p;
}

int run_skinny(const gemm_plan& pl, int dev, const Problem& q, cudaStream_t stream) {
  CUtensorMap tmW, tmX;
  int st;
  if ((st = operand_map(&tmW, q.B, q.in_dtype, q.K, q.N, q.batch, q.ldb, q.sb, kSkinnyRows)) !=
      GEMM_OK)
    return st;
  if ((st = operand_map(&tmX, q.A, q.in_dtype, q.K, q.M, q.batch, q.lda, q.sa, kSkinnyNX)) !=
      GEMM_OK)
    return st;
  SkinnyParams p = skinny_params(pl, q);
  auto kern = gemm_skinny_kernel<kSkinnyStages>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), CfgSkinny::kSmemBytes)) !=
        GEMM_OK)
      return st;
    if (p.splits > 1) {
      const size_t ws_bytes =
          static_cast<size_t>(q.batch) * p.splits * q.M * q.N * sizeof(float);
      const size_t counters = static_cast<size_t>(q.batch) * p.n_blocks * 4;
      if ((st = ensure_workspace(dev, ws_bytes, counters, stream)) != GEMM_OK) return st;
      p.ws = g_dev[dev].ws;
      p.counters = g_dev[dev].counters;
    }
  }
  return launch(kern, pl.grid, kThreads, CfgSkinny::kSmemBytes, stream, tmW, tmW, tmX, p);
}

// The decode-sized gate/up: the split-K kernel with Wg (as B) and Wu.
int run_skinny_gate_up(const gemm_plan& pl, int dev, const Problem& q, const void* Wu,
                       cudaStream_t stream) {
  CUtensorMap tmWg, tmWu, tmX;
  int st;
  if ((st = operand_map(&tmWg, q.B, GEMM_IN_BF16, q.K, q.N, 1, q.ldb, 0, kSkinnyRows)) != GEMM_OK)
    return st;
  if ((st = operand_map(&tmWu, Wu, GEMM_IN_BF16, q.K, q.N, 1, q.ldb, 0, kSkinnyRows)) != GEMM_OK)
    return st;
  if ((st = operand_map(&tmX, q.A, GEMM_IN_BF16, q.K, q.M, 1, q.lda, 0, kSkinnyNX)) != GEMM_OK)
    return st;
  SkinnyParams p = skinny_params(pl, q);
  auto kern = gemm_skinny_kernel<kSkinnyGateUpStages, true>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern),
                               CfgSkinnyGU::kSmemBytes)) != GEMM_OK)
      return st;
    if (p.splits > 1) {
      const size_t ws_bytes = static_cast<size_t>(p.splits) * 2 * q.M * q.N * sizeof(float);
      const size_t counters = static_cast<size_t>(p.n_blocks) * 4;
      if ((st = ensure_workspace(dev, ws_bytes, counters, stream)) != GEMM_OK) return st;
      p.ws = g_dev[dev].ws;
      p.counters = g_dev[dev].counters;
    }
  }
  return launch(kern, pl.grid, kThreads, CfgSkinnyGU::kSmemBytes, stream, tmWg, tmWu, tmX, p);
}

template <int NX>
int launch_smallm(const gemm_plan& pl, int dev, const CUtensorMap& tmW, const CUtensorMap& tmX,
                  const SmallMParams& p, cudaStream_t stream) {
  auto kern = gemm_smallm_kernel<NX>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const int st =
        ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), SmallMCfg<NX>::kSmemBytes);
    if (st != GEMM_OK) return st;
  }
  return launch(kern, pl.grid, kThreads, SmallMCfg<NX>::kSmemBytes, stream, tmW, tmX, p);
}

int run_smallm(const gemm_plan& pl, int dev, const Problem& q, cudaStream_t stream) {
  const int nx = pl.tile_n;
  CUtensorMap tmW, tmX;
  int st;
  if ((st = operand_map(&tmW, q.B, q.in_dtype, q.K, q.N, q.batch, q.ldb, q.sb, kSmallRows)) !=
      GEMM_OK)
    return st;
  if ((st = operand_map(&tmX, q.A, q.in_dtype, q.K, q.M, q.batch, q.lda, q.sa, nx)) != GEMM_OK)
    return st;
  SmallMParams p;
  p.M = static_cast<int>(q.M);
  p.N = static_cast<int>(q.N);
  p.K = static_cast<int>(q.K);
  p.n_blocks = static_cast<int>(ceil_div(q.N, kSmallRows));
  p.k_blocks = static_cast<int>(ceil_div(q.K, kBK));
  p.batch = static_cast<int>(q.batch);
  p.num_tiles = static_cast<int>(pl.tiles);
  smallm_divide(pl.tiles, p.k_blocks, pl.grid, &p);
  p.alpha = q.alpha;
  p.beta = q.beta;
  p.C = q.C;
  p.ldc = q.ldc;
  p.c_stride = q.batch > 1 ? q.sc : 0;
  p.out_kind = q.out_dtype;
  p.idesc = idesc_f32_acc(kSmallRows, nx, q.in_dtype == GEMM_IN_F16);
  p.ws = nullptr;
  p.counters = nullptr;
  if (p.max_pieces > 1) {
    std::lock_guard<std::mutex> lk(g_mu);
    const size_t ws_bytes = smallm_workspace_bytes(pl.grid, pl.tiles, q.M);
    const size_t counters = static_cast<size_t>(pl.tiles);
    if ((st = ensure_workspace(dev, ws_bytes, counters, stream)) != GEMM_OK) return st;
    p.ws = g_dev[dev].ws;
    p.counters = g_dev[dev].counters;
  }
  switch (nx) {
    case 16: return launch_smallm<16>(pl, dev, tmW, tmX, p, stream);
    case 32: return launch_smallm<32>(pl, dev, tmW, tmX, p, stream);
    case 64: return launch_smallm<64>(pl, dev, tmW, tmX, p, stream);
    case 128: return launch_smallm<128>(pl, dev, tmW, tmX, p, stream);
    default: return GEMM_ERR_UNSUPPORTED;
  }
}

// ----------------------------------------------------------------------------
// Attention
// ----------------------------------------------------------------------------
int validate_attention(int64_t heads, int64_t Nq, int64_t Nk, int64_t D, float scale,
                       const void* Q, int64_t ldq, int64_t sq, const void* K, int64_t ldk,
                       int64_t sk, const void* V, int64_t ldv, int64_t sv, const void* O,
                       int64_t ldo, int64_t so, int out_dtype) {
  if (heads < 0 || Nq < 0 || Nk < 0 || heads > kMaxDim || Nq > kMaxDim || Nk > kMaxDim)
    return GEMM_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GEMM_ERR_INVALID_ARG;
  if (out_dtype != GEMM_OUT_F32 && out_dtype != GEMM_OUT_BF16) return GEMM_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GEMM_ERR_INVALID_ARG;
  if (heads == 0 || Nq == 0) return GEMM_OK;
  if (Nk == 0) return GEMM_ERR_INVALID_ARG;   // a softmax over no keys is undefined
  if (heads * ceil_div(Nq, kAttnBR) > kMaxDim) return GEMM_ERR_INVALID_ARG;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return GEMM_ERR_INVALID_ARG;
  if (ldq < D || ldk < D || ldv < D || ldo < D) return GEMM_ERR_INVALID_ARG;
  if (heads > 1 && (sq < Nq * ldq || sk < Nk * ldk || sv < Nk * ldv || so < Nq * ldo))
    return GEMM_ERR_INVALID_ARG;
  const int64_t oe = out_elem_bytes(out_dtype);
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return GEMM_ERR_ALIGNMENT;
  if ((ldq * 2) % 16 != 0 || (ldk * 2) % 16 != 0 || (ldv * 2) % 16 != 0 || (ldo * oe) % 16 != 0)
    return GEMM_ERR_ALIGNMENT;
  if (heads > 1 && ((sq * 2) % 16 != 0 || (sk * 2) % 16 != 0 || (sv * 2) % 16 != 0 ||
                    (so * oe) % 16 != 0))
    return GEMM_ERR_ALIGNMENT;
  return GEMM_OK;
}

template <int D>
int launch_attention(int dev, int grid, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                     const CUtensorMap& tmV, const AttnParams& p, cudaStream_t stream) {
  auto kern = attention_kernel<D>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const int st =
        ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), AttnCfg<D>::kSmemBytes);
    if (st != GEMM_OK) return st;
  }
  return launch(kern, grid, kAttnThreads, AttnCfg<D>::kSmemBytes, stream, tmQ, tmK, tmV, p);
}

int run_problem(const Problem& q, void* stream_) {
  int st = validate_problem(q);
  if (st != GEMM_OK) return st;
  if (q.batch == 0 || q.M == 0 || q.N == 0) return GEMM_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  int sms, slots;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
    sms = g_dev[dev].sms;
    slots = query_pair_slots(dev);
  }
  gemm_plan pl;
  plan_gemm(q.batch, q.M, q.N, q.K, sms, &pl, slots, true, q.stats());
  switch (pl.kernel) {
    case K_SCALE:
      if (q.stats()) {
        const int64_t warps = q.batch * q.M;
        const int grid = static_cast<int>(std::min<int64_t>(ceil_div(warps, 8), 4 * sms));
        st = launch(row_stats_k0_kernel, grid, 256, 0, stream, static_cast<const void*>(q.C),
                    static_cast<long long>(q.ldc), static_cast<long long>(q.batch > 1 ? q.sc : 0),
                    static_cast<int>(q.batch), static_cast<int>(q.M), static_cast<int>(q.N),
                    q.beta, q.out_dtype, q.row_sum, q.row_max, q.row_min);
        if (st != GEMM_OK) return st;
      }
      return run_scale(pl, q.C, q.ldc, q.batch > 1 ? q.sc : 0, q.batch, q.M, q.N, q.beta,
                       q.out_dtype, stream);
    case K_PAIR:
      return run_pair(pl, dev, slots, q, stream);
    case K_SKINNY:
      return run_skinny(pl, dev, q, stream);
    case K_SMALL_M:
      return run_smallm(pl, dev, q, stream);
    default:
      return run_single(pl, dev, q, stream);
  }
}

}  // namespace

// ============================================================================
// C ABI
// ============================================================================
extern "C" {

const char* gemm_status_string(int status) {
  switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_ALIGNMENT: return "pointer or row pitch not 16-byte aligned";
    case GEMM_ERR_UNSUPPORTED: return "unsupported device (needs compute capability 10.3)";
    case GEMM_ERR_CUDA: return "CUDA runtime or driver call failed";
    case GEMM_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    default: return "unknown status";
  }
}

int gemm_batched_plan(int64_t batch, int64_t M, int64_t N, int64_t K, int in_dtype,
                      int out_dtype, int num_sms, gemm_plan* plan) {
  if (plan == nullptr) return GEMM_ERR_INVALID_ARG;
  if (bad_dims(batch, M, N, K)) return GEMM_ERR_INVALID_ARG;
  if (in_dtype != GEMM_IN_BF16 && in_dtype != GEMM_IN_F16) return GEMM_ERR_INVALID_ARG;
  if (out_dtype != GEMM_OUT_F32 && out_dtype != GEMM_OUT_BF16 && out_dtype != GEMM_OUT_F16)
    return GEMM_ERR_INVALID_ARG;
  int slots = 0;
  if (num_sms <= 0) {
    int dev;
    int st = current_device(&dev);
    if (st != GEMM_OK) return st;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
    num_sms = g_dev[dev].sms;
    slots = query_pair_slots(dev);
  }
  return plan_gemm(batch, M, N, K, num_sms, plan, slots);
}

int gemm_bf16_plan(int64_t M, int64_t N, int64_t K, int out_dtype, int num_sms,
                   gemm_plan* plan) {
  return gemm_batched_plan(1, M, N, K, GEMM_IN_BF16, out_dtype, num_sms, plan);
}

int gemm_gate_up_plan(int64_t M, int64_t N, int64_t K, int num_sms, gemm_plan* plan) {
  if (plan == nullptr) return GEMM_ERR_INVALID_ARG;
  if (bad_dims(1, M, N, K)) return GEMM_ERR_INVALID_ARG;
  int slots = 0;
  if (num_sms <= 0) {
    int dev;
    int st = current_device(&dev);
    if (st != GEMM_OK) return st;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
    num_sms = g_dev[dev].sms;
    slots = query_pair_slots(dev);
  }
  return plan_gate_up(M, N, K, num_sms, plan, slots);
}

int gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
              const void* B, int64_t ldb, float beta, void* C, int64_t ldc, int out_dtype,
              void* stream) {
  const Problem q{1, M, N, K, alpha, beta, A, lda, 0, B, ldb, 0, C, ldc, 0, GEMM_IN_BF16,
                  out_dtype};
  return run_problem(q, stream);
}

int gemm_batched(int64_t batch, int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                 int64_t lda, int64_t stride_a, const void* B, int64_t ldb, int64_t stride_b,
                 float beta, void* C, int64_t ldc, int64_t stride_c, int in_dtype, int out_dtype,
                 void* stream) {
  const Problem q{batch, M,        N,   K,   alpha, beta,     A,        lda,      stride_a,
                  B,     ldb,      stride_b, C, ldc, stride_c, in_dtype, out_dtype};
  return run_problem(q, stream);
}

int gemm_row_stats(int64_t batch, int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                   int64_t lda, int64_t stride_a, const void* B, int64_t ldb, int64_t stride_b,
                   float beta, void* C, int64_t ldc, int64_t stride_c, int in_dtype,
                   int out_dtype, float* row_sum, float* row_max, float* row_min,
                   void* stream) {
  Problem q{batch, M,        N,   K,   alpha, beta,     A,        lda,      stride_a,
            B,     ldb,      stride_b, C, ldc, stride_c, in_dtype, out_dtype};
  q.row_sum = row_sum;
  q.row_max = row_max;
  q.row_min = row_min;
  for (const float* r : {row_sum, row_max, row_min})
    if (reinterpret_cast<uintptr_t>(r) % alignof(float) != 0) return GEMM_ERR_ALIGNMENT;
  const int st = validate_problem(q);
  if (st != GEMM_OK || !q.stats() || batch == 0 || M == 0 || N > 0) return run_problem(q, stream);
  // N == 0: each row's reductions are over no values: sum 0, maximum -inf,
  // minimum +inf (C is not touched).
  int dev, sms;
  int s2 = current_device(&dev);
  if (s2 != GEMM_OK) return s2;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((s2 = probe_device(dev)) != GEMM_OK) return s2;
    sms = g_dev[dev].sms;
  }
  const int grid = static_cast<int>(std::min<int64_t>(ceil_div(batch * M, 8), 4 * sms));
  return launch(row_stats_k0_kernel, grid, 256, 0, static_cast<cudaStream_t>(stream),
                static_cast<const void*>(nullptr), 0LL, 0LL, static_cast<int>(batch),
                static_cast<int>(M), 0, 0.0f, out_dtype, row_sum, row_max, row_min);
}

int gemm_row_stats_plan(int64_t batch, int64_t M, int64_t N, int64_t K, int in_dtype,
                        int out_dtype, int num_sms, gemm_plan* plan) {
  if (plan == nullptr) return GEMM_ERR_INVALID_ARG;
  if (bad_dims(batch, M, N, K)) return GEMM_ERR_INVALID_ARG;
  if (in_dtype != GEMM_IN_BF16 && in_dtype != GEMM_IN_F16) return GEMM_ERR_INVALID_ARG;
  if (out_dtype != GEMM_OUT_F32 && out_dtype != GEMM_OUT_BF16 && out_dtype != GEMM_OUT_F16)
    return GEMM_ERR_INVALID_ARG;
  int slots = 0;
  if (num_sms <= 0) {
    int dev;
    int st = current_device(&dev);
    if (st != GEMM_OK) return st;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
    num_sms = g_dev[dev].sms;
    slots = query_pair_slots(dev);
  }
  const int st = plan_gemm(batch, M, N, K, num_sms, plan, slots, true, true);
  if (st == GEMM_OK && batch > 0 && M > 0 && N == 0) {
    plan->kernel = K_SCALE;   // the empty-row reductions alone
    plan->launches = 1;
  }
  return st;
}

int gemm_gate_up_silu(int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx,
                      const void* Wg, const void* Wu, int64_t ldw, void* Y, int64_t ldy,
                      void* stream_) {
  int st = validate_gate_up(M, N, K, X, ldx, Wg, Wu, ldw, Y, ldy);
  if (st != GEMM_OK) return st;
  if (M == 0 || N == 0) return GEMM_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  int sms, slots;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
    sms = g_dev[dev].sms;
    slots = query_pair_slots(dev);
  }
  gemm_plan pl;
  plan_gate_up(M, N, K, sms, &pl, slots);
  if (pl.kernel == K_SCALE) return run_scale(pl, Y, ldy, 0, 1, M, N, 0.0f, GEMM_OUT_BF16, stream);
  // Wg and Wu play the part of B; the output is BF16.
  const Problem q{1, M, N, K, 1.0f, 0.0f, X, ldx, 0, Wg, ldw, 0, Y, ldy, 0, GEMM_IN_BF16,
                  GEMM_OUT_BF16};
  if (pl.kernel == K_SKINNY_GATE_UP) return run_skinny_gate_up(pl, dev, q, Wu, stream);
  const bool pair = pl.kernel == K_PAIR_GATE_UP;
  const int out_cols = pair ? CfgPairGU::kOutCols : CfgGU::kOutCols;
  CUtensorMap tmX, tmWg, tmWu, tmY;
  if ((st = operand_map(&tmX, X, GEMM_IN_BF16, K, M, 1, ldx, 0, pair ? 128 : kBM)) != GEMM_OK)
    return st;
  if ((st = operand_map(&tmWg, Wg, GEMM_IN_BF16, K, N, 1, ldw, 0, out_cols)) != GEMM_OK) return st;
  if ((st = operand_map(&tmWu, Wu, GEMM_IN_BF16, K, N, 1, ldw, 0, out_cols)) != GEMM_OK) return st;
  if ((st = output_map(&tmY, Y, 1, M, N, ldy, 0, GEMM_OUT_BF16, out_cols)) != GEMM_OK) return st;
  if (pair) {
    TileParams p = tile_params(q, kPairBM, out_cols, idesc_f32_acc(kPairBM, 256, false));
    pair_units(dev, &pl, q, out_cols, &p, stream, true, slots);
    return launch_pair_gemm<256, EPI_GATE_UP>(pl, dev, tmX, tmWg, tmWu, tmY, p, stream);
  }
  const TileParams p = tile_params(q, kBM, out_cols, idesc_f32_acc(kBM, 256, false));
  return launch_single_gemm<256, kGateUpStages, EPI_GATE_UP>(pl, dev, tmX, tmWg, tmWu, tmY, p,
                                                             stream);
}

int gemm_rmsnorm_gate_up_silu(int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx,
                              const float* G, float eps, const void* Wg, const void* Wu,
                              int64_t ldw, void* Xn, int64_t ldxn, void* Y, int64_t ldy,
                              void* stream_) {
  // Every argument is checked before anything is enqueued.
  int st = validate_gate_up(M, N, K, Xn, ldxn, Wg, Wu, ldw, Y, ldy);
  if (st != GEMM_OK) return st;
  if ((st = rms_norm_check(M, K, X, ldx, GEMM_OUT_BF16, G, eps, Xn, ldxn, GEMM_OUT_BF16)) !=
      GEMM_OK)
    return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (M > 0 && N > 0 && K > 0) {
    int dev;
    if ((st = current_device(&dev)) != GEMM_OK) return st;
    int sms, slots;
    unsigned int* sync = nullptr;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if ((st = probe_device(dev)) != GEMM_OK) return st;
      sms = g_dev[dev].sms;
      slots = query_pair_slots(dev);
      if ((st = grid_sync_counters(dev, &sync)) != GEMM_OK) return st;
    }
    gemm_plan pl;
    plan_gate_up(M, N, K, sms, &pl, slots);
    // GB3_RMSNORM_SINGLE_LAUNCH = 1: one launch, the pair gate/up kernel
    // normalising its activation first.  It copies the gains and whole rows
    // of X into the pipeline's shared memory: rows of whole 16-byte vectors,
    // three chunks of at least one row beside the gains.  Not the default:
    // measured on GB300 (4096 x 14336 x 4096, same box) at 512.7 us against
    // 508.5 us for the two launches and 490.4 us for the plain gate/up.
    // Both are bound by writing Xn (32 MB): from every SM at once, with
    // nothing else to overlap, it runs at about 3 TB/s in the single launch,
    // while the standalone normalisation overlaps it with its reads.
    const bool rows_fit =
        (K * 2) % 16 == 0 && K * (4 + 3 * 2) <= PairCfg<256, kPairStages, EPI_GATE_UP>::kBarOffset &&
        env_int("GB3_RMSNORM_SINGLE_LAUNCH", 0) == 1;
    const int norm = rows_fit ? fused_norm_geometry(K) : 0;
    if (pl.kernel == K_PAIR_GATE_UP && norm != 0) {
      // One launch: the pair gate/up kernel normalises X into Xn first.
      const Problem q{1, M, N, K, 1.0f, 0.0f, Xn, ldxn, 0, Wg, ldw, 0, Y, ldy, 0, GEMM_IN_BF16,
                      GEMM_OUT_BF16};
      const int out_cols = CfgPairGU::kOutCols;
      CUtensorMap tmX, tmWg, tmWu, tmY;
      if ((st = operand_map(&tmX, Xn, GEMM_IN_BF16, K, M, 1, ldxn, 0, 128)) != GEMM_OK) return st;
      if ((st = operand_map(&tmWg, Wg, GEMM_IN_BF16, K, N, 1, ldw, 0, out_cols)) != GEMM_OK)
        return st;
      if ((st = operand_map(&tmWu, Wu, GEMM_IN_BF16, K, N, 1, ldw, 0, out_cols)) != GEMM_OK)
        return st;
      if ((st = output_map(&tmY, Y, 1, M, N, ldy, 0, GEMM_OUT_BF16, out_cols)) != GEMM_OK)
        return st;
      TileParams p = tile_params(q, kPairBM, out_cols, idesc_f32_acc(kPairBM, 256, false));
      pair_units(dev, &pl, q, out_cols, &p, stream, true, slots);
      const NormParams nrm{X,  ldx, G, eps, Xn, ldxn, static_cast<int>(M), static_cast<int>(K),
                           sync};
      return norm == 2 ? launch_pair_gemm<256, EPI_GATE_UP, false, false, 2>(
                             pl, dev, tmX, tmWg, tmWu, tmY, p, stream, RowStatsParams{}, nrm)
                       : launch_pair_gemm<256, EPI_GATE_UP, false, false, 1>(
                             pl, dev, tmX, tmWg, tmWu, tmY, p, stream, RowStatsParams{}, nrm);
    }
  }
  if ((st = rms_norm_run(M, K, X, ldx, GEMM_OUT_BF16, G, eps, Xn, ldxn, GEMM_OUT_BF16, stream)) !=
      GEMM_OK)
    return st;
  return gemm_gate_up_silu(M, N, K, Xn, ldxn, Wg, Wu, ldw, Y, ldy, stream_);
}

int gemm_attention(int64_t heads, int64_t Nq, int64_t Nk, int64_t D, float scale, const void* Q,
                   int64_t ldq, int64_t stride_q, const void* K, int64_t ldk, int64_t stride_k,
                   const void* V, int64_t ldv, int64_t stride_v, void* O, int64_t ldo,
                   int64_t stride_o, int out_dtype, void* stream_) {
  int st = validate_attention(heads, Nq, Nk, D, scale, Q, ldq, stride_q, K, ldk, stride_k, V, ldv,
                              stride_v, O, ldo, stride_o, out_dtype);
  if (st != GEMM_OK || heads == 0 || Nq == 0) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
  }
  CUtensorMap tmQ, tmK, tmV;
  const uint64_t pq = static_cast<uint64_t>(ldq) * 2, pk = static_cast<uint64_t>(ldk) * 2,
                 pv = static_cast<uint64_t>(ldv) * 2;
  if ((st = tensor_map_3d(&tmQ, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, Nq, heads, pq,
                          heads > 1 ? static_cast<uint64_t>(stride_q) * 2 : pq * Nq, 64,
                          kAttnBR)) != GEMM_OK)
    return st;
  if ((st = tensor_map_3d(&tmK, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, Nk, heads, pk,
                          heads > 1 ? static_cast<uint64_t>(stride_k) * 2 : pk * Nk, 64,
                          kAttnBC)) != GEMM_OK)
    return st;
  if ((st = tensor_map_3d(&tmV, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, Nk, heads, pv,
                          heads > 1 ? static_cast<uint64_t>(stride_v) * 2 : pv * Nk, 64,
                          kAttnBC)) != GEMM_OK)
    return st;
  AttnParams p;
  p.heads = static_cast<int>(heads);
  p.Nq = static_cast<int>(Nq);
  p.Nk = static_cast<int>(Nk);
  p.q_blocks = static_cast<int>(ceil_div(Nq, kAttnBR));
  p.k_blocks = static_cast<int>(ceil_div(Nk, kAttnBC));
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.O = O;
  p.ldo = ldo;
  p.o_stride = heads > 1 ? stride_o : 0;
  p.out_kind = out_dtype;
  p.idesc_s = idesc_f32_acc(kAttnBR, kAttnBC, false);
  p.idesc_o = idesc_f32_acc(kAttnBR, static_cast<int>(D), false) | (1u << 16);  // B MN-major
  const int grid = static_cast<int>(heads * p.q_blocks);
  return D == 64 ? launch_attention<64>(dev, grid, tmQ, tmK, tmV, p, stream)
                 : launch_attention<128>(dev, grid, tmQ, tmK, tmV, p, stream);
}

int gemm_get_device_status(void* stream, int* site) {
  int dev;
  int st = current_device(&dev);
  if (st != GEMM_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  int h[4] = {0, 0, 0, 0};
  const int zero[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(h, g_gemm_status, sizeof(h)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_gemm_status, zero, sizeof(zero)) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (site != nullptr) *site = h[1];
  if (h[0] != GEMM_OK) {
    // A kernel gave up mid-way: arrival counters of split work may be left
    // non-zero; clear them so that later calls start from a clean state.
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& d = g_dev[dev];
    if (d.counters != nullptr &&
        cudaMemset(d.counters, 0, d.counter_count * sizeof(int)) != cudaSuccess)
      cudaGetLastError();
    if (d.grid_sync != nullptr && cudaMemset(d.grid_sync, 0, 2 * sizeof(unsigned int)) != cudaSuccess)
      cudaGetLastError();
    if (d.stats_counters != nullptr &&
        cudaMemset(d.stats_counters, 0, d.stats_counter_count * sizeof(int)) != cudaSuccess)
      cudaGetLastError();
  }
  return h[0];
}

int gemm_selftest_wait_timeout(int64_t limit_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000) return GEMM_ERR_INVALID_ARG;
  int dev;
  int st = current_device(&dev);
  if (st != GEMM_OK) return st;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
  }
  return launch(wait_timeout_probe_kernel, 1, 32, 0, static_cast<cudaStream_t>(stream),
                static_cast<unsigned long long>(limit_ns));
}

int gemm_selftest_pipeline_timeout(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                   const void* B, int64_t ldb, void* C, int64_t ldc,
                                   int stall_after, void* stream_) {
  const Problem q{1, M, N, K, 1.0f, 0.0f, A, lda, 0, B, ldb, 0, C, ldc, 0, GEMM_IN_BF16,
                  GEMM_OUT_BF16};
  int st = validate_problem(q);
  if (st != GEMM_OK) return st;
  if (M < 1 || M > kSkinnyMaxM || N < 1 || K < 1 || stall_after < 0 ||
      stall_after >= ceil_div(K, kBK))
    return GEMM_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  auto kern = gemm_skinny_kernel<kSkinnyStages>;
  int sms;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
    sms = g_dev[dev].sms;
    if ((st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), CfgSkinny::kSmemBytes)) !=
        GEMM_OK)
      return st;
  }
  // Whole K per unit (no split, so no workspace or arrival counter is
  // touched), one unit per CTA at most; every unit stops inside its K range.
  gemm_plan pl;
  std::memset(&pl, 0, sizeof(pl));
  pl.split_k = 1;
  pl.tiles = ceil_div(N, kSkinnyRows);
  pl.grid = static_cast<int>(std::min<int64_t>(pl.tiles, sms));
  SkinnyParams p = skinny_params(pl, q);
  p.stall_after = stall_after;
  CUtensorMap tmW, tmX;
  if ((st = operand_map(&tmW, B, GEMM_IN_BF16, K, N, 1, ldb, 0, kSkinnyRows)) != GEMM_OK)
    return st;
  if ((st = operand_map(&tmX, A, GEMM_IN_BF16, K, M, 1, lda, 0, kSkinnyNX)) != GEMM_OK)
    return st;
  return launch(kern, pl.grid, kThreads, CfgSkinny::kSmemBytes, stream, tmW, tmW, tmX, p);
}

uint64_t gemm_layout_smem_descriptor(uint32_t smem_address, uint32_t mn_chunk_bytes) {
  return mn_chunk_bytes == 0 ? smem_desc_sw128(smem_address)
                             : smem_desc_mn_sw128(smem_address, mn_chunk_bytes);
}

uint32_t gemm_layout_instr_descriptor(int M, int N, int in_dtype) {
  return idesc_f32_acc(M, N, in_dtype == GEMM_IN_F16);
}

uint32_t gemm_layout_swizzle128_offset(int row, int chunk) {
  return staging_offset<true>(row, static_cast<uint32_t>(chunk));
}

uint32_t gemm_layout_tmem_address(uint32_t base, int lane, int column) {
  return tmem_addr(base, static_cast<uint32_t>(lane), static_cast<uint32_t>(column));
}

int gemm_prepare(int64_t max_N, void* stream) {
  if (max_N < 0 || max_N > kMaxDim) return GEMM_ERR_INVALID_ARG;
  int dev;
  int st = current_device(&dev);
  if (st != GEMM_OK) return st;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((st = probe_device(dev)) != GEMM_OK) return st;
  // M <= 16: the largest split the planner can choose is 32.
  const int64_t nb = ceil_div(std::max<int64_t>(max_N, 1), kSkinnyRows);
  const size_t skinny_bytes = static_cast<size_t>(32) * kSkinnyMaxM * max_N * sizeof(float);
  // 16 < M <= 128: the small-M kernel, which the planner picks only while its
  // tiles number at most the SMs, on at most one CTA per SM.
  const int64_t tiles =
      std::min<int64_t>(ceil_div(std::max<int64_t>(max_N, 1), kSmallRows), g_dev[dev].sms);
  const size_t small_bytes = smallm_workspace_bytes(g_dev[dev].sms, tiles, kSmallMMaxM);
  return ensure_workspace(dev, std::max(skinny_bytes, small_bytes),
                          static_cast<size_t>(std::max(nb * 4, tiles)),
                          static_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ============================================================================
// Decode-shaped GEMM without any allocation
// ============================================================================
// Some callers cannot allocate device memory at the moment they call: code
// running under a custom allocator or memory pool that forbids stray
// cudaMalloc, code inside a region where allocation would synchronize the
// device, or callers whose memory budget is fixed up front.  For them the
// split-K partial sums of the M <= 16 path live in one fixed array in the
// library's device image instead of an allocated workspace.  The array is
// created when the library is loaded onto a GPU and held until the process
// exits, on every GPU that loads the library.
namespace {

// 8 MiB: arrival counters first (rounded up to 256 bytes), FP32 partial sums
// after them.  Enough for split * M * N * 4 bytes up to about 8 MB, e.g. two
// splits of a 16 x 28672 output (3.7 MB).
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
unsigned char* g_noalloc_base[kMaxDevices];  // device address of the array, per device
// Whether the split-K kernel's shared-memory attribute was set by this entry
// point (guarded by g_mu, as ensure_smem_attr is; a fixed array rather than
// ensure_smem_attr's list, whose growth would allocate host memory).
bool g_noalloc_smem_set[kMaxDevices];

}  // namespace

extern "C" int gemm_bf16_skinny_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                        const void* A, int64_t lda, const void* B, int64_t ldb,
                                        float beta, void* C, int64_t ldc, int out_dtype,
                                        void* stream_) {
  const Problem q{1, M, N, K, alpha, beta, A, lda, 0, B, ldb, 0, C, ldc, 0, GEMM_IN_BF16,
                  out_dtype};
  int st = validate_problem(q);
  if (st != GEMM_OK) return st;
  if (M == 0 || N == 0) return GEMM_OK;
  if (M > kSkinnyMaxM) return GEMM_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  auto kern = gemm_skinny_kernel<kSkinnyStages>;
  int sms;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
    sms = g_dev[dev].sms;
    if (!g_noalloc_smem_set[dev]) {
      if (cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               CfgSkinny::kSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
      }
      g_noalloc_smem_set[dev] = true;
    }
  }
  gemm_plan pl;
  if (K == 0) {
    plan_gemm(1, M, N, K, sms, &pl);   // the scaling of C alone
    return run_scale(pl, C, ldc, 0, 1, M, N, beta, out_dtype, stream);
  }
  // Always the split-K kernel, with its own plan and shared-memory size.
  std::memset(&pl, 0, sizeof(pl));
  plan_skinny(1, M, N, K, sms, &pl);

  SkinnyParams p = skinny_params(pl, q);
  const size_t counter_bytes =
      (static_cast<size_t>(p.n_blocks) * 4 * sizeof(int) + 255) & ~static_cast<size_t>(255);
  const size_t partial_bytes =
      p.splits > 1 ? static_cast<size_t>(p.splits) * M * N * sizeof(float) : 0;
  if (counter_bytes + partial_bytes > kNoAllocScratchBytes) return GEMM_ERR_INVALID_ARG;

  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_base[dev] == nullptr) {
      // One-time set-up on this device (the device is current): the host-side
      // name of the array is not a device address; ask the runtime for it.
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
      }
      g_noalloc_base[dev] = static_cast<unsigned char*>(addr);
    }
    base = g_noalloc_base[dev];
  }
  p.counters = reinterpret_cast<int*>(base);
  p.ws = reinterpret_cast<float*>(base + counter_bytes);

  // Descriptors encoded straight into the parameter block (no cache, no allocation).
  CUtensorMap tmW, tmX;
  if ((st = encode_map_3d(&tmW, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, 1, ldb * 2,
                          static_cast<uint64_t>(ldb) * 2 * N, kBK, kSkinnyRows,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_OK)
    return st;
  if ((st = encode_map_3d(&tmX, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, 1, lda * 2,
                          static_cast<uint64_t>(lda) * 2 * M, kBK, kSkinnyNX,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != GEMM_OK)
    return st;
  // The arrival counters must start at zero; the array keeps whatever the
  // previous call left, so clear them on the stream first.
  if (p.splits > 1 && cudaMemsetAsync(p.counters, 0, counter_bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return launch(kern, pl.grid, kThreads, CfgSkinny::kSmemBytes, stream, tmW, tmW, tmX, p);
}
