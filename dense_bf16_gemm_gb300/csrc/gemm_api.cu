// gemm_api.cu -- host side of the library: argument validation, tile
// planning, TMA descriptor encoding (cuTensorMapEncodeTiled, 128-byte
// swizzle) with a descriptor cache, kernel launch and the C ABI declared in
// include/gemm_bf16.h.
//
// Descriptor contract ("TMA and Hopper WGMMA", section "The same storage
// contract on both sides"): a descriptor names the element type, the tile
// (box) shape, the inner axis and a 128-byte swizzle row; the box's inner
// extent is one swizzle row (64 BF16 or 32 FP32) and its outer extent is at
// most 256.  Section "The same storage contract on both sides" also states
// that a descriptor stays valid while values change and must be re-encoded
// for a new address or new dimensions: the cache key is therefore (address,
// element type, dimensions, row pitch, box).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/gemm_bf16.h"
#include "gemm_kernels.cuh"
#include "gemm_kernels_pair.cuh"
#include "gemm_skinny.cuh"

namespace {

using namespace gb3;

// ----------------------------------------------------------------------------
// Kernel configurations
// ----------------------------------------------------------------------------
constexpr int kTileN = 256;        // output columns per tile of the tiled GEMM
constexpr int kStages = 4;         // ring depth of the tiled GEMM (48 KB per stage)
constexpr int kGateUpStages = 4;   // gate/up: 16 KB X + 16 KB Wg + 16 KB Wu per stage
constexpr int kSkinnyStages = 12;  // 18 KB per stage
constexpr int kSkinnyMaxM = 16;
constexpr int kGroupM = 16;

constexpr int kPairStages = 6;     // CTA-pair kernels: 16 KB A + BN*64 B per stage and CTA
constexpr int kPairMinM = 129;     // pair tiles (256 rows) from this M on

using CfgF32 = GemmCfg<kTileN, kStages, EPI_F32>;
using CfgBF16 = GemmCfg<kTileN, kStages, EPI_BF16>;
using CfgGU = GemmCfg<256, kGateUpStages, EPI_GATE_UP>;
using CfgSkinny = SkinnyCfg<kSkinnyStages>;
using CfgPairGU = PairCfg<256, kPairStages, EPI_GATE_UP>;

// Tile widths compiled for the CTA-pair GEMM.
constexpr int kPairWidths[] = {256, 224};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

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
  K_PAIR_GATE_UP = 6
};

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

int pair_stage_bytes(int bn) { return 128 * kBK * 2 + (bn / 2) * kBK * 2; }

// Split of K for the skinny path: minimise the k-blocks of the busiest CTA,
// ceil(units / grid) * ceil(k_blocks / S), with a small charge per extra split
// for the partial-sum traffic.
void choose_split(int64_t n_blocks, int64_t k_blocks, int sms, int* splits, int* kb_per) {
  int best_s = 1;
  double best = 1e300;
  for (int s = 1; s <= 32; ++s) {
    const int64_t kbp = ceil_div(k_blocks, s);
    if (s > 1 && kbp < 4) break;
    const int64_t real_s = ceil_div(k_blocks, kbp);  // splits that get work
    if (real_s != s) continue;
    const int64_t units = n_blocks * s;
    const double cost = static_cast<double>(ceil_div(units, sms)) * static_cast<double>(kbp) +
                        0.5 * static_cast<double>(s - 1);
    if (cost < best) {
      best = cost;
      best_s = s;
    }
  }
  *splits = best_s;
  *kb_per = static_cast<int>(ceil_div(k_blocks, best_s));
}

constexpr int kMinPieceKb = 24;       // shortest K piece of a split tail tile (1536 of K)
constexpr int kMaxTailSplit = 2;      // more pieces cost more partial-sum traffic than they save
constexpr double kSplitCharge = 0.1;  // partial-sum traffic of a split tail, in waves
constexpr int kWidthCostOffset = 320;  // per-wave time model of a pair tile: width + 320

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : fallback;
}

struct PairChoice {
  int bn = 256;
  int64_t tiles = 0;
  int64_t full = 0;      // tiles run whole
  int split = 1;         // K pieces per tail tile
  int kb_per_piece = 0;
};

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
  int64_t s = std::min<int64_t>({static_cast<int64_t>(kMaxTailSplit), slots / tail,
                                  k_blocks / kMinPieceKb});
  if (s < 2) return;
  const int64_t kbp = ceil_div(k_blocks, s);
  c->full = tiles - tail;
  c->kb_per_piece = static_cast<int>(kbp);
  c->split = static_cast<int>(ceil_div(k_blocks, kbp));
}

// Tile width of the CTA-pair GEMM and its tail split: the fewest waves of
// pair tiles (a split tail wave counts 1/split of a wave plus a charge for its
// partial sums) weighted by the time a wave of that width takes.
PairChoice choose_pair(int64_t M, int64_t N, int64_t K, int slots, bool allow_split) {
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
    PairChoice c;
    c.bn = bn;
    plan_tail(mb * ceil_div(N, bn), kb, slots, allow_split, &c);
    double waves = static_cast<double>(c.full / slots);
    const int64_t left = c.tiles - (c.full / slots) * slots;
    if (left > 0) waves += c.split > 1 ? 1.0 / c.split + kSplitCharge : 1.0;
    // Measured on GB300 (8192^3): a wave of 256-wide pair tiles takes 1.057x
    // the time of 224-wide ones for 1.143x the work, i.e. time ~ width + 320.
    const double cost = waves * static_cast<double>(bn + kWidthCostOffset);
    if (cost < best_cost) {
      best_cost = cost;
      best = c;
    }
  }
  return best;
}

int64_t pair_workspace_bytes(const PairChoice& c) {
  if (c.split <= 1) return 0;
  return (c.tiles - c.full) * c.split * static_cast<int64_t>(kPairBM) * c.bn * 4;
}

// pair_slots: CTA pairs that fit on the device at once (0: assume sms / 2,
// negative: pair kernels unavailable).
int plan_gemm(int64_t M, int64_t N, int64_t K, int sms, gemm_plan* pl, int pair_slots = 0,
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
  pl->tile_k = kBK;
  if (M <= kSkinnyMaxM) {
    const int64_t nb = ceil_div(N, kSkinnyRows), kb = ceil_div(K, kBK);
    int s, kbp;
    choose_split(nb, kb, sms, &s, &kbp);
    pl->kernel = K_SKINNY;
    pl->tile_m = kSkinnyRows;
    pl->tile_n = kSkinnyNX;
    pl->stages = kSkinnyStages;
    pl->split_k = s;
    pl->tiles = nb * s;
    pl->grid = static_cast<int>(std::min<int64_t>(pl->tiles, sms));
    pl->smem_bytes = CfgSkinny::kSmemBytes;
    pl->launches = 1;
    pl->stage_tx_bytes = CfgSkinny::kStageBytes;
    return GEMM_OK;
  }
  if (M >= kPairMinM && pair_slots >= 0) {
    const int slots = pair_slots > 0 ? pair_slots : std::max(1, sms / 2);
    const PairChoice c = choose_pair(M, N, K, slots, allow_split);
    const int64_t units = c.full + (c.tiles - c.full) * c.split;
    pl->kernel = K_PAIR;
    pl->tile_m = kPairBM;
    pl->tile_n = c.bn;
    pl->stages = kPairStages;
    pl->split_k = c.split;
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
  pl->tiles = ceil_div(M, kBM) * ceil_div(N, kTileN);
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
    PairChoice c;
    c.bn = 256;
    plan_tail(ceil_div(M, kPairBM) * ceil_div(N, CfgPairGU::kOutCols), ceil_div(K, kBK), slots,
              allow_split, &c);
    const int64_t units = c.full + (c.tiles - c.full) * c.split;
    pl->kernel = K_PAIR_GATE_UP;
    pl->tile_m = kPairBM;
    pl->tile_n = CfgPairGU::kOutCols;
    pl->tile_k = kBK;
    pl->stages = kPairStages;
    pl->split_k = c.split;
    pl->tiles = units;
    pl->grid = 2 * static_cast<int>(std::min<int64_t>(units, slots));
    pl->smem_bytes = CfgPairGU::kSmemBytes;
    pl->launches = 1;
    pl->stage_tx_bytes = 2 * CfgPairGU::kStageBytes;
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
constexpr int64_t kMaxDim = 0x7FFFFFFF;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate_gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                  int64_t ldb, float beta, const void* C, int64_t ldc, int out_dtype) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return GEMM_ERR_INVALID_ARG;
  if (out_dtype != GEMM_OUT_F32 && out_dtype != GEMM_OUT_BF16) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  const int64_t esize = out_dtype == GEMM_OUT_F32 ? 4 : 2;
  if (C == nullptr || ldc < N) return GEMM_ERR_INVALID_ARG;
  if (K > 0) {
    if (A == nullptr || B == nullptr || lda < K || ldb < K) return GEMM_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || (lda * 2) % 16 != 0 || (ldb * 2) % 16 != 0)
      return GEMM_ERR_ALIGNMENT;
  }
  if (!aligned16(C) || (ldc * esize) % 16 != 0) return GEMM_ERR_ALIGNMENT;
  (void)beta;
  return GEMM_OK;
}

int validate_gate_up(int64_t M, int64_t N, int64_t K, const void* X, int64_t ldx, const void* Wg,
                     const void* Wu, int64_t ldw, const void* Y, int64_t ldy) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return GEMM_ERR_INVALID_ARG;
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
  // kernels whose shared-memory limit has been raised on this device
  std::vector<const void*> configured;
  // CTA pairs that fit on the device at once (0: not queried yet, -1: none)
  int pair_slots = 0;
  // split-K workspace of the skinny path
  float* ws = nullptr;
  size_t ws_bytes = 0;
  int* counters = nullptr;
  size_t counter_count = 0;
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

int device_sms(int* sms) {
  int dev;
  int st = current_device(&dev);
  if (st != GEMM_OK) return st;
  std::lock_guard<std::mutex> lk(g_mu);
  st = probe_device(dev);
  if (st != GEMM_OK) return st;
  *sms = g_dev[dev].sms;
  return GEMM_OK;
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
  uint64_t inner, outer, pitch;
  uint32_t box_inner, box_outer;
  int swizzle;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && dtype == o.dtype && inner == o.inner && outer == o.outer &&
           pitch == o.pitch && box_inner == o.box_inner && box_outer == o.box_outer &&
           swizzle == o.swizzle;
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

// 2-D map over a row-major matrix of `outer` rows of `inner` elements with a
// row pitch of `pitch` bytes; box of box_inner x box_outer elements, 128-byte
// swizzle, out-of-bounds elements read as zero.
int tensor_map_2d(CUtensorMap* out, const void* ptr, CUtensorMapDataType dtype, uint64_t inner,
                  uint64_t outer, uint64_t pitch, uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const MapKey key{ptr, static_cast<int>(dtype), inner, outer, pitch, box_inner, box_outer,
                   static_cast<int>(swizzle)};
  std::lock_guard<std::mutex> lk(g_map_mu);
  for (MapEntry& e : g_maps) {
    if (e.key == key) {
      e.used = ++g_map_clock;
      *out = e.map;
      return GEMM_OK;
    }
  }
  auto fn = encode_fn();
  if (fn == nullptr) return GEMM_ERR_CUDA;
  CUtensorMap map;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estrides[2] = {1, 1};
  const CUresult r = fn(&map, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estrides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return GEMM_ERR_CUDA;
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

template <typename... ExpT, typename... ActT>
int launch_pair(void (*kernel)(ExpT...), int grid, int smem, cudaStream_t stream,
                ActT&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(kThreads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
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

// C = beta * C (K == 0); C is not read when beta == 0.
__global__ void scale_kernel(void* C, long long ldc, int M, int N, float beta, int bf16) {
  const long long total = static_cast<long long>(M) * N;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long m = i / N, n = i % N;
    const long long off = m * ldc + n;
    if (bf16) {
      uint16_t* c = static_cast<uint16_t*>(C);
      const float v = beta == 0.0f ? 0.0f : beta * bf16_bits_to_float(c[off]);
      c[off] = static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xFFFFu);
    } else {
      float* c = static_cast<float*>(C);
      c[off] = beta == 0.0f ? 0.0f : beta * c[off];
    }
  }
}

int run_scale(const gemm_plan& pl, void* C, int64_t ldc, int64_t M, int64_t N, float beta,
              bool bf16, cudaStream_t stream) {
  return launch(scale_kernel, pl.grid, 256, 0, stream, C, static_cast<long long>(ldc),
                static_cast<int>(M), static_cast<int>(N), beta, bf16 ? 1 : 0);
}

TileParams tile_params(int64_t M, int64_t N, int64_t K, int tile_m, int tile_n_out, float alpha,
                       float beta, const void* C, int64_t ldc, int64_t tiles) {
  TileParams p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_blocks = static_cast<int>(ceil_div(M, tile_m));
  p.n_blocks = static_cast<int>(ceil_div(N, tile_n_out));
  p.k_blocks = static_cast<int>(ceil_div(K, kBK));
  p.num_tiles = static_cast<int>(tiles);
  p.group_m = kGroupM;
  p.alpha = alpha;
  p.beta = beta;
  p.C = C;
  p.ldc = ldc;
  p.num_full = p.num_tiles;
  p.tail_split = 1;
  p.kb_per_piece = p.k_blocks;
  p.num_units = p.num_tiles;
  p.ws = nullptr;
  p.counters = nullptr;
  return p;
}

// Work units of a pair plan (whole tiles, then split tail pieces) and the
// workspace they need.  A plan that needs a workspace the device cannot get
// (the stream is being captured) is redone without the split.
int pair_units(int dev, gemm_plan* pl, int64_t M, int64_t N, int64_t K, int bn_out_cols,
               TileParams* p, cudaStream_t stream, bool gate_up, int slots) {
  const int64_t tiles = ceil_div(M, kPairBM) * ceil_div(N, bn_out_cols);
  p->num_tiles = static_cast<int>(tiles);
  PairChoice c;
  if (gate_up) {
    c.bn = 256;
    plan_tail(tiles, p->k_blocks, slots, true, &c);
  } else {
    c = choose_pair(M, N, K, slots, true);
  }
  if (c.split > 1) {
    const size_t ws = static_cast<size_t>(pair_workspace_bytes(c));
    const size_t counters = static_cast<size_t>(c.tiles - c.full) * 8;
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
      // Without a workspace (graph capture): the same tiles, all whole.
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
  p->num_units = static_cast<int>(c.full + (c.tiles - c.full) * c.split);
  return GEMM_OK;
}

template <int BN, int EPI>
int launch_pair_gemm(const gemm_plan& pl, int dev, const CUtensorMap& tmA, const CUtensorMap& tmB,
                     const CUtensorMap& tmB2, const CUtensorMap& tmOut, const TileParams& p,
                     cudaStream_t stream) {
  using Cfg = PairCfg<BN, kPairStages, EPI>;
  auto kern = gemm_pair_kernel<BN, kPairStages, EPI>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const int st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), Cfg::kSmemBytes);
    if (st != GEMM_OK) return st;
  }
  return launch_pair(kern, pl.grid, Cfg::kSmemBytes, stream, tmA, tmB, tmB2, tmOut, p);
}

// Output descriptor of an epilogue box: FP32 32 x 32 (128-byte swizzle);
// BF16 64 x 32 (128-byte swizzle) or, for tile widths not a multiple of 64,
// 32 x 32 (64-byte swizzle).  Must match EpiBox in gemm_kernels.cuh.
int output_map(CUtensorMap* out, void* C, int64_t M, int64_t N, int64_t ldc, bool bf16,
               int tile_out_cols) {
  if (!bf16)
    return tensor_map_2d(out, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, N, M, ldc * 4, 32, 32);
  if (tile_out_cols % 64 == 0)
    return tensor_map_2d(out, C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldc * 2, 64, 32);
  return tensor_map_2d(out, C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldc * 2, 32, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B);
}

int run_pair(gemm_plan& pl, int dev, int sms, int slots, int64_t M, int64_t N, int64_t K,
             float alpha, const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
             void* C, int64_t ldc, bool bf16, cudaStream_t stream) {
  const int bn = pl.tile_n;
  CUtensorMap tmA, tmB, tmOut;
  int st;
  if ((st = tensor_map_2d(&tmA, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, lda * 2, kBK, 128)) !=
      GEMM_OK)
    return st;
  if ((st = tensor_map_2d(&tmB, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, ldb * 2, kBK,
                          bn / 2)) != GEMM_OK)
    return st;
  if ((st = output_map(&tmOut, C, M, N, ldc, bf16, bn)) != GEMM_OK) return st;
  TileParams p = tile_params(M, N, K, kPairBM, bn, alpha, beta, C, ldc, pl.tiles);
  pair_units(dev, &pl, M, N, K, bn, &p, stream, false, slots);
  switch (bn) {
    case 256:
      return bf16 ? launch_pair_gemm<256, EPI_BF16>(pl, dev, tmA, tmB, tmB, tmOut, p, stream)
                  : launch_pair_gemm<256, EPI_F32>(pl, dev, tmA, tmB, tmB, tmOut, p, stream);
    case 224:
      return bf16 ? launch_pair_gemm<224, EPI_BF16>(pl, dev, tmA, tmB, tmB, tmOut, p, stream)
                  : launch_pair_gemm<224, EPI_F32>(pl, dev, tmA, tmB, tmB, tmOut, p, stream);
    default:
      return GEMM_ERR_UNSUPPORTED;
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

int gemm_bf16_plan(int64_t M, int64_t N, int64_t K, int out_dtype, int num_sms,
                   gemm_plan* plan) {
  if (plan == nullptr) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return GEMM_ERR_INVALID_ARG;
  if (out_dtype != GEMM_OUT_F32 && out_dtype != GEMM_OUT_BF16) return GEMM_ERR_INVALID_ARG;
  if (num_sms <= 0) {
    const int st = device_sms(&num_sms);
    if (st != GEMM_OK) return st;
  }
  return plan_gemm(M, N, K, num_sms, plan);
}

int gemm_gate_up_plan(int64_t M, int64_t N, int64_t K, int num_sms, gemm_plan* plan) {
  if (plan == nullptr) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return GEMM_ERR_INVALID_ARG;
  if (num_sms <= 0) {
    const int st = device_sms(&num_sms);
    if (st != GEMM_OK) return st;
  }
  return plan_gate_up(M, N, K, num_sms, plan);
}

int gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha, const void* A, int64_t lda,
              const void* B, int64_t ldb, float beta, void* C, int64_t ldc, int out_dtype,
              void* stream_) {
  int st = validate_gemm(M, N, K, A, lda, B, ldb, beta, C, ldc, out_dtype);
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
  plan_gemm(M, N, K, sms, &pl, slots);
  const bool bf16 = out_dtype == GEMM_OUT_BF16;

  if (pl.kernel == K_SCALE) return run_scale(pl, C, ldc, M, N, beta, bf16, stream);
  if (pl.kernel == K_PAIR)
    return run_pair(pl, dev, sms, slots, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bf16,
                    stream);

  if (pl.kernel == K_SKINNY) {
    CUtensorMap tmW, tmX;
    if ((st = tensor_map_2d(&tmW, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, ldb * 2, kBK,
                            kSkinnyRows)) != GEMM_OK)
      return st;
    if ((st = tensor_map_2d(&tmX, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, lda * 2, kBK,
                            kSkinnyNX)) != GEMM_OK)
      return st;
    SkinnyParams p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.n_blocks = static_cast<int>(ceil_div(N, kSkinnyRows));
    p.k_blocks = static_cast<int>(ceil_div(K, kBK));
    p.splits = pl.split_k;
    p.kb_per_split = static_cast<int>(ceil_div(p.k_blocks, p.splits));
    p.num_units = static_cast<int>(pl.tiles);
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.out_bf16 = bf16 ? 1 : 0;
    p.ws = nullptr;
    p.counters = nullptr;
    auto kern = gemm_skinny_kernel<kSkinnyStages>;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if ((st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), pl.smem_bytes)) !=
          GEMM_OK)
        return st;
      if (p.splits > 1) {
        const size_t ws_bytes = static_cast<size_t>(p.splits) * M * N * sizeof(float);
        const size_t counters = static_cast<size_t>(p.n_blocks) * 4;
        if ((st = ensure_workspace(dev, ws_bytes, counters, stream)) != GEMM_OK) return st;
        p.ws = g_dev[dev].ws;
        p.counters = g_dev[dev].counters;
      }
    }
    return launch(kern, pl.grid, kThreads, pl.smem_bytes, stream, tmW, tmX, p);
  }

  // Tiled tcgen05 GEMM.
  CUtensorMap tmA, tmB, tmOut;
  if ((st = tensor_map_2d(&tmA, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, lda * 2, kBK, kBM)) !=
      GEMM_OK)
    return st;
  if ((st = tensor_map_2d(&tmB, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, ldb * 2, kBK,
                          kTileN)) != GEMM_OK)
    return st;
  if (bf16) {
    st = tensor_map_2d(&tmOut, C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldc * 2, 64, 32);
  } else {
    st = tensor_map_2d(&tmOut, C, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, N, M, ldc * 4, 32, 32);
  }
  if (st != GEMM_OK) return st;
  const TileParams p = tile_params(M, N, K, kBM, kTileN, alpha, beta, C, ldc, pl.tiles);
  if (bf16) {
    auto kern = gemm_tc_kernel<kTileN, kStages, EPI_BF16>;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      if ((st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern),
                                 CfgBF16::kSmemBytes)) != GEMM_OK)
        return st;
    }
    return launch(kern, pl.grid, kThreads, CfgBF16::kSmemBytes, stream, tmA, tmB, tmB, tmOut, p);
  }
  auto kern = gemm_tc_kernel<kTileN, kStages, EPI_F32>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), CfgF32::kSmemBytes)) !=
        GEMM_OK)
      return st;
  }
  return launch(kern, pl.grid, kThreads, CfgF32::kSmemBytes, stream, tmA, tmB, tmB, tmOut, p);
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
  if (pl.kernel == K_SCALE) return run_scale(pl, Y, ldy, M, N, 0.0f, true, stream);
  if (pl.kernel == K_PAIR_GATE_UP) {
    CUtensorMap tmX, tmWg, tmWu, tmY;
    if ((st = tensor_map_2d(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, ldx * 2, kBK, 128)) !=
        GEMM_OK)
      return st;
    if ((st = tensor_map_2d(&tmWg, Wg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, ldw * 2, kBK,
                            CfgPairGU::kOutCols)) != GEMM_OK)
      return st;
    if ((st = tensor_map_2d(&tmWu, Wu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, ldw * 2, kBK,
                            CfgPairGU::kOutCols)) != GEMM_OK)
      return st;
    if ((st = output_map(&tmY, Y, M, N, ldy, true, CfgPairGU::kOutCols)) != GEMM_OK) return st;
    TileParams p = tile_params(M, N, K, kPairBM, CfgPairGU::kOutCols, 1.0f, 0.0f, nullptr, ldy,
                               pl.tiles);
    pair_units(dev, &pl, M, N, K, CfgPairGU::kOutCols, &p, stream, true, slots);
    return launch_pair_gemm<256, EPI_GATE_UP>(pl, dev, tmX, tmWg, tmWu, tmY, p, stream);
  }

  CUtensorMap tmX, tmWg, tmWu, tmY;
  if ((st = tensor_map_2d(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, ldx * 2, kBK, kBM)) !=
      GEMM_OK)
    return st;
  if ((st = tensor_map_2d(&tmWg, Wg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, ldw * 2, kBK,
                          CfgGU::kOutCols)) != GEMM_OK)
    return st;
  if ((st = tensor_map_2d(&tmWu, Wu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, ldw * 2, kBK,
                          CfgGU::kOutCols)) != GEMM_OK)
    return st;
  if ((st = tensor_map_2d(&tmY, Y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldy * 2, 64, 32)) !=
      GEMM_OK)
    return st;
  const TileParams p =
      tile_params(M, N, K, kBM, CfgGU::kOutCols, 1.0f, 0.0f, nullptr, ldy, pl.tiles);
  auto kern = gemm_tc_kernel<256, kGateUpStages, EPI_GATE_UP>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = ensure_smem_attr(dev, reinterpret_cast<const void*>(kern), CfgGU::kSmemBytes)) !=
        GEMM_OK)
      return st;
  }
  return launch(kern, pl.grid, kThreads, CfgGU::kSmemBytes, stream, tmX, tmWg, tmWu, tmY, p);
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
    if (d.counters != nullptr && cudaMemset(d.counters, 0, d.counter_count * sizeof(int)) != cudaSuccess)
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

int gemm_prepare(int64_t max_N, void* stream) {
  if (max_N < 0 || max_N > kMaxDim) return GEMM_ERR_INVALID_ARG;
  int dev;
  int st = current_device(&dev);
  if (st != GEMM_OK) return st;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((st = probe_device(dev)) != GEMM_OK) return st;
  // Largest split the planner can choose is 32.
  const int64_t nb = ceil_div(std::max<int64_t>(max_N, 1), kSkinnyRows);
  const size_t ws_bytes = static_cast<size_t>(32) * kSkinnyMaxM * max_N * sizeof(float);
  return ensure_workspace(dev, ws_bytes, static_cast<size_t>(nb) * 4,
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
bool g_noalloc_smem_set[kMaxDevices];

// Encodes a 2-D map straight into *out (no descriptor cache, no allocation).
int encode_map_2d_direct(CUtensorMap* out, const void* ptr, CUtensorMapDataType dtype,
                         uint64_t inner, uint64_t outer, uint64_t pitch, uint32_t box_inner,
                         uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return GEMM_ERR_CUDA;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estrides[2] = {1, 1};
  const CUresult r = fn(out, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estrides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

extern "C" int gemm_bf16_skinny_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                        const void* A, int64_t lda, const void* B, int64_t ldb,
                                        float beta, void* C, int64_t ldc, int out_dtype,
                                        void* stream_) {
  int st = validate_gemm(M, N, K, A, lda, B, ldb, beta, C, ldc, out_dtype);
  if (st != GEMM_OK) return st;
  if (M == 0 || N == 0) return GEMM_OK;
  if (M > kSkinnyMaxM) return GEMM_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev;
  if ((st = current_device(&dev)) != GEMM_OK) return st;
  int sms;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((st = probe_device(dev)) != GEMM_OK) return st;
    sms = g_dev[dev].sms;
  }
  gemm_plan pl;
  plan_gemm(M, N, K, sms, &pl);
  const bool bf16 = out_dtype == GEMM_OUT_BF16;
  if (pl.kernel == K_SCALE) return run_scale(pl, C, ldc, M, N, beta, bf16, stream);

  SkinnyParams p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.n_blocks = static_cast<int>(ceil_div(N, kSkinnyRows));
  p.k_blocks = static_cast<int>(ceil_div(K, kBK));
  p.splits = pl.split_k;
  p.kb_per_split = static_cast<int>(ceil_div(p.k_blocks, p.splits));
  p.num_units = static_cast<int>(pl.tiles);
  p.alpha = alpha;
  p.beta = beta;
  p.C = C;
  p.ldc = ldc;
  p.out_bf16 = bf16 ? 1 : 0;
  const size_t counter_bytes =
      (static_cast<size_t>(p.n_blocks) * 4 * sizeof(int) + 255) & ~static_cast<size_t>(255);
  const size_t partial_bytes =
      p.splits > 1 ? static_cast<size_t>(p.splits) * M * N * sizeof(float) : 0;
  if (counter_bytes + partial_bytes > kNoAllocScratchBytes) return GEMM_ERR_INVALID_ARG;

  auto kern = gemm_skinny_kernel<kSkinnyStages>;
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
    if (!g_noalloc_smem_set[dev]) {
      if (cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               pl.smem_bytes) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
      }
      g_noalloc_smem_set[dev] = true;
    }
    base = g_noalloc_base[dev];
  }
  p.counters = reinterpret_cast<int*>(base);
  p.ws = reinterpret_cast<float*>(base + counter_bytes);

  CUtensorMap tmW, tmX;
  if ((st = encode_map_2d_direct(&tmW, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, N, ldb * 2, kBK,
                                 kSkinnyRows)) != GEMM_OK)
    return st;
  if ((st = encode_map_2d_direct(&tmX, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, lda * 2, kBK,
                                 kSkinnyNX)) != GEMM_OK)
    return st;
  // The arrival counters must start at zero; the array keeps whatever the
  // previous call left, so clear them on the stream first.
  if (p.splits > 1 && cudaMemsetAsync(p.counters, 0, counter_bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return launch(kern, pl.grid, kThreads, pl.smem_bytes, stream, tmW, tmX, p);
}
