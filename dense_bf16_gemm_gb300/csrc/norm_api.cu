// norm_api.cu -- host side of the row normalisation ("Tiles and shared
// memory", section "A complete kernel"): argument checks, the launch shape
// and the C ABI entry gemm_rms_norm declared in include/gemm_bf16.h.
//
// The kernel is bound by HBM bandwidth, so the launch fills every SM with as
// many resident blocks as its registers allow (a persistent grid of
// SMs x resident blocks) and lets the warps stride over the rows.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/gemm_bf16.h"
#include "norm_api.h"
#include "rms_norm.cuh"

namespace {

using namespace gb3;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = 0x7FFFFFFF;

struct NormDevice {
  bool probed = false;
  bool supported = false;
  int sms = 0;
  // resident blocks per SM of each kernel instantiation used so far
  std::vector<std::pair<const void*, int>> occupancy;
};

std::mutex g_norm_mu;
NormDevice g_norm_dev[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t elem_bytes(int code) { return code == GEMM_OUT_F32 ? 4 : 2; }

bool valid_code(int code) {
  return code == GEMM_OUT_F32 || code == GEMM_OUT_BF16 || code == GEMM_OUT_F16;
}

// Caller holds g_norm_mu.
int probe(int* dev_out, int* sms) {
  int dev;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
  NormDevice& d = g_norm_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    d.probed = true;
    d.supported = (major == 10 && minor == 3);
    d.sms = n;
  }
  *dev_out = dev;
  *sms = d.sms;
  return d.supported ? GEMM_OK : GEMM_ERR_UNSUPPORTED;
}

// Caller holds g_norm_mu.
int resident_blocks(int dev, const void* fn) {
  NormDevice& d = g_norm_dev[dev];
  for (const auto& e : d.occupancy)
    if (e.first == fn) return e.second;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, kNormThreads, 0) != cudaSuccess) {
    cudaGetLastError();
    blocks = 1;
  }
  blocks = std::max(1, blocks);
  d.occupancy.emplace_back(fn, blocks);
  return blocks;
}

template <int XK, int YK, int CACHE, int RW = 1>
int launch_norm(int64_t rows, int64_t D, const void* X, int64_t ldx, const float* G, float eps,
                void* Y, int64_t ldy, cudaStream_t stream) {
  auto kern = rms_norm_kernel<XK, YK, CACHE, RW>;
  int dev, sms, per_sm;
  {
    std::lock_guard<std::mutex> lk(g_norm_mu);
    const int st = probe(&dev, &sms);
    if (st != GEMM_OK) return st;
    per_sm = resident_blocks(dev, reinterpret_cast<const void*>(kern));
  }
  constexpr int kGroups = kNormThreads / 32 / RW;   // rows a block works on at a time
  const int64_t want = (rows + kGroups - 1) / kGroups;
  const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sms) * per_sm));
  kern<<<grid, kNormThreads, 0, stream>>>(X, static_cast<long long>(ldx), G, eps, Y,
                                          static_cast<long long>(ldy), static_cast<int>(rows),
                                          static_cast<int>(D));
  if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
  return GEMM_OK;
}

// Rows whose 16-byte vectors fit in 4 registers per lane take one warp and
// the small cache; longer rows take two warps of 8 cached vectors each
// (GB3_NORM_ROW_WARPS = 1 keeps them on one warp of 16, for comparison).
template <int XK, int YK>
int launch_sized(int64_t rows, int64_t D, const void* X, int64_t ldx, const float* G, float eps,
                 void* Y, int64_t ldy, cudaStream_t stream) {
  const int64_t vecs_per_lane = (D * NormElems<XK>::kBytes + 32 * 16 - 1) / (32 * 16);
  if (vecs_per_lane <= 4) return launch_norm<XK, YK, 4>(rows, D, X, ldx, G, eps, Y, ldy, stream);
  const char* env = std::getenv("GB3_NORM_ROW_WARPS");
  if (env != nullptr && std::atoi(env) == 1)
    return launch_norm<XK, YK, 16>(rows, D, X, ldx, G, eps, Y, ldy, stream);
  return launch_norm<XK, YK, 8, 2>(rows, D, X, ldx, G, eps, Y, ldy, stream);
}

template <int XK>
int launch_x(int y_dtype, int64_t rows, int64_t D, const void* X, int64_t ldx, const float* G,
             float eps, void* Y, int64_t ldy, cudaStream_t stream) {
  switch (y_dtype) {
    case GEMM_OUT_F32: return launch_sized<XK, NORM_F32>(rows, D, X, ldx, G, eps, Y, ldy, stream);
    case GEMM_OUT_BF16: return launch_sized<XK, NORM_BF16>(rows, D, X, ldx, G, eps, Y, ldy, stream);
    default: return launch_sized<XK, NORM_F16>(rows, D, X, ldx, G, eps, Y, ldy, stream);
  }
}

}  // namespace

namespace gb3 {

int rms_norm_check(int64_t rows, int64_t D, const void* X, int64_t ldx, int x_dtype,
                   const float* G, float eps, const void* Y, int64_t ldy, int y_dtype) {
  if (rows < 0 || D < 0 || rows > kMaxDim || D > kMaxDim) return GEMM_ERR_INVALID_ARG;
  if (!valid_code(x_dtype) || !valid_code(y_dtype)) return GEMM_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || std::isinf(eps)) return GEMM_ERR_INVALID_ARG;
  if (rows == 0 || D == 0) return GEMM_OK;
  if (X == nullptr || Y == nullptr || G == nullptr || ldx < D || ldy < D)
    return GEMM_ERR_INVALID_ARG;
  const int64_t xe = elem_bytes(x_dtype), ye = elem_bytes(y_dtype);
  if (!aligned16(X) || !aligned16(Y) || !aligned16(G) || (ldx * xe) % 16 != 0 ||
      (ldy * ye) % 16 != 0)
    return GEMM_ERR_ALIGNMENT;
  // Y may be X itself (same element size and pitch); any other overlap is refused.
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(X), y0 = reinterpret_cast<uintptr_t>(Y);
  const uintptr_t x1 = x0 + static_cast<uintptr_t>(((rows - 1) * ldx + D) * xe);
  const uintptr_t y1 = y0 + static_cast<uintptr_t>(((rows - 1) * ldy + D) * ye);
  const bool overlap = x0 < y1 && y0 < x1;
  if (overlap && !(x0 == y0 && ldx * xe == ldy * ye && xe == ye)) return GEMM_ERR_INVALID_ARG;
  return GEMM_OK;
}

int rms_norm_run(int64_t rows, int64_t D, const void* X, int64_t ldx, int x_dtype,
                 const float* G, float eps, void* Y, int64_t ldy, int y_dtype,
                 cudaStream_t stream) {
  const int st = rms_norm_check(rows, D, X, ldx, x_dtype, G, eps, Y, ldy, y_dtype);
  if (st != GEMM_OK || rows == 0 || D == 0) return st;
  switch (x_dtype) {
    case GEMM_OUT_F32: return launch_x<NORM_F32>(y_dtype, rows, D, X, ldx, G, eps, Y, ldy, stream);
    case GEMM_OUT_BF16: return launch_x<NORM_BF16>(y_dtype, rows, D, X, ldx, G, eps, Y, ldy, stream);
    default: return launch_x<NORM_F16>(y_dtype, rows, D, X, ldx, G, eps, Y, ldy, stream);
  }
}

}  // namespace gb3

extern "C" int gemm_rms_norm(int64_t rows, int64_t D, const void* X, int64_t ldx, int x_dtype,
                             const float* G, float eps, void* Y, int64_t ldy, int y_dtype,
                             void* stream) {
  return gb3::rms_norm_run(rows, D, X, ldx, x_dtype, G, eps, Y, ldy, y_dtype,
                           static_cast<cudaStream_t>(stream));
}
