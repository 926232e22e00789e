// rms_norm.cuh -- row normalisation for sm_103a ("Tiles and shared memory",
// section "A complete kernel"):
//
//   ss(m) = sum_k x(m,k)^2,   inv(m) = 1 / sqrt(ss(m)/D + eps),
//   y(m,k) = x(m,k) * inv(m) * g(k)
//
// The operation reads each element once and writes it once, so it is bound by
// HBM bandwidth, not arithmetic: one warp (short rows) or two warps (long
// rows) own one row at a time (rows are visited group-stride over the grid),
// lanes read 16-byte vectors so that every warp-wide load moves 512
// contiguous bytes, and the first CACHE vectors of each lane stay in registers
// between the sum of squares and the scaling pass (two warps with CACHE = 8
// hold a BF16 row of 4096 elements whole; short rows use one warp and
// CACHE = 4).  Fewer registers per warp keep more warps, and so more loads,
// in flight.  Longer rows are read a second time, from L1/L2.
//
// Arithmetic (FP32): each lane adds the squares of its elements in order
// (vector v = (i*RW + sub)*32 + lane, elements of a vector in order, then the
// scalar tail k = tail0 + lane + 32 j in the first warp), the 32 lane sums
// are combined by a butterfly of 5 shuffle steps and the RW warp sums in
// warp order, then ss / D, + eps, sqrtf and the reciprocal are each
// correctly rounded; y = (x * inv) * g, rounded to the output type (nearest
// even for BF16/FP16).
#pragma once

#include "ptx.cuh"

namespace gb3 {

// Element kinds of the normalisation's input and output.
enum NormKind : int { NORM_F32 = 0, NORM_BF16 = 1, NORM_F16 = 2 };

constexpr int kNormThreads = 256;   // 8 warps, one row each at a time

template <int KIND>
struct NormElems {
  static constexpr int kPerVec = (KIND == NORM_F32) ? 4 : 8;  // elements per 16 bytes
  static constexpr int kBytes = (KIND == NORM_F32) ? 4 : 2;
};

// Loads of X are plain (not the read-only path): Y may be X itself.
template <int KIND>
__device__ __forceinline__ float norm_scalar(const void* base, long long idx) {
  if constexpr (KIND == NORM_F32) {
    return static_cast<const float*>(base)[idx];
  } else {
    const uint32_t bits = static_cast<const unsigned short*>(base)[idx];
    return KIND == NORM_F16 ? f16_bits_to_float(bits) : bf16_bits_to_float(bits);
  }
}

// The elements of one 16-byte vector in FP32 (4 or 8 of them).
template <int KIND>
__device__ __forceinline__ void unpack_vec(const uint4& q, float (&x)[8]) {
  if constexpr (KIND == NORM_F32) {
    x[0] = __uint_as_float(q.x);
    x[1] = __uint_as_float(q.y);
    x[2] = __uint_as_float(q.z);
    x[3] = __uint_as_float(q.w);
  } else {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = half16_to_float(w[j] & 0xFFFFu, KIND == NORM_F16);
      x[2 * j + 1] = half16_to_float(w[j] >> 16, KIND == NORM_F16);
    }
  }
}

template <int KIND>
__device__ __forceinline__ float sum_squares(const uint4& q, float ss) {
  float x[8];
  unpack_vec<KIND>(q, x);
#pragma unroll
  for (int j = 0; j < NormElems<KIND>::kPerVec; ++j) ss = fmaf(x[j], x[j], ss);
  return ss;
}

// y = (x * inv) * g for one vector; `gv` points at the vector's gains.
template <int XK, int YK>
__device__ __forceinline__ void scale_store(const uint4& q, float inv, const float* gv, void* dst) {
  constexpr int V = NormElems<XK>::kPerVec;
  float x[8];
  unpack_vec<XK>(q, x);
  float y[8];
  const float4 g0 = __ldg(reinterpret_cast<const float4*>(gv));
  y[0] = x[0] * inv * g0.x;
  y[1] = x[1] * inv * g0.y;
  y[2] = x[2] * inv * g0.z;
  y[3] = x[3] * inv * g0.w;
  if constexpr (V == 8) {
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(gv) + 1);
    y[4] = x[4] * inv * g1.x;
    y[5] = x[5] * inv * g1.y;
    y[6] = x[6] * inv * g1.z;
    y[7] = x[7] * inv * g1.w;
  }
  if constexpr (YK == NORM_F32) {
    float4* d = static_cast<float4*>(dst);
    d[0] = make_float4(y[0], y[1], y[2], y[3]);
    if constexpr (V == 8) d[1] = make_float4(y[4], y[5], y[6], y[7]);
  } else {
    const bool f16 = YK == NORM_F16;
    if constexpr (V == 8) {
      *static_cast<uint4*>(dst) = make_uint4(pack_half16x2(y[0], y[1], f16), pack_half16x2(y[2], y[3], f16),
                                             pack_half16x2(y[4], y[5], f16), pack_half16x2(y[6], y[7], f16));
    } else {
      *static_cast<uint2*>(dst) = make_uint2(pack_half16x2(y[0], y[1], f16), pack_half16x2(y[2], y[3], f16));
    }
  }
}

template <int YK>
__device__ __forceinline__ void store_scalar(void* base, long long idx, float y) {
  if constexpr (YK == NORM_F32) {
    static_cast<float*>(base)[idx] = y;
  } else {
    const uint32_t packed = pack_half16x2(y, 0.0f, YK == NORM_F16);
    static_cast<unsigned short*>(base)[idx] = static_cast<unsigned short>(packed & 0xFFFFu);
  }
}

// X(m,k) at X[m*ldx + k], Y(m,k) at Y[m*ldy + k], G(k) at G[k].  X, Y and G
// are 16-byte aligned and ldx, ldy keep every row 16-byte aligned (checked on
// the host).  Y may be X itself (same pitch): every element is read by the
// thread that writes it, before it writes it.
//
// RW warps share a row (RW = 2 for long rows: half the registers per warp, so
// twice the warps, and twice the bytes, in flight per SM).  Warp `sub` of a
// row takes vectors v = (i*RW + sub)*32 + lane; the warps' sums meet in
// shared memory (double-buffered by row parity, one named barrier per row)
// and are added in sub order, so both warps hold the same value.
template <int XK, int YK, int CACHE, int RW = 1>
// Resident blocks per SM the registers must allow: 4 for short rows, 2 for
// one warp holding 16 vectors, 3 for two warps holding 8 each.
__global__ void __launch_bounds__(kNormThreads, RW == 2 ? 3 : (CACHE <= 4 ? 4 : 2))
    rms_norm_kernel(const void* X, long long ldx, const float* __restrict__ G, float eps, void* Y,
                    long long ldy, int rows, int D) {
  static_assert(RW == 1 || RW == 2, "warps per row");
  constexpr int V = NormElems<XK>::kPerVec;
  constexpr int kWarps = kNormThreads / 32;
  constexpr int kGroups = kWarps / RW;  // rows a block works on at a time
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int grp = warp / RW, sub = warp % RW;
  const int groups = gridDim.x * kGroups;
  const int nvec = D / V;          // whole vectors per row
  const int tail0 = nvec * V;      // first element of the scalar tail
  __shared__ float partial[2][kWarps];
  int parity = 0;
  for (int m = blockIdx.x * kGroups + grp; m < rows; m += groups, parity ^= 1) {
    const uint4* xrow = reinterpret_cast<const uint4*>(
        static_cast<const uint8_t*>(X) + static_cast<long long>(m) * ldx * NormElems<XK>::kBytes);
    uint8_t* yrow = static_cast<uint8_t*>(Y) + static_cast<long long>(m) * ldy * NormElems<YK>::kBytes;
    uint4 cache[CACHE];
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < CACHE; ++i) {
      const int v = (i * RW + sub) * 32 + lane;
      if (v < nvec) cache[i] = xrow[v];
    }
#pragma unroll
    for (int i = 0; i < CACHE; ++i) {
      const int v = (i * RW + sub) * 32 + lane;
      if (v < nvec) ss = sum_squares<XK>(cache[i], ss);
    }
    for (int v = (CACHE * RW + sub) * 32 + lane; v < nvec; v += 32 * RW)
      ss = sum_squares<XK>(xrow[v], ss);
    const void* xr = static_cast<const uint8_t*>(X) + static_cast<long long>(m) * ldx * NormElems<XK>::kBytes;
    if (sub == 0) {
      for (int k = tail0 + lane; k < D; k += 32) {
        const float x = norm_scalar<XK>(xr, k);
        ss = fmaf(x, x, ss);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if constexpr (RW > 1) {
      if (lane == 0) partial[parity][warp] = ss;
      asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(32 * RW) : "memory");
      ss = 0.0f;
#pragma unroll
      for (int w = 0; w < RW; ++w) ss += partial[parity][grp * RW + w];
    }
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + eps);

#pragma unroll
    for (int i = 0; i < CACHE; ++i) {
      const int v = (i * RW + sub) * 32 + lane;
      if (v < nvec)
        scale_store<XK, YK>(cache[i], inv, G + static_cast<long long>(v) * V,
                            yrow + static_cast<long long>(v) * V * NormElems<YK>::kBytes);
    }
    for (int v = (CACHE * RW + sub) * 32 + lane; v < nvec; v += 32 * RW)
      scale_store<XK, YK>(xrow[v], inv, G + static_cast<long long>(v) * V,
                          yrow + static_cast<long long>(v) * V * NormElems<YK>::kBytes);
    if (sub == 0)
      for (int k = tail0 + lane; k < D; k += 32)
        store_scalar<YK>(yrow, k, norm_scalar<XK>(xr, k) * inv * __ldg(G + k));
  }
}

}  // namespace gb3
