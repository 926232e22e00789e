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

// y = (x * inv) * g for one vector; `gv` points at the vector's gains (in
// global memory, read through the read-only path, or with G_GENERIC a
// generic address, e.g. a copy in shared memory: the same values).
template <int XK, int YK, bool G_GENERIC = false>
__device__ __forceinline__ void scale_store(const uint4& q, float inv, const float* gv, void* dst) {
  constexpr int V = NormElems<XK>::kPerVec;
  float x[8];
  unpack_vec<XK>(q, x);
  float y[8];
  const float4 g0 = G_GENERIC ? *reinterpret_cast<const float4*>(gv)
                              : __ldg(reinterpret_cast<const float4*>(gv));
  y[0] = x[0] * inv * g0.x;
  y[1] = x[1] * inv * g0.y;
  y[2] = x[2] * inv * g0.z;
  y[3] = x[3] * inv * g0.w;
  if constexpr (V == 8) {
    const float4 g1 = G_GENERIC ? reinterpret_cast<const float4*>(gv)[1]
                                : __ldg(reinterpret_cast<const float4*>(gv) + 1);
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
// shared memory (`partial`, double-buffered by row parity, one named barrier
// per row group: id bar0 + group) and are added in sub order, so both warps
// hold the same value.
//
// The rows a group normalises: m = group0, group0 + group_stride, ... up to
// `rows`.  Row m is read from X + (m - src_row0) * ldx (elements), written to
// Y + m * ldy: the normalisation kernel reads X itself (src_row0 = 0); the
// gate/up kernel that normalises its activation first reads a batch of rows
// it copied into shared memory (X = the copy, src_row0 its first row), and
// with G_GENERIC the gains from a copy in shared memory too.  ROWS rows
// (1 or 2, m and m + group_stride) go through the steps together, so that
// their independent work overlaps; every row takes exactly the operations,
// in the same order, of ROWS = 1, so the bits are the same in every case.
// Y_BULK (X a copy in shared memory, YK == XK): each normalised row is
// written over its copy and sent to Y by one bulk copy of row_bytes bytes
// (issued by the group's first lane, committed as one bulk group); the
// caller waits for those copies before it reuses the shared memory.
template <int XK, int YK, int CACHE, int RW, int WARPS, bool G_GENERIC = false, int ROWS = 1,
          bool Y_BULK = false>
__device__ __forceinline__ void rms_norm_rows(const void* X, long long ldx,
                                              const float* __restrict__ G, float eps, void* Y,
                                              long long ldy, int rows, int D, int group0,
                                              int group_stride, float (&partial)[2][ROWS][WARPS],
                                              int bar0, int src_row0 = 0,
                                              uint32_t row_bytes = 0) {
  static_assert(RW == 1 || RW == 2, "warps per row");
  static_assert(ROWS == 1 || ROWS == 2, "rows together");
  static_assert(!Y_BULK || XK == YK, "the row is normalised in place before its copy");
  constexpr int V = NormElems<XK>::kPerVec;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int grp = warp / RW, sub = warp % RW;
  const int nvec = D / V;          // whole vectors per row
  const int tail0 = nvec * V;      // first element of the scalar tail
  int parity = 0;
  for (int m0 = group0; m0 < rows; m0 += ROWS * group_stride, parity ^= 1) {
    const uint4* xrow[ROWS];
    uint8_t* yrow[ROWS];
    bool live[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      const int m = m0 + r * group_stride;
      live[r] = m < rows;
      xrow[r] = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(X) +
          static_cast<long long>(m - src_row0) * ldx * NormElems<XK>::kBytes);
      yrow[r] = Y_BULK ? const_cast<uint8_t*>(reinterpret_cast<const uint8_t*>(xrow[r]))
                       : static_cast<uint8_t*>(Y) +
                             static_cast<long long>(m) * ldy * NormElems<YK>::kBytes;
    }
    uint4 cache[ROWS][CACHE];
    float ss[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      ss[r] = 0.0f;
#pragma unroll
      for (int i = 0; i < CACHE; ++i) {
        const int v = (i * RW + sub) * 32 + lane;
        if (live[r] && v < nvec) cache[r][i] = xrow[r][v];
      }
    }
#pragma unroll
    for (int i = 0; i < CACHE; ++i) {
      const int v = (i * RW + sub) * 32 + lane;
#pragma unroll
      for (int r = 0; r < ROWS; ++r)
        if (live[r] && v < nvec) ss[r] = sum_squares<XK>(cache[r][i], ss[r]);
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      if (!live[r]) continue;
      for (int v = (CACHE * RW + sub) * 32 + lane; v < nvec; v += 32 * RW)
        ss[r] = sum_squares<XK>(xrow[r][v], ss[r]);
      if (sub == 0) {
        for (int k = tail0 + lane; k < D; k += 32) {
          const float x = norm_scalar<XK>(xrow[r], k);
          ss[r] = fmaf(x, x, ss[r]);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int r = 0; r < ROWS; ++r) ss[r] += __shfl_xor_sync(0xffffffffu, ss[r], off);
    if constexpr (RW > 1) {
      if (lane == 0)
#pragma unroll
        for (int r = 0; r < ROWS; ++r) partial[parity][r][warp] = ss[r];
      asm volatile("bar.sync %0, %1;" ::"r"(bar0 + grp), "r"(32 * RW) : "memory");
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        ss[r] = 0.0f;
#pragma unroll
        for (int w = 0; w < RW; ++w) ss[r] += partial[parity][r][grp * RW + w];
      }
    }
    float inv[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) inv[r] = 1.0f / sqrtf(ss[r] / static_cast<float>(D) + eps);

#pragma unroll
    for (int i = 0; i < CACHE; ++i) {
      const int v = (i * RW + sub) * 32 + lane;
#pragma unroll
      for (int r = 0; r < ROWS; ++r)
        if (live[r] && v < nvec)
          scale_store<XK, YK, G_GENERIC>(cache[r][i], inv[r], G + static_cast<long long>(v) * V,
                                         yrow[r] + static_cast<long long>(v) * V * NormElems<YK>::kBytes);
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
      if (!live[r]) continue;
      for (int v = (CACHE * RW + sub) * 32 + lane; v < nvec; v += 32 * RW)
        scale_store<XK, YK, G_GENERIC>(xrow[r][v], inv[r], G + static_cast<long long>(v) * V,
                                       yrow[r] + static_cast<long long>(v) * V * NormElems<YK>::kBytes);
      if (sub == 0)
        for (int k = tail0 + lane; k < D; k += 32)
          store_scalar<YK>(yrow[r], k,
                           norm_scalar<XK>(xrow[r], k) * inv[r] * (G_GENERIC ? G[k] : __ldg(G + k)));
    }
    if constexpr (Y_BULK) {
      // The group's normalised rows are in shared memory: one lane sends each.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("bar.sync %0, %1;" ::"r"(bar0 + grp), "r"(32 * RW) : "memory");
      if (sub == 0 && lane == 0) {
        // Kept in L2: the rows are read again right away (by TMA, every CTA).
        const uint64_t keep = l2_policy_evict_last();
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
          if (!live[r]) continue;
          bulk_store_hint(static_cast<uint8_t*>(Y) + static_cast<long long>(m0 + r * group_stride) *
                                                         ldy * NormElems<YK>::kBytes,
                          static_cast<uint32_t>(__cvta_generic_to_shared(yrow[r])), row_bytes,
                          keep);
        }
        bulk_commit_group();
      }
    }
  }
}

template <int XK, int YK, int CACHE, int RW = 1>
// Resident blocks per SM the registers must allow: 4 for short rows, 2 for
// one warp holding 16 vectors, 3 for two warps holding 8 each.
__global__ void __launch_bounds__(kNormThreads, RW == 2 ? 3 : (CACHE <= 4 ? 4 : 2))
    rms_norm_kernel(const void* X, long long ldx, const float* __restrict__ G, float eps, void* Y,
                    long long ldy, int rows, int D) {
  constexpr int kWarps = kNormThreads / 32;
  constexpr int kGroups = kWarps / RW;  // rows a block works on at a time
  __shared__ float partial[2][1][kWarps];
  const int grp = (threadIdx.x >> 5) / RW;
  rms_norm_rows<XK, YK, CACHE, RW, kWarps>(X, ldx, G, eps, Y, ldy, rows, D,
                                           blockIdx.x * kGroups + grp, gridDim.x * kGroups,
                                           partial, 1);
}

}  // namespace gb3
