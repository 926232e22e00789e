// norm_api.h -- library-internal entry points of the row normalisation
// (norm_api.cu), used by the fused normalisation + gate/up call in
// gemm_api.cu.  Not exported from the shared library.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace gb3 {

// Checks the arguments of gemm_rms_norm (sizes, element codes, eps, null
// pointers, alignment, aliasing) without touching the device.
int rms_norm_check(int64_t rows, int64_t D, const void* X, int64_t ldx, int x_dtype,
                   const float* G, float eps, const void* Y, int64_t ldy, int y_dtype);

// Checks as rms_norm_check, then enqueues the normalisation on `stream`.
int rms_norm_run(int64_t rows, int64_t D, const void* X, int64_t ldx, int x_dtype,
                 const float* G, float eps, void* Y, int64_t ldy, int y_dtype,
                 cudaStream_t stream);

}  // namespace gb3
