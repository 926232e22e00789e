/*
 * gemm_bf16.h -- C ABI of the GB300 (sm_103a) dense BF16 GEMM library.
 *
 * Every entry point takes plain pointers and sizes.  Device buffers are owned
 * by the caller: the library never frees them, never keeps them past the call
 * (beyond caching the tensor-map descriptor keyed by address and shape) and
 * does not check for aliasing between inputs and outputs (the tile
 * abstractions of "TMEM tiles and transfers", section "Completion and
 * validation", leave allocation, bounds and lifetime to the caller in the same
 * way).
 *
 * Compute calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and never synchronize the host.  A status other
 * than GEMM_OK means nothing was launched.  Errors raised by a kernel while
 * it runs (a pipeline wait that exceeded its limit) are recorded in a device
 * status word and read back with gemm_get_device_status().
 *
 * Storage convention ("TMA and Hopper WGMMA", section "The same storage
 * contract on both sides": A(M,K) has K contiguous and B(K,N) is stored with
 * K as its inner axis, so both operands are K-contiguous):
 *   a(m,k) = A[m*lda + k]      BF16
 *   b(k,n) = B[n*ldb + k]      BF16
 *   c(m,n) = C[m*ldc + n]      FP32 or BF16 (out_dtype), row-major
 * TMA requires 16-byte aligned base addresses and row pitches that are
 * multiples of 16 bytes ("TMA and Hopper WGMMA", section "Copy and
 * completion": the inner origin starts a 16-byte chunk).
 */
#ifndef GEMM_BF16_H
#define GEMM_BF16_H

#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,  /* negative or too large sizes, ld < extent, NULL with nonzero size, bad dtype */
    GEMM_ERR_ALIGNMENT = 2,    /* pointer not 16-byte aligned or row pitch not a multiple of 16 bytes */
    GEMM_ERR_UNSUPPORTED = 3,  /* current device is not compute capability 10.3 (GB300) */
    GEMM_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (descriptor encode, launch, allocation) */
    GEMM_ERR_TIMEOUT = 5       /* a kernel's bounded pipeline wait expired (read via gemm_get_device_status) */
};

/* Output element type. */
enum gemm_out_dtype {
    GEMM_OUT_F32 = 0,
    GEMM_OUT_BF16 = 1,
    GEMM_OUT_F16 = 2   /* rounded to nearest-even FP16 ("TMEM tiles and transfers",
                          section "Representation and windows": pack(Float16, f)) */
};

/* Operand element type of gemm_batched (A and B always share it). */
enum gemm_in_dtype {
    GEMM_IN_BF16 = 0,
    GEMM_IN_F16 = 1
};

/*
 * C = alpha * A.B + beta * C            ("Tiles and shared memory", section
 *                                        "var and let": the tile epilogue
 *                                        writes alpha*acc + beta*c_old over
 *                                        the slice of C it read)
 *
 * M, N, K    problem sizes, 0 <= M, N, K < 2^31, and at most 2^25 blocks of
 *            128 x 128 outputs per call (ceil(M/128) * ceil(N/128), times the
 *            batch in gemm_batched: more output than any GPU memory holds).
 *            M == 0 or N == 0 does nothing and returns GEMM_OK.  K == 0 gives
 *            C = beta * C.
 * A, lda     device BF16 matrix, a(m,k) = A[m*lda + k], lda >= K.
 * B, ldb     device BF16 matrix, b(k,n) = B[n*ldb + k], ldb >= K.
 * C, ldc     device matrix of type out_dtype, c(m,n) = C[m*ldc + n],
 *            ldc >= N.  Read only when beta != 0 (with beta == 0 it may hold
 *            NaN or garbage), always written.
 * out_dtype  GEMM_OUT_F32, GEMM_OUT_BF16 or GEMM_OUT_F16.  Accumulation is
 *            FP32; a 16-bit output is rounded to nearest-even once, from the
 *            FP32 value of alpha*acc + beta*c.
 * stream     cudaStream_t the work is enqueued on.
 *
 * Split K: for M <= 16, for the small-M kernel (16 < M <= 128, tiles shared
 * by several CTAs), and for the tiles of a last, partial wave of the
 * CTA-pair kernel, K is cut into pieces whose FP32 partial sums live in a
 * per-device workspace the library allocates on first use; the last piece
 * of each tile adds them in a fixed order, so results do not depend on
 * timing.  A call made while `stream` is being captured into a CUDA graph
 * cannot allocate: the M <= 128 paths then return GEMM_ERR_CUDA (make one
 * such call, or gemm_prepare(), before capturing) and the tiled path runs its
 * tiles whole.  Calls that use the workspace and run concurrently on
 * different streams share it and must not overlap on the GPU.
 */
GEMM_API int gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha,
              const void *A, int64_t lda,
              const void *B, int64_t ldb,
              float beta, void *C, int64_t ldc,
              int out_dtype, void *stream);

/*
 * A batch of independent GEMMs: C_b = alpha * A_b.B_b + beta * C_b for
 * b = 0 .. batch-1 ("TMA and Hopper WGMMA", section "The same storage
 * contract on both sides": a three-dimensional binding whose third
 * coordinate selects one matrix of a batch, each bounded separately).
 *
 * batch      number of matrices, 0 <= batch < 2^31 (0 does nothing); the
 *            2^25 limit on 128 x 128 output blocks counts every matrix.
 * M, N, K, lda, ldb, ldc, alpha, beta, out_dtype  as gemm_bf16, per matrix.
 * stride_a   elements between A_b and A_(b+1), >= M*lda when batch > 1;
 * stride_b   elements between B_b and B_(b+1), >= N*ldb when batch > 1;
 * stride_c   elements between C_b and C_(b+1), >= M*ldc when batch > 1;
 *            (stride * element size) must be a multiple of 16 bytes.
 *            Ignored when batch == 1.
 * in_dtype   GEMM_IN_BF16 or GEMM_IN_F16: the type of both A and B.
 * Rows and columns past a matrix's edges never read or write the next
 * matrix.  With batch == 1 and GEMM_IN_BF16 this is gemm_bf16.
 */
GEMM_API int gemm_batched(int64_t batch, int64_t M, int64_t N, int64_t K, float alpha,
                          const void *A, int64_t lda, int64_t stride_a,
                          const void *B, int64_t ldb, int64_t stride_b,
                          float beta, void *C, int64_t ldc, int64_t stride_c,
                          int in_dtype, int out_dtype, void *stream);

/*
 * Y = silu(X.Wg) * (X.Wu), elementwise product, silu(t) = t / (1 + exp(-t)).
 * ("TMA and Hopper WGMMA", sections "TMA and Hopper WGMMA" and "Worked
 * consumers and current validation": the fused gate/up projection epilogue.)
 *
 * X, ldx     device BF16, x(m,k) = X[m*ldx + k], ldx >= K.
 * Wg, Wu     device BF16, wg(k,n) = Wg[n*ldw + k], wu(k,n) = Wu[n*ldw + k],
 *            ldw >= K (both K-contiguous like B of gemm_bf16).
 * Y, ldy     device BF16 output, y(m,n) = Y[m*ldy + n], ldy >= N.
 * M, N, K    as gemm_bf16 (the same limits).
 * Both products accumulate in FP32; silu(g)*u is evaluated in FP32 and
 * rounded to BF16 once.  K == 0 gives Y = 0.
 */
GEMM_API int gemm_gate_up_silu(int64_t M, int64_t N, int64_t K,
                      const void *X, int64_t ldx,
                      const void *Wg, const void *Wu, int64_t ldw,
                      void *Y, int64_t ldy, void *stream);

/*
 * gemm_batched with reductions along each row of every result:
 *
 *   v_b(m,n)       = alpha * A_b.B_b(m,n) + beta * C_b(m,n)   (FP32, before the
 *                    output rounding)
 *   row_sum[b*M+m] = sum over n of v_b(m,n)
 *   row_max[b*M+m] = max over n,   row_min[b*M+m] = min over n
 *
 * ("TMEM tiles and transfers", section "Storage and a transfer": a reduction
 * along the second axis of a loaded accumulator, which each thread holds
 * whole for its row; "TMA and Hopper WGMMA", section "WGMMA values and
 * ownership": sum, maximum and minimum along axis 2 of a finished
 * accumulator.  The pages reduce one tile; here the reduction covers the
 * whole row, n = 0 .. N-1.)
 *
 * All arguments up to out_dtype are those of gemm_batched, and C is written
 * as there.  row_sum, row_max, row_min: device arrays of batch*M FP32 values
 * (4-byte aligned, owned by the caller); any of them may be NULL (not
 * written).  Maxima and minima ignore NaN values (IEEE maxNum); sums
 * propagate them.  N == 0 (with batch, M > 0) writes sum 0, max -inf and
 * min +inf without touching C.
 *
 * Order and determinism: each tile's epilogue adds its row's values in column
 * order in FP32; the per-tile partials are combined in column-tile order by
 * the last tile of each 32-row band to finish, so the results do not depend
 * on timing.  The partials live in a per-device workspace allocated on first
 * use; a call made while `stream` is being captured returns GEMM_ERR_CUDA
 * unless an earlier call of at least the same batch*M*N/256 size allocated
 * it.  Problems with M <= 16 run on the 128-row tiled kernel instead of the
 * swapped-operand one.
 */
GEMM_API int gemm_row_stats(int64_t batch, int64_t M, int64_t N, int64_t K, float alpha,
                   const void *A, int64_t lda, int64_t stride_a,
                   const void *B, int64_t ldb, int64_t stride_b,
                   float beta, void *C, int64_t ldc, int64_t stride_c,
                   int in_dtype, int out_dtype,
                   float *row_sum, float *row_max, float *row_min, void *stream);

/*
 * Row normalisation ("Tiles and shared memory", section "A complete kernel":
 * each row is scaled by the inverse root of the mean of its squares plus a
 * small constant, then by a per-column gain):
 *
 *   inv(m) = 1 / sqrt((sum_k x(m,k)^2) / D + eps),   y(m,k) = x(m,k) * inv(m) * g(k)
 *
 * rows, D    0 <= rows, D < 2^31 (either 0: nothing is done).
 * X          device, x(m,k) at X[m*ldx + k], element type x_dtype.
 * x_dtype, y_dtype  element codes GEMM_OUT_F32, GEMM_OUT_BF16, GEMM_OUT_F16.
 * G          device, D FP32 gains.
 * eps        finite, >= 0.
 * Y          device, y(m,k) at Y[m*ldy + k], element type y_dtype; may be X
 *            itself when both element types have the same size and ldy ==
 *            ldx; any other overlap with X is refused (GEMM_ERR_INVALID_ARG).
 * X, Y and G must be 16-byte aligned and ldx, ldy keep rows 16-byte aligned
 * (GEMM_ERR_ALIGNMENT otherwise); D itself may be any size.
 *
 * Arithmetic is FP32: per row, 32 lanes each add the squares of their
 * elements in order and a 5-step butterfly combines them; the division,
 * the addition of eps, the square root and the reciprocal are correctly
 * rounded; y = (x * inv) * g, rounded to nearest even for a 16-bit output.
 * Asynchronous on `stream`; allocates nothing.
 */
GEMM_API int gemm_rms_norm(int64_t rows, int64_t D, const void *X, int64_t ldx, int x_dtype,
                  const float *G, float eps, void *Y, int64_t ldy, int y_dtype,
                  void *stream);

/*
 * The gate/up projection of a normalised activation, the two steps on
 * either side of it in one call:
 *
 *   Xn = rms_norm(X, G, eps)  (BF16, as gemm_rms_norm)
 *   Y  = silu(Xn.Wg) * (Xn.Wu)  (as gemm_gate_up_silu)
 *
 * ("Tiles and shared memory", section "A complete kernel" for the
 * normalisation; "TMA and Hopper WGMMA", sections "TMA and Hopper WGMMA" and
 * "Worked consumers and current validation" for the fused gate/up
 * projection.)  X (M, K) BF16 with pitch ldx; G K FP32 gains; Wg, Wu, Y as
 * gemm_gate_up_silu.  Xn (M, K) BF16 with pitch ldxn is caller-owned scratch
 * that also receives the normalised activation (it may be X itself, ldxn ==
 * ldx).  The tensor cores take 16-bit operands, so the normalised values are
 * rounded to BF16 (nearest even) before the contraction.  Two launches on
 * `stream`, the normalisation then the projection; every argument is
 * checked before either is enqueued.  Allocates nothing beyond what
 * gemm_gate_up_silu does.  With GB3_RMSNORM_SINGLE_LAUNCH = 1 (M > 128, K a
 * multiple of 8 and at most 22937) it is one cooperative launch instead: the
 * pair gate/up kernel normalises X into Xn, meets at a grid-wide barrier
 * (status site 10 if it times out) and then reads Xn; the same bits, but
 * measured slower on GB300 than the two launches, hence not the default.
 * Calls of this form on one device must not overlap (they share the
 * barrier's counters).
 */
GEMM_API int gemm_rmsnorm_gate_up_silu(int64_t M, int64_t N, int64_t K,
                              const void *X, int64_t ldx, const float *G, float eps,
                              const void *Wg, const void *Wu, int64_t ldw,
                              void *Xn, int64_t ldxn, void *Y, int64_t ldy, void *stream);

/*
 * Softmax attention, per head h = 0 .. heads-1:
 *
 *   O_h = softmax(scale * Q_h . K_h^T) . V_h        (softmax along each row, over Nk keys)
 *
 * ("Tiles and shared memory", section "How long a tile lives": the
 * flash-attention loop -- a query tile, a running maximum and a running sum
 * kept across the loop over key tiles, s = dot_t(q, k) per tile, acc / l at
 * the end.  The sketch shows no score scale; `scale` is a parameter, usually
 * 1/sqrt(D).)
 *
 * heads, Nq, Nk  sizes, 0 <= each < 2^31; heads == 0 or Nq == 0 does nothing;
 *            Nk == 0 is GEMM_ERR_INVALID_ARG (no keys to normalise over).
 * D          head dimension, 64 or 128 (else GEMM_ERR_INVALID_ARG).
 * scale      finite; the scores are s * scale.
 * Q          device, BF16: q(h,i,d) at Q[h*stride_q + i*ldq + d], ldq >= D.
 * K, V       device, BF16: k(h,j,d) at K[h*stride_k + j*ldk + d], V likewise.
 * O          device, FP32 or BF16 (out_dtype GEMM_OUT_F32 / GEMM_OUT_BF16):
 *            o(h,i,d) at O[h*stride_o + i*ldo + d]; written, never read.
 * Strides are in elements and keep heads apart when heads > 1; pointers are
 * 16-byte aligned and pitches / strides multiples of 16 bytes
 * (GEMM_ERR_ALIGNMENT otherwise).
 *
 * Arithmetic: scores accumulate in FP32 on the tensor cores (BF16 operands);
 * the softmax runs in FP32 in base 2 (exp2 of s * scale * log2 e minus a
 * running maximum that moves only when a key block's maximum exceeds it by
 * more than 8, so probabilities stay below 2^8); the probabilities enter the
 * second product as BF16 (nearest even) and the output accumulates over all
 * keys in FP32 on the tensor cores; the row sums, the rescaling of the
 * running output when the maximum moves and the final division are FP32; a
 * BF16 output is rounded to nearest even once.
 * One launch on `stream`; allocates nothing.
 */
GEMM_API int gemm_attention(int64_t heads, int64_t Nq, int64_t Nk, int64_t D, float scale,
                   const void *Q, int64_t ldq, int64_t stride_q,
                   const void *K, int64_t ldk, int64_t stride_k,
                   const void *V, int64_t ldv, int64_t stride_v,
                   void *O, int64_t ldo, int64_t stride_o, int out_dtype, void *stream);

/* Static, NUL-terminated description of a return code. */
GEMM_API const char *gemm_status_string(int status);

/*
 * Synchronizes `stream`, then returns and clears the device status word of
 * the current device (GEMM_OK if no kernel reported an error since the last
 * read).  The site of the failure (which pipeline wait) is written to
 * *site when site is not NULL: 1 producer waiting for a free stage, 2 MMA
 * waiting for a full stage, 3 MMA waiting for a free accumulator, 4 epilogue
 * waiting for a full accumulator, 5 a drain before exit, 6 the split-K kernel,
 * 7 gemm_selftest_wait_timeout, 8 epilogue waiting for a box of C, 10 the
 * grid-wide barrier of gemm_rmsnorm_gate_up_silu's single launch; with status
 * GEMM_ERR_CUDA, 9 a kernel launched with less dynamic shared memory than its
 * layout needs (it returned without touching shared memory).
 */
GEMM_API int gemm_get_device_status(void *stream, int *site);

/*
 * Allocates, on the current device, the split-K workspace that a gemm_bf16
 * call with M <= 128 and N <= max_N would need as planned (the GB3_* tuning
 * variables can force plans that need more), so that later calls (for
 * example inside CUDA-graph capture) allocate nothing.  Ordered on `stream`.
 */
GEMM_API int gemm_prepare(int64_t max_N, void *stream);

/*
 * gemm_bf16 for M <= 16 that allocates nothing.  The pages have no
 * counterpart of this call; it exists for callers that may not allocate
 * device memory while they run (a caching allocator or memory pool that must
 * stay in charge of every byte, a fixed memory budget, code that cannot
 * afford the device synchronization an allocation can cause).
 *
 * Same arguments, storage and results as gemm_bf16, restricted to
 * 1 <= M <= 16 (GEMM_ERR_INVALID_ARG otherwise; M == 0 or N == 0 still does
 * nothing).  The split-K partial sums live in one 8 MiB array compiled into
 * the library, which every GPU that loads the library holds until the process
 * exits.  A problem whose split * M * N * 4 bytes of partial sums plus its
 * arrival counters do not fit in that array is rejected with
 * GEMM_ERR_INVALID_ARG before anything is launched.
 *
 * The first call on each device looks the array's device address up (a
 * runtime query, not an allocation); make that first call before capturing
 * the stream into a CUDA graph.  Every call re-zeroes the counters on
 * `stream` before its kernel.  All calls on a device share the one array, so
 * calls that overlap on the GPU (different streams running at the same time)
 * race and must be serialized by the caller.
 */
GEMM_API int gemm_bf16_skinny_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                      const void *A, int64_t lda,
                                      const void *B, int64_t ldb,
                                      float beta, void *C, int64_t ldc,
                                      int out_dtype, void *stream);

/*
 * Self-test of failure detection: launches one thread that waits, through the
 * same bounded mbarrier wait the GEMM pipelines use, on a barrier nothing
 * arrives on.  After limit_ns (1 us .. 1 s) the wait gives up and records
 * GEMM_ERR_TIMEOUT in the device status word, so a following
 * gemm_get_device_status() returns GEMM_ERR_TIMEOUT.  Touches no memory of
 * the caller.  Returns GEMM_ERR_INVALID_ARG for a limit outside the range.
 */
GEMM_API int gemm_selftest_wait_timeout(int64_t limit_ns, void *stream);

/*
 * Self-test of a GEMM pipeline's abort path.  Launches the M <= 16 split-K
 * kernel (without a split: one CTA per 128 rows of B) on C = A . B^T with
 * BF16 operands and output, A row-major M x K (lda), B row-major N x K (ldb),
 * C row-major M x N (ldc), all device memory of the caller.  Its TMA producer
 * issues only `stall_after` k-blocks (64 columns of K each) and then stops,
 * as if the next copy never landed, so the MMA thread's wait for that stage
 * runs out after the pipelines' 2 s bound ("TMEM tiles and transfers",
 * section "Completion and validation": completion is observed through
 * mbarriers).  Each CTA then sets its abort flag, lets its epilogue warps
 * leave, waits (bounded) for the copies and MMAs it issued, frees its Tensor
 * Memory and returns; the device status word then reads GEMM_ERR_TIMEOUT at
 * wait site 2 (the MMA thread waiting for a full stage).  C is not written,
 * and no workspace or arrival counter is touched.  Takes about 2 s on the
 * GPU.  Returns GEMM_ERR_INVALID_ARG unless 1 <= M <= 16, N >= 1 and
 * 0 <= stall_after < ceil(K / 64); alignment as for gemm_bf16.
 */
GEMM_API int gemm_selftest_pipeline_timeout(int64_t M, int64_t N, int64_t K,
                                            const void *A, int64_t lda,
                                            const void *B, int64_t ldb,
                                            void *C, int64_t ldc,
                                            int stall_after, void *stream);

/* How a call would be executed (host-side planning only). */
typedef struct gemm_plan {
    int kernel;       /* 0 none, 1 single-CTA tiled GEMM, 2 skinny split-K, 3 scale only (K == 0),
                         4 single-CTA gate/up, 5 CTA-pair tiled GEMM, 6 CTA-pair gate/up,
                         7 small-M (128-row weight tiles; whole tiles per CTA, or
                           the k-blocks of all tiles divided evenly over the CTAs
                           with shared tiles summed in the workspace),
                         8 split-K gate/up (M <= 16: Wg and Wu rows streamed together) */
    int tile_m;       /* output rows per tile (tcgen05 M, or weight rows for kernels 2 and 7) */
    int tile_n;       /* output columns per tile (activation rows for kernels 2 and 7) */
    int tile_k;       /* K per pipeline stage */
    int stages;       /* shared-memory ring depth */
    int split_k;      /* K pieces of a split tile (skinny path; the CTA-pair kernel's
                         split last-wave tiles, or the most pieces of one tile under
                         its balanced division); most CTAs sharing one tile (small-M);
                         else 1 */
    int64_t tiles;    /* work units: whole tiles plus split pieces (and, for the
                         CTA-pair kernel, 64-column strips of last-wave tiles) */
    int grid;         /* CTAs launched (persistent: at most one per SM) */
    int smem_bytes;   /* dynamic shared memory per CTA */
    int launches;     /* kernels one call launches */
    int64_t stage_tx_bytes; /* bytes one pipeline stage receives through TMA */
} gemm_plan;

/*
 * Plan of gemm_bf16(M, N, K, ...) on a device with num_sms SMs (num_sms <= 0:
 * query the current device, including how many CTA pairs fit at once).  Pure
 * host logic otherwise; returns GEMM_INVALID_ARG for invalid sizes or dtype.
 * M > 128 runs on CTA pairs (256-row tiles) with the tile width that needs the
 * fewest waves; the environment variable GB3_GEMM_PAIR_TILE_N (256 or 224)
 * forces one width, for tuning and tests.  The tiles of a partial last wave
 * are cut into 2 K pieces when that shortens the wave; where K is too short
 * for that (pieces under 24 k-blocks) and four times the wave's 256-wide
 * tiles fit on the pairs, they run as 256 x 64 strips over all of K instead
 * (not with row statistics; `tiles` then counts the strips as units;
 * GB3_GEMM_STRIPS = 0 turns strips off, 1 takes them wherever the wave fits,
 * even in place of a K split); GB3_GEMM_BALANCED = 1
 * instead gives every CTA pair one contiguous range of all tiles' k-blocks
 * (measured slower on GB300, so off by default; split_k then reports the most
 * pieces of a tile and `tiles` the units), and GB3_GEMM_BALANCED = 2 runs all
 * whole waves but the last as whole tiles first and divides the rest (also
 * slower; not with beta != 0, whose C ring keeps the default division).  The plan is that of beta == 0: with
 * beta != 0 the CTA-pair kernel runs one stage fewer (its shared memory holds
 * a deeper staging ring for C) unless GB3_GEMM_C_RING = 0.  M <= 128 runs on
 * the small-M kernel when its 128-row weight tiles (batch * ceil(N / 128))
 * number at most the SMs (16 < M) or half the SMs (M <= 16); otherwise the
 * single-CTA tiled kernel (16 < M) or the split-K kernel (M <= 16, K split by
 * a time model of the weight stream).  The small-M kernel divides the
 * k-blocks of all tiles over every SM when its tiles fill at most half of
 * them (or exceed them), unless that gives a CTA fewer than 8 k-blocks; else
 * one CTA per tile.  GB3_GEMM_SMALL_M = 1 or 0 forces or forbids the small-M
 * kernel; GB3_SMALL_M_STREAM_K = 1 or 0 forces the division or whole tiles.
 */
GEMM_API int gemm_bf16_plan(int64_t M, int64_t N, int64_t K, int out_dtype, int num_sms,
                   gemm_plan *plan);

/* Plan of gemm_batched(batch, M, N, K, ..., in_dtype, out_dtype, ...), as gemm_bf16_plan. */
GEMM_API int gemm_batched_plan(int64_t batch, int64_t M, int64_t N, int64_t K, int in_dtype,
                               int out_dtype, int num_sms, gemm_plan *plan);

/* Plan of gemm_row_stats(batch, M, N, K, ..., in_dtype, out_dtype, ...), as gemm_bf16_plan. */
GEMM_API int gemm_row_stats_plan(int64_t batch, int64_t M, int64_t N, int64_t K, int in_dtype,
                                 int out_dtype, int num_sms, gemm_plan *plan);

/* Plan of gemm_gate_up_silu(M, N, K, ...), as gemm_bf16_plan. */
GEMM_API int gemm_gate_up_plan(int64_t M, int64_t N, int64_t K, int num_sms, gemm_plan *plan);

/* ------------------------------------------------------------------------
 * Layout inspection (host only, no GPU needed): the encodings the kernels
 * compute, returned by the same functions the kernels call, so that they can
 * be checked field by field without running a kernel.
 * ------------------------------------------------------------------------ */

/*
 * Shared-memory matrix descriptor of an operand tile stored as TMA writes it
 * with the 128-byte swizzle ("TMA and Hopper WGMMA", section "The same storage
 * contract on both sides": 16-byte chunk j of 128-byte row r at chunk
 * j xor (r mod 8), eight-row groups 1024 bytes apart).  smem_address: the
 * tile's shared-memory byte address (1024-byte aligned for a whole tile).
 * mn_chunk_bytes == 0: a K-major tile (rows of 64 K elements); otherwise an
 * MN-major tile whose 64-element MN chunks are mn_chunk_bytes apart.
 */
GEMM_API uint64_t gemm_layout_smem_descriptor(uint32_t smem_address, uint32_t mn_chunk_bytes);

/*
 * Instruction descriptor of one tcgen05.mma kind::f16 with FP32 accumulation
 * and K-major operands: M rows, N columns (M in {64, 128, 256}, N a multiple
 * of 8 or 16), both operands in_dtype (GEMM_IN_BF16 or GEMM_IN_F16).
 */
GEMM_API uint32_t gemm_layout_instr_descriptor(int M, int N, int in_dtype);

/*
 * Byte offset, inside one 32-row epilogue staging box or one operand tile
 * with 128-byte rows and the 128-byte swizzle, of 16-byte chunk `chunk` of
 * row `row` ("TMA and Hopper WGMMA", section "The same storage contract on
 * both sides": element (r, k) of a 16-bit tile at 64 r + (k xor 8 (r mod 8))).
 */
GEMM_API uint32_t gemm_layout_swizzle128_offset(int row, int chunk);

/*
 * Tensor Memory address of (lane, column) in an allocation whose address is
 * `base` ("TMEM tiles and transfers", section "Storage units": lane in bits
 * 31:16, 32-bit column in bits 15:0).
 */
GEMM_API uint32_t gemm_layout_tmem_address(uint32_t base, int lane, int column);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_BF16_H */
