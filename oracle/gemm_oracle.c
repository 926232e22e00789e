/*
 * CPU oracle for the dense BF16 GEMM and the fused gate/up projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes (the plain definitions, no blocking, no reordering):
 *
 *   GEMM   C_ref(m,n) = alpha * sum_k a(m,k) * b(k,n) + beta * c(m,n)
 *          ("Tiles and shared memory", section "var and let": the tile
 *          epilogue writes alpha * acc + beta * c_old over the C slice, so
 *          C is read and then overwritten.)
 *          Operands are stored K-contiguous: a(m,k) at A[m*lda + k] and
 *          b(k,n) at B[n*ldb + k] ("TMA and Hopper WGMMA", section "The same
 *          storage contract on both sides": A(M,K) with K contiguous, B(K,N)
 *          with K as the inner axis).  C(m,n) sits at C[m*ldc + n].
 *
 *   gate/up  g(m,n) = sum_k x(m,k) wg(k,n),  u(m,n) = sum_k x(m,k) wu(k,n),
 *            y(m,n) = silu(g) * u,  silu(t) = t / (1 + exp(-t))
 *          ("TMA and Hopper WGMMA", sections "TMA and Hopper WGMMA" and
 *          "Worked consumers and current validation" name the fused gate/up
 *          projection without defining it; it is read as the SwiGLU form
 *          above, with no bias and no scaling.)
 *
 *   rms_norm  ss(m) = sum_k x(m,k)^2,  inv(m) = 1 / sqrt(ss(m)/D + eps),
 *             y(m,k) = x(m,k) * inv(m) * g(k)
 *          ("Tiles and shared memory", section "A complete kernel": a row
 *          normalisation that sums the squares of each row, scales the row by
 *          the inverse root of their mean plus a small constant, then by a
 *          per-column gain).  The normalised activation then feeds the gate/up
 *          projection in oracle_gate_up_entries_f64.
 *
 *   attention  s(i,j) = sum_d q(i,d) k(j,d),  t = scale * s,
 *              o(i,d) = sum_j exp(t(i,j) - max_j t(i,j)) v(j,d) / sum_j exp(...)
 *          ("Tiles and shared memory", section "How long a tile lives": the
 *          flash-attention loop keeps a query tile, a running maximum m and a
 *          running sum l across the key loop, takes s = dot_t(q, k) per key
 *          tile and finishes with acc / l -- the online form of the softmax
 *          attention above, which the oracle evaluates directly, in one pass
 *          over all keys).
 *
 * Operands are BF16 or, for the FP16 variant, IEEE binary16 ("TMEM tiles and
 * transfers", section "Representation and windows": FP16 values packed with
 * pack(Float16, f)); the GEMM functions take the operand type as in_f16.
 *
 * Precision: every 16-bit input is widened exactly to double and every sum is
 * one running double accumulator over k = 0 .. K-1 in order.  Beside each
 * result the oracle also returns sum_k |a(m,k) b(k,n)|, which the tests use
 * to scale the rounding tolerance of the FP32-accumulating GPU path.
 *
 * Rows are spread over OpenMP threads; each output is still computed by one
 * thread in the order above, so the result does not depend on the thread
 * count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* A BF16 value is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE binary16: sign, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_to_double(uint16_t bits)
{
    int sign = bits >> 15, e = (bits >> 10) & 0x1F, m = bits & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* f16_to_double of every bit pattern, filled once (before any parallel
 * region) so the inner loops look values up instead of calling ldexp. */
static double f16_values[65536];
static int f16_values_ready;

static void prepare_decode(int in_f16)
{
    if (!in_f16 || f16_values_ready)
        return;
    for (uint32_t b = 0; b < 65536u; ++b)
        f16_values[b] = f16_to_double((uint16_t)b);
    f16_values_ready = 1;
}

/* Operand element decoding: in_f16 = 0 for BF16, 1 for FP16. */
static double to_double(uint16_t bits, int in_f16)
{
    return in_f16 ? f16_values[bits] : bf16_to_double(bits);
}

static void dot_16(int64_t K, const uint16_t *x, const uint16_t *y, int in_f16,
                   double *sum, double *abs_sum)
{
    double s = 0.0, a = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = to_double(x[k], in_f16) * to_double(y[k], in_f16);
        s += p;
        a += fabs(p);
    }
    *sum = s;
    *abs_sum = a;
}

static void dot_bf16(int64_t K, const uint16_t *x, const uint16_t *y,
                     double *sum, double *abs_sum)
{
    dot_16(K, x, y, 0, sum, abs_sum);
}

/* Exact value of one 16-bit pattern (for pinning the decoders). */
double oracle_decode16(uint16_t bits, int in_f16)
{
    return in_f16 ? f16_to_double(bits) : bf16_to_double(bits);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Entries (rows[i], cols[i]) of alpha*A*B + beta*C, i = 0 .. count-1.
 * C is read only when beta != 0 (it may be NULL otherwise).
 * out[i] receives the value, abs_out[i] (if not NULL) receives
 * sum_k |a(m,k) b(k,n)|.
 */
void oracle_gemm_entries(int64_t K, double alpha,
                         const uint16_t *A, int64_t lda,
                         const uint16_t *B, int64_t ldb,
                         double beta, const float *C, int64_t ldc,
                         int64_t count, const int64_t *rows, const int64_t *cols,
                         double *out, double *abs_out, int in_f16)
{
    prepare_decode(in_f16);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = rows[i], n = cols[i];
        double s, a;
        dot_16(K, A + m * lda, B + n * ldb, in_f16, &s, &a);
        double v = alpha * s;
        if (beta != 0.0)
            v += beta * (double)C[m * ldc + n];
        out[i] = v;
        if (abs_out)
            abs_out[i] = a;
    }
}

/*
 * Every entry of alpha*A*B + beta*C for an M x N result, written row-major
 * to out[m*N + n] (and abs_out likewise when not NULL).
 */
void oracle_gemm_full(int64_t M, int64_t N, int64_t K, double alpha,
                      const uint16_t *A, int64_t lda,
                      const uint16_t *B, int64_t ldb,
                      double beta, const float *C, int64_t ldc,
                      double *out, double *abs_out, int in_f16)
{
    prepare_decode(in_f16);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s, a;
            dot_16(K, A + m * lda, B + n * ldb, in_f16, &s, &a);
            double v = alpha * s;
            if (beta != 0.0)
                v += beta * (double)C[m * ldc + n];
            out[m * N + n] = v;
            if (abs_out)
                abs_out[m * N + n] = a;
        }
    }
}

/* silu(t) = t * sigmoid(t), written directly. */
double oracle_silu(double t)
{
    return t / (1.0 + exp(-t));
}

/*
 * Entries (rows[i], cols[i]) of the gate/up projection.  X(m,k) at
 * X[m*ldx + k]; Wg(k,n) at Wg[n*ldw + k] and Wu(k,n) at Wu[n*ldw + k]
 * (K-contiguous like B).  Outputs y, and the intermediates g, u with their
 * absolute sums; any of g, u, abs_g, abs_u may be NULL.
 */
void oracle_gate_up_entries(int64_t K,
                            const uint16_t *X, int64_t ldx,
                            const uint16_t *Wg, const uint16_t *Wu, int64_t ldw,
                            int64_t count, const int64_t *rows, const int64_t *cols,
                            double *y, double *g_out, double *u_out,
                            double *abs_g, double *abs_u)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = rows[i], n = cols[i];
        double g, ag, u, au;
        dot_bf16(K, X + m * ldx, Wg + n * ldw, &g, &ag);
        dot_bf16(K, X + m * ldx, Wu + n * ldw, &u, &au);
        y[i] = oracle_silu(g) * u;
        if (g_out) g_out[i] = g;
        if (u_out) u_out[i] = u;
        if (abs_g) abs_g[i] = ag;
        if (abs_u) abs_u[i] = au;
    }
}

/* One element of a normalisation input: x_kind 0 FP32, 1 BF16, 2 FP16. */
static double norm_input(const void *X, int64_t idx, int x_kind)
{
    if (x_kind == 0)
        return (double)((const float *)X)[idx];
    return x_kind == 1 ? bf16_to_double(((const uint16_t *)X)[idx])
                       : f16_values[((const uint16_t *)X)[idx]];
}

/*
 * Rows rows[i] of rms_norm(X) for i = 0 .. count-1: X(m,k) at X[m*ldx + k]
 * of kind x_kind, k = 0 .. D-1; G(k) FP32.  out[i*D + k] receives y and
 * inv_out[i] (if not NULL) receives inv.  The sum of squares is one running
 * double over k in order; sqrt and the divisions are double.
 */
void oracle_rms_norm_rows(int64_t D, const void *X, int64_t ldx, int x_kind,
                          const float *G, double eps, int64_t count,
                          const int64_t *rows, double *out, double *inv_out)
{
    prepare_decode(x_kind == 2);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < count; ++i) {
        const int64_t base = rows[i] * ldx;
        double ss = 0.0;
        for (int64_t k = 0; k < D; ++k) {
            double x = norm_input(X, base + k, x_kind);
            ss += x * x;
        }
        double inv = 1.0 / sqrt(ss / (double)D + eps);
        for (int64_t k = 0; k < D; ++k)
            out[i * D + k] = norm_input(X, base + k, x_kind) * inv * (double)G[k];
        if (inv_out)
            inv_out[i] = inv;
    }
}

/*
 * Entries of the gate/up projection whose activation is given in double:
 * row xrows[i] of Xd (at Xd[xrows[i]*ldx]) against weight column cols[i]
 * (Wg(k,n) at Wg[n*ldw + k], Wu likewise, BF16).  Same outputs as
 * oracle_gate_up_entries.
 */
void oracle_gate_up_entries_f64(int64_t K, const double *Xd, int64_t ldx,
                                const uint16_t *Wg, const uint16_t *Wu, int64_t ldw,
                                int64_t count, const int64_t *xrows, const int64_t *cols,
                                double *y, double *g_out, double *u_out,
                                double *abs_g, double *abs_u)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i) {
        const double *x = Xd + xrows[i] * ldx;
        const uint16_t *wg = Wg + cols[i] * ldw, *wu = Wu + cols[i] * ldw;
        double g = 0.0, ag = 0.0, u = 0.0, au = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double pg = x[k] * bf16_to_double(wg[k]);
            double pu = x[k] * bf16_to_double(wu[k]);
            g += pg;
            ag += fabs(pg);
            u += pu;
            au += fabs(pu);
        }
        y[i] = oracle_silu(g) * u;
        if (g_out) g_out[i] = g;
        if (u_out) u_out[i] = u;
        if (abs_g) abs_g[i] = ag;
        if (abs_u) abs_u[i] = au;
    }
}

/*
 * Attention rows.  For each i in 0..count-1, query row qi = qrow[i] of head
 * h = head[i]: Q(h,qi,d) at Q[(h*Nq + qi)*D + d], K(h,j,d) at K[(h*Nk + j)*D + d],
 * V likewise (all BF16, contiguous).  Writes o[i*D + d], abs_o[i*D + d] =
 * sum_j w_j |v(j,d)| (w the softmax weights) and smax[i] = scale *
 * max_j sum_d |q k| (both for the tolerance).  Scores are float64 dot
 * products in d order; the maximum is subtracted before exp (exact in real
 * arithmetic); sums run over j in order.  `work` holds Nk doubles per thread.
 */
void oracle_attention_rows(int64_t Nq, int64_t Nk, int64_t D, double scale,
                           const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                           int64_t count, const int64_t *head, const int64_t *qrow,
                           double *o, double *abs_o, double *smax)
{
#pragma omp parallel
    {
        double *t = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t i = 0; i < count; ++i) {
            const uint16_t *q = Q + (head[i] * Nq + qrow[i]) * D;
            const uint16_t *kb = K + head[i] * Nk * D, *vb = V + head[i] * Nk * D;
            double mx = -INFINITY, amax = 0.0;
            for (int64_t j = 0; j < Nk; ++j) {
                double sum = 0.0, a = 0.0;
                for (int64_t d = 0; d < D; ++d) {
                    double pr = bf16_to_double(q[d]) * bf16_to_double(kb[j * D + d]);
                    sum += pr;
                    a += fabs(pr);
                }
                t[j] = scale * sum;
                if (t[j] > mx) mx = t[j];
                if (a > amax) amax = a;
            }
            double l = 0.0;
            for (int64_t j = 0; j < Nk; ++j) {
                t[j] = exp(t[j] - mx);
                l += t[j];
            }
            for (int64_t d = 0; d < D; ++d) {
                double acc = 0.0, aa = 0.0;
                for (int64_t j = 0; j < Nk; ++j) {
                    double v = bf16_to_double(vb[j * D + d]);
                    acc += t[j] * v;
                    aa += t[j] * fabs(v);
                }
                o[i * D + d] = acc / l;
                abs_o[i * D + d] = aa / l;
            }
            smax[i] = fabs(scale) * amax;
        }
        free(t);
    }
}
