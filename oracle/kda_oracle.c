/*
 * kda_oracle.c -- plain, slow, fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant generator with the CUDA library; neither side
 * includes or links the other.
 *
 * What it computes (per head h of every packed sequence n), taken from
 *   "Kimi K3 Architecture: Scaling 2.8T Parameters for Long-Context
 *    Multimodal MoE" (dev.to), section "The Sequence Bottleneck: Hybrid KDA
 *    and Gated MLA" -- the display equation for the gate and the paragraph
 *    after it (g_min = -5, 16-token tiles, cumulative decay in (-80, 0)),
 * together with the state update named there ("adaptive Householder delta
 * updates and channel-wise forget gates", also on "Kimi K3 - Sparsity
 * Mechanics...", section 2 "Temporal Sequence (KDA)"):
 *
 *   g_t   = g_min * Sigmoid(exp(A_h) * z_t)            (per channel, dk of them)
 *   alpha = exp(g_t)
 *   S_t   = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t   = S_t^T q_t
 *
 * S is dk x dv, row i indexes the key channel, column j the value channel.
 * The arithmetic follows the definition step by step, per token:
 *   (1) S <- Diag(alpha) S                      (row i scaled by alpha_i)
 *   (2) a_j = sum_i k_i S_ij                    (k^T S)
 *   (3) S_ij <- S_ij + beta k_i (v_j - a_j)     (= S - beta k (k^T S) + beta k v^T)
 *   (4) o_j = sum_i S_ij q_i                    (S^T q)
 * Columns j never interact (steps 1-4 touch column j only through S[:, j]
 * and v_j), so work is split over (sequence, head, column block) without
 * changing a single floating-point operation of any column.
 *
 * Inputs are read in the exact storage precision the GPU consumed (fp32 or
 * bf16 bit patterns, or fp64) and widened to fp64 element by element.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

static double ld(const void *p, int dt, int64_t i) {
    if (dt == ORC_F64) return ((const double *)p)[i];
    if (dt == ORC_F32) return (double)((const float *)p)[i];
    {
        uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
}

/* widen a bf16/fp32 bit pattern to double (exposed for the tests) */
void kda_oracle_widen(const void *src, int dt, int64_t n, double *dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = ld(src, dt, i);
}

/* The gate: g = g_min * Sigmoid(exp(A) * z), Sigmoid(x) = 1 / (1 + exp(-x)). */
static double gate(double z, double A, double g_min) {
    double x = exp(A) * z;
    return g_min / (1.0 + exp(-x));
}

/*
 * The unbounded baseline the lower-bounded gate replaces ("Kimi K3
 * Architecture...", section "The Sequence Bottleneck": "replaces unbounded
 * negative Softplus decay"): g = -Softplus(exp(A) * z), Softplus(x) =
 * log(1 + exp(x)), read with the same argument as the bounded gate.
 */
static double gate_softplus(double z, double A) {
    double x = exp(A) * z;
    return x > 40.0 ? -x : -log1p(exp(x));
}

int kda_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Gate and in-tile cumulative decay.
 *   mode   0: the lower-bounded gate; 1: the Softplus baseline
 *   z      [T_tot, H, dk] in dtype dt
 *   A_log  [H] (the per-head A^h)
 *   g_out  [T_tot, H, dk] fp64 (may be NULL)
 *   G_out  [T_tot, H, dk] fp64 (may be NULL): inclusive cumulative sum of g
 *          restarted at every tile of `tile` tokens; tiles start at each
 *          sequence's first token, the last tile of a sequence may be short.
 * Returns the number of tile prefix sums that are not finite or lie outside
 * the closed interval [-80, 0] (the bound on 16-token tiles).
 */
int64_t kda_oracle_gate(const void *z, int dt, const double *A_log, const int64_t *cu_seqlens,
                        int32_t N, int32_t H, int32_t dk, int32_t tile, double g_min,
                        int mode, double *g_out, double *G_out) {
    int64_t bad = 0;
    for (int32_t n = 0; n < N; ++n) {
        for (int32_t h = 0; h < H; ++h) {
            for (int32_t c = 0; c < dk; ++c) {
                double run = 0.0;
                for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
                    if ((t - cu_seqlens[n]) % tile == 0) run = 0.0;
                    int64_t idx = (t * H + h) * (int64_t)dk + c;
                    double g = mode == 1 ? gate_softplus(ld(z, dt, idx), A_log[h])
                                         : gate(ld(z, dt, idx), A_log[h], g_min);
                    run += g;
                    if (g_out) g_out[idx] = g;
                    if (G_out) G_out[idx] = run;
                    if (!(isfinite(run) && run >= -80.0 && run <= 0.0)) ++bad;
                }
            }
        }
    }
    return bad;
}

/*
 * The sequential recurrence over packed variable-length sequences.
 *
 *   q, k, z     [T_tot, H, dk]   dtype dt
 *   v           [T_tot, H, dv]   dtype dt
 *   beta        [T_tot, H]       dtype dt
 *   A_log       [H]              fp64
 *   cu_seqlens  [N+1]            int64, cu[0] = 0, non-decreasing
 *   h0          [N, H, dk, dv]   fp64 or NULL (zeros)
 *   hT          [N, H, dk, dv]   fp64 or NULL (not written); may alias h0
 *   o           [T_tot, H, dv]   fp64 or NULL (not written)
 *   o_cmp       [T_tot, H, dv]   dtype cmp_dt or NULL: a result to score
 *   err         [N, H, ncb, 2]   fp64 or NULL: per (n, h, column block) the
 *                                sums of (o - o_cmp)^2 and o^2
 *   col_block   columns per work unit (ncb = ceil(dv / col_block))
 *   nthreads    <= 0: OpenMP default
 * Returns 0, or -1 on a bad argument.
 */
int kda_oracle_forward(const void *q, const void *k, const void *v, const void *z,
                       const void *beta, int dt, const double *A_log, const int64_t *cu_seqlens,
                       int32_t N, int32_t H, int32_t dk, int32_t dv, const double *h0, double *hT,
                       double *o, const void *o_cmp, int cmp_dt, double *err, int32_t col_block,
                       double g_min, int nthreads) {
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || col_block <= 0) return -1;
    const int32_t ncb = (dv + col_block - 1) / col_block;
    const int64_t units = (int64_t)N * H * ncb;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    (void)nthreads;
#endif

#pragma omp parallel num_threads(nthreads)
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)dk * col_block);
        double *alpha = (double *)malloc(sizeof(double) * (size_t)dk);
        double *kk = (double *)malloc(sizeof(double) * (size_t)dk);
        double *qq = (double *)malloc(sizeof(double) * (size_t)dk);
        double *a = (double *)malloc(sizeof(double) * (size_t)col_block);

#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int32_t n = (int32_t)(u / ((int64_t)H * ncb));
            const int32_t h = (int32_t)((u / ncb) % H);
            const int32_t j0 = (int32_t)(u % ncb) * col_block;
            const int32_t nj = (j0 + col_block <= dv) ? col_block : dv - j0;
            const int64_t sbase = ((int64_t)n * H + h) * (int64_t)dk * dv;
            double e2 = 0.0, r2 = 0.0;

            for (int32_t i = 0; i < dk; ++i)
                for (int32_t j = 0; j < nj; ++j)
                    S[(int64_t)i * nj + j] = h0 ? h0[sbase + (int64_t)i * dv + j0 + j] : 0.0;

            for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
                const int64_t kb = (t * H + h) * (int64_t)dk;
                const int64_t vb = (t * H + h) * (int64_t)dv;
                const double b = ld(beta, dt, t * H + h);
                for (int32_t i = 0; i < dk; ++i) {
                    alpha[i] = exp(gate(ld(z, dt, kb + i), A_log[h], g_min));
                    kk[i] = ld(k, dt, kb + i);
                    qq[i] = ld(q, dt, kb + i);
                }
                /* (1) Diag(alpha) S */
                for (int32_t i = 0; i < dk; ++i)
                    for (int32_t j = 0; j < nj; ++j) S[(int64_t)i * nj + j] *= alpha[i];
                /* (2) a = k^T S */
                for (int32_t j = 0; j < nj; ++j) {
                    double s = 0.0;
                    for (int32_t i = 0; i < dk; ++i) s += kk[i] * S[(int64_t)i * nj + j];
                    a[j] = s;
                }
                /* (3) S += beta k (v^T - a^T) */
                for (int32_t i = 0; i < dk; ++i)
                    for (int32_t j = 0; j < nj; ++j)
                        S[(int64_t)i * nj + j] += b * kk[i] * (ld(v, dt, vb + j0 + j) - a[j]);
                /* (4) o = S^T q */
                for (int32_t j = 0; j < nj; ++j) {
                    double s = 0.0;
                    for (int32_t i = 0; i < dk; ++i) s += S[(int64_t)i * nj + j] * qq[i];
                    if (o) o[vb + j0 + j] = s;
                    if (o_cmp) {
                        double d = s - ld(o_cmp, cmp_dt, vb + j0 + j);
                        e2 += d * d;
                        r2 += s * s;
                    }
                }
            }
            if (hT)
                for (int32_t i = 0; i < dk; ++i)
                    for (int32_t j = 0; j < nj; ++j)
                        hT[sbase + (int64_t)i * dv + j0 + j] = S[(int64_t)i * nj + j];
            if (err) {
                err[2 * u] = e2;
                err[2 * u + 1] = r2;
            }
        }
        free(S);
        free(alpha);
        free(kk);
        free(qq);
        free(a);
    }
    return 0;
}

/*
 * One decode step: every sequence n advances by exactly one token against
 * its resident state, in place.  This is the recurrence above with a single
 * token per sequence:
 *   q, k, z [N, H, dk], v [N, H, dv], beta [N, H] (dtype dt), state [N, H, dk, dv] fp64
 *   o [N, H, dv] fp64.
 */
int kda_oracle_decode(const void *q, const void *k, const void *v, const void *z,
                      const void *beta, int dt, const double *A_log, int32_t N, int32_t H,
                      int32_t dk, int32_t dv, double *state, double *o, double g_min,
                      int nthreads) {
    int64_t *cu = (int64_t *)malloc(sizeof(int64_t) * ((size_t)N + 1));
    if (!cu) return -1;
    for (int32_t n = 0; n <= N; ++n) cu[n] = n;
    int rc = kda_oracle_forward(q, k, v, z, beta, dt, A_log, cu, N, H, dk, dv, state, state, o,
                                NULL, 0, NULL, dv, g_min, nthreads);
    free(cu);
    return rc;
}
