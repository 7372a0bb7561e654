/*
 * oracle.c -- plain float64 CPU reference for the exact attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with
 * the CUDA library (no headers, helpers, tables or constants).
 *
 * What it computes is the textbook definition that the FlashAttention pages
 * say the fused kernels reproduce exactly ("FlashAttention -- one, two,
 * three!", section "Standard Attention"; comrad404 review, "Коротко" and FAQ):
 *
 *   s_ij  = scale * sum_c q_ic k_jc          for the visible keys j of row i
 *   m_i   = max_j s_ij
 *   l_i   = sum_j exp(s_ij - m_i)
 *   o_ic  = sum_j exp(s_ij - m_i) v_jc / l_i
 *   lse_i = m_i + ln l_i
 *
 * Queries i < Nq, keys j < Nk.  Visible keys: every j (no mask); j <= i
 * (causal mode 1, queries and keys aligned at their first positions, which is
 * the causal mask of self-attention when Nq = Nk); j <= i + Nk - Nq (causal
 * mode 2, aligned at their last positions: the queries are the last Nq of the
 * Nk positions).  The pages define the causal mask for self-attention only;
 * both modes are the readings this library takes for Nq != Nk.
 *
 * Each query row is independent, so rows are spread over POSIX threads; every
 * row is computed whole (no blocking, no online softmax).
 *
 * FP8 helpers follow the OCP 8-bit floating point specification for E4M3
 * (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, subnormals,
 * S.1111.111 is NaN, no infinities, largest finite 448), plus the two
 * pre-processing steps named in "Incoherent Processing for FP8 Accuracy"
 * (FlashAttention-3 podcast page) and "Метод", item 3 (comrad404 review):
 * a random-sign Hadamard rotation of Q and K, and block quantisation.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ---------------------------------------------------------------- attention */

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int64_t BH, Nq, Nk, d, R;   /* R = number of rows computed per head */
    const int64_t *rows;         /* NULL: rows 0..Nq-1 */
    int causal;                  /* 0 none, 1 aligned at the start, 2 at the end */
    double scale;
    int tid, nthreads;
    int status;
} att_job;

/* Keys 0 .. visible_keys(...) - 1 are the ones query row i sees. */
static int64_t visible_keys(int64_t i, int64_t Nq, int64_t Nk, int causal) {
    if (causal == 1) return i + 1 < Nk ? i + 1 : Nk;
    if (causal == 2) return i + 1 + (Nk - Nq);
    return Nk;
}

static void *att_worker(void *arg) {
    att_job *J = (att_job *)arg;
    double *w = (double *)malloc(sizeof(double) * (size_t)(J->Nk > 0 ? J->Nk : 1));
    if (!w) { J->status = 1; return NULL; }
    const int64_t total = J->BH * J->R;
    for (int64_t item = J->tid; item < total; item += J->nthreads) {
        const int64_t bh = item / J->R, r = item % J->R;
        const int64_t i = J->rows ? J->rows[r] : r;          /* query row index */
        const double *qi = J->q + (bh * J->Nq + i) * J->d;
        const double *kh = J->k + bh * J->Nk * J->d;
        const double *vh = J->v + bh * J->Nk * J->d;
        const int64_t nkeys = visible_keys(i, J->Nq, J->Nk, J->causal);
        double m = -INFINITY;
        for (int64_t j = 0; j < nkeys; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < J->d; ++c) dot += qi[c] * kh[j * J->d + c];
            w[j] = J->scale * dot;
            if (w[j] > m) m = w[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            w[j] = exp(w[j] - m);
            l += w[j];
        }
        double *oi = J->o + (bh * J->R + r) * J->d;
        for (int64_t c = 0; c < J->d; ++c) oi[c] = 0.0;
        for (int64_t j = 0; j < nkeys; ++j)
            for (int64_t c = 0; c < J->d; ++c) oi[c] += w[j] * vh[j * J->d + c];
        for (int64_t c = 0; c < J->d; ++c) oi[c] /= l;
        if (J->lse) J->lse[bh * J->R + r] = m + log(l);
    }
    free(w);
    return NULL;
}

/* q: [BH, Nq, d], k, v: [BH, Nk, d] float64.  o: [BH, R, d], lse: [BH, R]
 * (may be NULL), where R = nrows if rows != NULL (row indices in [0, Nq)),
 * else Nq.  causal: 0, 1 or 2 as above; a row with no visible key (Nk = 0, or
 * mode 2 with Nq > Nk) has no softmax and is rejected.  nthreads <= 0 uses
 * every online core.  Returns 0 on success (2: bad arguments); writes the
 * number of threads used to *threads_used (may be NULL). */
ORACLE_API int oracle_attention_qk(const double *q, const double *k, const double *v,
                                   double *o, double *lse, int64_t BH, int64_t Nq, int64_t Nk,
                                   int64_t d, int causal, double scale, const int64_t *rows,
                                   int64_t nrows, int nthreads, int *threads_used) {
    if (!q || !k || !v || !o || BH < 0 || Nq < 0 || Nk < 0 || d < 1) return 2;
    if (causal < 0 || causal > 2) return 2;
    if (Nq > 0 && (Nk == 0 || (causal == 2 && Nq > Nk))) return 2;
    const int64_t R = rows ? nrows : Nq;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= Nq) return 2;
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (BH * R < nthreads) nthreads = (int)(BH * R > 0 ? BH * R : 1);
    if (threads_used) *threads_used = nthreads;
    att_job *jobs = (att_job *)calloc((size_t)nthreads, sizeof(att_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 1; }
    for (int t = 0; t < nthreads; ++t) {
        att_job J = {q, k, v, o, lse, BH, Nq, Nk, d, R, rows, causal, scale, t, nthreads, 0};
        jobs[t] = J;
    }
    int st = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, att_worker, &jobs[t]) != 0) { jobs[t].status = 1; th[t] = 0; }
    att_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t) st |= jobs[t].status;
    free(jobs);
    free(th);
    return st;
}

/* Self-attention (Nq = Nk = N); causal: 0 none, nonzero the causal mask. */
ORACLE_API int oracle_attention(const double *q, const double *k, const double *v,
                                double *o, double *lse, int64_t BH, int64_t N, int64_t d,
                                int causal, double scale, const int64_t *rows, int64_t nrows,
                                int nthreads, int *threads_used) {
    return oracle_attention_qk(q, k, v, o, lse, BH, N, N, d, causal ? 1 : 0, scale, rows, nrows,
                               nthreads, threads_used);
}

/* ----------------------------------------------------------- backward */

/* Gradients of the attention above with respect to Q, K and V, given
 * dout = dL/dO for a scalar loss L (lse is treated as an auxiliary output:
 * no gradient flows through it).  The pages only say that the fused kernels
 * recompute the forward intermediates in the backward pass ("FlashAttention --
 * one, two, three!", section "FlashAttention v1."); the gradients themselves
 * are the chain rule through the definition, row by row:
 *
 *   p_ij  = softmax over the visible keys j of s_ij = scale q_i . k_j
 *   dv_j += p_ij g_i                                  (g_i = dout row i)
 *   dp_ij = g_i . v_j
 *   ds_ij = p_ij (dp_ij - sum_l p_il dp_il)          (softmax Jacobian)
 *   dq_i  = scale sum_j ds_ij k_j
 *   dk_j += scale ds_ij q_i
 *
 * Heads are spread over POSIX threads (each head's dk, dv are its own). */
typedef struct {
    const double *q, *k, *v, *g;
    double *dq, *dk, *dv;
    int64_t BH, Nq, Nk, d;
    int causal;
    double scale;
    int tid, nthreads;
    int status;
} bwd_job;

static void *bwd_worker(void *arg) {
    bwd_job *J = (bwd_job *)arg;
    double *p = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    double *dp = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    if (!p || !dp) { free(p); free(dp); J->status = 1; return NULL; }
    for (int64_t bh = J->tid; bh < J->BH; bh += J->nthreads) {
        const int64_t qoff = bh * J->Nq * J->d, koff = bh * J->Nk * J->d;
        const double *qh = J->q + qoff, *gh = J->g + qoff, *kh = J->k + koff, *vh = J->v + koff;
        double *dqh = J->dq + qoff, *dkh = J->dk + koff, *dvh = J->dv + koff;
        for (int64_t x = 0; x < J->Nk * J->d; ++x) { dkh[x] = 0.0; dvh[x] = 0.0; }
        for (int64_t i = 0; i < J->Nq; ++i) {
            const double *qi = qh + i * J->d, *gi = gh + i * J->d;
            const int64_t nkeys = visible_keys(i, J->Nq, J->Nk, J->causal);
            double m = -INFINITY;
            for (int64_t j = 0; j < nkeys; ++j) {
                const double *kj = kh + j * J->d;
                double sij = 0.0;
                for (int64_t c = 0; c < J->d; ++c) sij += qi[c] * kj[c];
                p[j] = J->scale * sij;
                if (p[j] > m) m = p[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j < nkeys; ++j) {
                p[j] = exp(p[j] - m);
                l += p[j];
            }
            double rowdot = 0.0;                             /* sum_l p_il dp_il */
            for (int64_t j = 0; j < nkeys; ++j) {
                p[j] /= l;
                double dot = 0.0;
                for (int64_t c = 0; c < J->d; ++c) dot += gi[c] * vh[j * J->d + c];
                dp[j] = dot;
                rowdot += p[j] * dp[j];
            }
            double *dqi = dqh + i * J->d;
            for (int64_t c = 0; c < J->d; ++c) dqi[c] = 0.0;
            for (int64_t j = 0; j < nkeys; ++j) {
                const double ds = p[j] * (dp[j] - rowdot);
                for (int64_t c = 0; c < J->d; ++c) {
                    dqi[c] += J->scale * ds * kh[j * J->d + c];
                    dkh[j * J->d + c] += J->scale * ds * qi[c];
                    dvh[j * J->d + c] += p[j] * gi[c];
                }
            }
        }
    }
    free(p);
    free(dp);
    return NULL;
}

/* q, dout, dq: [BH, Nq, d]; k, v, dk, dv: [BH, Nk, d]; float64.  causal as for
 * oracle_attention_qk (rows without a visible key are rejected).  Returns 0
 * on success (2: bad arguments). */
ORACLE_API int oracle_attention_bwd(const double *q, const double *k, const double *v,
                                    const double *dout, double *dq, double *dk, double *dv,
                                    int64_t BH, int64_t Nq, int64_t Nk, int64_t d, int causal,
                                    double scale, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || BH < 0 || Nq < 0 || Nk < 0 || d < 1) return 2;
    if (causal < 0 || causal > 2) return 2;
    if (Nq > 0 && (Nk == 0 || (causal == 2 && Nq > Nk))) return 2;
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (BH < nthreads) nthreads = (int)(BH > 0 ? BH : 1);
    bwd_job *jobs = (bwd_job *)calloc((size_t)nthreads, sizeof(bwd_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return 1; }
    for (int t = 0; t < nthreads; ++t) {
        bwd_job J = {q, k, v, dout, dq, dk, dv, BH, Nq, Nk, d, causal, scale, t, nthreads, 0};
        jobs[t] = J;
    }
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, bwd_worker, &jobs[t]) != 0) { jobs[t].status = 1; th[t] = 0; }
    bwd_worker(&jobs[0]);
    int st = 0;
    for (int t = 1; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t) st |= jobs[t].status;
    free(jobs);
    free(th);
    return st;
}

/* ------------------------------------------------------------ E4M3 codec */

ORACLE_API double oracle_e4m3_decode1(uint8_t code) {
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);          /* subnormal: 0.m * 2^-6 */
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);        /* normal: 1.m * 2^(e-7) */
    return sign ? -mag : mag;
}

/* Round to nearest, ties to even; finite values beyond 448 saturate to +-448;
 * NaN maps to 0x7F. */
ORACLE_API uint8_t oracle_e4m3_encode1(double x) {
    if (isnan(x)) return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                 /* subnormal grid: multiples of 2^-9 */
        double n = nearbyint(ldexp(a, 9));    /* ties to even (default FP mode) */
        return sign | (uint8_t)n;             /* n == 8 is the smallest normal, code 0x08 */
    }
    int ex;
    double fr = frexp(a, &ex);                /* a = fr * 2^ex, fr in [0.5, 1) */
    int e = ex - 1;                           /* a = (2 fr) * 2^e, 2 fr in [1, 2) */
    double mq = nearbyint((2.0 * fr - 1.0) * 8.0);
    if (mq == 8.0) { mq = 0.0; e += 1; }
    int biased = e + 7;
    if (biased > 15 || (biased == 15 && mq == 7.0)) return sign | 0x7E;
    return sign | (uint8_t)((biased << 3) | (int)mq);
}

ORACLE_API void oracle_e4m3_decode(const uint8_t *codes, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode1(codes[i]);
}

ORACLE_API void oracle_e4m3_encode(const double *x, uint8_t *codes, int64_t n) {
    for (int64_t i = 0; i < n; ++i) codes[i] = oracle_e4m3_encode1(x[i]);
}

/* ------------------------------------------------------- Hadamard rotation */

/* Sylvester Hadamard matrix entry: H[i][j] = (-1)^popcount(i & j). */
ORACLE_API int oracle_hadamard_entry(int64_t i, int64_t j) {
    return (__builtin_popcountll((unsigned long long)(i & j)) & 1) ? -1 : 1;
}

/* x: [BH, N, d] with d a power of two; signs: [H, d] (+-1), head h = bh % H.
 * out_row = (x_row * sigma_h) . H_d / sqrt(d)   (a dense product, O(d^2)). */
ORACLE_API int oracle_hadamard_rotate(const double *x, const int8_t *signs, double *out,
                                      int64_t BH, int64_t H, int64_t N, int64_t d) {
    if (d < 1 || (d & (d - 1)) || H < 1) return 2;
    const double inv = 1.0 / sqrt((double)d);
    for (int64_t bh = 0; bh < BH; ++bh) {
        const int8_t *sg = signs + (bh % H) * d;
        for (int64_t n = 0; n < N; ++n) {
            const double *xr = x + (bh * N + n) * d;
            double *yr = out + (bh * N + n) * d;
            for (int64_t j = 0; j < d; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < d; ++i)
                    acc += xr[i] * (double)sg[i] * (double)oracle_hadamard_entry(i, j);
                yr[j] = acc * inv;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------ rotary */

/* Rotary position embedding (RoFormer: each pair of features of the row at
 * position n is rotated by the angle n * theta_i), with the angles given as
 * tables: cos_t, sin_t [N, d/2] (float32, widened exactly), entry (n, i) for
 * pair i of row n.  Pair i is (2i, 2i+1) when interleaved != 0, else
 * (i, i + d/2).  A pair (a, b) becomes (a cos - b sin, a sin + b cos).
 * x, out: [BH, N, d] float64. */
ORACLE_API int oracle_rotary(const double *x, const float *cos_t, const float *sin_t, double *out,
                             int64_t BH, int64_t N, int64_t d, int interleaved) {
    if (d < 2 || (d & 1)) return 2;
    const int64_t half = d / 2;
    for (int64_t bh = 0; bh < BH; ++bh)
        for (int64_t n = 0; n < N; ++n) {
            const double *xr = x + (bh * N + n) * d;
            double *yr = out + (bh * N + n) * d;
            for (int64_t i = 0; i < half; ++i) {
                const int64_t ia = interleaved ? 2 * i : i;
                const int64_t ib = interleaved ? 2 * i + 1 : i + half;
                const double c = (double)cos_t[n * half + i], s = (double)sin_t[n * half + i];
                const double a = xr[ia], b = xr[ib];
                yr[ia] = a * c - b * s;
                yr[ib] = a * s + b * c;
            }
        }
    return 0;
}

/* ------------------------------------------------------ block quantisation */

/* x: [BH, N, d].  For every (bh, block of `block` rows) -- or for the whole
 * tensor when per_tensor != 0 -- the scale is s = amax / 448 in float32 (1 when
 * amax == 0) and each element is encoded as E4M3(x / s), the division and the
 * rounding decision taken in float32.  scales: [BH, ceil(N / block)] float32,
 * or a single float when per_tensor != 0. */
ORACLE_API int oracle_block_quantize(const double *x, uint8_t *codes, float *scales,
                                     int64_t BH, int64_t N, int64_t d, int64_t block,
                                     int per_tensor) {
    if (block < 1) return 2;
    const int64_t nblk = per_tensor ? 1 : (N + block - 1) / block;
    for (int64_t bh = 0; bh < (per_tensor ? 1 : BH); ++bh) {
        for (int64_t b = 0; b < nblk; ++b) {
            int64_t r0 = per_tensor ? 0 : bh * N + b * block;
            int64_t r1 = per_tensor ? BH * N : bh * N + ((b + 1) * block < N ? (b + 1) * block : N);
            float amax = 0.0f;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = 0; c < d; ++c) {
                    float a = fabsf((float)x[r * d + c]);
                    if (a > amax) amax = a;
                }
            float s = amax > 0.0f ? amax / 448.0f : 1.0f;
            if (per_tensor) scales[0] = s; else scales[bh * nblk + b] = s;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = 0; c < d; ++c)
                    codes[r * d + c] = oracle_e4m3_encode1((double)((float)x[r * d + c] / s));
        }
    }
    return 0;
}
