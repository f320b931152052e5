/*
 * Exact-attention oracle: plain, slow, fp64 CPU code.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
 * leg may load this library.  The product path (the CUDA library) never calls
 * it and shares no code with it.
 *
 * What it computes follows the pages of "exact_attention_online":
 *   - Standard attention, FlashAttention blog (NeurIPS 2022 summary),
 *     "From Online Softmax to FlashAttention": S = Q K^T (scaled), P = softmax(S),
 *     O = P V, with the score matrix materialised (here one full row of S at a
 *     time; softmax is defined row by row).
 *   - Safe softmax with three loops (max, sum, normalise), same page,
 *     "(Safe) Softmax".
 *   - Online softmax (running max m and running denominator d', d_N = d'_N),
 *     same page, "Online Softmax", after Milakov & Gimelshein; and the
 *     one-pass output recurrence o'_i with o_N = o'_N, same page,
 *     "FlashAttention" (the tiled version over blocks of b keys).
 *   - The deferred normalisation of FlashAttention-2 (rescale without dividing
 *     by l, divide once at the end), FlashAttention-2 review thread, author
 *     answer "How does the tweaks reduce non-matmul FLOPs".
 *   - The per-row log-sum-exp saved for the backward pass, FlashAttention-2
 *     review thread, review 2 ("Save a logsumexp ...").
 *   - Backward: dV = P^T dO (FlashAttention-2 review thread, public comment on
 *     page 3 of the paper), and the remaining gradients by the calculus of
 *     softmax attention (the pages cite Appendix B without reproducing it):
 *       dP = dO V^T, D_i = sum_c dO_ic O_ic, dS = P o (dP - D),
 *       dQ = scale * dS K, dK = scale * dS^T Q.
 *
 * Layout (plain reading; the pages give none): Q, O, dO, dQ are
 * [B][H][N][d] row-major; K, V, dK, dV are [B][Hkv][N][d]; LSE and D are
 * [B][H][N].  Query head h reads key/value head h / (H / Hkv).
 * LSE is the natural-log log-sum-exp of the scaled scores.
 *
 * Causal: key j is visible to query i iff j <= i (N_q == N_k, so top-left and
 * bottom-right alignment coincide).  A row with no visible key (not reachable
 * when N_q == N_k) gets O = 0 and LSE = -inf.
 *
 * ORACLE_MUTANT: compile-time switch used only by the mutation tests, which
 * build deliberately wrong copies of this file to show that the pins catch
 * each plausible mistake.  The default build has ORACLE_MUTANT == 0.
 *
 * Parity pins for every function here live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif
#define MUT(n) (ORACLE_MUTANT == (n))

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

static int check_shape(int B, int H, int Hkv, int N, int d) {
    if (B < 1 || H < 1 || Hkv < 1 || N < 1 || d < 1) return ORACLE_EINVAL;
    if (H % Hkv != 0) return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* Query head h reads key/value head h / (H / Hkv) (consecutive grouping). */
static int kv_head_of(int h, int H, int Hkv) {
    if (MUT(6)) return h % Hkv;
    return h / (H / Hkv);
}

/* Visibility of key j to query i.  window > 0 (with causal): a sliding
 * window of the window most recent keys, i - window < j <= i. */
static int visible(int i, int j, int causal, int window) {
    if (!causal) return 1;
    if (window > 0 && i - j >= (MUT(16) ? window + 1 : window)) return 0;
    if (MUT(2)) return j < i;
    return j <= i;
}

/* One row of scaled scores: s[j] = scale * <q_i, k_j>, -inf where masked. */
static void score_row(const double* qi, const double* kh, int N, int d, int i,
                      int causal, int window, double scale, double* s) {
    for (int j = 0; j < N; ++j) {
        if (!visible(i, j, causal, window)) { s[j] = -INFINITY; continue; }
        const double* kj = kh + (size_t)j * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += qi[c] * kj[c];
        s[j] = MUT(1) ? acc : scale * acc;
    }
}

/* Safe softmax, three loops over the row: max, sum of exp(s - m), normalise.
 * Writes p (may alias nothing) and returns the row statistics m and l. */
static void safe_softmax_row(const double* s, int N, double* p, double* m_out, double* l_out) {
    double m = -INFINITY;
    for (int j = 0; j < N; ++j) if (s[j] > m) m = s[j];              /* loop 1 */
    double l = 0.0;
    if (m != -INFINITY)
        for (int j = 0; j < N; ++j) l += exp(s[j] - m);              /* loop 2 */
    for (int j = 0; j < N; ++j)                                       /* loop 3 */
        p[j] = (m == -INFINITY) ? 0.0 : exp(s[j] - m) / (MUT(3) ? 1.0 : l);
    *m_out = m;
    *l_out = l;
}

/*
 * Standard attention forward for a set of rows.
 *   rows == NULL: every row (b, h, i), outputs written at their full-tensor
 *   positions.  Otherwise rows[r] is a flat row index (b*H + h)*N + i, and the
 *   outputs are written compactly: o[r*d ...], lse[r].
 *   p_out (optional, only with rows == NULL) receives P as [B][H][N][N].
 */
static int attn_fwd_impl(const double* q, const double* k, const double* v,
                         double* o, double* lse, double* p_out,
                         int B, int H, int Hkv, int N, int d, int causal, int window,
                         double scale, const long long* rows, long long n_rows) {
    int rc = check_shape(B, H, Hkv, N, d);
    if (rc) return rc;
    if (rows && p_out) return ORACLE_EINVAL;
    long long total = rows ? n_rows : (long long)B * H * N;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)N);
        double* p = (double*)malloc(sizeof(double) * (size_t)N);
        if (!s || !p) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long long r = 0; r < total; ++r) {
                long long flat = rows ? rows[r] : r;
                if (flat < 0 || flat >= (long long)B * H * N) {
#pragma omp atomic write
                    err = 2;
                    continue;
                }
                int i = (int)(flat % N);
                long long bh = flat / N;
                int h = (int)(bh % H), b = (int)(bh / H);
                int g = kv_head_of(h, H, Hkv);
                const double* qi = q + (size_t)flat * d;
                const double* kh = k + ((size_t)b * Hkv + g) * (size_t)N * d;
                const double* vh = v + ((size_t)b * Hkv + g) * (size_t)N * d;
                double m, l;
                score_row(qi, kh, N, d, i, causal, window, scale, s);
                safe_softmax_row(s, N, p, &m, &l);
                double* oi = o + (size_t)(rows ? r : flat) * d;
                for (int c = 0; c < d; ++c) oi[c] = 0.0;
                for (int j = 0; j < N; ++j) {
                    if (p[j] == 0.0) continue;
                    int jj = MUT(4) ? (j == 0 ? 0 : j - 1) : j;   /* mutant: off-by-one V row */
                    const double* vj = vh + (size_t)jj * d;
                    for (int c = 0; c < d; ++c) oi[c] += p[j] * vj[c];
                }
                lse[rows ? r : flat] =
                    (m == -INFINITY) ? -INFINITY : (MUT(5) ? log(l) : m + log(l));
                if (p_out) memcpy(p_out + (size_t)flat * N, p, sizeof(double) * (size_t)N);
            }
        }
        free(s);
        free(p);
    }
    if (err == 1) return ORACLE_ENOMEM;
    if (err == 2) return ORACLE_EINVAL;
    return ORACLE_OK;
}

int oracle_attn_fwd(const double* q, const double* k, const double* v,
                    double* o, double* lse, double* p_out,
                    int B, int H, int Hkv, int N, int d, int causal, double scale,
                    const long long* rows, long long n_rows) {
    return attn_fwd_impl(q, k, v, o, lse, p_out, B, H, Hkv, N, d, causal, 0, scale, rows, n_rows);
}

/* The same with a causal sliding window (window > 0: query i sees keys
 * i - window < j <= i, local attention). */
int oracle_attn_fwd_window(const double* q, const double* k, const double* v,
                           double* o, double* lse, int B, int H, int Hkv, int N, int d,
                           int window, double scale) {
    if (window < 1) return ORACLE_EINVAL;
    return attn_fwd_impl(q, k, v, o, lse, NULL, B, H, Hkv, N, d, 1, window, scale, NULL, 0);
}

/*
 * One-pass (online) attention forward, every row, visiting keys in blocks of
 * `block` (block == 1 is the element-by-element recurrence).
 *   deferred == 0: the normalised recurrence of the FlashAttention blog: after
 *     each block the running output o' is already divided by the running
 *     denominator d'; at the end o_N = o'_N.
 *   deferred == 1: the FlashAttention-2 form: rescale the unnormalised output
 *     by exp(m_old - m_new) only and divide by l once at the end.
 * Both are exact in exact arithmetic; they differ from the three-pass path only
 * by rounding.
 */
int oracle_attn_fwd_online(const double* q, const double* k, const double* v,
                           double* o, double* lse,
                           int B, int H, int Hkv, int N, int d, int causal, double scale,
                           int block, int deferred) {
    int rc = check_shape(B, H, Hkv, N, d);
    if (rc) return rc;
    if (block < 1) return ORACLE_EINVAL;
    long long total = (long long)B * H * N;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)block);
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s || !acc) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long long flat = 0; flat < total; ++flat) {
                int i = (int)(flat % N);
                long long bh = flat / N;
                int h = (int)(bh % H), b = (int)(bh / H);
                int g = kv_head_of(h, H, Hkv);
                const double* qi = q + (size_t)flat * d;
                const double* kh = k + ((size_t)b * Hkv + g) * (size_t)N * d;
                const double* vh = v + ((size_t)b * Hkv + g) * (size_t)N * d;
                double m = -INFINITY, l = 0.0;
                for (int c = 0; c < d; ++c) acc[c] = 0.0;
                for (int j0 = 0; j0 < N; j0 += block) {
                    int nb = (N - j0 < block) ? (N - j0) : block;
                    double mb = -INFINITY;
                    for (int t = 0; t < nb; ++t) {
                        int j = j0 + t;
                        if (!visible(i, j, causal, 0)) { s[t] = -INFINITY; continue; }
                        const double* kj = kh + (size_t)j * d;
                        double a = 0.0;
                        for (int c = 0; c < d; ++c) a += qi[c] * kj[c];
                        s[t] = scale * a;
                        if (s[t] > mb) mb = s[t];
                    }
                    double m_new = (mb > m) ? mb : m;
                    if (m_new == -INFINITY) continue;       /* nothing visible yet */
                    double alpha = exp(m - m_new);          /* exp(-inf) = 0 on first block */
                    double lb = 0.0;
                    for (int t = 0; t < nb; ++t) lb += exp(s[t] - m_new);
                    double l_new = l * alpha + lb;
                    if (deferred) {
                        for (int c = 0; c < d; ++c) acc[c] *= alpha;
                        for (int t = 0; t < nb; ++t) {
                            double e = exp(s[t] - m_new);
                            if (e == 0.0) continue;
                            const double* vj = vh + (size_t)(j0 + t) * d;
                            for (int c = 0; c < d; ++c) acc[c] += e * vj[c];
                        }
                    } else {
                        double keep = l * alpha / l_new;
                        for (int c = 0; c < d; ++c) acc[c] *= keep;
                        for (int t = 0; t < nb; ++t) {
                            double e = exp(s[t] - m_new) / l_new;
                            if (e == 0.0) continue;
                            const double* vj = vh + (size_t)(j0 + t) * d;
                            for (int c = 0; c < d; ++c) acc[c] += e * vj[c];
                        }
                    }
                    m = m_new;
                    l = l_new;
                }
                double* oi = o + (size_t)flat * d;
                if (m == -INFINITY) {
                    for (int c = 0; c < d; ++c) oi[c] = 0.0;
                    lse[flat] = -INFINITY;
                } else {
                    for (int c = 0; c < d; ++c) oi[c] = deferred ? acc[c] / l : acc[c];
                    lse[flat] = m + log(l);
                }
            }
        }
        free(s);
        free(acc);
    }
    return err ? ORACLE_ENOMEM : ORACLE_OK;
}

/*
 * Analytic backward of standard attention, from the definitions (no saved
 * statistics are trusted: P and O are recomputed here from Q, K, V).
 *   P_i = softmax(S_i), O_i = sum_j P_ij V_j
 *   dV_j = sum_{i, heads of the group} P_ij dO_i
 *   dP_ij = <dO_i, V_j>,  D_i = <dO_i, O_i>,  dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i = scale * sum_j dS_ij K_j
 *   dK_j = scale * sum_{i, heads of the group} dS_ij Q_i
 * D_out (optional) receives D as [B][H][N].
 * Work is split over query rows; dK and dV are summed from per-thread
 * accumulators (a plain reduction, no change to what is summed).
 */
static int attn_bwd_impl(const double* q, const double* k, const double* v, const double* dout,
                         double* dq, double* dk, double* dv, double* D_out,
                         int B, int H, int Hkv, int N, int d, int causal, int window,
                         double scale) {
    int rc = check_shape(B, H, Hkv, N, d);
    if (rc) return rc;
    size_t kv_elems = (size_t)B * Hkv * N * d;
    memset(dk, 0, sizeof(double) * kv_elems);
    memset(dv, 0, sizeof(double) * kv_elems);
    int G = H / Hkv;
    int err = 0;
    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < Hkv; ++g) {
            const double* kh = k + ((size_t)b * Hkv + g) * (size_t)N * d;
            const double* vh = v + ((size_t)b * Hkv + g) * (size_t)N * d;
            double* dkh = dk + ((size_t)b * Hkv + g) * (size_t)N * d;
            double* dvh = dv + ((size_t)b * Hkv + g) * (size_t)N * d;
#pragma omp parallel
            {
                double* s = (double*)malloc(sizeof(double) * (size_t)N);
                double* p = (double*)malloc(sizeof(double) * (size_t)N);
                double* ds = (double*)malloc(sizeof(double) * (size_t)N);
                double* oi = (double*)malloc(sizeof(double) * (size_t)d);
                double* ldk = (double*)calloc((size_t)N * d, sizeof(double));
                double* ldv = (double*)calloc((size_t)N * d, sizeof(double));
                int ok = s && p && ds && oi && ldk && ldv;
                if (!ok) {
#pragma omp atomic write
                    err = 1;
                } else {
#pragma omp for schedule(dynamic, 8)
                    for (long long r = 0; r < (long long)H * N; ++r) {
                        int h = (int)(r / N), i = (int)(r % N);
                        if (kv_head_of(h, H, Hkv) != g) continue;
                        size_t flat = ((size_t)b * H + h) * (size_t)N + i;
                        const double* qi = q + flat * d;
                        const double* doi = dout + flat * d;
                        double m, l;
                        score_row(qi, kh, N, d, i, causal, window, scale, s);
                        safe_softmax_row(s, N, p, &m, &l);
                        for (int c = 0; c < d; ++c) oi[c] = 0.0;
                        for (int j = 0; j < N; ++j) {
                            if (p[j] == 0.0) continue;
                            const double* vj = vh + (size_t)j * d;
                            for (int c = 0; c < d; ++c) oi[c] += p[j] * vj[c];
                        }
                        double Di = 0.0;
                        for (int c = 0; c < d; ++c) Di += doi[c] * oi[c];
                        if (D_out) D_out[flat] = Di;
                        for (int j = 0; j < N; ++j) {
                            if (p[j] == 0.0) { ds[j] = 0.0; continue; }
                            const double* vj = vh + (size_t)j * d;
                            double dp = 0.0;
                            for (int c = 0; c < d; ++c) dp += doi[c] * vj[c];
                            ds[j] = MUT(7) ? p[j] * dp : p[j] * (dp - Di);
                            if (MUT(8)) ds[j] = -ds[j];
                        }
                        double* dqi = dq + flat * d;
                        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
                        for (int j = 0; j < N; ++j) {
                            if (ds[j] == 0.0 && p[j] == 0.0) continue;
                            const double* kj = kh + (size_t)j * d;
                            for (int c = 0; c < d; ++c) dqi[c] += ds[j] * kj[c];
                            double* ldvj = ldv + (size_t)j * d;
                            double* ldkj = ldk + (size_t)j * d;
                            for (int c = 0; c < d; ++c) ldvj[c] += p[j] * doi[c];
                            for (int c = 0; c < d; ++c) ldkj[c] += ds[j] * qi[c];
                        }
                        for (int c = 0; c < d; ++c) dqi[c] *= scale;
                    }
#pragma omp critical
                    {
                        for (size_t e = 0; e < (size_t)N * d; ++e) {
                            dvh[e] += ldv[e];
                            dkh[e] += (MUT(9) ? 1.0 : scale) * ldk[e];
                        }
                    }
                }
                free(s); free(p); free(ds); free(oi); free(ldk); free(ldv);
            }
            if (err) return ORACLE_ENOMEM;
            (void)G;
        }
    }
    return ORACLE_OK;
}

int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv, double* D_out,
                    int B, int H, int Hkv, int N, int d, int causal, double scale) {
    return attn_bwd_impl(q, k, v, dout, dq, dk, dv, D_out, B, H, Hkv, N, d, causal, 0, scale);
}

/* Backward with a causal sliding window (see oracle_attn_fwd_window). */
int oracle_attn_bwd_window(const double* q, const double* k, const double* v, const double* dout,
                           double* dq, double* dk, double* dv, double* D_out,
                           int B, int H, int Hkv, int N, int d, int window, double scale) {
    if (window < 1) return ORACLE_EINVAL;
    return attn_bwd_impl(q, k, v, dout, dq, dk, dv, D_out, B, H, Hkv, N, d, 1, window, scale);
}

/* Number of OpenMP threads the oracle uses (reported beside its timings). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * ---------------------------------------------------------------------------
 * FP8 (e4m3) block quantisation, for the FP8 forward (FlashAttention-3 summary,
 * "block quantization" named in the abstract; the granularity is this
 * repository's reading: one scale per (batch, head, block of 128 rows) of each
 * of Q, K and V, scale = amax / 448).
 *
 * The e4m3 format, from its definition: 1 sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits; exponent field 0 holds subnormals m * 2^-9; no
 * infinities; the all-ones magnitude S.1111.111 is NaN, so the largest finite
 * magnitude is 1.110b * 2^8 = 448.  Encoding rounds to the nearest
 * representable value, ties to an even mantissa, and saturates magnitudes at
 * or beyond 448 to 448 (no NaN is produced from a finite input).
 * ---------------------------------------------------------------------------
 */

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double x) {
    if (MUT(10)) return floor(x + 0.5);            /* planted: ties away from zero */
    const double f = floor(x);
    const double r = x - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

unsigned char oracle_e4m3_encode(float x) {
    const unsigned char sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return (unsigned char)(sign | (MUT(11) ? 0x7F : 0x7E));  /* 11: no saturation */
    if (a < ldexp(1.0, -6)) {                      /* subnormal range: m * 2^-9 */
        const double m = round_half_even(a * (MUT(12) ? 256.0 : 512.0));   /* m = 8: smallest normal */
        return (unsigned char)(sign | (unsigned char)m);
    }
    int e = (int)floor(log2(a));
    /* guard against log2 landing one off at exact powers of two */
    if (ldexp(1.0, e) > a) --e;
    if (ldexp(1.0, e + 1) <= a) ++e;
    double m = round_half_even((a / ldexp(1.0, e) - 1.0) * 8.0);
    if (m == 8.0) { m = 0.0; ++e; }
    if (e > 8 || (e == 8 && m > 6.0)) return (unsigned char)(sign | 0x7E);
    return (unsigned char)(sign | (unsigned char)(((e + 7) << 3) | (int)m));
}

/* Value of a code; NaN for S.1111.111. */
double oracle_e4m3_decode(unsigned char c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = m * ldexp(1.0, -9);
    else v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return s ? -v : v;
}

/*
 * One block: x is rows x cols fp32 values (the bf16 inputs, exactly), row
 * stride ld.  amax = max |x|; scale = amax / 448 and inv = 448 / amax, both as
 * fp32 divisions (1 and 1 for an all-zero block); code = encode(fp32(x * inv)).
 * out is written with row stride ld_out; out_t (if given) receives the
 * transpose, [cols][rows] with row stride ld_t.
 */
int oracle_fp8_quant_block(const float* x, int rows, int cols, long long ld,
                           unsigned char* out, long long ld_out,
                           unsigned char* out_t, long long ld_t, float* scale) {
    if (!x || rows < 0 || cols <= 0 || !scale) return ORACLE_EINVAL;
    float amax = 0.0f;
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            const float a = fabsf(x[r * ld + c]);
            if (a > amax) amax = a;
        }
    volatile float num = MUT(13) ? 240.0f : 448.0f, den = amax;   /* fp32 divisions, as written */
    float inv = 1.0f, sc = 1.0f;
    if (amax > 0.0f) {
        inv = num / den;
        sc = den / num;
    }
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            volatile float y = x[r * ld + c] * inv;
            const unsigned char code = oracle_e4m3_encode(y);
            if (out) out[r * ld_out + c] = code;
            if (out_t) out_t[MUT(14) ? (r * ld_t + c) : (c * ld_t + r)] = code;
        }
    *scale = sc;
    return ORACLE_OK;
}

/*
 * Incoherent processing (FlashAttention-3 summary, abstract: FP8 "with block
 * quantization and incoherent processing"; the pages do not define it, and
 * this is the reading from its name): multiply Q and K by one random
 * orthogonal matrix M, Q -> Q M and K -> K M, which leaves every score
 * (Q M)(K M)^T = Q K^T unchanged while spreading a large entry of a row over
 * all d channels.  M = diag(signs) Hd / sqrt(d), Hd the Sylvester Hadamard
 * matrix, entry (c, j) = (-1)^popcount(c & j), d a power of two, signs +-1.
 * x and out are rows x d, row-major (out may not alias x).
 */
int oracle_hadamard_rotate(const double* x, int rows, int d, const signed char* signs,
                           double* out) {
    if (!x || !out || !signs || rows < 0 || d < 1 || (d & (d - 1)) != 0) return ORACLE_EINVAL;
    const double norm = MUT(18) ? 1.0 : 1.0 / sqrt((double)d);   /* 18: not normalised */
    for (int r = 0; r < rows; ++r) {
        const double* xr = x + (size_t)r * d;
        double* orow = out + (size_t)r * d;
        for (int j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) {
                const double h = (__builtin_popcount((unsigned)(c & j)) & 1) ? -1.0 : 1.0;
                acc += xr[c] * signs[c] * h;
            }
            orow[j] = acc * norm;
        }
    }
    return ORACLE_OK;
}

/*
 * Attention forward with fewer queries than keys, as in decoding with a cache
 * of Nk keys (the decoding setting of the FlashAttention blog and FA2 review
 * thread: few new query rows against a long key/value sequence).  q is
 * [B][H][Nq][d], k and v [B][Hkv][Nk][d], o [B][H][Nq][d], lse [B][H][Nq].
 * The queries are the last Nq positions of the sequence: under the causal
 * mask query r sees key j iff j <= r + (Nk - Nq) (bottom-right alignment,
 * which is the j <= i rule of oracle_attn_fwd when Nq == Nk).  Scores, the
 * three-loop safe softmax, O and LSE as in oracle_attn_fwd.
 */
int oracle_attn_fwd_decode(const double* q, const double* k, const double* v,
                           double* o, double* lse, int B, int H, int Hkv, int Nq, int Nk,
                           int d, int causal, double scale) {
    if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < Nq || d < 1 || H % Hkv) return ORACLE_EINVAL;
    const long long total = (long long)B * H * Nq;
    int err = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
        double* p = (double*)malloc(sizeof(double) * (size_t)Nk);
        if (!s || !p) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long long flat = 0; flat < total; ++flat) {
                const int r = (int)(flat % Nq);
                const long long bh = flat / Nq;
                const int h = (int)(bh % H), b = (int)(bh / H);
                const int g = kv_head_of(h, H, Hkv);
                const double* qr = q + (size_t)flat * d;
                const double* kh = k + ((size_t)b * Hkv + g) * (size_t)Nk * d;
                const double* vh = v + ((size_t)b * Hkv + g) * (size_t)Nk * d;
                const int last = MUT(15) ? r : r + (Nk - Nq);   /* 15: top-left alignment */
                for (int j = 0; j < Nk; ++j) {
                    if (causal && j > last) { s[j] = -INFINITY; continue; }
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += qr[c] * kh[(size_t)j * d + c];
                    s[j] = scale * acc;
                }
                double m, l;
                safe_softmax_row(s, Nk, p, &m, &l);
                double* orow = o + (size_t)flat * d;
                for (int c = 0; c < d; ++c) orow[c] = 0.0;
                for (int j = 0; j < Nk; ++j) {
                    if (p[j] == 0.0) continue;
                    for (int c = 0; c < d; ++c) orow[c] += p[j] * vh[(size_t)j * d + c];
                }
                lse[flat] = (m == -INFINITY) ? -INFINITY : m + log(l);
            }
        }
        free(s);
        free(p);
    }
    return err ? ORACLE_ENOMEM : ORACLE_OK;
}
