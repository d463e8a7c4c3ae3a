/*
 * swiattn_oracle.c -- plain fp64 CPU oracle for the SwiAttn routed-attention
 * hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library: it is a direct, slow, readable restatement of the definitions on
 * the pages, evaluated in double precision on the exact input values.
 *
 * Sources (page title, section):
 *  - SwiAttn report (paper-daily.com retrieval report of 2026-03-31),
 *    section 2 "方法详解" (method details): the linear router R(H), the soft
 *    gate sigmoid(R(H)), the hard gate 1(sigmoid > 0.5), the two branches
 *    sharing one Q/K/V, the gated output O = sigma*O_FULL + (1-sigma)*O_SWA,
 *    the branch divergence ||o_FULL - o_SWA||_2^2, the adaptive weight
 *    gamma = gamma_base / (eps + NLL + alpha*||.||^2) and the regulariser
 *    L = gamma * softplus(R(h)); the KV cache shared by both branches at
 *    decode time.
 *  - "滑窗注意力 Sliding Window Attention 是什么" (weimeta.cn glossary),
 *    "详细解释" (definition): row i attends to keys [i-W+1, i], W keys
 *    including itself, clipped at 0 (the W=4, 7-token visualisation);
 *    "常见问题" (FAQ): W = N is the causal mask; GQA groups query heads on
 *    fewer KV heads.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - rows are 0-based; the window is clipped at key 0;
 *  - the gate compares the logit with 0 (sigmoid(x) > 0.5 <=> x > 0), strict;
 *  - R(h) = w.h + b, one scalar per token, shared by every head;
 *  - the softmax scale is a parameter (callers pass 1/sqrt(d));
 *  - GQA: query head h reads KV head h / (Hq/Hkv) (contiguous groups);
 *  - ||o_FULL - o_SWA||^2 sums over all Hq*d output elements of the token;
 *  - decode: the cache already holds the new token, whose position is L-1.
 *
 * Layouts (row-major, contiguous): q [B,N,Hq,d], k/v [B,N,Hkv,d],
 * decode caches [B,Lmax,Hkv,d], per-token arrays [B,N].
 * Every function returns 0, or -1 on an argument it cannot evaluate.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Visited key range of row i: full branch [0, i], window branch
 * [max(0, i-W+1), i].  The window bound is the glossary's definition. */
static void key_range(int routed, int64_t i, int64_t W, int64_t *lo, int64_t *hi)
{
    *hi = i;
    if (routed) {
        *lo = 0;
    } else {
        int64_t a = i - W + 1;
        *lo = a > 0 ? a : 0;
    }
}

/* Softmax attention of one query over keys [lo, hi] (inclusive):
 *   s_j = scale * <q, k_j>,  p_j = exp(s_j - max_j s_j),
 *   o   = sum_j p_j v_j / sum_j p_j,   lse = max + log(sum_j p_j).
 * kstride/vstride: distance in elements between consecutive keys.
 * s is scratch of at least hi-lo+1 doubles. */
static void attend(const double *q, const double *k, const double *v,
                   int64_t kstride, int64_t vstride, int64_t lo, int64_t hi,
                   int64_t d, double scale, double *s, double *o, double *lse)
{
    int64_t n = hi - lo + 1;
    double mx = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        const double *kj = k + (lo + t) * kstride;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += q[c] * kj[c];
        s[t] = scale * dot;
        if (s[t] > mx) mx = s[t];
    }
    double den = 0.0;
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        double p = exp(s[t] - mx);
        den += p;
        const double *vj = v + (lo + t) * vstride;
        for (int64_t c = 0; c < d; ++c) o[c] += p * vj[c];
    }
    for (int64_t c = 0; c < d; ++c) o[c] /= den;
    if (lse) *lse = mx + log(den);
}

static int shapes_ok(int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d, int64_t W)
{
    return B > 0 && N > 0 && Hq > 0 && Hkv > 0 && d > 0 && W > 0 && Hq % Hkv == 0;
}

/* Visited range of every row of a [B,N] gate array. */
int oracle_row_ranges(const uint8_t *gate, int64_t B, int64_t N, int64_t W,
                      int64_t *lo, int64_t *hi)
{
    if (B <= 0 || N <= 0 || W <= 0) return -1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t i = 0; i < N; ++i)
            key_range(gate[b * N + i] != 0, i, W, &lo[b * N + i], &hi[b * N + i]);
    return 0;
}

/* Router: logit_t = <h_t, w> + bias; gate_t = 1(sigmoid(logit_t) > 0.5),
 * evaluated as logit_t > 0 (report section 2, router design). */
int oracle_route(const double *h, const double *w, double bias, int64_t T, int64_t D,
                 double *logits, uint8_t *gate)
{
    if (T < 0 || D <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double acc = 0.0;
        for (int64_t j = 0; j < D; ++j) acc += h[t * D + j] * w[j];
        acc += bias;
        logits[t] = acc;
        gate[t] = acc > 0.0 ? 1 : 0;
    }
    return 0;
}

/* One output row (b, i, head) of the routed prefill: keys per key_range. */
static void prefill_row(const double *q, const double *k, const double *v, int routed,
                        int64_t b, int64_t i, int64_t h, int64_t N, int64_t Hq, int64_t Hkv,
                        int64_t d, int64_t W, double scale, double *s, double *o, double *lse)
{
    int64_t kvh = h / (Hq / Hkv);
    int64_t lo, hi;
    key_range(routed, i, W, &lo, &hi);
    const double *qr = q + ((b * N + i) * Hq + h) * d;
    const double *kb = k + (b * N * Hkv + kvh) * d;
    const double *vb = v + (b * N * Hkv + kvh) * d;
    attend(qr, kb, vb, Hkv * d, Hkv * d, lo, hi, d, scale, s, o, lse);
}

/* Routed prefill, every row: O = gate ? O_FULL : O_SWA (the gated sum with a
 * 0/1 gate selects one branch exactly).  o [B,N,Hq,d]; lse [B,N,Hq] or NULL. */
int oracle_prefill(const double *q, const double *k, const double *v, const uint8_t *gate,
                   int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d, int64_t W,
                   double scale, double *o, double *lse)
{
    if (!shapes_ok(B, N, Hq, Hkv, d, W)) return -1;
    int64_t rows = B * N * Hq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t h = r % Hq, bi = r / Hq, i = bi % N, b = bi / N;
            prefill_row(q, k, v, gate[b * N + i] != 0, b, i, h, N, Hq, Hkv, d, W, scale, s,
                        o + r * d, lse ? lse + r : NULL);
        }
        free(s);
    }
    return 0;
}

/* Routed prefill on selected rows only: sel holds nsel triples (b, i, h);
 * o_sel [nsel, d], lse_sel [nsel] or NULL.  Same arithmetic as above. */
int oracle_prefill_rows(const double *q, const double *k, const double *v, const uint8_t *gate,
                        int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d, int64_t W,
                        double scale, const int64_t *sel, int64_t nsel, double *o_sel,
                        double *lse_sel)
{
    if (!shapes_ok(B, N, Hq, Hkv, d, W) || nsel < 0) return -1;
    for (int64_t r = 0; r < nsel; ++r) {
        int64_t b = sel[3 * r], i = sel[3 * r + 1], h = sel[3 * r + 2];
        if (b < 0 || b >= B || i < 0 || i >= N || h < 0 || h >= Hq) return -1;
    }
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nsel; ++r) {
            int64_t b = sel[3 * r], i = sel[3 * r + 1], h = sel[3 * r + 2];
            prefill_row(q, k, v, gate[b * N + i] != 0, b, i, h, N, Hq, Hkv, d, W, scale, s,
                        o_sel + r * d, lse_sel ? lse_sel + r : NULL);
        }
        free(s);
    }
    return 0;
}

/* Decode: sequence b has L_b = seq_lens[b] cached tokens, the newest (its own)
 * at position L_b - 1.  A window token reads the last W entries, a routed token
 * the whole cache (report section 2: both branches share the KV cache).
 * q [B,Hq,d], caches [B,Lmax,Hkv,d], o [B,Hq,d]; lse [B,Hq] or NULL. */
int oracle_decode(const double *q, const double *kc, const double *vc, const int32_t *seq_lens,
                  const uint8_t *gate, int64_t B, int64_t Lmax, int64_t Hq, int64_t Hkv,
                  int64_t d, int64_t W, double scale, double *o, double *lse)
{
    if (!shapes_ok(B, Lmax, Hq, Hkv, d, W)) return -1;
    for (int64_t b = 0; b < B; ++b)
        if (seq_lens[b] < 1 || seq_lens[b] > Lmax) return -1;
    int64_t rows = B * Hq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Lmax);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t b = r / Hq, h = r % Hq, kvh = h / (Hq / Hkv);
            int64_t lo, hi;
            key_range(gate[b] != 0, (int64_t)seq_lens[b] - 1, W, &lo, &hi);
            const double *kb = kc + (b * Lmax * Hkv + kvh) * d;
            const double *vb = vc + (b * Lmax * Hkv + kvh) * d;
            attend(q + r * d, kb, vb, Hkv * d, Hkv * d, lo, hi, d, scale, s, o + r * d,
                   lse ? lse + r : NULL);
        }
        free(s);
    }
    return 0;
}

/* softplus(x) = log(1 + e^x), written in the overflow-free form
 * max(x, 0) + log1p(exp(-|x|)). */
double oracle_softplus(double x)
{
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* Adaptive regulariser of the report's section 2, per token:
 *   gamma_t = gamma_base / (eps + NLL_t + alpha * mse_t)
 *   L_t     = gamma_t * softplus(logit_t). */
int oracle_regulariser(const double *logits, const double *nll, const double *mse, int64_t n,
                       double gamma_base, double eps, double alpha, double *gamma, double *reg)
{
    if (n < 0) return -1;
    for (int64_t t = 0; t < n; ++t) {
        double g = gamma_base / (eps + nll[t] + alpha * mse[t]);
        gamma[t] = g;
        reg[t] = g * oracle_softplus(logits[t]);
    }
    return 0;
}

/* Both branches of one token (b, i) over every query head, then the divergence
 * mse = sum_{h,c} (o_FULL - o_SWA)^2 and the regulariser terms.
 * of, os: [Hq, d] outputs for this token. */
static void dual_token(const double *q, const double *k, const double *v, const double *logits,
                       const double *nll, int64_t b, int64_t i, int64_t N, int64_t Hq,
                       int64_t Hkv, int64_t d, int64_t W, double scale, double gamma_base,
                       double eps, double alpha, double *s, double *of, double *os,
                       double *mse, double *gamma, double *reg)
{
    double acc = 0.0;
    for (int64_t h = 0; h < Hq; ++h) {
        prefill_row(q, k, v, 1, b, i, h, N, Hq, Hkv, d, W, scale, s, of + h * d, NULL);
        prefill_row(q, k, v, 0, b, i, h, N, Hq, Hkv, d, W, scale, s, os + h * d, NULL);
        for (int64_t c = 0; c < d; ++c) {
            double e = of[h * d + c] - os[h * d + c];
            acc += e * e;
        }
    }
    *mse = acc;
    oracle_regulariser(logits + b * N + i, nll + b * N + i, mse, 1, gamma_base, eps, alpha,
                       gamma, reg);
}

/* Dual-branch training forward, every token.  o_full/o_swa [B,N,Hq,d];
 * mse/gamma/reg [B,N]. */
int oracle_dual(const double *q, const double *k, const double *v, const double *logits,
                const double *nll, int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d,
                int64_t W, double scale, double gamma_base, double eps, double alpha,
                double *o_full, double *o_swa, double *mse, double *gamma, double *reg)
{
    if (!shapes_ok(B, N, Hq, Hkv, d, W)) return -1;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < B * N; ++t) {
            int64_t b = t / N, i = t % N;
            dual_token(q, k, v, logits, nll, b, i, N, Hq, Hkv, d, W, scale, gamma_base, eps,
                       alpha, s, o_full + t * Hq * d, o_swa + t * Hq * d, mse + t, gamma + t,
                       reg + t);
        }
        free(s);
    }
    return 0;
}

/* Dual branch on selected tokens: sel holds nsel pairs (b, i); outputs
 * of_sel/os_sel [nsel,Hq,d], mse/gamma/reg [nsel]. */
int oracle_dual_rows(const double *q, const double *k, const double *v, const double *logits,
                     const double *nll, int64_t B, int64_t N, int64_t Hq, int64_t Hkv, int64_t d,
                     int64_t W, double scale, double gamma_base, double eps, double alpha,
                     const int64_t *sel, int64_t nsel, double *of_sel, double *os_sel,
                     double *mse, double *gamma, double *reg)
{
    if (!shapes_ok(B, N, Hq, Hkv, d, W) || nsel < 0) return -1;
    for (int64_t r = 0; r < nsel; ++r)
        if (sel[2 * r] < 0 || sel[2 * r] >= B || sel[2 * r + 1] < 0 || sel[2 * r + 1] >= N)
            return -1;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nsel; ++r)
            dual_token(q, k, v, logits, nll, sel[2 * r], sel[2 * r + 1], N, Hq, Hkv, d, W,
                       scale, gamma_base, eps, alpha, s, of_sel + r * Hq * d,
                       os_sel + r * Hq * d, mse + r, gamma + r, reg + r);
        free(s);
    }
    return 0;
}

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
