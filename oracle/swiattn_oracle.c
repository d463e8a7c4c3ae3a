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
 *  - decode: the cache already holds the new token, whose position is L-1;
 *  - training backward: the straight-through gate's forward value is the hard
 *    0/1, so dO reaches the selected branch only; the adaptive weight gamma
 *    is a coefficient of the regulariser and carries no gradient.
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

/* ---------------------------------------------------------------------------
 * Global anchors (SWA glossary, "详细解释", the platform note on 全局锚点重注入,
 * and "SWA 落地的四个常见坑", pitfall 1, fix 2): besides its window, every
 * query also attends the first S tokens of the sequence (S = 256 there),
 * which the window never evicts.  Attention stays causal, so a window row i
 * visits [0, min(S, i+1)) together with [max(0, i-W+1), i]; a routed row
 * still visits [0, i].  S = 0 is plain sliding-window attention.
 * ------------------------------------------------------------------------- */

/* Visited keys of row i, in ascending order, into idx (capacity >= i+1);
 * returns their count. */
static int64_t anchored_keys(int routed, int64_t i, int64_t W, int64_t S, int64_t *idx)
{
    int64_t n = 0;
    int64_t lo = routed ? 0 : (i - W + 1 > 0 ? i - W + 1 : 0);
    for (int64_t j = 0; j < lo && j < S; ++j) idx[n++] = j;
    for (int64_t j = lo; j <= i; ++j) idx[n++] = j;
    return n;
}

/* Softmax attention of one query over an explicit ascending key list. */
static void attend_list(const double *q, const double *k, const double *v, int64_t stride,
                        const int64_t *idx, int64_t n, int64_t d, double scale, double *s,
                        double *o, double *lse)
{
    double mx = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        const double *kj = k + idx[t] * stride;
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
        const double *vj = v + idx[t] * stride;
        for (int64_t c = 0; c < d; ++c) o[c] += p * vj[c];
    }
    for (int64_t c = 0; c < d; ++c) o[c] /= den;
    if (lse) *lse = mx + log(den);
}

/* Routed prefill with S global anchors; arguments as oracle_prefill. */
int oracle_prefill_anchored(const double *q, const double *k, const double *v,
                            const uint8_t *gate, int64_t B, int64_t N, int64_t Hq, int64_t Hkv,
                            int64_t d, int64_t W, int64_t S, double scale, double *o, double *lse)
{
    if (!shapes_ok(B, N, Hq, Hkv, d, W) || S < 0) return -1;
    int64_t rows = B * N * Hq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)N);
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t h = r % Hq, bi = r / Hq, i = bi % N, b = bi / N, kvh = h / (Hq / Hkv);
            int64_t n = anchored_keys(gate[b * N + i] != 0, i, W, S, idx);
            attend_list(q + r * d, k + (b * N * Hkv + kvh) * d, v + (b * N * Hkv + kvh) * d,
                        Hkv * d, idx, n, d, scale, s, o + r * d, lse ? lse + r : NULL);
        }
        free(s);
        free(idx);
    }
    return 0;
}

/* Decode with S global anchors; arguments as oracle_decode. */
int oracle_decode_anchored(const double *q, const double *kc, const double *vc,
                           const int32_t *seq_lens, const uint8_t *gate, int64_t B, int64_t Lmax,
                           int64_t Hq, int64_t Hkv, int64_t d, int64_t W, int64_t S, double scale,
                           double *o, double *lse)
{
    if (!shapes_ok(B, Lmax, Hq, Hkv, d, W) || S < 0) return -1;
    for (int64_t b = 0; b < B; ++b)
        if (seq_lens[b] < 1 || seq_lens[b] > Lmax) return -1;
    int64_t rows = B * Hq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Lmax);
        int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)Lmax);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t b = r / Hq, h = r % Hq, kvh = h / (Hq / Hkv);
            int64_t n = anchored_keys(gate[b] != 0, (int64_t)seq_lens[b] - 1, W, S, idx);
            attend_list(q + r * d, kc + (b * Lmax * Hkv + kvh) * d, vc + (b * Lmax * Hkv + kvh) * d,
                        Hkv * d, idx, n, d, scale, s, o + r * d, lse ? lse + r : NULL);
        }
        free(s);
        free(idx);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Training backward.
 *
 * Report section 2 (router design): the hard gate is formed with the
 * straight-through estimator, sigma = 1(sigmoid(R) > 0.5) + sigmoid(R)
 * - sg(sigmoid(R)).  Its forward value is exactly 0 or 1, so in
 * O = sigma*O_FULL + (1-sigma)*O_SWA the output gradient dO reaches only the
 * branch the gate selected; the gate itself receives dO.(O_FULL - O_SWA)
 * times the derivative of the soft sigmoid.  The adaptive weight gamma is a
 * coefficient of the regulariser (like NLL, it carries no gradient), so
 * dL_t/dR_t = gamma_t * sigmoid(R_t).
 * ------------------------------------------------------------------------- */

/* Gradient of one row's softmax attention over keys [lo, hi] (chain rule):
 *   p_j = softmax_j(scale <q, k_j>),  o = sum_j p_j v_j,  D = <dO, o>,
 *   dS_j = p_j (<dO, v_j> - D),
 *   dq  += scale sum_j dS_j k_j,  dk_j += scale dS_j q,  dv_j += p_j dO.
 * dq is (d) for this row, or NULL; dk/dv point at key 0 of this (b, kv head)
 * with stride kstride, or are NULL.  s, o are scratch (n and d doubles). */
static void attend_backward(const double *q, const double *k, const double *v, const double *dout,
                            int64_t kstride, int64_t lo, int64_t hi, int64_t d, double scale,
                            double *s, double *o, double *dq, double *dk, double *dv)
{
    int64_t n = hi - lo + 1;
    double lse;
    attend(q, k, v, kstride, kstride, lo, hi, d, scale, s, o, &lse);
    double D = 0.0;
    for (int64_t c = 0; c < d; ++c) D += dout[c] * o[c];
    for (int64_t t = 0; t < n; ++t) {
        int64_t j = lo + t;
        const double *kj = k + j * kstride, *vj = v + j * kstride;
        double p = exp(s[t] - lse);
        double dp = 0.0;
        for (int64_t c = 0; c < d; ++c) dp += dout[c] * vj[c];
        double ds = p * (dp - D);
        if (dq)
            for (int64_t c = 0; c < d; ++c) dq[c] += scale * ds * kj[c];
        if (dk)
            for (int64_t c = 0; c < d; ++c) dk[j * kstride + c] += scale * ds * q[c];
        if (dv)
            for (int64_t c = 0; c < d; ++c) dv[j * kstride + c] += p * dout[c];
    }
}

/* Backward of the routed prefill: dq [B,N,Hq,d], dk/dv [B,N,Hkv,d] (zeroed
 * here, then accumulated).  One thread per (b, kv head) owns every dk/dv row
 * it writes and the dq rows of that head group. */
int oracle_prefill_backward(const double *q, const double *k, const double *v,
                            const uint8_t *gate, const double *dout, int64_t B, int64_t N,
                            int64_t Hq, int64_t Hkv, int64_t d, int64_t W, double scale,
                            double *dq, double *dk, double *dv)
{
    if (!shapes_ok(B, N, Hq, Hkv, d, W)) return -1;
    memset(dq, 0, sizeof(double) * (size_t)(B * N * Hq * d));
    memset(dk, 0, sizeof(double) * (size_t)(B * N * Hkv * d));
    memset(dv, 0, sizeof(double) * (size_t)(B * N * Hkv * d));
    int64_t G = Hq / Hkv;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < B * Hkv; ++u) {
            int64_t b = u / Hkv, kvh = u % Hkv;
            const double *kb = k + (b * N * Hkv + kvh) * d;
            const double *vb = v + (b * N * Hkv + kvh) * d;
            double *dkb = dk + (b * N * Hkv + kvh) * d;
            double *dvb = dv + (b * N * Hkv + kvh) * d;
            for (int64_t h = kvh * G; h < (kvh + 1) * G; ++h)
                for (int64_t i = 0; i < N; ++i) {
                    int64_t lo, hi, r = (b * N + i) * Hq + h;
                    key_range(gate[b * N + i] != 0, i, W, &lo, &hi);
                    attend_backward(q + r * d, kb, vb, dout + r * d, Hkv * d, lo, hi, d, scale,
                                    s, o, dq + r * d, dkb, dvb);
                }
        }
        free(s);
        free(o);
    }
    return 0;
}

/* dq of selected rows: sel holds nsel triples (b, i, h); dq_sel [nsel, d]. */
int oracle_prefill_backward_rows(const double *q, const double *k, const double *v,
                                 const uint8_t *gate, const double *dout, int64_t B, int64_t N,
                                 int64_t Hq, int64_t Hkv, int64_t d, int64_t W, double scale,
                                 const int64_t *sel, int64_t nsel, double *dq_sel)
{
    if (!shapes_ok(B, N, Hq, Hkv, d, W) || nsel < 0) return -1;
    for (int64_t r = 0; r < nsel; ++r) {
        int64_t b = sel[3 * r], i = sel[3 * r + 1], h = sel[3 * r + 2];
        if (b < 0 || b >= B || i < 0 || i >= N || h < 0 || h >= Hq) return -1;
    }
    memset(dq_sel, 0, sizeof(double) * (size_t)(nsel * d));
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nsel; ++r) {
            int64_t b = sel[3 * r], i = sel[3 * r + 1], h = sel[3 * r + 2];
            int64_t kvh = h / (Hq / Hkv), lo, hi, row = (b * N + i) * Hq + h;
            key_range(gate[b * N + i] != 0, i, W, &lo, &hi);
            attend_backward(q + row * d, k + (b * N * Hkv + kvh) * d, v + (b * N * Hkv + kvh) * d,
                            dout + row * d, Hkv * d, lo, hi, d, scale, s, o, dq_sel + r * d, NULL,
                            NULL);
        }
        free(s);
        free(o);
    }
    return 0;
}

/* dk and dv of selected keys: sel holds nsel triples (b, j, kv head);
 * dk_sel/dv_sel [nsel, d].  Every row i >= j of the head group whose visited
 * range holds key j contributes scale*dS_ij*q_i and p_ij*dO_i; each such row's
 * softmax is recomputed in full. */
int oracle_prefill_backward_keys(const double *q, const double *k, const double *v,
                                 const uint8_t *gate, const double *dout, int64_t B, int64_t N,
                                 int64_t Hq, int64_t Hkv, int64_t d, int64_t W, double scale,
                                 const int64_t *sel, int64_t nsel, double *dk_sel,
                                 double *dv_sel)
{
    if (!shapes_ok(B, N, Hq, Hkv, d, W) || nsel < 0) return -1;
    for (int64_t r = 0; r < nsel; ++r) {
        int64_t b = sel[3 * r], j = sel[3 * r + 1], kvh = sel[3 * r + 2];
        if (b < 0 || b >= B || j < 0 || j >= N || kvh < 0 || kvh >= Hkv) return -1;
    }
    int64_t G = Hq / Hkv;
    for (int64_t r = 0; r < nsel; ++r) {
        int64_t b = sel[3 * r], j = sel[3 * r + 1], kvh = sel[3 * r + 2];
        const double *kb = k + (b * N * Hkv + kvh) * d;
        const double *vb = v + (b * N * Hkv + kvh) * d;
        const double *vj = vb + j * Hkv * d;
        double *dk_r = dk_sel + r * d, *dv_r = dv_sel + r * d;
        for (int64_t c = 0; c < d; ++c) dk_r[c] = dv_r[c] = 0.0;
#pragma omp parallel
        {
            double *s = (double *)malloc(sizeof(double) * (size_t)N);
            double *o = (double *)malloc(sizeof(double) * (size_t)d);
            double *pk = (double *)calloc((size_t)d, sizeof(double));
            double *pv = (double *)calloc((size_t)d, sizeof(double));
#pragma omp for schedule(dynamic, 4)
            for (int64_t u = 0; u < G * (N - j); ++u) {
                int64_t h = kvh * G + u % G, i = j + u / G, lo, hi, row = (b * N + i) * Hq + h;
                key_range(gate[b * N + i] != 0, i, W, &lo, &hi);
                if (j < lo) continue;
                double lse, D = 0.0, dp = 0.0;
                attend(q + row * d, kb, vb, Hkv * d, Hkv * d, lo, hi, d, scale, s, o, &lse);
                for (int64_t c = 0; c < d; ++c) D += dout[row * d + c] * o[c];
                for (int64_t c = 0; c < d; ++c) dp += dout[row * d + c] * vj[c];
                double p = exp(s[j - lo] - lse), ds = p * (dp - D);
                for (int64_t c = 0; c < d; ++c) {
                    pk[c] += scale * ds * q[row * d + c];
                    pv[c] += p * dout[row * d + c];
                }
            }
#pragma omp critical
            for (int64_t c = 0; c < d; ++c) {
                dk_r[c] += pk[c];
                dv_r[c] += pv[c];
            }
            free(s);
            free(o);
            free(pk);
            free(pv);
        }
    }
    return 0;
}

static double sigmoid(double x)
{
    return 1.0 / (1.0 + exp(-x));
}

/* Router backward through the straight-through gate and the regulariser.
 * Per token t (T tokens; per-token rows of HD = Hq*d attention outputs):
 *   d_logit_t = s_t (1 - s_t) * <dO_t, O_FULL,t - O_SWA,t>
 *             + d_reg_t * gamma_t * sigmoid(logit_t),     s_t = sigmoid(logit_t)
 * (d_reg may be NULL: no regulariser gradient).  Then through the linear
 * router logit_t = <h_t, w> + b:
 *   dh_t = d_logit_t w,   dw = sum_t d_logit_t h_t,   db = sum_t d_logit_t.
 * dh [T, D], dw [D], db [1] may each be NULL (h and w then unused). */
int oracle_route_backward(const double *logits, const double *o_full, const double *o_swa,
                          const double *dout, const double *gamma, const double *d_reg,
                          const double *h, const double *w, int64_t T, int64_t HD, int64_t D,
                          double *d_logits, double *dh, double *dw, double *db)
{
    if (T < 0 || HD <= 0 || ((dh || dw) && D <= 0)) return -1;
    for (int64_t t = 0; t < T; ++t) {
        double acc = 0.0;
        for (int64_t c = 0; c < HD; ++c)
            acc += dout[t * HD + c] * (o_full[t * HD + c] - o_swa[t * HD + c]);
        double sg = sigmoid(logits[t]);
        double g = sg * (1.0 - sg) * acc;
        if (d_reg) g += d_reg[t] * gamma[t] * sg;
        d_logits[t] = g;
    }
    if (dh)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t j = 0; j < D; ++j) dh[t * D + j] = d_logits[t] * w[j];
    if (dw)
        for (int64_t j = 0; j < D; ++j) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t) acc += d_logits[t] * h[t * D + j];
            dw[j] = acc;
        }
    if (db) {
        double acc = 0.0;
        for (int64_t t = 0; t < T; ++t) acc += d_logits[t];
        *db = acc;
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

/* Threads for the calls that follow (n >= 1; no effect without OpenMP).
 * Timing only: the results do not depend on the thread count. */
int oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
    return 0;
}
