/*
 * sfi_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the Slow-Fast Inference (SFI)
 * decode-attention path computes. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path never does. It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Sources (pages about arXiv 2603.12038, "Slow-Fast Inference: Training-Free Inference
 * Acceleration via Within-Sentence Support Stability"):
 *   [Blog]    "Training-Free LLM Inference Acceleration by Exploiting Attention Stability
 *             Within Sentences", section "How SFI Works: Two Gears for Decoding".
 *   [Abs]     the arXiv abstract page of the paper.
 *   [Sum 2A]  gist.science technical summary, section 2 "Methodik", A "Das Slow-Fast
 *             Paradigma" (sparse state = sinks + recent window + selected memory).
 *   [Sum 2B]  same summary, 2 B "Der Training-Free Selector" (evidence, prior, closed-form
 *             fusion s = (1 - lambda) f + lambda r, Top-K).
 *   [Sum 2C]  same summary, 2 C "Trigger-Policy" (trigger token, T_max refresh).
 *   [Sum 3]   same summary, 3 "Systemdesign und Kernel-Optimierung" (packed sink+selected
 *             buffer, recent tokens from the KV cache).
 *
 * Readings of points the pages leave open are stated beside the function that takes
 * them. Arithmetic is double precision unless a step is defined in fp32 (the fused
 * score, whose fp32 recipe both sides evaluate identically). Compile with
 * -ffp-contract=off and without fast-math.
 *
 * Parity status: every function below is pinned by the CPU tests (closed forms,
 * library special cases, brute force); none is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bit pattern -> double. Exact: a bf16 value is the fp32 value with the low 16
 * mantissa bits zero, and every fp32 value is a double. */
double sfi_oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------------------ */
/* Attention                                                                              */
/* ------------------------------------------------------------------------------------ */

/*
 * Attention of G query heads over a set of key/value rows.
 *
 * [Blog] slow step = full dense attention over the whole KV cache; fast step = the same
 * attention restricted to the support kept from the last slow step. For each head h:
 *     z_hj = (q_h . k_j) / sqrt(D)
 *     p_hj = exp(z_hj - max_i z_hi) / sum_i exp(z_hi - max_i z_hi)
 *     o_h  = sum_j p_hj v_j
 * q: bf16 [G][D]; k, v: bf16 rows of D elements; rows[0..n_rows) index those rows (NULL
 * means rows 0..n_rows-1 in order). o: double [G][D]. p (optional): double [G][n_rows],
 * the weights in the order of `rows`. Returns 0, or -1 when n_rows < 1 or on allocation
 * failure.
 */
int sfi_oracle_attend(int G, int D, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const int32_t *rows, int n_rows, double *o, double *p)
{
    if (n_rows < 1)
        return -1;
    double *z = (double *)malloc(sizeof(double) * (size_t)n_rows);
    if (!z)
        return -1;
    const double scale = 1.0 / sqrt((double)D);
    for (int h = 0; h < G; ++h) {
        const uint16_t *qh = q + (size_t)h * D;
        double zmax = -INFINITY;
        for (int j = 0; j < n_rows; ++j) {
            const int64_t r = rows ? rows[j] : j;
            const uint16_t *kr = k + (size_t)r * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += sfi_oracle_bf16_to_double(qh[d]) * sfi_oracle_bf16_to_double(kr[d]);
            z[j] = dot * scale;
            if (z[j] > zmax)
                zmax = z[j];
        }
        double sum = 0.0;
        for (int j = 0; j < n_rows; ++j) {
            z[j] = exp(z[j] - zmax);
            sum += z[j];
        }
        double *oh = o + (size_t)h * D;
        for (int d = 0; d < D; ++d)
            oh[d] = 0.0;
        for (int j = 0; j < n_rows; ++j) {
            const double w = z[j] / sum;
            if (p)
                p[(size_t)h * n_rows + j] = w;
            const int64_t r = rows ? rows[j] : j;
            const uint16_t *vr = v + (size_t)r * D;
            for (int d = 0; d < D; ++d)
                oh[d] += w * sfi_oracle_bf16_to_double(vr[d]);
        }
    }
    free(z);
    return 0;
}

/*
 * The same attention computed in consecutive chunks of `split` rows, each chunk keeping
 * (m, l, acc) = (its max logit, sum exp(z - m), sum exp(z - m) v), merged at the end:
 *     M = max_c m_c,  o = sum_c exp(m_c - M) acc_c / sum_c exp(m_c - M) l_c.
 * This is the split-KV (flash-decoding) decomposition the GPU dense step uses, restated
 * so a test can check it equals the unsplit definition above.
 */
int sfi_oracle_attend_split(int G, int D, const uint16_t *q, const uint16_t *k,
                            const uint16_t *v, int n_rows, int split, double *o)
{
    if (n_rows < 1 || split < 1)
        return -1;
    const int n_chunks = (n_rows + split - 1) / split;
    double *m = (double *)malloc(sizeof(double) * (size_t)n_chunks);
    double *l = (double *)malloc(sizeof(double) * (size_t)n_chunks);
    double *acc = (double *)malloc(sizeof(double) * (size_t)n_chunks * D);
    if (!m || !l || !acc) {
        free(m); free(l); free(acc);
        return -1;
    }
    const double scale = 1.0 / sqrt((double)D);
    for (int h = 0; h < G; ++h) {
        const uint16_t *qh = q + (size_t)h * D;
        for (int c = 0; c < n_chunks; ++c) {
            const int j0 = c * split;
            const int j1 = j0 + split < n_rows ? j0 + split : n_rows;
            m[c] = -INFINITY;
            for (int j = j0; j < j1; ++j) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += sfi_oracle_bf16_to_double(qh[d]) *
                           sfi_oracle_bf16_to_double(k[(size_t)j * D + d]);
                if (dot * scale > m[c])
                    m[c] = dot * scale;
            }
            l[c] = 0.0;
            for (int d = 0; d < D; ++d)
                acc[(size_t)c * D + d] = 0.0;
            for (int j = j0; j < j1; ++j) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += sfi_oracle_bf16_to_double(qh[d]) *
                           sfi_oracle_bf16_to_double(k[(size_t)j * D + d]);
                const double e = exp(dot * scale - m[c]);
                l[c] += e;
                for (int d = 0; d < D; ++d)
                    acc[(size_t)c * D + d] += e * sfi_oracle_bf16_to_double(v[(size_t)j * D + d]);
            }
        }
        double M = -INFINITY;
        for (int c = 0; c < n_chunks; ++c)
            if (m[c] > M)
                M = m[c];
        double L = 0.0;
        for (int c = 0; c < n_chunks; ++c)
            L += exp(m[c] - M) * l[c];
        for (int d = 0; d < D; ++d) {
            double s = 0.0;
            for (int c = 0; c < n_chunks; ++c)
                s += exp(m[c] - M) * acc[(size_t)c * D + d];
            o[(size_t)h * D + d] = s / L;
        }
    }
    free(m); free(l); free(acc);
    return 0;
}

/*
 * Selector evidence ([Sum 2B], "Evidenz": the attention of the current slow step).
 * Reading: the evidence of a KV head is the attention probability its G query heads put
 * on each position, averaged over the group:  f_j = (1/G) sum_h p_hj.
 * p: [G][L]; f: [L]. Each f is a probability distribution over the L positions.
 */
void sfi_oracle_evidence(int G, int L, const double *p, double *f)
{
    for (int j = 0; j < L; ++j) {
        double s = 0.0;
        for (int h = 0; h < G; ++h)
            s += p[(size_t)h * L + j];
        f[j] = s / (double)G;
    }
}

/* ------------------------------------------------------------------------------------ */
/* Selector                                                                               */
/* ------------------------------------------------------------------------------------ */

/* Number of selection candidates C = [S, L - W): n_C = max(0, L - W - S). */
int sfi_oracle_num_candidates(int L, int S, int W)
{
    const int n = L - W - S;
    return n > 0 ? n : 0;
}

/*
 * Positional prior ([Sum 2B], "Prior": a light cache-based prior that counters the
 * over-concentration on very recent tokens). Reading: on the candidates j in [S, L-W),
 * with distance d_j = (L - W) - j in [1, n_C] to the recent window,
 *     r_j = min(1, d_j / tau) / Z,   Z = sum_{j in C} min(1, d_j / tau),
 * i.e. a ramp that damps the candidates just before the window and is flat beyond tau.
 * This returns Z by summing the definition (exact in double for power-of-two tau).
 */
double sfi_oracle_prior_norm(int n_cand, int tau)
{
    double z = 0.0;
    for (int d = 1; d <= n_cand; ++d)
        z += d < tau ? (double)d / (double)tau : 1.0;
    return z;
}

/*
 * Fused score ([Sum 2B], closed form of the fusion: s = (1 - lambda) f + lambda r).
 * The fp32 recipe, evaluated identically by the GPU:
 *     c1 = fl32(1 - lambda), c2 = fl32(lambda / Z) (both from double),
 *     rt_j = fl32(min(1, d_j * (1/tau))),
 *     s_j  = fl32( fl32(c1 * f_j) + fl32(c2 * rt_j) ).
 * f: fp32 evidence [L] (positions 0..L-1); s: fp32 [n_C] for candidates S .. L-W-1.
 * Returns n_C.
 */
int sfi_oracle_fused_scores(int L, int S, int W, int tau, double lambda, const float *f,
                            float *s)
{
    const int n = sfi_oracle_num_candidates(L, S, W);
    if (n == 0)
        return 0;
    const float c1 = (float)(1.0 - lambda);
    const float c2 = (float)(lambda / sfi_oracle_prior_norm(n, tau));
    const float inv_tau = (float)(1.0 / (double)tau);
    for (int i = 0; i < n; ++i) {
        const int j = S + i;
        const int d = (L - W) - j;
        float rt = (float)d * inv_tau;
        if (rt > 1.0f)
            rt = 1.0f;
        const float a = c1 * f[j];
        const float b = c2 * rt;
        s[i] = a + b;
    }
    return n;
}

/*
 * log2 of an fp32 value in fp32, from the definition x = 2^e m, m in [1, 2):
 *     log2 x = e + (2/ln 2) * atanh(t),  t = (m - 1)/(m + 1) in [0, 1/3],
 * with atanh(t) = t + t^3/3 + ... + t^11/11 (truncation < 2e-7 relative). Every step is
 * an IEEE round-to-nearest fp32 operation in a fixed order, so any IEEE host computes the
 * same bits. log2(0) = -inf; negative or NaN input gives NaN.
 */
float sfi_oracle_log2f(float x)
{
    if (x != x || x < 0.0f)
        return NAN;
    if (x == 0.0f)
        return -INFINITY;
    if (isinf(x))
        return INFINITY;
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    int e = (int)((u >> 23) & 0xFFu);
    if (e == 0) { /* subnormal: scale by 2^32 first */
        const float y = x * 4294967296.0f;
        memcpy(&u, &y, sizeof u);
        e = (int)((u >> 23) & 0xFFu) - 32;
    }
    e -= 127;
    const uint32_t mb = (u & 0x007FFFFFu) | 0x3F800000u;
    float m;
    memcpy(&m, &mb, sizeof m);
    const float t = (m - 1.0f) / (m + 1.0f);
    const float t2 = t * t;
    /* fl32(1/11), fl32(1/9), ..., fl32(2/ln 2) as exact literals */
    float s = 0x1.745d18p-4f;
    s = s * t2 + 0x1.c71c72p-4f;
    s = s * t2 + 0x1.24924ap-3f;
    s = s * t2 + 0x1.99999ap-3f;
    s = s * t2 + 0x1.555556p-2f;
    s = s * t2 + 1.0f;
    const float two_over_ln2 = 0x1.715476p+1f;
    return (float)e + two_over_ln2 * (t * s);
}

/*
 * Selector refinements ([Sum 2B]): the pages name them without formulas; the readings:
 *   prior with a key-norm term (it steers the selection away from keys of very large norm):
 *       rt_j = fl32(min(1, d_j/tau)) * g_j,  g_j = min(1, fl32(nu / ||k_j||))  (nu = 0: g = 1),
 *       still divided by the closed-form Z of the plain ramp (the term only removes mass);
 *   fusion: arithmetic s = fl32(fl32(c1 f) + fl32(c2 rt)) as sfi_oracle_fused_scores, or the
 *       geometric (log-linear) mixture of the reverse-KL objective, scored in the log domain:
 *       s = fl32(fl32(fl32(1 - lambda) log2 f) + fl32(fl32(lambda) log2 fl32(c2 rt / lambda)))
 *       (lambda = 0: s = log2 f; the log score ranks like the geometric mixture);
 *   Soft-NMS within a head (nearby candidates whose scores are close damp one another): a
 *       candidate is scaled by gamma, s' = fl32(gamma s), when a candidate neighbour at
 *       distance 1..radius scores strictly higher and, with a similarity limit delta > 0,
 *       at most delta higher: fl32(s_i - s_j) <= delta (delta = 0: no limit);
 *   cross-head exclusivity: with T_j = s'_0j + ... + s'_(H-1)j summed in head order,
 *       s''_hj = fl32(s'_hj - fl32(mu' fl32(T_j - s'_hj))),  mu' = fl32(mu / (H - 1)).
 * f: fp32 [H][L] evidence of the H kv heads of one (layer, sequence); knorm: fp32 [H][L]
 * key norms or NULL; out: fp32 [H][n_C] refined scores of candidates S .. L-W-1.
 * Returns n_C.
 */
/* Soft-NMS: does the neighbour's score w suppress the score v? Strictly higher, and when
 * delta > 0 similar as well (the difference, rounded to fp32, at most delta). */
static int nms_neighbour_suppresses(float w, float v, float delta)
{
    if (!(w > v))
        return 0;
    return delta <= 0.0f || w - v <= delta;
}

int sfi_oracle_refine_scores(int H, int L, int S, int W, int tau, double lambda, int geometric,
                             float nu, const float *knorm, int radius, float gamma, float delta,
                             float mu, const float *f, float *out)
{
    const int n = sfi_oracle_num_candidates(L, S, W);
    if (n == 0)
        return 0;
    const double Z = sfi_oracle_prior_norm(n, tau);
    const float c1 = (float)(1.0 - lambda);
    const float c2 = (float)(lambda / Z);
    const float inv_tau = (float)(1.0 / (double)tau);
    const float lam_f = (float)lambda;
    float *s = (float *)malloc(sizeof(float) * (size_t)H * n);
    if (!s)
        return -1;
    for (int h = 0; h < H; ++h)
        for (int i = 0; i < n; ++i) {
            const int j = S + i;
            const int d = (L - W) - j;
            float rt = (float)d * inv_tau;
            if (rt > 1.0f)
                rt = 1.0f;
            if (nu > 0.0f && knorm) {
                float g = nu / knorm[(size_t)h * L + j];
                if (g > 1.0f)
                    g = 1.0f;
                rt = rt * g;
            }
            const float fj = f[(size_t)h * L + j];
            float v;
            if (!geometric) {
                const float a = c1 * fj;
                const float b = c2 * rt;
                v = a + b;
            } else {
                const float a = c1 * sfi_oracle_log2f(fj);
                float b = 0.0f;
                if (lambda > 0.0) {
                    const float r = (c2 * rt) / lam_f;
                    b = lam_f * sfi_oracle_log2f(r);
                }
                v = lambda < 1.0 ? a + b : b;
            }
            s[(size_t)h * n + i] = v;
        }
    /* Soft-NMS within each head */
    for (int h = 0; h < H; ++h) {
        const float *sh = s + (size_t)h * n;
        for (int i = 0; i < n; ++i) {
            const float v = sh[i];
            int suppressed = 0;
            for (int k = 1; k <= radius; ++k) {
                if (i - k >= 0 && nms_neighbour_suppresses(sh[i - k], v, delta))
                    suppressed = 1;
                if (i + k < n && nms_neighbour_suppresses(sh[i + k], v, delta))
                    suppressed = 1;
            }
            out[(size_t)h * n + i] = suppressed ? gamma * v : v;
        }
    }
    /* cross-head exclusivity */
    if (mu != 0.0f && H > 1) {
        const float mu1 = (float)((double)mu / (double)(H - 1));
        for (int i = 0; i < n; ++i) {
            float T = 0.0f;
            for (int h = 0; h < H; ++h)
                T = T + out[(size_t)h * n + i];
            for (int h = 0; h < H; ++h) {
                const float v = out[(size_t)h * n + i];
                const float others = T - v;
                const float pen = mu1 * others;
                s[(size_t)h * n + i] = v - pen;
            }
        }
        memcpy(out, s, sizeof(float) * (size_t)H * n);
    }
    free(s);
    return n;
}

/* Key norms ||k_j||_2 of bf16 rows: squares summed in fp32 in dimension order, then the
 * correctly rounded fp32 square root. k: [L][D]; out: [L]. */
void sfi_oracle_key_norms(int L, int D, const uint16_t *k, float *out)
{
    for (int j = 0; j < L; ++j) {
        float acc = 0.0f;
        for (int d = 0; d < D; ++d) {
            const float x = (float)sfi_oracle_bf16_to_double(k[(size_t)j * D + d]);
            const float sq = x * x;
            acc = acc + sq;
        }
        out[j] = sqrtf(acc);
    }
}

/* IEEE total order of an fp32 value as an unsigned key (NaN lowest): used so that the
 * order of scores is a total order on bit patterns. */
static uint32_t order_key(float x)
{
    if (x != x)
        return 0u;
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

typedef struct {
    uint32_t key;
    int32_t idx;
} keyed_t;

static int cmp_desc_key_asc_idx(const void *a, const void *b)
{
    const keyed_t *x = (const keyed_t *)a, *y = (const keyed_t *)b;
    if (x->key != y->key)
        return x->key > y->key ? -1 : 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

static int cmp_int32(const void *a, const void *b)
{
    const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * Top-K discretisation ([Sum 2B], final Top-K over the refined scores).
 * Order: i before j iff s_i > s_j, or s_i == s_j (same bits) and i < j -- ties go to the
 * lower index, so the chosen set is unique. Returns min(K, n) and writes the chosen
 * indices in ascending order to out.
 */
int sfi_oracle_topk(int n, const float *s, int K, int32_t *out)
{
    const int cnt = K < n ? K : n;
    if (cnt <= 0)
        return 0;
    keyed_t *a = (keyed_t *)malloc(sizeof(keyed_t) * (size_t)n);
    if (!a)
        return -1;
    for (int i = 0; i < n; ++i) {
        a[i].key = order_key(s[i]);
        a[i].idx = i;
    }
    qsort(a, (size_t)n, sizeof(keyed_t), cmp_desc_key_asc_idx);
    for (int i = 0; i < cnt; ++i)
        out[i] = a[i].idx;
    qsort(out, (size_t)cnt, sizeof(int32_t), cmp_int32);
    free(a);
    return cnt;
}

/*
 * The Selector for one (layer, sequence, kv head) at a slow step of length L
 * ([Sum 2B]): fused score over the candidates [S, L-W), Top-K, mapped back to positions.
 * The sinks [0, min(S, L)) and the window are kept by construction of the sparse state,
 * never by the selection. sel: ascending positions; returns the count min(K, n_C).
 */
int sfi_oracle_select(int L, int S, int W, int K, int tau, double lambda, const float *f,
                      int32_t *sel)
{
    const int n = sfi_oracle_num_candidates(L, S, W);
    if (n == 0)
        return 0;
    float *s = (float *)malloc(sizeof(float) * (size_t)n);
    if (!s)
        return -1;
    sfi_oracle_fused_scores(L, S, W, tau, lambda, f, s);
    const int cnt = sfi_oracle_topk(n, s, K, sel);
    for (int i = 0; i < cnt; ++i)
        sel[i] += S;
    free(s);
    return cnt;
}

/*
 * Rows a fast step attends to ([Sum 2A] sinks + sliding recent window + selected memory;
 * [Sum 3] sinks and selected packed after the slow step, recent tokens from the cache).
 * With L_slow the length at the last slow step and L_now the current length:
 *     sinks    [0, n_s) with n_s = min(S, L_slow)
 *     selected sel[0..cnt)  (ascending, inside [S, L_slow - W))
 *     window   [max(n_s, L_now - W), L_now)   -- slides with every step
 * Returns the row count; rows are written in that order.
 */
int sfi_oracle_sparse_rows(int L_slow, int L_now, int S, int W, const int32_t *sel, int cnt,
                           int32_t *rows)
{
    const int n_s = S < L_slow ? S : L_slow;
    int n = 0;
    for (int j = 0; j < n_s; ++j)
        rows[n++] = j;
    for (int i = 0; i < cnt; ++i)
        rows[n++] = sel[i];
    int w0 = L_now - W;
    if (w0 < n_s)
        w0 = n_s;
    for (int j = w0; j < L_now; ++j)
        rows[n++] = j;
    return n;
}

/*
 * Trigger policy ([Sum 2C]): step t is slow when the previous token is a trigger token
 * (mask[t-1] = 1), or when T_max steps have passed since the last slow step; the first
 * decode step is slow because no selection exists after the prefill (reading).
 * t_max <= 0 disables the forced refresh. slow: uint8 [steps].
 */
void sfi_oracle_schedule(int steps, const uint8_t *mask, int t_max, uint8_t *slow)
{
    int last = 0;
    for (int t = 0; t < steps; ++t) {
        int s = (t == 0) || mask[t - 1] || (t_max > 0 && t - last >= t_max);
        slow[t] = (uint8_t)s;
        if (s)
            last = t;
    }
}

/*
 * Trigger policy on a token stream ([Sum 2C]: a slow step follows a trigger token such as
 * '.', '?', '!' or a newline). tokens: host int32 [steps], the token emitted at each step;
 * trigger_ids: the n_trigger token ids that end a span. Step t is slow when t == 0, when
 * tokens[t-1] is a trigger id, or when t_max > 0 steps have passed since the last slow step.
 */
void sfi_oracle_schedule_tokens(int steps, const int32_t *tokens, const int32_t *trigger_ids,
                                int n_trigger, int t_max, uint8_t *slow)
{
    int last = 0;
    for (int t = 0; t < steps; ++t) {
        int trig = 0;
        if (t > 0)
            for (int i = 0; i < n_trigger; ++i)
                if (tokens[t - 1] == trigger_ids[i])
                    trig = 1;
        int s = (t == 0) || trig || (t_max > 0 && t - last >= t_max);
        slow[t] = (uint8_t)s;
        if (s)
            last = t;
    }
}

/* ------------------------------------------------------------------------------------ */
/* Batched drivers (independent units on a few threads; no change to the arithmetic)     */
/* ------------------------------------------------------------------------------------ */

typedef struct {
    int G, D, n_units, lmax, rmax;
    const uint16_t *q, *k, *v;       /* q [U][G][D]; k, v [U][lmax][D] */
    const int32_t *rows, *n_rows;    /* rows [U][rmax] or NULL; n_rows [U] */
    double *o, *f;                   /* o [U][G][D]; f [U][lmax] or NULL (evidence) */
    int next;
    pthread_mutex_t mu;
    int status;
} batch_job_t;

static void *batch_worker(void *arg)
{
    batch_job_t *j = (batch_job_t *)arg;
    double *p = NULL;
    size_t p_cap = 0;
    for (;;) {
        pthread_mutex_lock(&j->mu);
        const int u = j->next++;
        pthread_mutex_unlock(&j->mu);
        if (u >= j->n_units)
            break;
        const int n = j->n_rows[u];
        if (n < 1)
            continue;
        if (j->f) {
            const size_t need = (size_t)j->G * (size_t)n;
            if (need > p_cap) {
                free(p);
                p = (double *)malloc(sizeof(double) * need);
                p_cap = p ? need : 0;
            }
        }
        const int rc = sfi_oracle_attend(
            j->G, j->D, j->q + (size_t)u * j->G * j->D, j->k + (size_t)u * j->lmax * j->D,
            j->v + (size_t)u * j->lmax * j->D, j->rows ? j->rows + (size_t)u * j->rmax : NULL,
            n, j->o + (size_t)u * j->G * j->D, j->f ? p : NULL);
        if (rc == 0 && j->f)
            sfi_oracle_evidence(j->G, n, p, j->f + (size_t)u * j->lmax);
        if (rc != 0) {
            pthread_mutex_lock(&j->mu);
            j->status = rc;
            pthread_mutex_unlock(&j->mu);
        }
    }
    free(p);
    return NULL;
}

/*
 * Attention for many independent units on n_threads threads. With rows == NULL unit u
 * attends to its first n_rows[u] rows (dense); f, when given, receives the evidence of
 * each dense unit. Returns 0 or the first failing unit's status.
 */
int sfi_oracle_attend_batch(int n_units, int G, int D, int lmax, const uint16_t *q,
                            const uint16_t *k, const uint16_t *v, const int32_t *rows, int rmax,
                            const int32_t *n_rows, double *o, double *f, int n_threads)
{
    batch_job_t j;
    memset(&j, 0, sizeof j);
    j.G = G; j.D = D; j.n_units = n_units; j.lmax = lmax; j.rmax = rmax;
    j.q = q; j.k = k; j.v = v; j.rows = rows; j.n_rows = n_rows; j.o = o; j.f = f;
    pthread_mutex_init(&j.mu, NULL);
    if (n_threads < 1)
        n_threads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    int started = 0;
    for (int t = 0; th && t < n_threads; ++t)
        if (pthread_create(&th[t], NULL, batch_worker, &j) == 0)
            ++started;
    if (started == 0)
        batch_worker(&j);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&j.mu);
    return j.status;
}
