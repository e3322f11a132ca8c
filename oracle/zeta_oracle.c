/*
 * zeta_oracle.c -- plain, slow, single-threaded CPU oracle for the ZETA hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this code:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Method: "ZETA: Leveraging Z-order Curves for Efficient Top-k Attention"
 * (Zeng, Huang, Lu, Xu, Chen, Ling, Wang; arXiv 2501.14577).  Sources used:
 *   [RB-A2bin]  OpenReview discussion, reply A2 "Clarification of Binary
 *               Expansion and Precision" (normalise to [0,1], 4096-cell grid =
 *               12 bits per coordinate, interleave bits, fits a 64-bit integer).
 *   [RB-asym]   OpenReview discussion, reply on the dimension-ordering asymmetry
 *               and the multiple Z-order curves (K^1, K^2, K^3 ordering).
 *   [RB-A3eff]  OpenReview discussion, reply A3 "Chunking ... & Where efficiency
 *               is coming from" (radix sort of Z codes, binary search of the
 *               insertion position).
 *   [RB-A2win]  OpenReview discussion, reply A2 "Clarification" on the insertion
 *               position (the window centred at the insertion position holds
 *               the nearest neighbours).
 *   [RB-cauchy] OpenReview discussion, reply A2 "Discussion on its robustness"
 *               (trainable gamma in the Cauchy softmax acts as a temperature;
 *               gamma = 1 gives a Student-t kernel) and reply A3 "Justification
 *               for Euclidean Distance Claim".
 *   [SUM-app]   atlas.scime.ai summary, "Approach" (keys sorted and split into
 *               chunks, every query finds its top-k neighbours among its
 *               causal past; Adaptive Cauchy-Softmax).
 *
 * Readings where the pages are silent:
 *   - normalisation is the fixed affine map [-1,1) -> [0,1); quantisation is done
 *     in IEEE float32: t = (x + 1) * 2^(bits-1), u = clamp(floor(t), 0, 2^bits-1);
 *   - interleave: level j (LSB = 0) occupies code bits [j*d_K, (j+1)*d_K), and
 *     dimension 0 is the most significant bit inside each level;
 *   - keys are ordered by (code, token index); the query in chunk c searches the
 *     keys of chunks 0..c-1; its insertion rank r counts keys with code <= its
 *     code; the window is positions [clamp(r - ceil(k/2), 0, M - k), +k) of that
 *     sorted prefix of M = c*C keys (all M, padded with -1, when M < k);
 *   - every key j of the query's own chunk with j <= i joins the attended set;
 *   - Cauchy weight w = 1 / (1 + |q - k|^2 / gamma^2), normalised over the set;
 *     the ablation kernels (softmax of -|q - k|^2 / gamma^2, inverse Euclidean
 *     1 / sqrt(|q - k|^2 + 1e-12)) are described at orc_w below;
 *   - several curves [RB-asym]: curve m reads the coordinates in the order
 *     axes[m]; each curve's window holds k // curves keys (same centring rule);
 *     the union lists the windows in curve order, drops a key an earlier curve
 *     (or slot) already gave, and pads the row to k with -1.
 *
 * Floating point is double everywhere except the quantiser, which the reading
 * above fixes to float32.  Compile with -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- encode --- */

/* One coordinate -> grid cell, [RB-A2bin].  float32 arithmetic on purpose. */
uint32_t orc_quantise(float x, int bits)
{
    float scale = ldexpf(1.0f, bits - 1);           /* exact power of two */
    float t = (x + 1.0f) * scale;                   /* [-1,1) -> [0, 2^bits) */
    float f = floorf(t);
    f = fmaxf(f, 0.0f);                             /* NaN -> 0 as well */
    f = fminf(f, (float)((1u << bits) - 1u));       /* exact for bits <= 24 */
    return (uint32_t)f;
}

/* Interleave d_K cell indices into one Z-order code by a naive bit loop,
 * [RB-A2bin] and [RB-asym]. */
uint64_t orc_interleave(const uint32_t *u, int d_K, int bits)
{
    uint64_t code = 0;
    for (int j = 0; j < bits; ++j)
        for (int d = 0; d < d_K; ++d)
            if ((u[d] >> j) & 1u)
                code |= (uint64_t)1 << (j * d_K + (d_K - 1 - d));
    return code;
}

/* x: [ntok][d_K] float32 -> codes[ntok]. */
void orc_encode(const float *x, int64_t ntok, int d_K, int bits, uint64_t *codes)
{
    uint32_t u[64];
    for (int64_t t = 0; t < ntok; ++t) {
        for (int d = 0; d < d_K; ++d)
            u[d] = orc_quantise(x[t * d_K + d], bits);
        codes[t] = orc_interleave(u, d_K, bits);
    }
}

/* ------------------------------------------------------- sort / prefix --- */

typedef struct { uint64_t code; int32_t idx; } orc_pair;

static int orc_pair_cmp(const void *a, const void *b)
{
    const orc_pair *x = (const orc_pair *)a, *y = (const orc_pair *)b;
    if (x->code != y->code) return x->code < y->code ? -1 : 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

/* Sorted prefix of chunks 0..c-1 of one (b,h) slice: the M = c*C keys ordered
 * by (code, index), [RB-A3eff] and [SUM-app].  The library qsort is the sort
 * step; the (code, index) key makes the order unique. */
void orc_prefix(const uint64_t *key_codes, int64_t c, int64_t C,
                uint64_t *pcodes, int32_t *pidx)
{
    int64_t M = c * C;
    orc_pair *p = (orc_pair *)malloc((size_t)(M > 0 ? M : 1) * sizeof(orc_pair));
    for (int64_t j = 0; j < M; ++j) { p[j].code = key_codes[j]; p[j].idx = (int32_t)j; }
    qsort(p, (size_t)M, sizeof(orc_pair), orc_pair_cmp);
    for (int64_t j = 0; j < M; ++j) { pcodes[j] = p[j].code; pidx[j] = p[j].idx; }
    free(p);
}

/* All prefixes c = 1..n-1 of one slice, back to back: prefix c starts at entry
 * C*c*(c-1)/2; T = C*n*(n-1)/2 entries in all. */
void orc_prefix_table(const uint64_t *key_codes, int64_t N, int64_t C,
                      uint64_t *pcodes, int32_t *pidx)
{
    int64_t n = N / C;
    for (int64_t c = 1; c < n; ++c) {
        int64_t off = C * c * (c - 1) / 2;
        orc_prefix(key_codes, c, C, pcodes + off, pidx + off);
    }
}

/* Window of the query with code qc in a sorted prefix of M keys,
 * [RB-A3eff] insertion position by search, [RB-A2win] window centred on it.
 * The rank is found by a plain linear count. */
static void orc_window(uint64_t qc, const uint64_t *pcodes, const int32_t *pidx,
                       int64_t M, int k, int32_t *out)
{
    int64_t r = 0;
    for (int64_t p = 0; p < M; ++p)
        if (pcodes[p] <= qc) ++r;
    if (M <= k) {
        for (int t = 0; t < k; ++t) out[t] = t < M ? pidx[t] : -1;
        return;
    }
    int64_t start = r - (k + 1) / 2;
    if (start < 0) start = 0;
    if (start > M - k) start = M - k;
    for (int t = 0; t < k; ++t) out[t] = pidx[start + t];
}

/* Top-k window for the queries listed in rows[0..nrows) of one slice
 * (rows == NULL: all N queries, in order).  Rows must be grouped by chunk for
 * speed only; any order gives the same answer.  idx: [nrows][k], -1 padded;
 * chunk-0 queries select nothing. */
void orc_select(const uint64_t *q_codes, const uint64_t *key_codes, int64_t N,
                int64_t C, int k, const int64_t *rows, int64_t nrows, int32_t *idx)
{
    int64_t cnt = rows ? nrows : N;
    uint64_t *pc = (uint64_t *)malloc((size_t)(N > 0 ? N : 1) * sizeof(uint64_t));
    int32_t *pi = (int32_t *)malloc((size_t)(N > 0 ? N : 1) * sizeof(int32_t));
    int64_t built = -1;
    for (int64_t t = 0; t < cnt; ++t) {
        int64_t i = rows ? rows[t] : t;
        int64_t c = i / C;
        int32_t *out = idx + t * k;
        if (c == 0) { for (int s = 0; s < k; ++s) out[s] = -1; continue; }
        if (built != c) { orc_prefix(key_codes, c, C, pc, pi); built = c; }
        orc_window(q_codes[i], pc, pi, c * C, k, out);
    }
    free(pc);
    free(pi);
}

/* ------------------------------------------------------------- attend --- */

/* Weight kernels of the attended set, [RB-cauchy] and the ablation in reply A3
 * "Justification for Euclidean Distance Claim" (Cauchy softmax against
 * negative Euclidean with the usual softmax and inverse Euclidean):
 *   kind 0  Cauchy             w = 1 / (1 + d2 / gamma^2)
 *   kind 1  softmax of -d2/gamma^2: w = exp(-(d2 - m) / gamma^2), m the row's
 *           smallest d2 over the attended set (a shift that leaves w / sum w
 *           unchanged and keeps the largest weight at 1)
 *   kind 2  inverse Euclidean  w = 1 / sqrt(d2 + eps^2), eps = 1e-6
 * d2 = |q - k|^2.  For each kind, dw/d(d2) and dw/dgamma (m held fixed, which
 * changes no gradient because sum_j a_ij (g_ij - gbar_i) = 0). */
#define ORC_INV_EPS2 1e-12

static double orc_d2(const double *q, const double *kk, int d_K)
{
    double d2 = 0.0;
    for (int d = 0; d < d_K; ++d) { double e = q[d] - kk[d]; d2 += e * e; }
    return d2;
}

static double orc_w(int kind, double d2, double m, double gamma)
{
    if (kind == 1) return exp(-(d2 - m) / (gamma * gamma));
    if (kind == 2) return 1.0 / sqrt(d2 + ORC_INV_EPS2);
    return 1.0 / (1.0 + d2 / (gamma * gamma));
}

static double orc_dw_dd2(int kind, double w, double gamma)
{
    if (kind == 1) return -w / (gamma * gamma);
    if (kind == 2) return -0.5 * w * w * w;
    return -w * w / (gamma * gamma);
}

static double orc_dw_dgamma(int kind, double w, double d2, double m, double gamma)
{
    if (kind == 1) return w * 2.0 * (d2 - m) / (gamma * gamma * gamma);
    if (kind == 2) return 0.0;
    return 2.0 * w * (1.0 - w) / gamma;
}

/* Row shift m of kind 1: the smallest d2 over the set (0 for the other kinds). */
static double orc_shift(int kind, const double *qi, const double *kx, const int64_t *set,
                        int64_t n, int d_K)
{
    if (kind != 1) return 0.0;
    double m = INFINITY;
    for (int64_t a = 0; a < n; ++a) {
        double d2 = orc_d2(qi, kx + set[a] * d_K, d_K);
        if (d2 < m) m = d2;
    }
    return m;
}

/* Attended set of query i: its window keys (non-negative entries of idx row)
 * followed by its own chunk's keys cC..i.  Returns the count. */
static int64_t orc_set(const int32_t *idxrow, int k, int64_t i, int64_t C, int64_t *set)
{
    int64_t m = 0;
    for (int t = 0; t < k; ++t) if (idxrow[t] >= 0) set[m++] = idxrow[t];
    for (int64_t j = (i / C) * C; j <= i; ++j) set[m++] = j;
    return m;
}

/* Forward for one slice: out[i] = sum_j w_ij v_j / s_i, s_i = sum_j w_ij over the
 * attended set, [RB-cauchy], [SUM-app].  rows == NULL: all N queries.
 * q,k: [N][d_K]; v: [N][d_V]; idx: one row of k entries per listed query
 * ([nrows][k], or [N][k] when rows == NULL); out: [nrows][d_V]; rowsum: [nrows]. */
void orc_attend_fwd(const double *q, const double *kx, const double *v, double gamma,
                    const int32_t *idx, int64_t N, int64_t C, int d_K, int d_V, int k,
                    const int64_t *rows, int64_t nrows, double *out, double *rowsum, int kind)
{
    int64_t cnt = rows ? nrows : N;
    int64_t *set = (int64_t *)malloc((size_t)(k + C + 1) * sizeof(int64_t));
    for (int64_t t = 0; t < cnt; ++t) {
        int64_t i = rows ? rows[t] : t;
        int64_t m = orc_set(idx + t * k, k, i, C, set);
        double sh = orc_shift(kind, q + i * d_K, kx, set, m, d_K);
        double s = 0.0;
        double *o = out + t * d_V;
        for (int e = 0; e < d_V; ++e) o[e] = 0.0;
        for (int64_t a = 0; a < m; ++a) {
            int64_t j = set[a];
            double w = orc_w(kind, orc_d2(q + i * d_K, kx + j * d_K, d_K), sh, gamma);
            s += w;
            for (int e = 0; e < d_V; ++e) o[e] += w * v[j * d_V + e];
        }
        for (int e = 0; e < d_V; ++e) o[e] /= s;
        rowsum[t] = s;
    }
    free(set);
}

/* Backward for one slice with the selection held fixed.  With a_ij = w_ij / s_i,
 * g_ij = dO_i . v_j and gbar_i = dO_i . o_i:
 *   dL/dw_ij   = (g_ij - gbar_i) / s_i
 *   dq_i  += dL/dw_ij * dw/d(d2) * 2 (q_i - k_j),  dk_j gets the negation
 *   dv_j  += a_ij dO_i,                  dgamma += dL/dw_ij * dw/dgamma
 * (Cauchy: dw/d(d2) = -w^2 / gamma^2, dw/dgamma = 2 w (1 - w) / gamma.)
 * Outputs are overwritten.  dgamma is this slice's sum.  rows == NULL: every
 * query contributes (the gradient); otherwise only the queries listed in
 * rows[0..nrows) do, idx holding their rows ([nrows][k]), so the outputs are
 * those queries' shares of the sums (used to time a bounded sample). */
void orc_attend_bwd_rows(const double *q, const double *kx, const double *v, double gamma,
                         const int32_t *idx, const double *dout, int64_t N, int64_t C,
                         int d_K, int d_V, int k, const int64_t *rows, int64_t nrows,
                         double *dq, double *dk, double *dv, double *dgamma, int kind);

void orc_attend_bwd(const double *q, const double *kx, const double *v, double gamma,
                    const int32_t *idx, const double *dout, int64_t N, int64_t C,
                    int d_K, int d_V, int k,
                    double *dq, double *dk, double *dv, double *dgamma, int kind)
{
    orc_attend_bwd_rows(q, kx, v, gamma, idx, dout, N, C, d_K, d_V, k, NULL, 0,
                        dq, dk, dv, dgamma, kind);
}

void orc_attend_bwd_rows(const double *q, const double *kx, const double *v, double gamma,
                         const int32_t *idx, const double *dout, int64_t N, int64_t C,
                         int d_K, int d_V, int k, const int64_t *rows, int64_t nrows,
                         double *dq, double *dk, double *dv, double *dgamma, int kind)
{
    int64_t *set = (int64_t *)malloc((size_t)(k + C + 1) * sizeof(int64_t));
    double *w = (double *)malloc((size_t)(k + C + 1) * sizeof(double));
    double *o = (double *)malloc((size_t)d_V * sizeof(double));
    memset(dq, 0, (size_t)N * d_K * sizeof(double));
    memset(dk, 0, (size_t)N * d_K * sizeof(double));
    memset(dv, 0, (size_t)N * d_V * sizeof(double));
    double dg = 0.0;
    int64_t cnt = rows ? nrows : N;
    for (int64_t t = 0; t < cnt; ++t) {
        int64_t i = rows ? rows[t] : t;
        int64_t m = orc_set(idx + t * k, k, i, C, set);
        const double *qi = q + i * d_K;
        const double *doi = dout + i * d_V;
        double sh = orc_shift(kind, qi, kx, set, m, d_K);
        double s = 0.0;
        for (int e = 0; e < d_V; ++e) o[e] = 0.0;
        for (int64_t a = 0; a < m; ++a) {
            int64_t j = set[a];
            w[a] = orc_w(kind, orc_d2(qi, kx + j * d_K, d_K), sh, gamma);
            s += w[a];
            for (int e = 0; e < d_V; ++e) o[e] += w[a] * v[j * d_V + e];
        }
        for (int e = 0; e < d_V; ++e) o[e] /= s;
        double gbar = 0.0;
        for (int e = 0; e < d_V; ++e) gbar += doi[e] * o[e];
        for (int64_t a = 0; a < m; ++a) {
            int64_t j = set[a];
            const double *kj = kx + j * d_K;
            double g = 0.0;
            for (int e = 0; e < d_V; ++e) g += doi[e] * v[j * d_V + e];
            double dldw = (g - gbar) / s;
            /* d(d2)/dq_i = 2 (q_i - k_j) = -d(d2)/dk_j */
            double coef = dldw * orc_dw_dd2(kind, w[a], gamma) * 2.0;
            for (int d = 0; d < d_K; ++d) {
                double term = coef * (qi[d] - kj[d]);
                dq[i * d_K + d] += term;
                dk[j * d_K + d] -= term;
            }
            double aij = w[a] / s;
            for (int e = 0; e < d_V; ++e) dv[j * d_V + e] += aij * doi[e];
            dg += dldw * orc_dw_dgamma(kind, w[a], orc_d2(qi, kj, d_K), sh, gamma);
        }
    }
    *dgamma = dg;
    free(set);
    free(w);
    free(o);
}

/* ------------------------------------------------------------- recall --- */

typedef struct { double d2; int32_t idx; } orc_dist;

static int orc_dist_cmp(const void *a, const void *b)
{
    const orc_dist *x = (const orc_dist *)a, *y = (const orc_dist *)b;
    if (x->d2 != y->d2) return x->d2 < y->d2 ? -1 : 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

/* Exact Euclidean top-k among the same prefix keys 0..cC-1 the window is drawn
 * from (ties by lower index), for measuring how much of the true neighbour set
 * the window keeps, [RB-A2win] and the locality discussion of the pages.
 * q,k: float32 [N][d_K]; out: [nrows][k], -1 padded. */
void orc_exact_topk(const float *q, const float *kx, int64_t N, int64_t C, int d_K,
                    int k, const int64_t *rows, int64_t nrows, int32_t *out)
{
    int64_t cnt = rows ? nrows : N;
    orc_dist *buf = (orc_dist *)malloc((size_t)(N > 0 ? N : 1) * sizeof(orc_dist));
    for (int64_t t = 0; t < cnt; ++t) {
        int64_t i = rows ? rows[t] : t;
        int64_t M = (i / C) * C;
        for (int64_t j = 0; j < M; ++j) {
            double d2 = 0.0;
            for (int d = 0; d < d_K; ++d) {
                double e = (double)q[i * d_K + d] - (double)kx[j * d_K + d];
                d2 += e * e;
            }
            buf[j].d2 = d2;
            buf[j].idx = (int32_t)j;
        }
        qsort(buf, (size_t)M, sizeof(orc_dist), orc_dist_cmp);
        for (int s = 0; s < k; ++s) out[t * k + s] = s < M ? buf[s].idx : -1;
    }
    free(buf);
}

/* --------------------------------------------------- multiple Z curves --- */

/* Codes of the coordinates read in the order axes[0..d_K) (a permutation of
 * 0..d_K-1): the curve of the tuple (x[axes[0]], x[axes[1]], ...), OpenReview
 * discussion, follow-up reply on interleaving the bits of
 * different dimensions (several curves): shifted and permuted
 * coordinate orders (K^1,K^2,K^3), (K^2,K^3,K^1), ... */
void orc_encode_axes(const float *x, int64_t ntok, int d_K, int bits, const int32_t *axes,
                     uint64_t *codes)
{
    uint32_t u[64];
    for (int64_t t = 0; t < ntok; ++t) {
        for (int d = 0; d < d_K; ++d)
            u[d] = orc_quantise(x[t * d_K + axes[d]], bits);
        codes[t] = orc_interleave(u, d_K, bits);
    }
}

/* Union of M per-curve windows of one query, same reply ("each mapping
 * collects k//M tokens"): curve windows in curve order, an index already taken
 * from an earlier curve (or earlier in the same window) is dropped, the row is
 * filled to k with -1.  win: M rows of km entries; out: k entries. */
void orc_merge_windows(const int32_t *win, int M, int km, int k, int32_t *out)
{
    int n = 0;
    for (int m = 0; m < M; ++m)
        for (int t = 0; t < km; ++t) {
            int32_t j = win[m * km + t];
            if (j < 0) continue;
            int dup = 0;
            for (int s = 0; s < n; ++s)
                if (out[s] == j) { dup = 1; break; }
            if (!dup && n < k) out[n++] = j;
        }
    for (; n < k; ++n) out[n] = -1;
}

/* ------------------------------------------------------------ projection --- */

/* Two-layer projection of one token onto the d_K key (or query) coordinates of
 * every head, OpenReview discussion, reply A "LLMs impact the selection of
 * d_K" (the keys come out of a small network of two layers):
 *   h_f   = max(0, sum_e W1[hd*F + f][e] x[e] + b1[hd*F + f])     f < F
 *   y_c   = tanh(sum_f W2[hd][c][f] h_f + b2[hd][c])               c < d_K
 * tanh lands the coordinates in (-1, 1), the range the quantiser reads.
 * x: [M][D]; W1: [H*F][D]; b1: [H*F]; W2: [H][d_K][F]; b2: [H][d_K];
 * out: [M][H][d_K]. */
void orc_project(const double *x, int64_t M, int D, int H, int F, int d_K,
                 const double *W1, const double *b1, const double *W2, const double *b2,
                 double *out)
{
    double *h = (double *)malloc((size_t)F * sizeof(double));
    for (int64_t t = 0; t < M; ++t) {
        const double *xt = x + t * D;
        for (int hd = 0; hd < H; ++hd) {
            for (int f = 0; f < F; ++f) {
                const double *w = W1 + ((int64_t)hd * F + f) * D;
                double z = b1[hd * F + f];
                for (int e = 0; e < D; ++e) z += w[e] * xt[e];
                h[f] = z > 0.0 ? z : 0.0;
            }
            for (int c = 0; c < d_K; ++c) {
                const double *w = W2 + ((int64_t)hd * d_K + c) * F;
                double y = b2[hd * d_K + c];
                for (int f = 0; f < F; ++f) y += w[f] * h[f];
                out[(t * H + hd) * d_K + c] = tanh(y);
            }
        }
    }
    free(h);
}
