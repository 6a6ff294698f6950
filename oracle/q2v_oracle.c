/*
 * q2v_oracle.c -- the plain, slow, fp64 CPU oracle for the target-verifier step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library, its
 * Python binding, or the timed arm of the benchmark) may load or call this file.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes, and where the pages define it:
 *
 *  - Q2B32 dequantisation and the tiny-batch matmul Y = A * W^T.  The pages name
 *    only undefined 2-bit GGUF formats ("ds4-on-spark" README, section "Model");
 *    the stand-in block format used here is fixed by the project's problem
 *    statement: 32 weights per block, 8 bytes of 2-bit unsigned codes (4 per
 *    byte, low bits first), then an fp16 scale d and an fp16 offset m, w = d*q+m,
 *    rows over N with the K-blocks of a row contiguous.
 *  - The routed MoE FFN of the verify forward ("Optimizing DeepSeek-V4-Flash on a
 *    single NVIDIA GB10/GX10 with DSpark speculative decoding", page 2, the
 *    verifier-bottleneck reply: the verifier runs attention, routed MoE,
 *    projections and the vocabulary head over K+1 rows): top-k of the router
 *    softmax, silu(gate) * up, down projection, weighted combine.
 *  - The p/q rejection-sampling verify ("Optimizing DeepSeek-V4-Flash ...",
 *    page 1, opening post, paragraph after the analyzer output: drafts are drawn
 *    from q, the target defines p, a draft is accepted with probability
 *    min(1, p(x)/q(x)), and a rejected draft is replaced from the positive
 *    residual distribution; the same thread's posts #12 and #20 describe the
 *    correction as exact).  When every draft is accepted the one extra
 *    token is drawn from the last target row ("1x Spark tuned DSpark for
 *    DeepSeek-V4-Flash ...", deep-dive, "On losslessness": the verify forward is
 *    the only token source and the accept loop samples from the verify-row
 *    logits with the request's own sampler).
 *
 * Readings taken where the pages are silent (each one is listed with its reason
 * in the design notes of the repository):
 *   accept iff u < p(x)/q(x) (strict; min(1,.) is implied because u < 1);
 *   q(x) == 0 accepts;  residual and bonus draws use the inverse CDF in
 *   ascending token order, returning the smallest y with C(y) > u*Z;  a zero
 *   residual mass falls back to p_j;  one temperature T > 0 for p and q;  one
 *   final uniform per session serves whichever final draw happens;  MoE gate
 *   weights are the selected softmax probabilities, not renormalised unless
 *   asked;  routing ties go to the lower expert index.
 *
 * Every floating-point step is fp64; inputs (fp16, bf16, fp32) are widened exactly.
 * All accumulations run in natural index order.  Parity is pinned by the
 * tests under tests/ (closed forms, brute-force enumeration, library routines,
 * chi-square of the emitted-token law); see the oracle pin tests.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ scalars */

/* IEEE 754 binary16 -> double, written from the format's definition:
 * sign bit, 5 exponent bits (bias 15), 10 fraction bits. Exact. */
double orc_half_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-24      */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);  /* (1 + f/2^10) * 2^(e-15)   */
    return sign ? -v : v;
}

/* bfloat16 -> double: a bf16 value is the upper half of an IEEE binary32. Exact. */
double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------ Q2B32 */

#define ORC_BLOCK_BYTES 12
#define ORC_BLOCK_K 32

/* One weight w[n][k] of a Q2B32 matrix with K columns. */
double orc_q2b32_weight(const uint8_t *W, int K, int n, int k)
{
    const uint8_t *blk = W + ((size_t)n * (size_t)(K / ORC_BLOCK_K) + (size_t)(k / ORC_BLOCK_K)) * ORC_BLOCK_BYTES;
    int j = k % ORC_BLOCK_K;
    int q = (blk[j / 4] >> (2 * (j % 4))) & 3;          /* code j: byte j/4, bits 2(j%4)..+1 */
    uint16_t dh = (uint16_t)(blk[8] | (blk[9] << 8));   /* little-endian fp16 scale  */
    uint16_t mh = (uint16_t)(blk[10] | (blk[11] << 8)); /* little-endian fp16 offset */
    return orc_half_to_f64(dh) * (double)q + orc_half_to_f64(mh);
}

/* Dequantise a whole [N,K] matrix to fp64, row-major. */
void orc_q2b32_dequant(const uint8_t *W, int N, int K, double *out)
{
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            out[(size_t)n * K + k] = orc_q2b32_weight(W, K, n, k);
}

/* Y[m][n] = sum_k A[m][k] * w[n][k]   (Y = A W^T), fp64, natural k order.
 * absY[m][n] = sum_k |A[m][k] * w[n][k]|  (the scale of the GEMM tolerance).
 * A is bf16 bits [M][lda]; Y and absY are [M][N]. absY may be NULL. */
void orc_gemm(const uint8_t *W, int N, int K, const uint16_t *A, int M, int lda,
              double *Y, double *absY, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *wrow = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int n = 0; n < N; ++n) {
            for (int k = 0; k < K; ++k) wrow[k] = orc_q2b32_weight(W, K, n, k);
            for (int m = 0; m < M; ++m) {
                double s = 0.0, sa = 0.0;
                for (int k = 0; k < K; ++k) {
                    double t = orc_bf16_to_f64(A[(size_t)m * lda + k]) * wrow[k];
                    s += t;
                    sa += fabs(t);
                }
                Y[(size_t)m * N + n] = s;
                if (absY) absY[(size_t)m * N + n] = sa;
            }
        }
        free(wrow);
    }
}

/* ------------------------------------------------------------------ softmax */

/* p = softmax(x / T) over V entries, by log-sum-exp (subtract the max of x/T). */
void orc_softmax(const float *x, int V, double T, double *p)
{
    double mx = -INFINITY;
    for (int i = 0; i < V; ++i) {
        double z = (double)x[i] / T;
        if (z > mx) mx = z;
    }
    double Z = 0.0;
    for (int i = 0; i < V; ++i) {
        p[i] = exp((double)x[i] / T - mx);
        Z += p[i];
    }
    for (int i = 0; i < V; ++i) p[i] /= Z;
}

/* Inverse-CDF draw from unnormalised non-negative weights w[0..V):
 * the smallest y with C(y) = sum_{y'<=y} w[y'] > u * Z, Z = sum w, scanning in
 * ascending index.  Also returns the normalised cell [C(y-1)/Z, C(y)/Z) of y.
 * Returns -1 if Z is not positive. */
int orc_inverse_cdf(const double *w, int V, double u, double *cell_lo, double *cell_hi)
{
    double Z = 0.0;
    for (int y = 0; y < V; ++y) Z += w[y];
    if (!(Z > 0.0)) return -1;
    double target = u * Z, c = 0.0;
    int last_pos = -1;
    for (int y = 0; y < V; ++y) {
        double prev = c;
        c += w[y];
        if (w[y] > 0.0) last_pos = y;
        if (c > target) {
            if (cell_lo) *cell_lo = prev / Z;
            if (cell_hi) *cell_hi = c / Z;
            return y;
        }
    }
    /* Not reached for u in [0,1): C(V-1) is Z itself and u*Z < Z. */
    if (cell_lo) *cell_lo = 1.0;
    if (cell_hi) *cell_hi = 1.0;
    return last_pos;
}

/* ------------------------------------------------------------------ p/q verify */

/*
 * For each session s (independent):
 *   p_i = softmax(target[s][i] / T), i = 0..k;  q_i = softmax(draft[s][i] / T), i = 0..k-1.
 *   Walk i = 0..k-1 with x_i = drafts[s][i]: accept iff q_i(x_i) == 0 or
 *   u_acc[s][i] < p_i(x_i) / q_i(x_i); stop at the first rejection j.
 *   j < k: draw y from max(0, p_j - q_j) (from p_j if that mass is zero);
 *   j = k: draw y from p_k.  Both draws use u_fin[s] and the inverse CDF.
 *   tokens[s] = [x_0 .. x_{j-1}, y, -1 ...] (k+1 entries), n_acc[s] = j.
 *
 * Diagnostics for the tests (all nullable):
 *   probs   [S][2k+1][V]: p_0..p_k then q_0..q_{k-1};
 *   ratio   [S][k]: p_i(x_i)/q_i(x_i) for every evaluated i (+inf when q is 0), NaN otherwise;
 *   cell_lo, cell_hi [S]: the normalised CDF cell of the final token;
 *   fin_src [S]: 0 = residual, 1 = bonus from p_k, 2 = residual mass zero, drawn from p_j.
 * Returns 0, or 1 if a draft token lies outside [0, V) (that session's outputs are -1).
 */
/* Lowest index of the largest value of x[0..V) (the greedy choice; ties go to the lower
 * token, the plainest deterministic reading). */
static int orc_argmax(const float *x, int V)
{
    int best = 0;
    for (int y = 1; y < V; ++y)
        if (x[y] > x[best]) best = y;
    return best;
}

/*
 * The greedy verify of session s (temperature 0): p_i and q_i become one-hot at the
 * argmax of their logits, so a draft is accepted iff it equals argmax t_i, and the token
 * after the first rejection j (or the bonus, j = k) is argmax t_j.  Neither the draft
 * logits' values beyond their argmax nor the uniforms are used.
 */
static void orc_verify_greedy(const float *ts, const float *ds, const int32_t *xs, int k, int V,
                              int32_t *n_acc, int32_t *tok, double *ps, double *ratio,
                              double *cell_lo, double *cell_hi, int32_t *fin_src)
{
    if (ps) {
        for (size_t e = 0; e < (size_t)(2 * k + 1) * V; ++e) ps[e] = 0.0;
        for (int i = 0; i <= k; ++i) ps[(size_t)i * V + orc_argmax(ts + (size_t)i * V, V)] = 1.0;
        for (int i = 0; i < k; ++i) ps[(size_t)(k + 1 + i) * V + orc_argmax(ds + (size_t)i * V, V)] = 1.0;
    }
    int j = k;
    for (int i = 0; i < k; ++i) {
        const int am = orc_argmax(ts + (size_t)i * V, V);
        if (ratio) ratio[i] = (xs[i] == am) ? INFINITY : 0.0;
        if (xs[i] != am) { j = i; break; }
    }
    for (int i = 0; i < j; ++i) tok[i] = xs[i];
    tok[j] = orc_argmax(ts + (size_t)j * V, V);
    *n_acc = j;
    if (cell_lo) *cell_lo = NAN;
    if (cell_hi) *cell_hi = NAN;
    if (fin_src) *fin_src = 3;
}

/*
 * orc_pq_verify with one temperature per session: temps[s] (NULL: T for every session).
 * temps[s] = 0 selects the greedy verify for that session; a negative or non-finite
 * temperature marks the session bad (n_acc -1, tokens -1) and sets bit 2 of the return.
 */
int orc_pq_verify_ex(const float *target, const float *draft, const int32_t *drafts,
                     const float *u_acc, const float *u_fin, int S, int k, int V, double T,
                     const double *temps, int32_t *n_acc, int32_t *tokens, double *probs,
                     double *ratio, double *cell_lo, double *cell_hi, int32_t *fin_src, int nthreads)
{
    int bad = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads) reduction(| : bad)
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)V * (size_t)(k + 1));
        double *q = (double *)malloc(sizeof(double) * (size_t)V * (size_t)(k > 0 ? k : 1));
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
#pragma omp for schedule(dynamic, 1)
        for (int s = 0; s < S; ++s) {
            const float *ts = target + (size_t)s * (k + 1) * V;
            const float *ds = draft + (size_t)s * k * V;
            const double Ts = temps ? temps[s] : T;
            for (int i = 0; i <= k; ++i) tokens[(size_t)s * (k + 1) + i] = -1;
            if (ratio)
                for (int i = 0; i < k; ++i) ratio[(size_t)s * k + i] = NAN;
            if (!(Ts >= 0.0) || !isfinite(Ts)) {
                bad |= 2;
                n_acc[s] = -1;
                if (fin_src) fin_src[s] = -1;
                continue;
            }
            {
                int token_ok = 1;
                for (int i = 0; i < k; ++i) {
                    int32_t x = drafts[(size_t)s * k + i];
                    if (x < 0 || x >= V) token_ok = 0;
                }
                if (!token_ok) {
                    bad |= 1;
                    n_acc[s] = -1;
                    if (fin_src) fin_src[s] = -1;
                    continue;
                }
            }
            if (Ts == 0.0) {
                orc_verify_greedy(ts, ds, drafts + (size_t)s * k, k, V, n_acc + s, tokens + (size_t)s * (k + 1),
                                  probs ? probs + (size_t)s * (2 * k + 1) * V : NULL,
                                  ratio ? ratio + (size_t)s * k : NULL, cell_lo ? cell_lo + s : NULL,
                                  cell_hi ? cell_hi + s : NULL, fin_src ? fin_src + s : NULL);
                continue;
            }
            for (int i = 0; i <= k; ++i) orc_softmax(ts + (size_t)i * V, V, Ts, p + (size_t)i * V);
            for (int i = 0; i < k; ++i) orc_softmax(ds + (size_t)i * V, V, Ts, q + (size_t)i * V);
            if (probs) {
                double *ps = probs + (size_t)s * (2 * k + 1) * V;
                memcpy(ps, p, sizeof(double) * (size_t)V * (k + 1));
                if (k > 0) memcpy(ps + (size_t)(k + 1) * V, q, sizeof(double) * (size_t)V * k);
            }

            int j = k;
            for (int i = 0; i < k; ++i) {
                int32_t x = drafts[(size_t)s * k + i];
                double px = p[(size_t)i * V + x], qx = q[(size_t)i * V + x];
                double r = (qx == 0.0) ? INFINITY : px / qx;
                if (ratio) ratio[(size_t)s * k + i] = r;
                int accept = (qx == 0.0) || ((double)u_acc[(size_t)s * k + i] < r);
                if (!accept) { j = i; break; }
            }

            double u = (double)u_fin[s];
            double lo = 0.0, hi = 0.0;
            int y, src;
            if (j < k) {
                const double *pj = p + (size_t)j * V, *qj = q + (size_t)j * V;
                for (int v = 0; v < V; ++v) {
                    double d = pj[v] - qj[v];
                    w[v] = d > 0.0 ? d : 0.0;
                }
                y = orc_inverse_cdf(w, V, u, &lo, &hi);
                src = 0;
                if (y < 0) {
                    y = orc_inverse_cdf(pj, V, u, &lo, &hi);
                    src = 2;
                }
            } else {
                y = orc_inverse_cdf(p + (size_t)k * V, V, u, &lo, &hi);
                src = 1;
            }
            for (int i = 0; i < j; ++i) tokens[(size_t)s * (k + 1) + i] = drafts[(size_t)s * k + i];
            tokens[(size_t)s * (k + 1) + j] = y;
            n_acc[s] = j;
            if (cell_lo) cell_lo[s] = lo;
            if (cell_hi) cell_hi[s] = hi;
            if (fin_src) fin_src[s] = src;
        }
        free(p);
        free(q);
        free(w);
    }
    return bad;
}

int orc_pq_verify(const float *target, const float *draft, const int32_t *drafts,
                  const float *u_acc, const float *u_fin, int S, int k, int V, double T,
                  int32_t *n_acc, int32_t *tokens, double *probs, double *ratio,
                  double *cell_lo, double *cell_hi, int32_t *fin_src, int nthreads)
{
    return orc_pq_verify_ex(target, draft, drafts, u_acc, u_fin, S, k, V, T, NULL, n_acc, tokens, probs,
                            ratio, cell_lo, cell_hi, fin_src, nthreads) & 1;
}

/* ------------------------------------------------------------------ routed MoE */

static double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * Routed MoE FFN over M rows:
 *   prob[r] = softmax(router[r][0..E));  ids[r] = the topk experts by probability,
 *   ties to the lower index, in descending order of probability;  g = the selected
 *   probabilities (divided by their sum when renorm != 0);
 *   for each slot: gate = x Wg_e^T, up = x Wu_e^T (F outputs), h = silu(gate) * up,
 *   out = h Wd_e^T (H outputs);  Y[r] = sum over slots in slot order of g * out.
 * Weight tensors: Wg, Wu: [E][F rows][H/32 blocks]; Wd: [E][H rows][F/32 blocks].
 * X is bf16 bits [M][H]; router fp32 [M][E]; Y fp64 [M][H].
 * Diagnostics (nullable): ids [M][topk], gw [M][topk], tol [M][H] = the parity
 * bound 2e-3*sum_slot g*sum_f |h_f w_f| + sum_slot g*sum_f |w_f|*dh_f, with
 * dh_f = |dh/dgate|*2e-3*sum_k|x_k wg_fk| + |dh/dup|*2e-3*sum_k|x_k wu_fk|.
 */
void orc_moe(const uint8_t *Wg, const uint8_t *Wu, const uint8_t *Wd, int E, int H, int F,
             int topk, int renorm, const uint16_t *X, int M, const float *router,
             double *Y, int32_t *ids, double *gw, double *tol, int nthreads)
{
    const double rel = 2e-3;
    if (topk < 1 || topk > 256 || topk > E) return;
    size_t gu_bytes = (size_t)F * (H / ORC_BLOCK_K) * ORC_BLOCK_BYTES;
    size_t d_bytes = (size_t)H * (F / ORC_BLOCK_K) * ORC_BLOCK_BYTES;
    if (nthreads < 1) nthreads = 1;
    for (int r = 0; r < M; ++r) {
        double *prob = (double *)malloc(sizeof(double) * E);
        int *taken = (int *)calloc((size_t)E, sizeof(int));
        int sel[256];
        double g[256];
        orc_softmax(router + (size_t)r * E, E, 1.0, prob);
        double gsum = 0.0;
        for (int t = 0; t < topk; ++t) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || prob[e] > prob[best])) best = e;
            taken[best] = 1;
            sel[t] = best;
            g[t] = prob[best];
            gsum += prob[best];
        }
        if (renorm)
            for (int t = 0; t < topk; ++t) g[t] /= gsum;
        for (int t = 0; t < topk; ++t) {
            if (ids) ids[(size_t)r * topk + t] = sel[t];
            if (gw) gw[(size_t)r * topk + t] = g[t];
        }
        for (int n = 0; n < H; ++n) {
            Y[(size_t)r * H + n] = 0.0;
            if (tol) tol[(size_t)r * H + n] = 0.0;
        }

        double *x = (double *)malloc(sizeof(double) * H);
        for (int kk = 0; kk < H; ++kk) x[kk] = orc_bf16_to_f64(X[(size_t)r * H + kk]);
        double *h = (double *)malloc(sizeof(double) * F);
        double *dh = (double *)malloc(sizeof(double) * F);
        for (int t = 0; t < topk; ++t) {
            int e = sel[t];
            const uint8_t *wg = Wg + (size_t)e * gu_bytes, *wu = Wu + (size_t)e * gu_bytes;
            const uint8_t *wd = Wd + (size_t)e * d_bytes;
#pragma omp parallel for num_threads(nthreads) schedule(static)
            for (int f = 0; f < F; ++f) {
                double ga = 0.0, ua = 0.0, gabs = 0.0, uabs = 0.0;
                for (int kk = 0; kk < H; ++kk) {
                    double a = x[kk] * orc_q2b32_weight(wg, H, f, kk);
                    double b = x[kk] * orc_q2b32_weight(wu, H, f, kk);
                    ga += a; gabs += fabs(a);
                    ua += b; uabs += fabs(b);
                }
                h[f] = orc_silu(ga) * ua;
                double sg = 1.0 / (1.0 + exp(-ga));
                double dsilu = sg * (1.0 + ga * (1.0 - sg));
                dh[f] = fabs(dsilu * ua) * rel * gabs + fabs(orc_silu(ga)) * rel * uabs;
            }
#pragma omp parallel for num_threads(nthreads) schedule(static)
            for (int n = 0; n < H; ++n) {
                double o = 0.0, oabs = 0.0, prop = 0.0;
                for (int f = 0; f < F; ++f) {
                    double w = orc_q2b32_weight(wd, F, n, f);
                    o += h[f] * w;
                    oabs += fabs(h[f] * w);
                    prop += fabs(w) * dh[f];
                }
                Y[(size_t)r * H + n] += g[t] * o;
                if (tol) tol[(size_t)r * H + n] += g[t] * (rel * oabs + prop);
            }
        }
        free(x);
        free(h);
        free(dh);
        free(prob);
        free(taken);
    }
}

int orc_version(void) { return 1; }
