/*
 * moe_oracle.c -- plain, slow, scalar fp64 reference of the decode step of a
 * top-k mixture-of-experts FFN layer over affine group-quantised weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or constant with the CUDA library and must never be
 * used as a fallback for it.
 *
 * Sources (the web pages describing the method):
 *   [MC]  PureDrive-35B-A3B-MLX model card (huggingface.co), "Summary":
 *         256 experts, top-8 plus a shared expert, 6-bit experts, 8-bit
 *         shared weights; "How it works": fused add+RMSNorm, row-exact verify.
 *   [FM]  flash-moe (ja.news.hada.io topic 27758), "FMA最適化デクォントカーネル":
 *         the dequantised weight is nibble*scale+bias; "Metal Compute Shaders":
 *         dequant mat-vec, SwiGLU, RMS normalisation, MoE combine + residual +
 *         gate; "Deferred GPU Expert Compute": combine, norm and residual stay
 *         on the GPU and feed the next layer.
 *
 * The pages give no formulas.  The readings taken here are:
 *   - affine groups of 64 consecutive elements along the contraction (input)
 *     axis: w = q * s + b, s and b stored as bf16;
 *   - RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma;
 *   - router: logits = W_r . hn; p = softmax(logits); the k largest p are
 *     kept (ties to the lower expert id) and renormalised to sum to 1;
 *   - expert FFN: y = W_d (silu(W_g hn) * (W_u hn)), silu(z) = z / (1 + e^-z);
 *   - shared expert weighted by sigmoid(w_sg . hn);
 *   - out = bf16(x + sum_i w_i y_i + sigma y_s); out_n = bf16(RMSNorm(out) * gamma_next)
 *     computed from the bf16 out.
 * Everything is accumulated in fp64 with no intermediate rounding except the
 * quantiser, whose integer decisions are taken in fp32 like the kernel's.
 *
 * The second workload, decode attention with grouped query heads
 * (oracle_gqa_decode), is the plain softmax attention written out; see its
 * comment.
 *
 * Parity pins: every function here is pinned by tests/test_oracle.py
 * (hand-computed dequant, a hand-packed bit stream, closed forms, library
 * routines in fp64, brute force on tiny inputs).
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, ties to even). */
uint16_t oracle_bf16_from_double(double v)
{
    if (isnan(v)) return 0x7FC0;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    uint16_t sign = (uint16_t)(neg << 15);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int e = ilogb(a);                 /* a = m * 2^e, m in [1, 2) */
    if (e < -126) e = -126;           /* subnormal bf16: fixed quantum 2^-133 */
    double quantum = ldexp(1.0, e - 7);
    double r = rint(a / quantum) * quantum;   /* rint: ties to even */
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)r;               /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFF));
}

/* --------------------------------------------------- canonical bit stream */

/* Canonical packing of b-bit codes: one little-endian bit stream per row,
 * code i occupying bits [i*b, (i+1)*b), least significant bit first.  64
 * codes take 32, 48 or 64 bytes at 4, 6 or 8 bits. */
void oracle_pack_bits(const uint8_t *codes, int n, int bits, uint8_t *out)
{
    int nbytes = (n * bits + 7) / 8;
    memset(out, 0, (size_t)nbytes);
    for (int i = 0; i < n; ++i) {
        for (int t = 0; t < bits; ++t) {
            int bit = (codes[i] >> t) & 1;
            int pos = i * bits + t;
            out[pos / 8] |= (uint8_t)(bit << (pos % 8));
        }
    }
}

void oracle_unpack_bits(const uint8_t *packed, int n, int bits, uint8_t *codes)
{
    for (int i = 0; i < n; ++i) {
        int v = 0;
        for (int t = 0; t < bits; ++t) {
            int pos = i * bits + t;
            v |= ((packed[pos / 8] >> (pos % 8)) & 1) << t;
        }
        codes[i] = (uint8_t)v;
    }
}

/* ------------------------------------------------------------- quantiser */

/* Affine quantisation of one group of 64 fp32 weights to b bits:
 *   s = bf16((max - min) / (2^b - 1)), b = bf16(min),
 *   q = clamp(rint((w - b) / s), 0, 2^b - 1), q = 0 when s == 0.
 * The arithmetic that decides each code is fp32, as in the kernel. */
void oracle_quantize_group(int bits, const float *w, uint8_t *q, uint16_t *s_out, uint16_t *b_out)
{
    float mn = w[0], mx = w[0];
    for (int i = 1; i < 64; ++i) {
        if (w[i] < mn) mn = w[i];
        if (w[i] > mx) mx = w[i];
    }
    const int qmax = (1 << bits) - 1;
    float range = mx - mn;
    float sf = range / (float)qmax;
    uint16_t sbits = oracle_bf16_from_double((double)sf);
    uint16_t bbits = oracle_bf16_from_double((double)mn);
    float s = (float)oracle_bf16_to_double(sbits);
    float b = (float)oracle_bf16_to_double(bbits);
    for (int i = 0; i < 64; ++i) {
        int code = 0;
        if (s != 0.0f) {
            float t = (w[i] - b) / s;
            float r = rintf(t);
            if (r < 0.0f) r = 0.0f;
            if (r > (float)qmax) r = (float)qmax;
            code = (int)r;
        }
        q[i] = (uint8_t)code;
    }
    *s_out = sbits;
    *b_out = bbits;
}

/* Row-major [rows, cols] fp32 -> codes [rows, cols], scales/biases [rows, cols/64]. */
void oracle_quantize_matrix(int bits, const float *w, int rows, int cols,
                            uint8_t *codes, uint16_t *scales, uint16_t *biases)
{
    int groups = cols / 64;
    for (int r = 0; r < rows; ++r)
        for (int g = 0; g < groups; ++g)
            oracle_quantize_group(bits, w + (size_t)r * cols + (size_t)g * 64,
                                  codes + (size_t)r * cols + (size_t)g * 64,
                                  scales + (size_t)r * groups + g,
                                  biases + (size_t)r * groups + g);
}

/* ------------------------------------------------------------ dequantise */

typedef struct {
    int bits;                 /* 4, 6 or 8; 0 = plain fp32 weights */
    int rows, cols;           /* logical [rows, cols], groups along cols */
    const uint8_t *codes;     /* [rows * cols], one code per byte */
    const uint16_t *scales;   /* [rows * cols / 64], bf16 patterns */
    const uint16_t *biases;   /* [rows * cols / 64], bf16 patterns */
    const float *w;           /* [rows * cols] when bits == 0 */
} oq_matrix;

/* Element (r, c) of a matrix: q * s + b for its group (c / 64). */
double oracle_weight(const oq_matrix *m, int r, int c)
{
    if (m->bits == 0) return (double)m->w[(size_t)r * m->cols + c];
    size_t gi = (size_t)r * (m->cols / 64) + (size_t)(c / 64);
    double q = (double)m->codes[(size_t)r * m->cols + c];
    return q * oracle_bf16_to_double(m->scales[gi]) + oracle_bf16_to_double(m->biases[gi]);
}

static int matrix_present(const oq_matrix *m)
{
    return m->bits == 0 ? m->w != NULL : (m->codes && m->scales && m->biases);
}

/* Threads of the all-cores timing run (1 = the single-core parity
 * reference).  Only the output rows of a mat-vec are spread over threads:
 * each y[r] is still summed by one thread in column order, so any thread
 * count gives the same bits. */
static int g_threads = 1;

void oracle_set_threads(int n) { g_threads = n < 1 ? 1 : n; }

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_num_procs();
#else
    return 1;
#endif
}

/* y[r] = sum_c W[r, c] * x[c] */
static void matvec(const oq_matrix *m, const double *x, double *y)
{
#ifdef _OPENMP
#pragma omp parallel for num_threads(g_threads) if (g_threads > 1) schedule(static)
#endif
    for (int r = 0; r < m->rows; ++r) {
        double acc = 0.0;
        for (int c = 0; c < m->cols; ++c) acc += oracle_weight(m, r, c) * x[c];
        y[r] = acc;
    }
}

/* Fused Q/K/V (or Gated-DeltaNet input) projection of M token rows: the
 * rows of Q, K and V stacked into one [rows, H] matrix, read once for the
 * input row ("Qwen3.5-397B on M5 Max" (openclawradar), "効果的な最適化":
 * fused QKV projection, the input read once).  x bf16 [M, H] is the layer's
 * normalised input (the MoE layer's fused out_n); y[m, r] = sum_c W[r, c]
 * x[m, c] in fp64. */
void oracle_qkv(const oq_matrix *w, const uint16_t *x, int M, double *y)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)w->cols);
    for (int m = 0; m < M; ++m) {
        for (int c = 0; c < w->cols; ++c) xd[c] = oracle_bf16_to_double(x[(size_t)m * w->cols + c]);
        matvec(w, xd, y + (size_t)m * w->rows);
    }
    free(xd);
}

/* --------------------------------------------------------------- layer */

typedef struct {
    int H, I, E, k;
    int has_shared, I_shared;
    double eps;
    oq_matrix router;         /* [E, H] */
    oq_matrix sgate;          /* [1, H] (has_shared) */
    const oq_matrix *gate;    /* E entries of [I, H]; unselected experts may be empty */
    const oq_matrix *up;      /* E entries of [I, H] */
    const oq_matrix *down;    /* E entries of [H, I] */
    oq_matrix shared_gate;    /* [I_s, H] */
    oq_matrix shared_up;      /* [I_s, H] */
    oq_matrix shared_down;    /* [H, I_s] */
    const uint16_t *gamma;    /* [H] bf16 */
    const uint16_t *gamma_next; /* [H] bf16 or NULL */
} oq_layer;

/* RMSNorm of one bf16 row: hn = x / sqrt(mean(x^2) + eps) * gamma
 * (flash-moe "Metal Compute Shaders": RMS normalisation). */
void oracle_rmsnorm(const uint16_t *x, const uint16_t *gamma, int H, double eps, double *hn)
{
    double ss = 0.0;
    for (int j = 0; j < H; ++j) {
        double v = oracle_bf16_to_double(x[j]);
        ss += v * v;
    }
    double rms = sqrt(ss / (double)H + eps);
    for (int j = 0; j < H; ++j)
        hn[j] = oracle_bf16_to_double(x[j]) / rms * oracle_bf16_to_double(gamma[j]);
}

/* Top-k routing of one row ([MC] "Summary": top-8 of 256 kept in full).
 * p = softmax(logits) over all E experts; the experts are ordered by a full
 * brute-force sort on (logit descending, expert id ascending); the first k
 * are kept and w_i = p_i / sum of the k kept p.  margin = smallest gap between
 * consecutive logits among the k+1 largest (k largest when k == E). */
void oracle_topk(const double *logits, int E, int k, int *idx, double *w, double *probs, double *margin)
{
    double mx = logits[0];
    for (int e = 1; e < E; ++e) if (logits[e] > mx) mx = logits[e];
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    double z = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp(logits[e] - mx); z += p[e]; }
    for (int e = 0; e < E; ++e) p[e] /= z;
    if (probs) for (int e = 0; e < E; ++e) probs[e] = p[e];
    /* insertion sort: obviously correct, O(E^2) */
    for (int e = 0; e < E; ++e) order[e] = e;
    for (int i = 1; i < E; ++i) {
        int cur = order[i];
        int j = i - 1;
        while (j >= 0 && (logits[order[j]] < logits[cur] ||
                          (logits[order[j]] == logits[cur] && order[j] > cur))) {
            order[j + 1] = order[j];
            --j;
        }
        order[j + 1] = cur;
    }
    double ps = 0.0;
    for (int i = 0; i < k; ++i) ps += p[order[i]];
    for (int i = 0; i < k; ++i) { idx[i] = order[i]; w[i] = p[order[i]] / ps; }
    if (margin) {
        int last = k < E ? k : E - 1;
        double m = INFINITY;
        for (int i = 0; i < last; ++i) {
            double gap = logits[order[i]] - logits[order[i + 1]];
            if (gap < m) m = gap;
        }
        *margin = m;
    }
    free(p);
    free(order);
}

static double silu(double z) { return z / (1.0 + exp(-z)); }
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* One expert FFN: y = W_d (silu(W_g hn) * (W_u hn)), [FM] "Metal Compute
 * Shaders" (dequant mat-vec and SwiGLU). */
void oracle_expert_ffn(const oq_matrix *gate, const oq_matrix *up, const oq_matrix *down,
                       const double *hn, double *y)
{
    int I = gate->rows;
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    double *a = (double *)malloc(sizeof(double) * (size_t)I);
    matvec(gate, hn, g);
    matvec(up, hn, u);
    for (int j = 0; j < I; ++j) a[j] = silu(g[j]) * u[j];
    matvec(down, a, y);
    free(g);
    free(u);
    free(a);
}

/* Routing for M rows: logits [M, E], idx/w [M, k], sigma [M] (shared-expert
 * gate, 0 without a shared expert), margin [M].  Needs only the router, the
 * shared-gate vector and gamma. */
void oracle_route(const oq_layer *L, const uint16_t *x, int M,
                  double *logits, int *idx, double *w, double *sigma, double *margin)
{
    double *hn = (double *)malloc(sizeof(double) * (size_t)L->H);
    for (int m = 0; m < M; ++m) {
        oracle_rmsnorm(x + (size_t)m * L->H, L->gamma, L->H, L->eps, hn);
        matvec(&L->router, hn, logits + (size_t)m * L->E);
        oracle_topk(logits + (size_t)m * L->E, L->E, L->k, idx + (size_t)m * L->k,
                    w + (size_t)m * L->k, NULL, margin ? margin + m : NULL);
        double sg = 0.0;
        if (L->has_shared) matvec(&L->sgate, hn, &sg);
        sigma[m] = L->has_shared ? sigmoid(sg) : 0.0;
    }
    free(hn);
}

/* The whole layer for M rows (rows never interact).
 *   o      [M, H]  x + sum_i w_i y_i + sigma y_s, before rounding
 *   out    [M, H]  bf16(o)
 *   on     [M, H]  RMSNorm(out) * gamma_next before rounding (NULL to skip)
 *   out_n  [M, H]  bf16(on) (NULL to skip)
 * plus the routing outputs of oracle_route.  Returns 0, or -(1 + e) when the
 * data of a selected expert e was not supplied. */
int oracle_layer(const oq_layer *L, const uint16_t *x, int M,
                 double *o, uint16_t *out, double *on, uint16_t *out_n,
                 double *logits, int *idx, double *w, double *sigma, double *margin)
{
    const int H = L->H;
    oracle_route(L, x, M, logits, idx, w, sigma, margin);
    for (int m = 0; m < M; ++m)
        for (int i = 0; i < L->k; ++i) {
            int e = idx[(size_t)m * L->k + i];
            if (!matrix_present(&L->gate[e]) || !matrix_present(&L->up[e]) || !matrix_present(&L->down[e]))
                return -(1 + e);
        }
    double *hn = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *ys = (double *)malloc(sizeof(double) * (size_t)H);
    for (int m = 0; m < M; ++m) {
        const uint16_t *xm = x + (size_t)m * H;
        double *om = o + (size_t)m * H;
        oracle_rmsnorm(xm, L->gamma, H, L->eps, hn);
        for (int h = 0; h < H; ++h) om[h] = oracle_bf16_to_double(xm[h]);   /* residual */
        for (int i = 0; i < L->k; ++i) {
            int e = idx[(size_t)m * L->k + i];
            oracle_expert_ffn(&L->gate[e], &L->up[e], &L->down[e], hn, y);
            for (int h = 0; h < H; ++h) om[h] += w[(size_t)m * L->k + i] * y[h];
        }
        if (L->has_shared) {
            oracle_expert_ffn(&L->shared_gate, &L->shared_up, &L->shared_down, hn, ys);
            for (int h = 0; h < H; ++h) om[h] += sigma[m] * ys[h];
        }
        for (int h = 0; h < H; ++h) out[(size_t)m * H + h] = oracle_bf16_from_double(om[h]);
        if (on && L->gamma_next) {
            /* fused next RMSNorm on the bf16 residual ([MC] "How it works":
             * fused add+RMSNorm) */
            double ss = 0.0;
            for (int h = 0; h < H; ++h) {
                double v = oracle_bf16_to_double(out[(size_t)m * H + h]);
                ss += v * v;
            }
            double rms = sqrt(ss / (double)H + L->eps);
            for (int h = 0; h < H; ++h) {
                double v = oracle_bf16_to_double(out[(size_t)m * H + h]) / rms *
                           oracle_bf16_to_double(L->gamma_next[h]);
                on[(size_t)m * H + h] = v;
                if (out_n) out_n[(size_t)m * H + h] = oracle_bf16_from_double(v);
            }
        }
    }
    free(hn);
    free(y);
    free(ys);
    return 0;
}

/* ------------------------------------------------ GQA decode attention */
/*
 * Decode-step attention over a bf16 key/value cache with grouped query
 * heads ([MC] "How it works": one attention kernel serves the one-row decode
 * and the multi-row verify, reading K/V once for all 8 query heads of a
 * key/value head and all verify rows; "Beyond this checkpoint": 16 query
 * heads, 2 key/value heads, head dimension 256).  The verify rows sit at
 * consecutive positions: row m is at position pos0 + m and attends to keys
 * 0 .. pos0 + m (its own included), the plain softmax attention
 *     o[m][h] = sum_t softmax_t(q[m][h] . k[g][t] / sqrt(D)) v[g][t],
 * g = h / (Hq / Hkv).  Layouts: q [M][Hq][D]; k [Hkv][T_cap][D]; v stored
 * transposed, vt [Hkv][D][T_cap] (position fastest); o and oabs [M][Hq][D],
 * oabs the same softmax-weighted sum of |v| (a scale for tolerances).
 * fp64 throughout; the softmax subtracts the row maximum before exp.
 * Returns 0, or -1 when the arguments are inconsistent or memory runs out.
 */
int oracle_gqa_decode(const uint16_t *q, const uint16_t *k, const uint16_t *vt, int T_cap, int pos0, int M,
                      int Hq, int Hkv, int D, double *o, double *oabs)
{
    if (M < 1 || Hkv < 1 || Hq % Hkv != 0 || D < 1 || pos0 < 0 || pos0 + M > T_cap) return -1;
    const int grp = Hq / Hkv, n_all = pos0 + M;
    const double scale = 1.0 / sqrt((double)D);
    double *s = (double *)malloc(sizeof(double) * (size_t)n_all);
    if (!s) return -1;
    for (int m = 0; m < M; ++m) {
        const int n = pos0 + m + 1;
        for (int h = 0; h < Hq; ++h) {
            const int g = h / grp;
            const uint16_t *qv = q + ((size_t)m * Hq + h) * D;
            double mx = -INFINITY;
            for (int t = 0; t < n; ++t) {
                const uint16_t *kv = k + ((size_t)g * T_cap + t) * D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += oracle_bf16_to_double(qv[d]) * oracle_bf16_to_double(kv[d]);
                s[t] = acc * scale;
                if (s[t] > mx) mx = s[t];
            }
            double z = 0.0;
            for (int t = 0; t < n; ++t) {
                s[t] = exp(s[t] - mx);
                z += s[t];
            }
            for (int d = 0; d < D; ++d) {
                const uint16_t *vrow = vt + ((size_t)g * D + d) * T_cap;
                double acc = 0.0, aacc = 0.0;
                for (int t = 0; t < n; ++t) {
                    const double v = oracle_bf16_to_double(vrow[t]);
                    acc += s[t] * v;
                    aacc += s[t] * fabs(v);
                }
                o[((size_t)m * Hq + h) * D + d] = acc / z;
                oabs[((size_t)m * Hq + h) * D + d] = aacc / z;
            }
        }
    }
    free(s);
    return 0;
}
