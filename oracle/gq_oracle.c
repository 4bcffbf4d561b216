/*
 * gq_oracle.c -- plain, slow, obviously correct CPU oracle for the
 * block-quantized matvec path.  TEST INFRASTRUCTURE ONLY: it is used by the
 * test suite, by the smoke check and by the benchmark's CPU-baseline leg,
 * and never by the product path.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Every weight is decoded from the CANONICAL block bytes into double, and
 * every sum is accumulated in double, in the order the definition states.
 *
 * Sources (page title, section):
 *   [ROADMAP]  "Gemma 4 M4 Max kernel roadmap" (gem, docs/research/
 *              kernel-roadmap.md): K1 "reference correctness core" (scalar F32
 *              dequantization, matrix-vector, GELU-gated FFN, logit
 *              soft-capping, compared against a high-precision reference);
 *              K2 "Metal decode path" steps 1, 5 and 6 (fused-dequant Q4_0
 *              matvec with F32 accumulation, gated GELU FFN pair, Q8_0 tied
 *              logit projection with top-k); K3 "prefill path" (batched Q4_0
 *              matrix-matrix); K4/K5 (top-k selection, exact full-sort parity).
 *   [LARQL]    "Metal kernel capability table (Phase B ground truth)":
 *              section 1 "Quant matvec family" (Q4_0 18 B, Q4_K 144 B,
 *              Q8_0 int8 blocks), section 2 (quantize_q8: f32 -> int8 plus
 *              per-32 scales), section 4 "FFN family" (GELU-tanh, clamp at
 *              +-15), section 8 findings F1, F6, F17.
 *
 * Block formats (the GGUF conventions; the pages fix only the byte sizes):
 *   Q4_0 (18 B / 32 weights): fp16 d, then 16 bytes; byte j holds element j
 *        in its low nibble and element j+16 in its high nibble;
 *        w = (q - 8) * d.
 *   Q8_0 (34 B / 32 weights): fp16 d, then 32 int8 q; w = q * d.
 *   Q4_K (144 B / 256 weights): fp16 d, fp16 dmin, 12 bytes of packed 6-bit
 *        sub-scales sc[8] and mins m[8], then 128 bytes of nibbles in four
 *        32-byte chunks; chunk c holds sub-block 2c in its low nibbles and
 *        sub-block 2c+1 in its high nibbles; w = d*sc*q - dmin*m.
 *   Q6_K (210 B / 256 weights; [LARQL] section 1 "Q6_K 210B"): 128 bytes ql
 *        (low 4 bits of the codes), 64 bytes qh (top 2 bits), 16 int8
 *        sub-scales (one per 16 weights), then fp16 d.  Each half of 128
 *        weights uses 64 bytes of ql and 32 of qh; in a half, weight 32*c + l
 *        (c = 0..3, l = 0..31) takes its low bits from ql byte l + 32*(c%2)
 *        (low nibble for c < 2, high nibble otherwise) and its top bits from
 *        bits 2c, 2c+1 of qh byte l; w = d * sc[weight/16] * (q - 32).
 *
 * Parity unpinned: bit compatibility with real GGUF files (nibble order of
 * Q4_0, 6-bit packing of Q4_K, bit placement of Q6_K) -- no GGUF file is
 * available to compare with.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GQO_Q4_0 0
#define GQO_Q8_0 1
#define GQO_Q4_K 2
#define GQO_Q6_K 3

/* IEEE binary16 -> double, exact (every half is a double). */
static double half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24); /* subnormal: mant * 2^-24 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(mant | 0x400), expo - 25); /* (1024+mant) * 2^(e-25) */
    return sign ? -v : v;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

double gqo_half_to_double(uint16_t h) { return half_to_double(h); }

/* ---- block decoding ------------------------------------------------------ */

/* Q4_0: w = (q - 8) * d. */
void gqo_dequant_q4_0(const uint8_t *blocks, int64_t nblocks, double *out)
{
    for (int64_t b = 0; b < nblocks; ++b) {
        const uint8_t *blk = blocks + b * 18;
        double d = half_to_double(rd16(blk));
        const uint8_t *qs = blk + 2;
        for (int j = 0; j < 16; ++j) {
            int lo = qs[j] & 0x0f;
            int hi = qs[j] >> 4;
            out[b * 32 + j] = (double)(lo - 8) * d;
            out[b * 32 + j + 16] = (double)(hi - 8) * d;
        }
    }
}

/* Q8_0: w = q * d. */
void gqo_dequant_q8_0(const uint8_t *blocks, int64_t nblocks, double *out)
{
    for (int64_t b = 0; b < nblocks; ++b) {
        const uint8_t *blk = blocks + b * 34;
        double d = half_to_double(rd16(blk));
        const int8_t *qs = (const int8_t *)(blk + 2);
        for (int j = 0; j < 32; ++j)
            out[b * 32 + j] = (double)qs[j] * d;
    }
}

/* Q4_K sub-scale and min of sub-block s (0..7) from the 12 packed bytes.
 * Sub-blocks 0..3 keep their 6 bits in the low bits of bytes s (scale) and
 * s+4 (min).  Sub-blocks 4..7 take their low 4 bits from byte s+4 (scale in
 * the low nibble, min in the high nibble) and their top 2 bits from the top
 * 2 bits of bytes s-4 (scale) and s (min). */
void gqo_q4_k_scale_min(const uint8_t *sc12, int s, int *sc, int *m)
{
    if (s < 4) {
        *sc = sc12[s] & 63;
        *m = sc12[s + 4] & 63;
    } else {
        *sc = (sc12[s + 4] & 0x0f) | ((sc12[s - 4] >> 6) << 4);
        *m = (sc12[s + 4] >> 4) | ((sc12[s] >> 6) << 4);
    }
}

/* Q4_K: w = d * sc_s * q - dmin * m_s for an element of sub-block s. */
void gqo_dequant_q4_k(const uint8_t *blocks, int64_t nsuper, double *out)
{
    for (int64_t b = 0; b < nsuper; ++b) {
        const uint8_t *blk = blocks + b * 144;
        double d = half_to_double(rd16(blk));
        double dmin = half_to_double(rd16(blk + 2));
        const uint8_t *sc12 = blk + 4;
        const uint8_t *qs = blk + 16;
        for (int s = 0; s < 8; ++s) {
            int sc, m;
            gqo_q4_k_scale_min(sc12, s, &sc, &m);
            const uint8_t *chunk = qs + 32 * (s / 2);
            for (int l = 0; l < 32; ++l) {
                int q = (s % 2 == 0) ? (chunk[l] & 0x0f) : (chunk[l] >> 4);
                out[b * 256 + s * 32 + l] = d * (double)sc * (double)q - dmin * (double)m;
            }
        }
    }
}

/* Q6_K: w = d * sc[e/16] * (q_e - 32), q_e from 4 bits of ql and 2 of qh. */
void gqo_dequant_q6_k(const uint8_t *blocks, int64_t nsuper, double *out)
{
    for (int64_t b = 0; b < nsuper; ++b) {
        const uint8_t *blk = blocks + b * 210;
        const uint8_t *ql = blk, *qh = blk + 128;
        const int8_t *sc = (const int8_t *)(blk + 192);
        double d = half_to_double(rd16(blk + 208));
        for (int e = 0; e < 256; ++e) {
            int half = e / 128, c = (e % 128) / 32, l = e % 32;
            int lowbyte = ql[64 * half + l + 32 * (c % 2)];
            int lo = (c < 2) ? (lowbyte & 0x0f) : (lowbyte >> 4);
            int hi = (qh[32 * half + l] >> (2 * c)) & 3;
            int q = lo | (hi << 4);
            out[b * 256 + e] = d * (double)sc[e / 16] * (double)(q - 32);
        }
    }
}

static int64_t row_bytes(int fmt, int64_t K)
{
    switch (fmt) {
    case GQO_Q4_0: return K / 32 * 18;
    case GQO_Q8_0: return K / 32 * 34;
    case GQO_Q4_K: return K / 256 * 144;
    case GQO_Q6_K: return K / 256 * 210;
    }
    return -1;
}

/* Decode one whole row of K weights into w[K]. */
static void dequant_row(int fmt, const uint8_t *row, int64_t K, double *w)
{
    switch (fmt) {
    case GQO_Q4_0: gqo_dequant_q4_0(row, K / 32, w); break;
    case GQO_Q8_0: gqo_dequant_q8_0(row, K / 32, w); break;
    case GQO_Q4_K: gqo_dequant_q4_k(row, K / 256, w); break;
    case GQO_Q6_K: gqo_dequant_q6_k(row, K / 256, w); break;
    }
}

/* ---- matvec -------------------------------------------------------------- */

/* y_i = sum_j w_ij x_j, accumulated in double in ascending j, and the
 * tolerance scale a_i = sum_j |w_ij x_j| ([ROADMAP] K1; K2 step 1).
 * row_idx lists the rows to compute (NULL: all rows 0..n_sel-1).
 * Returns 0, or -1 for an unknown format or a K that is not whole blocks. */
int gqo_matvec(int fmt, const uint8_t *W, int64_t rows, int64_t K, const float *x,
               const int64_t *row_idx, int64_t n_sel, double *y, double *a)
{
    int64_t rb = row_bytes(fmt, K);
    if (rb < 0 || K <= 0 || K % ((fmt == GQO_Q4_K || fmt == GQO_Q6_K) ? 256 : 32) != 0)
        return -1;
    (void)rows;
#pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t i = 0; i < n_sel; ++i) {
            int64_t r = row_idx ? row_idx[i] : i;
            dequant_row(fmt, W + r * rb, K, w);
            double acc = 0.0, aacc = 0.0;
            for (int64_t j = 0; j < K; ++j) {
                double p = w[j] * (double)x[j];
                acc += p;
                aacc += fabs(p);
            }
            y[i] = acc;
            if (a)
                a[i] = aacc;
        }
        free(w);
    }
    return 0;
}

/* ---- epilogues ------------------------------------------------------------ */

/* GELU, tanh form: 0.5 a (1 + tanh(sqrt(2/pi) (a + 0.044715 a^3))), with the
 * tanh argument clamped to +-15 as the separated GELU-tanh kernels of [LARQL]
 * section 4 do (finding F1 is the NaN an unclamped tanh gave). */
double gqo_gelu_tanh(double a)
{
    const double k = sqrt(2.0 / acos(-1.0)); /* sqrt(2/pi) */
    double t = k * (a + 0.044715 * a * a * a);
    if (t > 15.0) t = 15.0;
    if (t < -15.0) t = -15.0;
    return 0.5 * a * (1.0 + tanh(t));
}

/* Logit soft-cap c * tanh(v / c) ([ROADMAP] K1); c <= 0 leaves v unchanged. */
double gqo_softcap(double v, double cap)
{
    if (!(cap > 0.0))
        return v;
    return cap * tanh(v / cap);
}

/* Gated GELU FFN gate/up pair ([ROADMAP] K1 and K2 step 5):
 * g = W_gate x, u = W_up x, h = gelu_tanh(g) * u, for the selected rows.
 * ag, au are the tolerance scales of g and u (any of g/u/ag/au may be NULL). */
int gqo_ffn_gate_up(const uint8_t *Wg, const uint8_t *Wu, int64_t rows, int64_t K,
                    const float *x, const int64_t *row_idx, int64_t n_sel,
                    double *g, double *u, double *ag, double *au, double *h)
{
    double *gg = (double *)malloc(sizeof(double) * (size_t)(n_sel > 0 ? n_sel : 1));
    double *uu = (double *)malloc(sizeof(double) * (size_t)(n_sel > 0 ? n_sel : 1));
    int rc = gqo_matvec(GQO_Q4_0, Wg, rows, K, x, row_idx, n_sel, gg, ag);
    if (rc == 0)
        rc = gqo_matvec(GQO_Q4_0, Wu, rows, K, x, row_idx, n_sel, uu, au);
    if (rc == 0) {
        for (int64_t i = 0; i < n_sel; ++i) {
            if (g) g[i] = gg[i];
            if (u) u[i] = uu[i];
            h[i] = gqo_gelu_tanh(gg[i]) * uu[i];
        }
    }
    free(gg);
    free(uu);
    return rc;
}

/* Down projection of a gated GELU FFN with the gate applied to its input
 * ([LARQL] section 4: the fused GELU-tanh down kernels, which take the gate
 * and up vectors; finding F1: the tanh argument is clamped, as
 * gqo_gelu_tanh does):
 *   h_j = gelu_tanh(g_j) * u_j,   y_i = sum_j w_ij h_j   (double, ascending j)
 * for the selected rows, with the tolerance scales
 *   a_i = sum_j |w_ij h_j|,   b_i = sum_j |w_ij| (|g_j u_j| + |h_j|)
 * (a or b may be NULL).  Returns 0, or -1 as gqo_matvec. */
int gqo_geglu_down(int fmt, const uint8_t *W, int64_t rows, int64_t K, const float *g,
                   const float *u, const int64_t *row_idx, int64_t n_sel, double *y, double *a,
                   double *b)
{
    int64_t rb = row_bytes(fmt, K);
    if (rb < 0 || K <= 0 || K % ((fmt == GQO_Q4_K || fmt == GQO_Q6_K) ? 256 : 32) != 0)
        return -1;
    (void)rows;
    double *h = (double *)malloc(sizeof(double) * (size_t)K);
    double *e = (double *)malloc(sizeof(double) * (size_t)K);
    for (int64_t j = 0; j < K; ++j) {
        h[j] = gqo_gelu_tanh((double)g[j]) * (double)u[j];
        e[j] = fabs((double)g[j] * (double)u[j]) + fabs(h[j]);
    }
#pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t i = 0; i < n_sel; ++i) {
            int64_t r = row_idx ? row_idx[i] : i;
            dequant_row(fmt, W + r * rb, K, w);
            double acc = 0.0, aacc = 0.0, bacc = 0.0;
            for (int64_t j = 0; j < K; ++j) {
                double p = w[j] * h[j];
                acc += p;
                aacc += fabs(p);
                bacc += fabs(w[j]) * e[j];
            }
            y[i] = acc;
            if (a) a[i] = aacc;
            if (b) b[i] = bacc;
        }
        free(w);
    }
    free(h);
    free(e);
    return 0;
}

/* ---- top-k ------------------------------------------------------------- */

typedef struct {
    double v;
    int64_t i;
} gqo_pair;

/* Ranking rule: larger value first; equal values by lower index; NaN after
 * every number (NaNs among themselves by lower index); -0 equals +0. */
static int pair_cmp(const void *pa, const void *pb)
{
    const gqo_pair *a = (const gqo_pair *)pa, *b = (const gqo_pair *)pb;
    int an = isnan(a->v), bn = isnan(b->v);
    if (an != bn)
        return an ? 1 : -1;
    if (!an) {
        if (a->v > b->v) return -1;
        if (a->v < b->v) return 1;
    }
    return (a->i < b->i) ? -1 : (a->i > b->i) ? 1 : 0;
}

/* Top-k by a full sort of all n (value, index) pairs -- the exhaustive
 * selection that [ROADMAP] K4 keeps as the parity reference for its bounded
 * selection.  Writes the first k pairs (k <= n). */
int gqo_topk(const double *v, int64_t n, int64_t k, int64_t *idx, double *val)
{
    if (k < 0 || k > n)
        return -1;
    gqo_pair *p = (gqo_pair *)malloc(sizeof(gqo_pair) * (size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i) {
        p[i].v = v[i];
        p[i].i = i;
    }
    qsort(p, (size_t)n, sizeof(gqo_pair), pair_cmp);
    for (int64_t i = 0; i < k; ++i) {
        idx[i] = p[i].i;
        val[i] = p[i].v;
    }
    free(p);
    return 0;
}

/* ---- Q8_0 activation quantization --------------------------------------- */

/* For every token t and 32-element block b of X (M x K, row-major f32):
 *   amax = max |x|;  d = amax / 127;  q = clamp(round(x / d), -127, 127)
 * in f32 arithmetic with IEEE-rounded division and round-half-away-from-zero;
 * an all-zero block gives d = 0 and q = 0 ([LARQL] section 2 quantize_q8:
 * f32 -> int8 plus per-32 external f32 scales; F6: every block's scale is
 * written).  q is M x K int8, d is M x (K/32) f32. */
int gqo_quantize_q8_0(const float *X, int64_t M, int64_t K, int8_t *q, float *d)
{
    if (K <= 0 || K % 32 != 0)
        return -1;
    int64_t nb = K / 32;
    for (int64_t t = 0; t < M; ++t) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = X + t * K + b * 32;
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                float ax = fabsf(xb[j]);
                if (ax > amax)
                    amax = ax;
            }
            volatile float dd = amax / 127.0f; /* f32 division, no excess precision */
            float dv = dd;
            d[t * nb + b] = dv;
            for (int j = 0; j < 32; ++j) {
                int qi = 0;
                if (dv != 0.0f) {
                    volatile float r = xb[j] / dv;
                    float rr = roundf(r);
                    if (rr > 127.0f) rr = 127.0f;
                    if (rr < -127.0f) rr = -127.0f;
                    qi = (int)rr;
                }
                q[t * K + b * 32 + j] = (int8_t)qi;
            }
        }
    }
    return 0;
}

/* ---- Q4_0 x Q8_0 prefill contraction ------------------------------------ */

/* Integer block dot products ([ROADMAP] K3 batched Q4_0 matrix-matrix, with
 * the activations in Q8_0):
 *   D[t][r][b] = sum_{j<32} qx[t, 32b+j] * (qw[r, 32b+j] - 8)
 * for tokens t0..t0+nt-1 and rows r0..r0+nr-1, all blocks b, in int32.
 * D is nt x nr x (K/32). */
int gqo_block_dots(const uint8_t *W, const int8_t *Xq, int64_t rows, int64_t K, int64_t M,
                   int64_t t0, int64_t nt, int64_t r0, int64_t nr, int32_t *D)
{
    if (K <= 0 || K % 32 != 0 || t0 < 0 || t0 + nt > M || r0 < 0 || r0 + nr > rows)
        return -1;
    int64_t nb = K / 32;
    for (int64_t ti = 0; ti < nt; ++ti) {
        const int8_t *xq = Xq + (t0 + ti) * K;
        for (int64_t ri = 0; ri < nr; ++ri) {
            const uint8_t *row = W + (r0 + ri) * nb * 18;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *qs = row + b * 18 + 2;
                int32_t acc = 0;
                for (int j = 0; j < 16; ++j) {
                    int lo = (qs[j] & 0x0f) - 8;
                    int hi = (qs[j] >> 4) - 8;
                    acc += (int32_t)xq[b * 32 + j] * lo;
                    acc += (int32_t)xq[b * 32 + j + 16] * hi;
                }
                D[(ti * nr + ri) * nb + b] = acc;
            }
        }
    }
    return 0;
}

/* Y[t][r] = sum_b d_w[r,b] * d_x[t,b] * D[t][r][b], summed in double, and
 * A[t][r] = sum_b |d_w d_x D| (the tolerance scale), for the selected tokens
 * and rows (NULL index lists select all).  Y and A are n_tok x n_row. */
int gqo_gemm_q8act(const uint8_t *W, const int8_t *Xq, const float *dx, int64_t rows,
                   int64_t K, int64_t M, const int64_t *tok_idx, int64_t n_tok,
                   const int64_t *row_idx, int64_t n_row, double *Y, double *A)
{
    if (K <= 0 || K % 32 != 0)
        return -1;
    int64_t nb = K / 32;
    (void)M;
    (void)rows;
#pragma omp parallel for schedule(static)
    for (int64_t ri = 0; ri < n_row; ++ri) {
        int64_t r = row_idx ? row_idx[ri] : ri;
        const uint8_t *row = W + r * nb * 18;
        for (int64_t ti = 0; ti < n_tok; ++ti) {
            int64_t t = tok_idx ? tok_idx[ti] : ti;
            const int8_t *xq = Xq + t * K;
            double acc = 0.0, aacc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *blk = row + b * 18;
                double dw = half_to_double(rd16(blk));
                int32_t dot = 0;
                for (int j = 0; j < 16; ++j) {
                    dot += (int32_t)xq[b * 32 + j] * ((blk[2 + j] & 0x0f) - 8);
                    dot += (int32_t)xq[b * 32 + j + 16] * ((blk[2 + j] >> 4) - 8);
                }
                double term = dw * (double)dx[t * nb + b] * (double)dot;
                acc += term;
                aacc += fabs(term);
            }
            Y[ti * n_row + ri] = acc;
            if (A)
                A[ti * n_row + ri] = aacc;
        }
    }
    return 0;
}

/* Threads of the row-parallel loops above (OpenMP builds; a no-op otherwise):
 * lets a caller time the oracle on one core and on all of them in one process.
 * Test and measurement infrastructure only; no arithmetic depends on it. */
#ifdef _OPENMP
#include <omp.h>
#endif
void gqo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
