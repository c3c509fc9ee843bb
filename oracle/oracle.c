/*
 * oracle.c — plain CPU oracle for one decode step of a Llama-style decoder
 * stack plus LM head.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  The product decode path never
 * calls it and shares no code with it.
 *
 * What it computes.  The MegaKernel papers fuse "the Transformer Decoder and
 * LM Head" of one decode step into one persistent kernel without changing
 * what is computed (Ada-MK technical summary, gist.science, Methodology,
 * Phase I; AutoMegaKernel abstract: the fused kernel reproduces HuggingFace
 * greedy decode token for token).  So the oracle is the plain, unfused
 * definition of that step for a HuggingFace Llama-family decoder, with
 * 16-bit activations (the A16 of W4A16/W8A16 in the Ada-MK summary,
 * Contribution 4, and the AutoMegaKernel abstract's W8A16 kernel):
 *
 *   x  = E[token]
 *   per layer:
 *     h  = bf16(rmsnorm(x) * g_attn)
 *     q, k, v = Wq h, Wk h, Wv h            (int8: s_row * sum_i w_i h_i)
 *     rotate q and k by RoPE at position p   (rotate-half pairs (i, i+d/2))
 *     Kc[p], Vc[p] = bf16(k), bf16(v)
 *     o_j = softmax_m(q_j . Kc[m] / sqrt(d)) . Vc[m],  m = 0..p,
 *           q head j reading kv head j / (n_heads / n_kv_heads)
 *     x += Wo bf16(o)
 *     h2 = bf16(rmsnorm(x) * g_mlp)
 *     a  = bf16(silu(Wg h2) * (Wu h2))
 *     x += Wd a
 *   logits = W_lm bf16(rmsnorm(x) * g_final)
 *
 * Arithmetic: every sum, product and transcendental is taken in IEEE double,
 * in the plain loop order (one accumulator per output, index ascending);
 * the only roundings are the bf16 ones written above.  There is no tiling,
 * fusion, split or reordering.  OpenMP splits independent outputs (matrix
 * rows, attention heads) across threads; no sum is split.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* GEMV accumulator.  The oracle accumulates in double.  Built with
 * -DORC_ACC_FLOAT it rounds every partial sum to float instead: that build is
 * not the oracle, it measures how far a plain fp32 implementation of the same
 * definition lands from it (the model's own rounding sensitivity). */
#ifdef ORC_ACC_FLOAT
typedef float acc_t;
#else
typedef double acc_t;
#endif

/* ------------------------------------------------------------ bf16 */

double orc_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to the nearest bf16 (8-bit significand), ties to even.
 * y = f * 2^e with f in [0.5, 1); the bf16 significand is f * 2^8 rounded to
 * an integer (nearbyint in the default to-nearest-even mode; the scaling by a
 * power of two is exact).  The result is a bf16 value, hence exactly
 * representable as float; its top 16 bits are the bf16 pattern. */
uint16_t orc_double_to_bf16(double y) {
    if (isnan(y)) return 0x7fc0;
    float f;
    if (y == 0.0 || isinf(y)) {
        f = (float)y;
    } else {
        int e;
        double m = frexp(y, &e);
        if (e < -125) {
            /* |y| < 2^-126: bf16 subnormal range, spacing 2^-133 */
            f = (float)ldexp(nearbyint(ldexp(y, 133)), -133);
        } else {
            double v = ldexp(nearbyint(ldexp(m, 8)), e - 8);
            const double bf16_max = 3.3895313892515355e38; /* (2 - 2^-7) * 2^127 */
            f = (v > bf16_max) ? INFINITY : (v < -bf16_max) ? -INFINITY : (float)v;
        }
    }
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static double round_bf16(double y) { return orc_bf16_to_double(orc_double_to_bf16(y)); }

/* ------------------------------------------------------------ operators */

/* RMSNorm (Zhang & Sennrich 2019) with gain, unrounded:
 *   y_i = x_i * g_i / sqrt(mean_j x_j^2 + eps) */
void orc_rmsnorm(int n, const double *x, const uint16_t *gain, double eps, double *y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * r * orc_bf16_to_double(gain[i]);
}

/* y[o] = sum_i W[o][i] * h[i] for a bf16 [rows, K] row-major W, or
 * y[o] = s[o] * sum_i W8[o][i] * h[i] for int8 W with per-row scales. */
void orc_gemv(int rows, int K, const void *W, int w_int8, const float *scales,
              const uint16_t *h, double *y) {
    double *hd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int i = 0; i < K; ++i) hd[i] = orc_bf16_to_double(h[i]);
#pragma omp parallel for schedule(static)
    for (int o = 0; o < rows; ++o) {
        acc_t acc = 0;
        if (w_int8) {
            const int8_t *w = (const int8_t *)W + (size_t)o * K;
            for (int i = 0; i < K; ++i) acc += (double)w[i] * hd[i];
            y[o] = (double)scales[o] * acc;
        } else {
            const uint16_t *w = (const uint16_t *)W + (size_t)o * K;
            for (int i = 0; i < K; ++i) acc += orc_bf16_to_double(w[i]) * hd[i];
            y[o] = acc;
        }
    }
    free(hd);
}

/* y[o] = sum_g s[o][g] * sum_{i in group g} (u[o][i] - 8) * h[i] for 4-bit
 * weight codes u in [0, 15] around the zero point 8 (the symmetric 4-bit
 * weight-only quantisation of W4A16), packed two per byte with element 2j in
 * the low nibble of byte j, and one fp32 scale per `group` weights along K
 * (scales [rows][K / group]). */
void orc_gemv_int4(int rows, int K, int group, const uint8_t *W, const float *scales, const uint16_t *h,
                   double *y) {
    double *hd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int i = 0; i < K; ++i) hd[i] = orc_bf16_to_double(h[i]);
    const int ng = K / group;
#pragma omp parallel for schedule(static)
    for (int o = 0; o < rows; ++o) {
        const uint8_t *w = W + (size_t)o * (K / 2);
        double tot = 0.0;
        for (int g = 0; g < ng; ++g) {
            acc_t acc = 0;
            for (int i = g * group; i < (g + 1) * group; ++i) {
                const int u = (w[i / 2] >> (4 * (i & 1))) & 15;
                acc += (double)(u - 8) * hd[i];
            }
            tot += (double)scales[(size_t)o * ng + g] * acc;
        }
        y[o] = tot;
    }
    free(hd);
}

/* Rotary position embedding (Su et al., RoFormer 2021), rotate-half pairing:
 * for i < d/2, theta_i = pos * base^(-2i/d) and the pair (u_i, u_{i+d/2}) is
 * rotated by theta_i. */
void orc_rope(int d, int pos, double base, double *u) {
    int half = d / 2;
    for (int i = 0; i < half; ++i) {
        double th = (double)pos * pow(base, -2.0 * (double)i / (double)d);
        double c = cos(th), s = sin(th);
        double a = u[i], b = u[i + half];
        u[i] = a * c - b * s;
        u[i + half] = b * c + a * s;
    }
}

/* Single-query attention over n_pos cached positions (rows of Kc, Vc, each d
 * bf16 values): w = softmax(q . Kc[m] / sqrt(d)), o = sum_m w_m Vc[m].
 * w may be NULL; otherwise it receives the n_pos softmax weights. */
void orc_attention(int n_pos, int d, const double *q, const uint16_t *Kc, const uint16_t *Vc,
                   double *w, double *o) {
    double *s = (double *)malloc(sizeof(double) * (size_t)(n_pos > 0 ? n_pos : 1));
    double scale = 1.0 / sqrt((double)d);
    double mx = -INFINITY;
    for (int m = 0; m < n_pos; ++m) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += q[i] * orc_bf16_to_double(Kc[(size_t)m * d + i]);
        s[m] = acc * scale;
        if (s[m] > mx) mx = s[m];
    }
    double den = 0.0;
    for (int m = 0; m < n_pos; ++m) {
        s[m] = exp(s[m] - mx);
        den += s[m];
    }
    for (int m = 0; m < n_pos; ++m) s[m] /= den;
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int m = 0; m < n_pos; ++m) acc += s[m] * orc_bf16_to_double(Vc[(size_t)m * d + i]);
        o[i] = acc;
    }
    if (w) memcpy(w, s, sizeof(double) * (size_t)n_pos);
    free(s);
}

/* SiLU / swish (Elfwing et al. 2018; SwiGLU per Shazeer 2020): z * sigmoid(z) */
double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* Greedy choice: index of the largest value, the lowest index on ties. */
int orc_argmax(int n, const double *v) {
    int best = 0;
    for (int i = 1; i < n; ++i)
        if (v[i] > v[best]) best = i;
    return best;
}

/* ------------------------------------------------------------ model */

typedef struct {
    int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab;
    int32_t weight_int8;  /* 0: bf16 layer matrices; 1: int8 layer matrices + fp32 per-row scales */
    int32_t lm_head_int8; /* 1: the LM head is int8 with per-row scales */
    double rms_eps, rope_theta;
    int32_t weight_int4;  /* 1: 4-bit layer matrices + fp32 scales per `group_size` weights (orc_gemv_int4) */
    int32_t lm_head_int4; /* 1: the LM head is 4-bit as well */
    int32_t group_size;
} orc_config;

typedef struct {
    const uint16_t *attn_norm, *mlp_norm;          /* [H] bf16 gains */
    const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;  /* [out, in] row-major */
    const float *sq, *sk, *sv, *so, *sg, *su, *sd; /* int8: per-row scales; int4: [out][in / group_size] */
} orc_layer;

/* one layer matrix in the model's weight format */
static void mat_vec(const orc_config *c, int lm, int rows, int K, const void *W, const float *s, const uint16_t *h,
                    double *y) {
    if (lm ? c->lm_head_int4 : c->weight_int4)
        orc_gemv_int4(rows, K, c->group_size, (const uint8_t *)W, s, h, y);
    else
        orc_gemv(rows, K, W, lm ? c->lm_head_int8 : c->weight_int8, s, h, y);
}

typedef struct {
    const uint16_t *embed;      /* [V, H] bf16 */
    const uint16_t *final_norm; /* [H] bf16 */
    const void *lm_head;        /* [V, H], bf16 or int8 */
    const float *s_lm;          /* [V], int8 only */
    const orc_layer *layers;    /* [n_layers] */
} orc_weights;

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

static void round_vec(int n, const double *y, uint16_t *out) {
    for (int i = 0; i < n; ++i) out[i] = orc_double_to_bf16(y[i]);
}

/*
 * Layer l of the decode step of sequence b at position p, applied in place to
 * the residual x[H].  Writes K/V slot p of (l, b) into the caches (layout
 * [L][Bmax][n_kv_heads][Smax][head_dim] bf16) before attending over slots
 * 0..p.  If x_mid is not NULL it receives the residual after attention.
 */
int orc_layer_forward(const orc_config *c, const orc_layer *w, int l, int b, int p, double *x,
                      uint16_t *kcache, uint16_t *vcache, int Bmax, int Smax, double *x_mid) {
    const int H = c->hidden, nq = c->n_heads, nkv = c->n_kv_heads, d = c->head_dim;
    const int I = c->intermediate;
    if (nkv < 1 || nq % nkv != 0 || d % 2 != 0 || p < 0 || p >= Smax || b < 0 || b >= Bmax) return -1;
    const int G = nq / nkv;
    double *y = malloc(sizeof(double) * (H > I ? H : I));
    double *q = malloc(sizeof(double) * nq * d), *k = malloc(sizeof(double) * nkv * d);
    double *v = malloc(sizeof(double) * nkv * d), *o = malloc(sizeof(double) * nq * d);
    double *gt = malloc(sizeof(double) * I), *up = malloc(sizeof(double) * I);
    uint16_t *hb = malloc(sizeof(uint16_t) * (H > I ? H : I));
    uint16_t *ob = malloc(sizeof(uint16_t) * nq * d);

    orc_rmsnorm(H, x, w->attn_norm, c->rms_eps, y);
    round_vec(H, y, hb);
    mat_vec(c, 0, nq * d, H, w->wq, w->sq, hb, q);
    mat_vec(c, 0, nkv * d, H, w->wk, w->sk, hb, k);
    mat_vec(c, 0, nkv * d, H, w->wv, w->sv, hb, v);
    for (int j = 0; j < nq; ++j) orc_rope(d, p, c->rope_theta, q + (size_t)j * d);
    for (int g = 0; g < nkv; ++g) orc_rope(d, p, c->rope_theta, k + (size_t)g * d);

    for (int g = 0; g < nkv; ++g) {
        size_t row = (((size_t)l * Bmax + b) * nkv + g) * (size_t)Smax;
        for (int i = 0; i < d; ++i) {
            kcache[(row + p) * d + i] = orc_double_to_bf16(k[(size_t)g * d + i]);
            vcache[(row + p) * d + i] = orc_double_to_bf16(v[(size_t)g * d + i]);
        }
    }
#pragma omp parallel for schedule(static)
    for (int j = 0; j < nq; ++j) {
        int g = j / G;
        size_t row = (((size_t)l * Bmax + b) * nkv + g) * (size_t)Smax;
        orc_attention(p + 1, d, q + (size_t)j * d, kcache + row * d, vcache + row * d, NULL,
                      o + (size_t)j * d);
    }
    round_vec(nq * d, o, ob);
    mat_vec(c, 0, H, nq * d, w->wo, w->so, ob, y);
    for (int i = 0; i < H; ++i) x[i] += y[i];
    if (x_mid) memcpy(x_mid, x, sizeof(double) * H);

    orc_rmsnorm(H, x, w->mlp_norm, c->rms_eps, y);
    round_vec(H, y, hb);
    mat_vec(c, 0, I, H, w->wg, w->sg, hb, gt);
    mat_vec(c, 0, I, H, w->wu, w->su, hb, up);
    for (int i = 0; i < I; ++i) hb[i] = orc_double_to_bf16(orc_silu(gt[i]) * up[i]);
    mat_vec(c, 0, H, I, w->wd, w->sd, hb, y);
    for (int i = 0; i < H; ++i) x[i] += y[i];

    free(y); free(q); free(k); free(v); free(o); free(gt); free(up); free(hb); free(ob);
    return 0;
}

/* Final RMSNorm and LM head: logits[V] = W_lm bf16(rmsnorm(x) * g_final). */
void orc_lm_head(const orc_config *c, const orc_weights *wt, const double *x, double *logits) {
    const int H = c->hidden;
    double *y = malloc(sizeof(double) * H);
    uint16_t *hb = malloc(sizeof(uint16_t) * H);
    orc_rmsnorm(H, x, wt->final_norm, c->rms_eps, y);
    round_vec(H, y, hb);
    mat_vec(c, 1, c->vocab, H, wt->lm_head, wt->s_lm, hb, logits);
    free(y);
    free(hb);
}

/*
 * One decode step for B sequences.  Sequence b decodes tokens[b] at
 * positions[b], reading and writing its own rows of the caches.
 * logits: [B][vocab] doubles.  x_trace, if not NULL, receives the residual
 * stream [B][L+1][H] at the input of every layer and after the last one.
 * Returns 0, or -1 on bad arguments.
 */
int orc_decode_step(const orc_config *c, const orc_weights *wt, int B, const int32_t *tokens,
                    const int32_t *positions, uint16_t *kcache, uint16_t *vcache, int Bmax, int Smax,
                    double *logits, double *x_trace) {
    const int L = c->n_layers, H = c->hidden, V = c->vocab;
    if (B < 1 || B > Bmax) return -1;
    for (int b = 0; b < B; ++b)
        if (tokens[b] < 0 || tokens[b] >= V || positions[b] < 0 || positions[b] >= Smax) return -1;
    double *x = malloc(sizeof(double) * H);
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        for (int i = 0; i < H; ++i) x[i] = orc_bf16_to_double(wt->embed[(size_t)tokens[b] * H + i]);
        for (int l = 0; l < L && rc == 0; ++l) {
            if (x_trace) memcpy(x_trace + ((size_t)b * (L + 1) + l) * H, x, sizeof(double) * H);
            rc = orc_layer_forward(c, &wt->layers[l], l, b, positions[b], x, kcache, vcache, Bmax, Smax, NULL);
        }
        if (x_trace) memcpy(x_trace + ((size_t)b * (L + 1) + L) * H, x, sizeof(double) * H);
        if (rc == 0) orc_lm_head(c, wt, x, logits + (size_t)b * V);
    }
    free(x);
    return rc;
}

/* exposed for pins of the rounding helper */
double orc_round_bf16(double y) { return round_bf16(y); }
