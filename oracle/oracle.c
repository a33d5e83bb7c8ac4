/*
 * oracle.c — plain, slow fp64 CPU reference of a Llama-style decoder: one
 * decode step over a KV cache, and a separate full-sequence causal forward.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * bench's CPU-baseline arm may load this code; the GPU library never does.
 * It shares no code, header or constant with the CUDA path.
 *
 * What it computes follows the decoder that the megakernel pages fuse into
 * their task lists:
 *   - "Llama-70B 向け…megakernel" (hakusoku.com/story/2591), section
 *     高スループットMegakernelの設計と工夫: fused instructions RMS norm, QKV
 *     matmul + RoPE, attention, O-proj matmul + residual;
 *   - "Cómo la fusión de kernels CUDA acelera la inferencia de LLM"
 *     (slavadubrov.com), section "Sigue los datos intermedios": residual add
 *     followed by RMSNorm, and the SwiGLU feed-forward (DeepFusionKernel);
 *   - "Compilar LLM en un MegaKernel…" (es.news.hada.io/topic?id=21563),
 *     "Parte 1. Compilador": the operator graph (matmul, attention) whose
 *     result the megakernel must reproduce exactly.
 * The pages fix no precision, norm epsilon, RoPE pairing or weight layout;
 * the readings taken here (rotate-half RoPE, eps inside the square root,
 * consecutive q heads sharing a kv head, causal window including the current
 * token, bf16 row-major [out][in] weights widened exactly) are the plainest
 * Llama readings and are listed with the design notes.
 *
 * Every floating-point operation is in double; weights and norm gains are
 * bf16 bit patterns widened exactly.  OpenMP only splits independent output
 * rows across threads; it never changes an individual sum.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    double rms_eps, rope_theta;
    /* nonzero: the cache stores each appended key and value as the nearest
     * bf16 value (the decoder's KV cache holds bf16; see orc_round_bf16) */
    int kv_bf16;
} orc_cfg;

/* Per-layer weights, bf16 bit patterns, row-major [out][in]. */
typedef struct {
    const uint16_t *attn_norm; /* [hidden] */
    const uint16_t *wq;        /* [n_q_heads*head_dim][hidden] */
    const uint16_t *wk;        /* [n_kv_heads*head_dim][hidden] */
    const uint16_t *wv;        /* [n_kv_heads*head_dim][hidden] */
    const uint16_t *wo;        /* [hidden][n_q_heads*head_dim] */
    const uint16_t *mlp_norm;  /* [hidden] */
    const uint16_t *w_gate;    /* [ffn_dim][hidden] */
    const uint16_t *w_up;      /* [ffn_dim][hidden] */
    const uint16_t *w_down;    /* [hidden][ffn_dim] */
} orc_layer_w;

typedef struct {
    const uint16_t *embed;      /* [vocab][hidden] */
    const uint16_t *lm_head;    /* [vocab][hidden]; equal to embed when tied */
    const uint16_t *final_norm; /* [hidden] */
    const orc_layer_w *layers;  /* [n_layers] */
} orc_weights;

/* Threads of the team that a parallel loop of this library runs with (what
 * a timed run of the oracle actually used; no arithmetic). */
int orc_num_threads(void) {
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
}

/* Team size of the later parallel loops of this library (timing only; no
 * arithmetic: every output row is still one sequential sum). */
void orc_set_num_threads(int n) {
    if (n > 0) omp_set_num_threads(n);
}

double orc_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* The bf16 value nearest to x, ties to the even significand: bf16 keeps 8
 * significant bits (1 implicit + 7 stored) over fp32's exponent range, so
 * for a finite nonzero x with 2^e <= |x| < 2^(e+1) the representable values
 * near x are the multiples of 2^(e-7).  (Every value here is far inside the
 * normal range; zeros and non-finite values pass through.) */
double orc_round_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    const double step = ldexp(1.0, ilogb(x) - 7);
    return nearbyint(x / step) * step; /* default rounding mode: to nearest, ties to even */
}

/* RMSNorm: y_i = g_i * x_i / sqrt(mean_j x_j^2 + eps). */
void orc_rmsnorm(int n, const double *x, const uint16_t *g, double eps, double *y) {
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; ++i) y[i] = orc_bf16(g[i]) * (x[i] * inv);
}

/* y = W x, W bf16 [rows][cols] row-major. */
void orc_matvec(int rows, int cols, const uint16_t *W, const double *x, double *y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const uint16_t *w = W + (size_t)r * cols;
        double acc = 0.0;
        for (int c = 0; c < cols; ++c) acc += orc_bf16(w[c]) * x[c];
        y[r] = acc;
    }
}

/* Rotary embedding of one head vector v[d] at position pos, rotate-half
 * pairing: element i is paired with i + d/2 (i < d/2), rotated by the angle
 * pos * theta^(-2i/d):  (a, b) -> (a cos - b sin, a sin + b cos). */
void orc_rope(int d, double *v, int pos, double theta) {
    int half = d / 2;
    for (int i = 0; i < half; ++i) {
        double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
        double ang = (double)pos * inv_freq;
        double c = cos(ang), s = sin(ang);
        double a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = a * s + b * c;
    }
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* One attention head over C cached positions: scores s_j = q.K_j / sqrt(d),
 * a = softmax(s), out = sum_j a_j V_j.  K and V rows are `stride` doubles
 * apart.  The max is subtracted before exp only to keep exp finite; it
 * cancels exactly in the normalisation. */
void orc_attention_head(int C, int d, const double *q, const double *K, const double *V, int stride,
                        double *out) {
    double *s = (double *)malloc(sizeof(double) * (size_t)(C > 0 ? C : 1));
    double scale = 1.0 / sqrt((double)d);
    double m = -INFINITY;
    for (int j = 0; j < C; ++j) {
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += q[e] * K[(size_t)j * stride + e];
        s[j] = acc * scale;
        if (s[j] > m) m = s[j];
    }
    double den = 0.0;
    for (int j = 0; j < C; ++j) {
        s[j] = exp(s[j] - m);
        den += s[j];
    }
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    for (int j = 0; j < C; ++j)
        for (int e = 0; e < d; ++e) out[e] += (s[j] / den) * V[(size_t)j * stride + e];
    free(s);
}

/* One decoder layer for one sequence at position pos.  x[hidden] is the
 * residual stream (updated in place).  kc/vc are this layer's cache,
 * [max_seq][n_kv_heads][head_dim]; row pos is written, rows 0..pos are read. */
int orc_layer_step(const orc_cfg *cfg, const orc_layer_w *w, double *kc, double *vc, int max_seq, int pos,
                   double *x) {
    const int H = cfg->hidden, nq = cfg->n_q_heads, nkv = cfg->n_kv_heads, d = cfg->head_dim, I = cfg->ffn_dim;
    if (pos < 0 || pos >= max_seq || nkv <= 0 || nq % nkv != 0) return -1;
    const int group = nq / nkv;
    double *xn = (double *)malloc(sizeof(double) * H);
    double *q = (double *)malloc(sizeof(double) * nq * d);
    double *k = (double *)malloc(sizeof(double) * nkv * d);
    double *v = (double *)malloc(sizeof(double) * nkv * d);
    double *att = (double *)malloc(sizeof(double) * nq * d);
    double *o = (double *)malloc(sizeof(double) * H);
    double *g = (double *)malloc(sizeof(double) * I);
    double *u = (double *)malloc(sizeof(double) * I);
    double *hm = (double *)malloc(sizeof(double) * I);

    /* attention block */
    orc_rmsnorm(H, x, w->attn_norm, cfg->rms_eps, xn);
    orc_matvec(nq * d, H, w->wq, xn, q);
    orc_matvec(nkv * d, H, w->wk, xn, k);
    orc_matvec(nkv * d, H, w->wv, xn, v);
    for (int h = 0; h < nq; ++h) orc_rope(d, q + (size_t)h * d, pos, cfg->rope_theta);
    for (int h = 0; h < nkv; ++h) orc_rope(d, k + (size_t)h * d, pos, cfg->rope_theta);
    if (cfg->kv_bf16)
        for (int i = 0; i < nkv * d; ++i) {
            k[i] = orc_round_bf16(k[i]);
            v[i] = orc_round_bf16(v[i]);
        }
    memcpy(kc + (size_t)pos * nkv * d, k, sizeof(double) * nkv * d);
    memcpy(vc + (size_t)pos * nkv * d, v, sizeof(double) * nkv * d);
    for (int h = 0; h < nq; ++h) {
        int hk = h / group; /* consecutive q heads share one kv head */
        orc_attention_head(pos + 1, d, q + (size_t)h * d, kc + (size_t)hk * d, vc + (size_t)hk * d, nkv * d,
                           att + (size_t)h * d);
    }
    orc_matvec(H, nq * d, w->wo, att, o);
    for (int i = 0; i < H; ++i) x[i] += o[i];

    /* feed-forward block (SwiGLU) */
    orc_rmsnorm(H, x, w->mlp_norm, cfg->rms_eps, xn);
    orc_matvec(I, H, w->w_gate, xn, g);
    orc_matvec(I, H, w->w_up, xn, u);
    for (int j = 0; j < I; ++j) hm[j] = orc_silu(g[j]) * u[j];
    orc_matvec(H, I, w->w_down, hm, o);
    for (int i = 0; i < H; ++i) x[i] += o[i];

    free(xn); free(q); free(k); free(v); free(att); free(o); free(g); free(u); free(hm);
    return 0;
}

/* x = embed[token] (widened). */
int orc_embed(const orc_cfg *cfg, const uint16_t *embed, int token, double *x) {
    if (token < 0 || token >= cfg->vocab) return -1;
    const uint16_t *row = embed + (size_t)token * cfg->hidden;
    for (int i = 0; i < cfg->hidden; ++i) x[i] = orc_bf16(row[i]);
    return 0;
}

/* logits = W_lm rmsnorm(x, g_final). */
void orc_head(const orc_cfg *cfg, const uint16_t *final_norm, const uint16_t *lm_head, const double *x,
              double *logits) {
    double *xn = (double *)malloc(sizeof(double) * cfg->hidden);
    orc_rmsnorm(cfg->hidden, x, final_norm, cfg->rms_eps, xn);
    orc_matvec(cfg->vocab, cfg->hidden, lm_head, xn, logits);
    free(xn);
}

/* One decode step for one sequence: token at position pos, caches
 * kcache/vcache [n_layers][max_seq][n_kv_heads][head_dim]. */
int orc_decode_step(const orc_cfg *cfg, const orc_weights *w, double *kcache, double *vcache, int max_seq, int token,
                    int pos, double *logits) {
    double *x = (double *)malloc(sizeof(double) * cfg->hidden);
    int rc = orc_embed(cfg, w->embed, token, x);
    size_t layer_elems = (size_t)max_seq * cfg->n_kv_heads * cfg->head_dim;
    for (int l = 0; rc == 0 && l < cfg->n_layers; ++l)
        rc = orc_layer_step(cfg, &w->layers[l], kcache + l * layer_elems, vcache + l * layer_elems, max_seq, pos, x);
    if (rc == 0) orc_head(cfg, w->final_norm, w->lm_head, x, logits);
    free(x);
    return rc;
}

/* Full-sequence causal forward over tokens[0..n): a separate code path that
 * keeps every position's activations and applies an explicit n x n causal
 * mask (key j visible to query i iff j <= i).  logits[n][vocab]. */
int orc_full_forward(const orc_cfg *cfg, const orc_weights *w, int n, const int *tokens, double *logits) {
    const int H = cfg->hidden, nq = cfg->n_q_heads, nkv = cfg->n_kv_heads, d = cfg->head_dim, I = cfg->ffn_dim;
    if (n <= 0 || nkv <= 0 || nq % nkv != 0) return -1;
    const int group = nq / nkv;
    double *X = (double *)malloc(sizeof(double) * (size_t)n * H);
    double *Xn = (double *)malloc(sizeof(double) * (size_t)n * H);
    double *Q = (double *)malloc(sizeof(double) * (size_t)n * nq * d);
    double *Kx = (double *)malloc(sizeof(double) * (size_t)n * nkv * d);
    double *Vx = (double *)malloc(sizeof(double) * (size_t)n * nkv * d);
    double *A = (double *)malloc(sizeof(double) * (size_t)n * nq * d);
    double *O = (double *)malloc(sizeof(double) * (size_t)n * H);
    double *Hm = (double *)malloc(sizeof(double) * (size_t)n * I);
    double *G = (double *)malloc(sizeof(double) * I);
    double *U = (double *)malloc(sizeof(double) * I);
    double *S = (double *)malloc(sizeof(double) * (size_t)n * n);
    int rc = 0;
    for (int t = 0; t < n && rc == 0; ++t) rc = orc_embed(cfg, w->embed, tokens[t], X + (size_t)t * H);
    const double scale = 1.0 / sqrt((double)d);
    for (int l = 0; l < cfg->n_layers && rc == 0; ++l) {
        const orc_layer_w *lw = &w->layers[l];
        for (int t = 0; t < n; ++t) {
            orc_rmsnorm(H, X + (size_t)t * H, lw->attn_norm, cfg->rms_eps, Xn + (size_t)t * H);
            orc_matvec(nq * d, H, lw->wq, Xn + (size_t)t * H, Q + (size_t)t * nq * d);
            orc_matvec(nkv * d, H, lw->wk, Xn + (size_t)t * H, Kx + (size_t)t * nkv * d);
            orc_matvec(nkv * d, H, lw->wv, Xn + (size_t)t * H, Vx + (size_t)t * nkv * d);
            for (int h = 0; h < nq; ++h) orc_rope(d, Q + ((size_t)t * nq + h) * d, t, cfg->rope_theta);
            for (int h = 0; h < nkv; ++h) orc_rope(d, Kx + ((size_t)t * nkv + h) * d, t, cfg->rope_theta);
            if (cfg->kv_bf16)
                for (int i = 0; i < nkv * d; ++i) {
                    Kx[(size_t)t * nkv * d + i] = orc_round_bf16(Kx[(size_t)t * nkv * d + i]);
                    Vx[(size_t)t * nkv * d + i] = orc_round_bf16(Vx[(size_t)t * nkv * d + i]);
                }
        }
        for (int h = 0; h < nq; ++h) {
            int hk = h / group;
            /* scores with an explicit mask, then a row softmax */
            for (int i = 0; i < n; ++i) {
                for (int j = 0; j < n; ++j) {
                    if (j > i) {
                        S[(size_t)i * n + j] = -INFINITY;
                        continue;
                    }
                    double acc = 0.0;
                    for (int e = 0; e < d; ++e)
                        acc += Q[((size_t)i * nq + h) * d + e] * Kx[((size_t)j * nkv + hk) * d + e];
                    S[(size_t)i * n + j] = acc * scale;
                }
                double m = -INFINITY, den = 0.0;
                for (int j = 0; j < n; ++j) m = fmax(m, S[(size_t)i * n + j]);
                for (int j = 0; j < n; ++j) {
                    double p = isinf(S[(size_t)i * n + j]) ? 0.0 : exp(S[(size_t)i * n + j] - m);
                    S[(size_t)i * n + j] = p;
                    den += p;
                }
                for (int e = 0; e < d; ++e) {
                    double acc = 0.0;
                    for (int j = 0; j < n; ++j) acc += (S[(size_t)i * n + j] / den) * Vx[((size_t)j * nkv + hk) * d + e];
                    A[((size_t)i * nq + h) * d + e] = acc;
                }
            }
        }
        for (int t = 0; t < n; ++t) {
            orc_matvec(H, nq * d, lw->wo, A + (size_t)t * nq * d, O + (size_t)t * H);
            for (int i = 0; i < H; ++i) X[(size_t)t * H + i] += O[(size_t)t * H + i];
            orc_rmsnorm(H, X + (size_t)t * H, lw->mlp_norm, cfg->rms_eps, Xn + (size_t)t * H);
            orc_matvec(I, H, lw->w_gate, Xn + (size_t)t * H, G);
            orc_matvec(I, H, lw->w_up, Xn + (size_t)t * H, U);
            for (int j = 0; j < I; ++j) Hm[(size_t)t * I + j] = orc_silu(G[j]) * U[j];
            orc_matvec(H, I, lw->w_down, Hm + (size_t)t * I, O + (size_t)t * H);
            for (int i = 0; i < H; ++i) X[(size_t)t * H + i] += O[(size_t)t * H + i];
        }
    }
    for (int t = 0; t < n && rc == 0; ++t)
        orc_head(cfg, w->final_norm, w->lm_head, X + (size_t)t * H, logits + (size_t)t * cfg->vocab);
    free(X); free(Xn); free(Q); free(Kx); free(Vx); free(A); free(O); free(Hm); free(G); free(U); free(S);
    return rc;
}
