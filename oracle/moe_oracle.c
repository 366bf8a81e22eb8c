/*
 * moe_oracle.c -- plain, slow CPU oracle for the top-k routed MoE FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY (see moe_oracle.h).  Plain nested loops, double accumulation,
 * no blocking, no fusion, no reordering beyond the definitions.  Each function names the
 * passage it follows.  The pages give the layer only in prose ("AI MAX+ 395部署Qwen3大模型：
 * GFX1151引擎实测优化解析", explanatory MoE paragraph under "MOE 内核优化": many experts,
 * few active per token; "AIMA AMD395 Qwen3.6 35B Windows Engine", "性能优化做了什么":
 * the selected-MoE kernel); the concrete steps are the standard top-k routed MoE FFN with
 * a SwiGLU expert and an always-on shared expert.  Readings where the pages are silent:
 *   - selection is made on the fp32 logits, lower expert index first on equal logits;
 *   - the router bias (if any) is an ordinary additive bias used for selection and weights;
 *   - silu acts on the gate projection, which multiplies the up projection;
 *   - the shared expert has weight 1 (no gate);
 *   - h is rounded to bf16 once, the layer output once.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 helpers -- */

double moe_ref_bf16_to_double(uint16_t b) {
    /* A bf16 value is the upper half of the binary32 with the same bits. */
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

uint16_t moe_ref_double_to_bf16(double v) {
    /* Round to nearest, ties to even, directly from double (one rounding).  bf16 has an
     * 8-bit exponent (the binary32 range) and 7 fraction bits, so its spacing at binade
     * [2^e, 2^(e+1)) is 2^(e-7); below 2^-126 the spacing stays 2^-133 (subnormals). */
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return 0x7FC0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int e2;
    (void)frexp(a, &e2);          /* a = m * 2^e2 with m in [0.5, 1)  => floor(log2 a) = e2-1 */
    int ex = e2 - 1;
    if (ex < -126) ex = -126;
    double spacing = ldexp(1.0, ex - 7);
    double q = a / spacing;        /* exact: division by a power of two */
    double r = nearbyint(q);       /* default rounding mode: nearest, ties to even */
    double res = r * spacing;
    if (res >= 0x1p128) return (uint16_t)(sign | 0x7F80u); /* overflow -> infinity */
    float f = (float)res;          /* exact: res has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

double moe_ref_silu(double g) {
    /* silu(g) = g * sigmoid(g) = g / (1 + e^-g). */
    return g / (1.0 + exp(-g));
}

#define BF(p) moe_ref_bf16_to_double(p)

int moe_ref_threads(int n_threads) {
#ifdef _OPENMP
    return n_threads > 0 ? n_threads : omp_get_max_threads();
#else
    (void)n_threads;
    return 1;
#endif
}

/* --------------------------------------------------------- step 1: router logits -- */

void moe_ref_router_logits(int H, int E, int T, const uint16_t *x, const uint16_t *w_router,
                           const float *b_router, float *logits) {
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += BF(x[(size_t)t * H + h]) * BF(w_router[(size_t)e * H + h]);
            float l = (float)acc;
            if (b_router) l = l + b_router[e]; /* fp32 addition of the bias */
            logits[(size_t)t * E + e] = l;
        }
    }
}

/* ------------------------------------------- steps 2-3: top-k and renormalisation -- */

static void route_one(int E, int k, const float *l, int32_t *ids, float *w) {
    /* Selection by rank: rank(e) = #{e' : l[e'] > l[e]} + #{e' < e : l[e'] == l[e]}.
     * The k experts of rank < k are the top-k with the lower index winning ties, and the
     * rank is also the output slot (descending logit). */
    for (int e = 0; e < E; ++e) {
        int rank = 0;
        for (int e2 = 0; e2 < E; ++e2) {
            if (l[e2] > l[e]) ++rank;
            else if (e2 < e && l[e2] == l[e]) ++rank;
        }
        if (rank < k) ids[rank] = e;
    }
    /* Softmax over all E logits in double, then renormalise over the k selected. */
    double m = l[0];
    for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp((double)l[e] - m);
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += exp((double)l[ids[j]] - m) / z;
    for (int j = 0; j < k; ++j) w[j] = (float)((exp((double)l[ids[j]] - m) / z) / s);
}

void moe_ref_route_from_logits(int E, int k, int T, const float *logits, int32_t *ids, float *w) {
    for (int t = 0; t < T; ++t)
        route_one(E, k, logits + (size_t)t * E, ids + (size_t)t * k, w + (size_t)t * k);
}

/* --------------------------------------------------------------- step 4: permute -- */

int moe_ref_permute(int E, int k, int T, const int32_t *ids, int32_t *offsets, int32_t *perm,
                    int32_t *inv) {
    /* Textbook stable counting sort of the pairs p = t*k + j by expert id:
     * counts, exclusive prefix sum, then each pair in increasing p goes to the next free
     * row of its expert, so row(p) = offsets[e] + #{p' < p : id(p') = e}. */
    const long P = (long)T * k;
    int32_t *cursor = (int32_t *)calloc((size_t)E + 1, sizeof(int32_t));
    if (!cursor) return -1;
    for (int e = 0; e <= E; ++e) offsets[e] = 0;
    for (long p = 0; p < P; ++p) {
        if (ids[p] < 0 || ids[p] >= E) { free(cursor); return -1; }
        offsets[ids[p] + 1] += 1;
    }
    for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (long p = 0; p < P; ++p) {
        int32_t row = cursor[ids[p]]++;
        perm[row] = (int32_t)p;
        inv[p] = row;
    }
    free(cursor);
    return 0;
}

/* ------------------------------------------------------ step 5/6: one SwiGLU FFN -- */

/* One SwiGLU expert applied to one token row: g = Wg x, u = Wu x (fp64 sums),
 * a = silu(g) * u, h = bf16(a) unless exact, y = Wd h (fp64 sum).
 * wg, wu: [I, H]; wd: [H, I].  hbuf: I doubles of scratch.  h_in (may be NULL) replaces
 * the computed h by given bf16 values. */
static void swiglu_ffn(int H, int I, const uint16_t *xrow, const uint16_t *wg, const uint16_t *wu,
                       const uint16_t *wd, int exact, const uint16_t *h_in, double *hbuf,
                       uint16_t *h_out, double *y) {
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            double xv = BF(xrow[h]);
            g += BF(wg[(size_t)i * H + h]) * xv;
            u += BF(wu[(size_t)i * H + h]) * xv;
        }
        double a = moe_ref_silu(g) * u;
        uint16_t hb = moe_ref_double_to_bf16(a);
        if (h_out) h_out[i] = hb;
        hbuf[i] = exact ? a : BF(hb);
        if (h_in) hbuf[i] = BF(h_in[i]);
    }
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += BF(wd[(size_t)n * I + i]) * hbuf[i];
        y[n] = acc;
    }
}

void moe_ref_expert_ffn(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                        const int32_t *offsets, const int32_t *perm, const uint16_t *w_gate,
                        const uint16_t *w_up, const uint16_t *w_down, const uint16_t *ws_gate,
                        const uint16_t *ws_up, const uint16_t *ws_down, const uint16_t *h_in,
                        uint16_t *h_rows, float *y_rows, float *shared_y) {
    int maxI = I > Is ? I : Is;
    double *hbuf = (double *)malloc(sizeof(double) * (size_t)(maxI > 0 ? maxI : 1));
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    /* Routed rows, expert by expert over the permuted order. */
    for (int e = 0; e < E; ++e) {
        for (int row = offsets[e]; row < offsets[e + 1]; ++row) {
            int t = perm[row] / k;
            swiglu_ffn(H, I, x + (size_t)t * H, w_gate + (size_t)e * I * H,
                       w_up + (size_t)e * I * H, w_down + (size_t)e * H * I, 0,
                       h_in ? h_in + (size_t)row * I : NULL, hbuf,
                       h_rows ? h_rows + (size_t)row * I : NULL, y);
            if (y_rows)
                for (int n = 0; n < H; ++n) y_rows[(size_t)row * H + n] = (float)y[n];
        }
    }
    /* Shared expert: every token, weight 1. */
    if (shared_y && Is > 0) {
        for (int t = 0; t < T; ++t) {
            swiglu_ffn(H, Is, x + (size_t)t * H, ws_gate, ws_up, ws_down, 0, NULL, hbuf, NULL, y);
            for (int n = 0; n < H; ++n) shared_y[(size_t)t * H + n] = (float)y[n];
        }
    }
    free(hbuf);
    free(y);
}

/* --------------------------------------------------------------- step 7: combine -- */

void moe_ref_combine(int H, int k, int T, const float *y_rows, const int32_t *inv,
                     const float *topk_w, const float *shared_y, uint16_t *out) {
    for (int t = 0; t < T; ++t) {
        for (int n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                long p = (long)t * k + j;
                acc += (double)topk_w[p] * (double)y_rows[(size_t)inv[p] * H + n];
            }
            if (shared_y) acc += (double)shared_y[(size_t)t * H + n];
            out[(size_t)t * H + n] = moe_ref_double_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------------- the whole layer -- */

void moe_ref_forward(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                     const uint16_t *w_router, const float *b_router, const uint16_t *w_gate,
                     const uint16_t *w_up, const uint16_t *w_down, const uint16_t *ws_gate,
                     const uint16_t *ws_up, const uint16_t *ws_down, const int32_t *ids_in,
                     const float *w_in, int exact, int n_threads, uint16_t *out,
                     double *out_f64, uint16_t *x_next, int32_t *ids_out, float *w_out) {
    int nt = moe_ref_threads(n_threads);
    (void)nt;
    int maxI = I > Is ? I : Is;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
    for (int t = 0; t < T; ++t) {
        const uint16_t *xrow = x + (size_t)t * H;
        float *l = (float *)malloc(sizeof(float) * (size_t)E);
        int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
        float *w = (float *)malloc(sizeof(float) * (size_t)k);
        double *hbuf = (double *)malloc(sizeof(double) * (size_t)(maxI > 0 ? maxI : 1));
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
        double *acc = (double *)calloc((size_t)H, sizeof(double));
        /* Steps 1-3, unless a routing is given. */
        if (ids_in) {
            for (int j = 0; j < k; ++j) {
                ids[j] = ids_in[(size_t)t * k + j];
                w[j] = w_in[(size_t)t * k + j];
            }
        } else {
            moe_ref_router_logits(H, E, 1, xrow, w_router, b_router, l);
            route_one(E, k, l, ids, w);
        }
        if (ids_out)
            for (int j = 0; j < k; ++j) ids_out[(size_t)t * k + j] = ids[j];
        if (w_out)
            for (int j = 0; j < k; ++j) w_out[(size_t)t * k + j] = w[j];
        /* Steps 5 and 7: the k selected experts in slot order, weighted. */
        for (int j = 0; j < k; ++j) {
            int e = ids[j];
            swiglu_ffn(H, I, xrow, w_gate + (size_t)e * I * H, w_up + (size_t)e * I * H,
                       w_down + (size_t)e * H * I, exact, NULL, hbuf, NULL, y);
            for (int n = 0; n < H; ++n) acc[n] += (double)w[j] * y[n];
        }
        /* Step 6: the shared expert, weight 1. */
        if (Is > 0) {
            swiglu_ffn(H, Is, xrow, ws_gate, ws_up, ws_down, exact, NULL, hbuf, NULL, y);
            for (int n = 0; n < H; ++n) acc[n] += y[n];
        }
        for (int n = 0; n < H; ++n) {
            uint16_t o = moe_ref_double_to_bf16(acc[n]);
            out[(size_t)t * H + n] = o;
            if (out_f64) out_f64[(size_t)t * H + n] = acc[n];
            if (x_next) x_next[(size_t)t * H + n] = moe_ref_double_to_bf16(BF(xrow[n]) + BF(o));
        }
        free(l); free(ids); free(w); free(hbuf); free(y); free(acc);
    }
}

/* ------------------------------------------- dense masked evaluation (second form) -- */

void moe_ref_dense_masked(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                          const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down,
                          const uint16_t *ws_gate, const uint16_t *ws_up,
                          const uint16_t *ws_down, const int32_t *ids, const float *w,
                          int exact, double *out_f64) {
    /* out[t] = sum over ALL experts e of mask[t,e] * FFN_e(x_t) + shared(x_t), where
     * mask[t,e] is the routing weight of e for token t if e is one of its k experts and
     * 0 otherwise.  Expert-major loop, no permutation. */
    int maxI = I > Is ? I : Is;
    double *hbuf = (double *)malloc(sizeof(double) * (size_t)(maxI > 0 ? maxI : 1));
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    for (size_t i = 0; i < (size_t)T * H; ++i) out_f64[i] = 0.0;
    for (int e = 0; e < E; ++e) {
        for (int t = 0; t < T; ++t) {
            double mask = 0.0;
            int hit = 0;
            for (int j = 0; j < k; ++j)
                if (ids[(size_t)t * k + j] == e) { mask += (double)w[(size_t)t * k + j]; hit = 1; }
            if (!hit) continue;
            swiglu_ffn(H, I, x + (size_t)t * H, w_gate + (size_t)e * I * H,
                       w_up + (size_t)e * I * H, w_down + (size_t)e * H * I, exact, NULL, hbuf,
                       NULL, y);
            for (int n = 0; n < H; ++n) out_f64[(size_t)t * H + n] += mask * y[n];
        }
    }
    if (Is > 0) {
        for (int t = 0; t < T; ++t) {
            swiglu_ffn(H, Is, x + (size_t)t * H, ws_gate, ws_up, ws_down, exact, NULL, hbuf, NULL, y);
            for (int n = 0; n < H; ++n) out_f64[(size_t)t * H + n] += y[n];
        }
    }
    free(hbuf);
    free(y);
}

/* ----------------------------------------------------- quantised expert weights -- */
/* "AI MAX+ 395部署Qwen3大模型：GFX1151引擎实测优化解析", "两种权重格式：HGN 与 GGUF 的统一支持":
 * one of the weight formats stores its large modules as 8-bit floats, with little precision
 * lost; the page gives no layout.  Reading: E4M3 codes with one fp32 scale per output row of
 * each expert matrix, weight = scale * code. */

double moe_ref_e4m3_to_double(uint8_t q) {
    int s = (q >> 7) & 1, e = (q >> 3) & 0xF, m = q & 7;
    if (e == 0xF && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

uint8_t moe_ref_float_to_e4m3(float v) {
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    double a = fabs((double)v);
    if (isnan(v)) return 0x7Fu;
    if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
    if (a < 0x1p-6) {
        /* subnormal step 2^-9; a rounded count of 8 is the smallest normal, code 0x08 */
        double c = nearbyint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)c);
    }
    int e2;
    (void)frexp(a, &e2);
    int ex = e2 - 1;                           /* 2^ex <= a < 2^(ex+1), -6 <= ex <= 8 */
    double c = nearbyint(a / ldexp(1.0, ex - 3)); /* 8 .. 16 steps of 2^(ex-3) */
    if (c == 16.0) { ex += 1; c = 8.0; }
    int code = ((ex + 7) << 3) | ((int)c - 8);
    if (code > 0x7E) code = 0x7E;              /* 480 would be the NaN pattern: saturate */
    return (uint8_t)(sign | code);
}

void moe_ref_quantize_e4m3_rows(int rows, int cols, const uint16_t *w, uint8_t *q, float *scale) {
    for (int r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < cols; ++c) {
            float a = (float)fabs(BF(w[(size_t)r * cols + c]));
            if (a > amax) amax = a;
        }
        float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[r] = s;
        for (int c = 0; c < cols; ++c) {
            float v = (float)BF(w[(size_t)r * cols + c]) / s;
            q[(size_t)r * cols + c] = moe_ref_float_to_e4m3(v);
        }
    }
}

/* h = bf16(silu(g) * u), y = Wd h with dequantised weights (fp64 sums); as swiglu_ffn. */
static void swiglu_ffn_q8(int H, int I, const uint16_t *xrow, const uint8_t *qg, const float *sg,
                          const uint8_t *qu, const float *su, const uint8_t *qd, const float *sd,
                          double *hbuf, double *y) {
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            double xv = BF(xrow[h]);
            g += (double)sg[i] * moe_ref_e4m3_to_double(qg[(size_t)i * H + h]) * xv;
            u += (double)su[i] * moe_ref_e4m3_to_double(qu[(size_t)i * H + h]) * xv;
        }
        hbuf[i] = BF(moe_ref_double_to_bf16(moe_ref_silu(g) * u));
    }
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += (double)sd[n] * moe_ref_e4m3_to_double(qd[(size_t)n * I + i]) * hbuf[i];
        y[n] = acc;
    }
}

void moe_ref_forward_q8(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                        const uint8_t *qg, const float *sg, const uint8_t *qu, const float *su,
                        const uint8_t *qd, const float *sd, const uint8_t *qsg, const float *ssg,
                        const uint8_t *qsu, const float *ssu, const uint8_t *qsd, const float *ssd,
                        const int32_t *ids, const float *w, uint16_t *out) {
    (void)E;
    int maxI = I > Is ? I : Is;
    double *hbuf = (double *)malloc(sizeof(double) * (size_t)(maxI > 0 ? maxI : 1));
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
    for (int t = 0; t < T; ++t) {
        const uint16_t *xrow = x + (size_t)t * H;
        for (int n = 0; n < H; ++n) acc[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            swiglu_ffn_q8(H, I, xrow, qg + (size_t)e * I * H, sg + (size_t)e * I, qu + (size_t)e * I * H,
                          su + (size_t)e * I, qd + (size_t)e * H * I, sd + (size_t)e * H, hbuf, y);
            for (int n = 0; n < H; ++n) acc[n] += (double)w[(size_t)t * k + j] * y[n];
        }
        if (Is > 0) {
            swiglu_ffn_q8(H, Is, xrow, qsg, ssg, qsu, ssu, qsd, ssd, hbuf, y);
            for (int n = 0; n < H; ++n) acc[n] += y[n];
        }
        for (int n = 0; n < H; ++n) out[(size_t)t * H + n] = moe_ref_double_to_bf16(acc[n]);
    }
    free(hbuf); free(y); free(acc);
}

/* ------------------------------------------------------------ 4-bit integer blocks -- */
/* GFX1151 page ("两种权重格式" section and its explanatory paragraph: Q4 is 4-bit integer
 * quantisation, FP8 8-bit floating point); the block layout is the reading stated in the header. */

void moe_ref_quantize_q4_rows(int rows, int cols, const uint16_t *w, uint8_t *q, float *scale) {
    const int nb = cols / 32;
    for (int r = 0; r < rows; ++r) {
        const uint16_t *wr = w + (size_t)r * cols;
        uint8_t *qr = q + (size_t)r * (cols / 2);
        for (int b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int c = 32 * b; c < 32 * b + 32; ++c) {
                float a = (float)fabs(BF(wr[c]));
                if (a > amax) amax = a;
            }
            float s = amax > 0.0f ? amax / 7.0f : 1.0f;
            scale[(size_t)r * nb + b] = s;
            for (int c = 32 * b; c < 32 * b + 32; ++c) {
                float v = rintf((float)BF(wr[c]) / s);
                if (v > 7.0f) v = 7.0f;
                if (v < -7.0f) v = -7.0f;
                int code = (int)v;
                uint8_t nib = (uint8_t)(code & 15);
                if (c % 2 == 0) qr[c / 2] = nib;
                else qr[c / 2] = (uint8_t)(qr[c / 2] | (nib << 4));
            }
        }
    }
}

int moe_ref_q4_code(const uint8_t *row, int c) {
    int nib = (c % 2 == 0) ? (row[c / 2] & 15) : (row[c / 2] >> 4);
    return nib >= 8 ? nib - 16 : nib;
}

/* One weight of a Q4 matrix with `cols` columns: scale * code. */
static double q4_weight(const uint8_t *q, const float *scale, int cols, int r, int c) {
    return (double)scale[(size_t)r * (cols / 32) + c / 32] * (double)moe_ref_q4_code(q + (size_t)r * (cols / 2), c);
}

/* h = bf16(silu(g) * u), y = Wd h with the Q4 weights (fp64 sums); as swiglu_ffn. */
static void swiglu_ffn_q4(int H, int I, const uint16_t *xrow, const uint8_t *qg, const float *sg,
                          const uint8_t *qu, const float *su, const uint8_t *qd, const float *sd,
                          double *hbuf, double *y) {
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            double xv = BF(xrow[h]);
            g += q4_weight(qg, sg, H, i, h) * xv;
            u += q4_weight(qu, su, H, i, h) * xv;
        }
        hbuf[i] = BF(moe_ref_double_to_bf16(moe_ref_silu(g) * u));
    }
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += q4_weight(qd, sd, I, n, i) * hbuf[i];
        y[n] = acc;
    }
}

void moe_ref_forward_q4(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                        const uint8_t *qg, const float *sg, const uint8_t *qu, const float *su,
                        const uint8_t *qd, const float *sd, const uint8_t *qsg, const float *ssg,
                        const uint8_t *qsu, const float *ssu, const uint8_t *qsd, const float *ssd,
                        const int32_t *ids, const float *w, uint16_t *out) {
    (void)E;
    int maxI = I > Is ? I : Is;
    double *hbuf = (double *)malloc(sizeof(double) * (size_t)(maxI > 0 ? maxI : 1));
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
    for (int t = 0; t < T; ++t) {
        const uint16_t *xrow = x + (size_t)t * H;
        for (int n = 0; n < H; ++n) acc[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            swiglu_ffn_q4(H, I, xrow, qg + (size_t)e * I * (H / 2), sg + (size_t)e * I * (H / 32),
                          qu + (size_t)e * I * (H / 2), su + (size_t)e * I * (H / 32),
                          qd + (size_t)e * H * (I / 2), sd + (size_t)e * H * (I / 32), hbuf, y);
            for (int n = 0; n < H; ++n) acc[n] += (double)w[(size_t)t * k + j] * y[n];
        }
        if (Is > 0) {
            swiglu_ffn_q4(H, Is, xrow, qsg, ssg, qsu, ssu, qsd, ssd, hbuf, y);
            for (int n = 0; n < H; ++n) acc[n] += y[n];
        }
        for (int n = 0; n < H; ++n) out[(size_t)t * H + n] = moe_ref_double_to_bf16(acc[n]);
    }
    free(hbuf); free(y); free(acc);
}
