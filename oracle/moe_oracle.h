/*
 * moe_oracle.h -- plain CPU oracle for the top-k routed Mixture-of-Experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or call this
 * code: only the tests, the smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no source, header, table or helper with the CUDA library.
 *
 * What the layer computes.  The pages define the layer only in prose: a sparse network of
 * many expert sub-networks of which each token activates a small part ("AI MAX+ 395部署
 * Qwen3大模型：GFX1151引擎实测优化解析", explanatory paragraph under "MOE 内核优化"), run on
 * the timed path as a "selected-MoE" kernel ("AIMA AMD395 Qwen3.6 35B Windows Engine",
 * section "性能优化做了什么").  The oracle follows the plainest standard reading of that
 * layer, step by step:
 *   1. router logits  l[t,e] = fp32( sum_h x[t,h] * Wr[e,h] )  (+ b[e], fp32 add)
 *   2. selection      S = the k largest logits, lower expert index first on ties
 *   3. weights        p = softmax over all E logits (fp64); w_j = p[S_j] / sum_i p[S_i] -> fp32
 *   4. permutation    stable counting sort of the T*k (token, slot) pairs by expert
 *   5. expert FFN     h = bf16( silu(Wg x) * (Wu x) ),  y = Wd h        (fp64 sums)
 *   6. shared expert  same as 5 with the shared weights, weight 1, every token
 *   7. combine        out[t] = bf16( sum_j w_j * y_j + y_shared )        (fp64 sum)
 * All sums are taken in double; the only roundings are the ones listed (fp32 logits,
 * fp32 weights, bf16 h, bf16 out).  "exact" mode skips the bf16 rounding of h.
 *
 * Layouts: row-major, [out, in] linear convention.  bf16 values travel as their 16-bit
 * patterns (uint16_t).  x [T,H]; Wr [E,H]; b [E] or NULL; Wg, Wu [E,I,H]; Wd [E,H,I];
 * Wsg, Wsu [Is,H]; Wsd [H,Is] (all NULL and Is = 0 when there is no shared expert).
 * Logits are assumed finite.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* bf16 pattern -> double (exact). */
double moe_ref_bf16_to_double(uint16_t b);
/* double -> bf16 pattern, round to nearest, ties to even, in one rounding step. */
uint16_t moe_ref_double_to_bf16(double v);
/* silu(g) = g / (1 + exp(-g)) in double. */
double moe_ref_silu(double g);

/* Step 1: router logits [T,E] (fp32). b may be NULL. */
void moe_ref_router_logits(int H, int E, int T, const uint16_t *x, const uint16_t *w_router,
                           const float *b_router, float *logits);

/* Steps 2-3 from given fp32 logits: ids [T,k] int32 in rank order, weights [T,k] fp32. */
void moe_ref_route_from_logits(int E, int k, int T, const float *logits, int32_t *ids, float *w);

/* Step 4: offsets [E+1], perm [T*k] (row -> pair index t*k+j), inv [T*k] (pair -> row).
 * Returns 0, or -1 if an id lies outside [0,E). */
int moe_ref_permute(int E, int k, int T, const int32_t *ids, int32_t *offsets, int32_t *perm,
                    int32_t *inv);

/* Step 5 for the rows of the permuted order: h_rows [T*k, I] (bf16 pattern) and
 * y_rows [T*k, H] (fp32 rounding of the fp64 sum), computed from x, the permutation and
 * the routed weights.  When h_in is not NULL the down projection uses those bf16 h rows
 * instead of the oracle's own (to isolate the down projection).  When shared_y is not
 * NULL and Is > 0, also step 6: shared_y [T,H] (fp32 rounding of the fp64 sum). */
void moe_ref_expert_ffn(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                        const int32_t *offsets, const int32_t *perm, const uint16_t *w_gate,
                        const uint16_t *w_up, const uint16_t *w_down, const uint16_t *ws_gate,
                        const uint16_t *ws_up, const uint16_t *ws_down, const uint16_t *h_in,
                        uint16_t *h_rows, float *y_rows, float *shared_y);

/* Step 7 from unfused rows: out[t] = bf16( sum_j w[t,j] * y_rows[inv[t*k+j]] + shared_y[t] ). */
void moe_ref_combine(int H, int k, int T, const float *y_rows, const int32_t *inv,
                     const float *topk_w, const float *shared_y, uint16_t *out);

/* The whole layer, token by token (steps 1-7).  When ids_in/w_in are not NULL they replace
 * steps 1-3 (the oracle then consumes a given routing).  exact != 0 skips the bf16 rounding
 * of h.  out [T,H] bf16 pattern; out_f64 [T,H] (may be NULL) receives the unrounded sum.
 * x_next (may be NULL) receives bf16( x + out ), the residual update of a layer stack.
 * ids_out / w_out (may be NULL) receive the routing used.  n_threads <= 0 uses OpenMP's
 * default; the loop over tokens is the only parallel loop. */
void moe_ref_forward(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                     const uint16_t *w_router, const float *b_router, const uint16_t *w_gate,
                     const uint16_t *w_up, const uint16_t *w_down, const uint16_t *ws_gate,
                     const uint16_t *ws_up, const uint16_t *ws_down, const int32_t *ids_in,
                     const float *w_in, int exact, int n_threads, uint16_t *out,
                     double *out_f64, uint16_t *x_next, int32_t *ids_out, float *w_out);

/* Second, independent evaluation of the combine: expert-major over all E experts with a
 * dense mask (weight w if the expert is among the token's k, else the expert is skipped),
 * no permutation.  Consumes the given routing ids/w.  out_f64 [T,H], unrounded. */
void moe_ref_dense_masked(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                          const uint16_t *w_gate, const uint16_t *w_up, const uint16_t *w_down,
                          const uint16_t *ws_gate, const uint16_t *ws_up,
                          const uint16_t *ws_down, const int32_t *ids, const float *w,
                          int exact, double *out_f64);

/* Number of threads the OpenMP loop of moe_ref_forward would use for n_threads. */
int moe_ref_threads(int n_threads);

/* ----------------------------------------------------- quantised expert weights -- */
/* The 8-bit float E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits, no infinities;
 * exponent and fraction all ones is NaN.  Exponent e > 0: (-1)^s * 2^(e-7) * (1 + m/8);
 * e = 0: (-1)^s * 2^-6 * (m/8).  Largest finite magnitude 448. */
double moe_ref_e4m3_to_double(uint8_t q);
/* float -> E4M3 pattern: round to nearest, ties to even; magnitudes past 448 saturate to 448. */
uint8_t moe_ref_float_to_e4m3(float v);
/* Row-wise quantisation of a bf16 matrix [rows, cols]: scale[r] = fp32(max_c |w[r,c]|) / 448
 * in fp32 (1 for an all-zero row), q[r,c] = E4M3 of fp32(w[r,c]) / scale[r] (fp32 division). */
void moe_ref_quantize_e4m3_rows(int rows, int cols, const uint16_t *w, uint8_t *q, float *scale);
/* The layer for T tokens with quantised expert weights, weight[r,c] = scale[r] * e4m3(q[r,c])
 * (exact in double), on a given routing ids/w [T,k]; the rounding points of moe_ref_forward
 * (h to bf16 once, out to bf16 once).  Routed: qg, qu [E,I,H] with sg, su [E,I]; qd [E,H,I]
 * with sd [E,H].  Shared (Is > 0): qsg, qsu [Is,H] with ssg, ssu [Is]; qsd [H,Is] with ssd [H]. */
void moe_ref_forward_q8(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                        const uint8_t *qg, const float *sg, const uint8_t *qu, const float *su,
                        const uint8_t *qd, const float *sd, const uint8_t *qsg, const float *ssg,
                        const uint8_t *qsu, const float *ssu, const uint8_t *qsd, const float *ssd,
                        const int32_t *ids, const float *w, uint16_t *out);

/* 4-bit integer block quantisation ("Q4": 4-bit integer codes, as the GFX1151 page's explanatory
 * paragraph on weight formats describes it).  Each row of a bf16 matrix [rows, cols] (cols a
 * multiple of 32) is cut into blocks of 32 consecutive columns.  Block b of row r: scale[r, b] =
 * fp32(max |w|) / 7 in fp32 (1 for an all-zero block); the code of w is round-half-even of
 * fp32(w) / scale (fp32 division), clamped to [-7, 7], stored as a two's-complement nibble:
 * column 2j in the low nibble and 2j+1 in the high nibble of byte j of the row (cols / 2 bytes a
 * row).  The weight the layer uses is scale * code (exact in double). */
void moe_ref_quantize_q4_rows(int rows, int cols, const uint16_t *w, uint8_t *q, float *scale);
/* The value of code nibble c (column c) of a row of packed codes. */
int moe_ref_q4_code(const uint8_t *row, int c);
/* The layer for T tokens with Q4 expert weights on a given routing, with the rounding points of
 * moe_ref_forward.  Routed: qg, qu [E, I, H/2] with sg, su [E, I, H/32]; qd [E, H, I/2] with
 * sd [E, H, I/32].  Shared (Is > 0): qsg, qsu [Is, H/2] with ssg, ssu [Is, H/32]; qsd [H, Is/2]
 * with ssd [H, Is/32]. */
void moe_ref_forward_q4(int H, int E, int k, int I, int Is, int T, const uint16_t *x,
                        const uint8_t *qg, const float *sg, const uint8_t *qu, const float *su,
                        const uint8_t *qd, const float *sd, const uint8_t *qsg, const float *ssg,
                        const uint8_t *qsu, const float *ssu, const uint8_t *qsd, const float *ssd,
                        const int32_t *ids, const float *w, uint16_t *out);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ORACLE_H */
