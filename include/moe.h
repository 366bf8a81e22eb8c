/*
 * moe.h -- C ABI of the GB300-native top-k routed Mixture-of-Experts FFN layer (libmoe.so).
 *
 * The layer.  The pages describe the layer only in prose: a network of many expert
 * sub-networks of which each token activates a small part ("AI MAX+ 395部署Qwen3大模型：
 * GFX1151引擎实测优化解析", explanatory MoE paragraph under "MOE 内核优化"), executed on the
 * timed path of a batch-1 BF16 engine by a "selected-MoE" kernel ("AIMA AMD395 Qwen3.6 35B
 * Windows Engine", section "性能优化做了什么").  This library computes the standard reading of
 * that layer, for T tokens of hidden size H, E routed experts, top-k, expert intermediate I
 * and a shared expert of intermediate Is:
 *   logits   l[t,e] = sum_h x[t,h] Wr[e,h] (+ b[e])                     fp32
 *   route    ids[t,0..k) = the k largest logits (lower index first on equal logits),
 *            descending; w[t,j] = exp(l[t,ids_j]) / sum_i exp(l[t,ids_i])   (softmax over
 *            all E followed by renormalisation over the k chosen; the full denominator cancels)
 *   permute  stable counting sort of the T*k pairs p = t*k + j by expert id
 *   experts  h = bf16( silu(Wg[e] x) * (Wu[e] x) ),  y = Wd[e] h        fp32 accumulate
 *   shared   the same SwiGLU with the shared weights, weight 1, for every token
 *   combine  out[t] = bf16( sum_j w[t,j] y[t,j] + y_shared[t] )
 * and composes long prompts from q8192 / q4096 / q2048 / q1024 pieces plus an exact tail
 * ("AIMA AMD395 Qwen3.6 35B Windows Engine", "性能优化做了什么": prompts split into a q8192
 * tile, q1024 and a tail; "AIMA AMD395 Qwen3.6 35B Linux Engine", "Read this boundary first":
 * resident q1024/q2048/q4096/q8192 buckets).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers (caller-allocated, caller-owned), row-major and
 *     contiguous, 16-byte aligned, in the [out, in] linear convention.  bf16 tensors are passed
 *     as moe_bf16 (the 16-bit pattern).  The library never allocates device memory and keeps no
 *     state between calls other than per-device launch attributes and the optional timing table.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call is
 *     asynchronous on that stream; inputs must stay valid until the stream reaches the work.
 *   - Arguments are validated on the host before any launch; an invalid call launches
 *     nothing and returns an error status.  T == 0 returns MOE_OK and does nothing.
 *   - Device-side failures (a bounded wait that ran out, an expert id out of range) are
 *     recorded in a status word in the workspace and read with moe_check_status().
 *   - Supported shapes: H % 128 == 0, I % 128 == 0, Is % 128 == 0 (or Is == 0: no shared
 *     expert), 1 <= k <= min(E, 32), E <= 1024, H <= 16384, I, Is <= 8192.  Router logits
 *     must be finite.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16; /* bit pattern of a bfloat16 value */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* null pointer, negative size, k > E, misalignment, ... */
    MOE_ERR_WORKSPACE_TOO_SMALL = 2,
    MOE_ERR_UNSUPPORTED_SHAPE = 3,  /* outside the supported shapes listed above */
    MOE_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed */
    MOE_ERR_TIMEOUT = 5,            /* a device-side bounded wait ran out (see moe_check_status) */
    MOE_ERR_NOT_IMPLEMENTED = 6
} moe_status;

/* Layer shape.  shared_inter == 0 means no shared expert. */
typedef struct {
    int hidden;       /* H */
    int n_experts;    /* E */
    int top_k;        /* k */
    int inter;        /* I */
    int shared_inter; /* Is */
} moe_config;

/* Device pointers to one layer's weights (bf16 unless noted). */
typedef struct {
    const moe_bf16 *w_router; /* [E, H] */
    const float *b_router;    /* [E] fp32 router bias, or NULL (no bias) */
    const moe_bf16 *w_gate;   /* [E, I, H] */
    const moe_bf16 *w_up;     /* [E, I, H] */
    const moe_bf16 *w_down;   /* [E, H, I] */
    const moe_bf16 *ws_gate;  /* [Is, H]  (NULL when Is == 0) */
    const moe_bf16 *ws_up;    /* [Is, H]  (NULL when Is == 0) */
    const moe_bf16 *ws_down;  /* [H, Is]  (NULL when Is == 0) */
} moe_weights;

/* One layer with quantised expert weights: every expert matrix as E4M3 codes (1 sign, 4
 * exponent bits with bias 7, 3 fraction bits; no infinities) with one fp32 scale per output row,
 * weight[r, c] = scale[r] * code[r, c].  The router stays bf16.  ("AI MAX+ 395部署Qwen3大模型：
 * GFX1151引擎实测优化解析", "两种权重格式：HGN 与 GGUF 的统一支持": 8-bit float weights for the large
 * modules; the row scales are this library's reading, the page gives no layout.)  Code arrays
 * 16-byte aligned; moe_quantize_e4m3 produces them from bf16 matrices. */
typedef struct {
    const moe_bf16 *w_router; /* [E, H] bf16 */
    const float *b_router;    /* [E] fp32, or NULL */
    const uint8_t *q_gate;    /* [E, I, H] codes */
    const uint8_t *q_up;      /* [E, I, H] */
    const uint8_t *q_down;    /* [E, H, I] */
    const float *s_gate;      /* [E, I] row scales */
    const float *s_up;        /* [E, I] */
    const float *s_down;      /* [E, H] */
    const uint8_t *qs_gate;   /* [Is, H] (NULL when Is == 0) */
    const uint8_t *qs_up;     /* [Is, H] */
    const uint8_t *qs_down;   /* [H, Is] */
    const float *ss_gate;     /* [Is] */
    const float *ss_up;       /* [Is] */
    const float *ss_down;     /* [H] */
} moe_weights_q8;

/* One layer with 4-bit integer expert weights ("Q4": 4-bit integer codes, as the GFX1151 page's
 * explanatory paragraph on weight formats calls them; the block layout is this library's
 * reading, the page gives none).  Each row of every expert matrix is cut into blocks of 32
 * consecutive columns; a block has one fp32 scale and 32 codes in [-7, 7], two's-complement
 * nibbles, column 2j in the low and 2j+1 in the high nibble of byte j of the row (cols / 2 bytes a
 * row); weight = scale * code.  The router stays bf16.  H and I (and Is) multiples of 128; code
 * arrays 16-byte aligned; moe_quantize_q4 produces them from bf16 matrices. */
typedef struct {
    const moe_bf16 *w_router; /* [E, H] bf16 */
    const float *b_router;    /* [E] fp32, or NULL */
    const uint8_t *q_gate;    /* [E, I, H/2] codes */
    const uint8_t *q_up;      /* [E, I, H/2] */
    const uint8_t *q_down;    /* [E, H, I/2] */
    const float *s_gate;      /* [E, I, H/32] block scales */
    const float *s_up;        /* [E, I, H/32] */
    const float *s_down;      /* [E, H, I/32] */
    const uint8_t *qs_gate;   /* [Is, H/2] (NULL when Is == 0) */
    const uint8_t *qs_up;     /* [Is, H/2] */
    const uint8_t *qs_down;   /* [H, Is/2] */
    const float *ss_gate;     /* [Is, H/32] */
    const float *ss_up;       /* [Is, H/32] */
    const float *ss_down;     /* [H, Is/32] */
} moe_weights_q4;

/* Text for a status code (static storage). */
const char *moe_status_string(moe_status s);

/* Bytes of device workspace needed by any call below for up to max_T tokens (moe_forward
 * needs only min(max_T, 8192) tokens' worth, since it works piece by piece).  Returns 0 for
 * an invalid or unsupported config.  The workspace must be 256-byte aligned.  Its first 256
 * bytes hold the device status word: zero them once after allocating the workspace (kernels
 * only ever change the word from 0 to an error code; moe_check_status clears it).  The rest
 * is scratch that every call overwrites. */
size_t moe_workspace_size(const moe_config *cfg, int max_T);

/* Router: logits, softmax, top-k and renormalisation.  Passage: each token activates only a few
 * of many experts ("AI MAX+ 395部署Qwen3大模型：GFX1151引擎实测优化解析", explanatory MoE
 * paragraph under "MOE 内核优化"); the selection rule (largest logits, lower index on ties,
 * weights renormalised over the k) is this library's reading, the pages give no formula.
 * x [T,H] bf16 -> topk_ids [T,k] int32 and topk_w [T,k] fp32, slots in descending logit
 * order.  logits_out [T,E] fp32 may be NULL; when given it receives the exact fp32 logits the
 * selection used.  ws: workspace of moe_workspace_size(cfg, T) bytes (holds the logits when
 * logits_out is NULL).  Computed on tensor cores (bf16 x bf16 -> fp32 accumulate); for the
 * 1 to 4 tokens moe_forward runs on the decode path, by that path's GEMV, so the logits are
 * the ones moe_forward selects on. */
moe_status moe_route(const moe_config *cfg, const moe_weights *w, const moe_bf16 *x, int T,
                     float *logits_out, int32_t *topk_ids, float *topk_w, void *ws,
                     size_t ws_bytes, void *stream);

/* Softmax + top-k + renormalisation only, from given fp32 logits [T,E] (the routing step of
 * the same passage as moe_route).  Bit-exact ids for
 * identical logits (the selection compares fp32 values exactly, lower index first on ties). */
moe_status moe_route_from_logits(const moe_config *cfg, const float *logits, int T,
                                 int32_t *topk_ids, float *topk_w, void *stream);

/* Permutation of the T*k (token, slot) pairs by expert: a stable counting sort.  Passage: the
 * "selected-MoE" kernel runs only the experts each token selected ("AIMA AMD395 Qwen3.6 35B
 * Windows Engine", "性能优化做了什么"), which needs each expert's tokens gathered together; the
 * page does not describe how, so the grouping is this library's (a textbook stable sort).
 * topk_ids [T,k] -> expert_offsets [E+1] (exclusive prefix sum of the per-expert counts,
 * offsets[E] == T*k), perm [T*k] (row of the expert-sorted order -> pair index t*k+j),
 * inv [T*k] (pair index -> row).  Pairs of one expert keep increasing pair order.  Bit-exact.
 * ws: workspace of moe_workspace_size(cfg, T) bytes.  Ids outside [0,E) are a caller error:
 * they are detected on the device, flagged in the status word, and the pair is dropped
 * (inv = -1). */
moe_status moe_permute(const moe_config *cfg, const int32_t *topk_ids, int T,
                       int32_t *expert_offsets, int32_t *perm, int32_t *inv, void *ws,
                       size_t ws_bytes, void *stream);

/* moe_permute without a workspace, for callers that cannot allocate device memory where
 * they route tokens (a serving process that reserves all device memory at start-up, host
 * code with no allocator at hand).  The pages have no counterpart: this is a convenience of
 * this library.  Same outputs as moe_permute (bit-identical), but the per-chunk count table
 * lives in a fixed array inside the library (160 KiB on every device that loads it, kept
 * until the process exits), so the call allocates nothing and takes no workspace.
 * Limits: T*k <= 65536 pairs, E <= 1024, k <= 32; larger problems return
 * MOE_ERR_UNSUPPORTED_SHAPE (use moe_permute).  Ids outside [0,E) get inv = -1 and are not
 * otherwise reported (no status word).  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array: calls that overlap on the GPU
 * (different streams or threads) race and must be serialised by the caller. */
moe_status moe_permute_noalloc(const moe_config *cfg, const int32_t *topk_ids, int T,
                               int32_t *expert_offsets, int32_t *perm, int32_t *inv,
                               void *stream);

/* Expert FFNs, unfused (for step-by-step checking).  Passage: the selected experts' own
 * sub-networks ("AI MAX+ 395部署Qwen3大模型：GFX1151引擎实测优化解析", "MOE 内核优化": the MoE
 * kernel that bounds prefill), read as SwiGLU experts plus an always-on shared expert.
 * Routed rows in the permuted order:
 * h_rows [T*k, I] bf16 = bf16(silu(Wg[e] x_t) * (Wu[e] x_t)) and y_rows [T*k, H] fp32 =
 * Wd[e] h, for row r of expert e holding pair perm[r] of token perm[r]/k.  When shared_y is not
 * NULL and Is > 0, also shared_y [T,H] fp32 = the shared expert applied to every token.
 * expert_offsets/perm as produced by moe_permute.  ws: moe_workspace_size(cfg, T) bytes. */
moe_status moe_expert_ffn(const moe_config *cfg, const moe_weights *w, const moe_bf16 *x, int T,
                          const int32_t *expert_offsets, const int32_t *perm, moe_bf16 *h_rows,
                          float *y_rows, float *shared_y, void *ws, size_t ws_bytes,
                          void *stream);

/* Weighted combine (the last step of the selected-MoE layer, "AIMA AMD395 Qwen3.6 35B Windows
 * Engine", "性能优化做了什么"; the weighting by the renormalised routing weights is this
 * library's reading): out[t] = bf16( sum_j topk_w[t,j] * y_rows[inv[t*k+j]] + shared_y[t] ).
 * shared_y may be NULL (no shared term).  Deterministic (fixed slot order, fp32). */
moe_status moe_combine(const moe_config *cfg, const float *y_rows, const int32_t *inv,
                       const float *topk_w, const float *shared_y, int T, moe_bf16 *out,
                       void *stream);

/* The whole layer, fused: x [T,H] -> out [T,H] bf16.  T is split greedily into pieces of
 * 8192, 4096, 2048 and 1024 tokens and an exact tail (no padding); every piece runs the same
 * kernels, so the result equals the concatenation of per-piece calls.  A call (or tail) of 1
 * to 4 tokens with T*H <= 32768 takes the decode path: a router GEMV, then every selected
 * expert's weights streamed once for all the tokens that chose it, its partial products
 * added in fp32 with atomics (so not bit-reproducible) and rounded to bf16 once.  x_next may
 * be NULL; when given it receives bf16(resid + out), the residual-stream update of a layer
 * stack, fused into the last kernel; resid [T,H] may be NULL, meaning x.  x_next may alias
 * resid (not x, when they differ).  ws: moe_workspace_size(cfg, T) bytes.  Rounding on the
 * prefill path: h is rounded to bf16 once, each weighted expert row w*y (and the shared
 * expert's row) is stored as bf16, the k+1 rows of a token are summed in fp32 in slot order,
 * and the sum is rounded to bf16 once.  No atomics there: the result is bit-reproducible.
 * Any T >= 0 (int) is accepted: the pieces are walked one after another, so there is no limit
 * on their number. */
moe_status moe_forward(const moe_config *cfg, const moe_weights *w, const moe_bf16 *x, int T,
                       moe_bf16 *out, const moe_bf16 *resid, moe_bf16 *x_next, void *ws,
                       size_t ws_bytes, void *stream);

/* moe_forward for a layer with quantised expert weights (moe_weights_q8): the same piece
 * composition, router (bf16 weights), selection, permutation, rounding points and combine, with
 * every expert matrix streamed as its E4M3 codes, one byte a weight ("AI MAX+ 395部署Qwen3大模型：
 * GFX1151引擎实测优化解析", "两种权重格式：HGN 与 GGUF 的统一支持": 8-bit float weights for the large
 * modules).  The grouped GEMMs widen each code exactly to bf16 in shared memory (every E4M3 value
 * is a bf16 value), multiply with bf16 tokens into fp32, and scale each weight row's accumulator
 * by its fp32 row scale; h = bf16(silu(g) * u) as in moe_forward.  Every piece, however short,
 * takes this grouped path (there is no E4M3 variant of the 1-4-token kernels in moe_forward;
 * moe_decode_chain_q8 is the quantised decode step).  Same arguments, workspace, alignment and
 * errors as moe_forward. */
moe_status moe_forward_q8(const moe_config *cfg, const moe_weights_q8 *w, const moe_bf16 *x, int T,
                          moe_bf16 *out, const moe_bf16 *resid, moe_bf16 *x_next, void *ws,
                          size_t ws_bytes, void *stream);

/* A layer stack captured once as a CUDA graph and replayed (the resident prefill buckets of
 * "AIMA AMD395 Qwen3.6 35B Linux Engine", release boundary v1.5.0: one graph per bucket size,
 * kept resident with its workspace).  The graph holds n_layers (1..64) moe_forward calls on T
 * tokens with these exact pointers: layer 0 reads x0; layer l writes out and
 * x_{l+1} = bf16(r + out_l), r = resid when given, else x_l; layer l+1 reads x_{l+1}.  The
 * intermediate x_l alternate between x_last and scratch so that x_last receives x_{n_layers};
 * both [T,H] bf16, required when n_layers > 1 (x_last may be NULL for one layer; scratch is
 * then unused), distinct from x0, resid and out.  Every buffer, the weights and ws must stay
 * allocated and unchanged in place while the graph lives; their contents may change between
 * launches (a new x0 is simply copied into x0's buffer).
 * moe_graph_create validates as moe_forward does, runs the stack once on `stream` (this
 * warms the library's per-device launch caches and writes the outputs), then captures it on a
 * private stream and instantiates it.  moe_graph_launch replays it on `stream`, asynchronously;
 * moe_launch_count() advances by the graph's kernel count.  Calls sharing ws must not overlap.
 * moe_graph_destroy frees the graph (NULL is a no-op). */
typedef struct moe_graph_s *moe_graph;
moe_status moe_graph_create(const moe_config *cfg, const moe_weights *layers, int n_layers, int T,
                            const moe_bf16 *x0, const moe_bf16 *resid, moe_bf16 *out, moe_bf16 *x_last,
                            moe_bf16 *scratch, void *ws, size_t ws_bytes, void *stream, moe_graph *graph);
moe_status moe_graph_launch(moe_graph graph, void *stream);
/* Kernel nodes in the graph (-1 for NULL). */
int moe_graph_kernel_count(moe_graph graph);
moe_status moe_graph_destroy(moe_graph graph);

/* One token through a stack of n_layers MoE layers (1 <= n_layers <= 64), each with its own
 * weights layers[l] (a host array of device pointers), in ONE cooperative kernel launch: the
 * batch-1 greedy decode step the pages run ("AIMA AMD395 Qwen3.6 35B Windows Engine",
 * "产品定位"), with the MoE layers back to back.  x_0 = x0 [H] bf16; for each layer
 * out_l = the layer applied to x_l (as moe_forward with T = 1: same router rows, selection and
 * rounding points) and x_{l+1} = bf16(r + out_l), r = resid [H] when given, else x_l (the
 * residual stream).  out [H] receives the last layer's out; x_last [H] (may be NULL) receives
 * x_{n_layers}.  The layers are separated by grid barriers instead of kernel boundaries; the
 * fp32 atomics of the split-K down projection make the last bit run-dependent, as at T = 1.
 * Requires T = 1 to fit the decode path (H <= 16384).  x0, resid, out, x_last 16-byte aligned;
 * out and x_last must not alias x0 or resid.  ws: moe_workspace_size(cfg, 1) bytes; the call
 * writes its barrier words there, so calls sharing a workspace must not overlap.  A barrier
 * wait that runs out (2 s) records MOE_ERR_TIMEOUT in the workspace status word and every
 * block returns.  MOE_ERR_UNSUPPORTED_SHAPE for more than 64 layers or a too-large H. */
moe_status moe_decode_chain(const moe_config *cfg, const moe_weights *layers, int n_layers,
                            const moe_bf16 *x0, const moe_bf16 *resid, moe_bf16 *out,
                            moe_bf16 *x_last, void *ws, size_t ws_bytes, void *stream);

/* moe_decode_chain for layers with quantised expert weights (moe_weights_q8): every expert
 * row streamed as its E4M3 codes (half the bytes of bf16) and its scale, widened exactly and
 * accumulated in fp32; otherwise the same steps, rounding points, barriers and errors. */
moe_status moe_decode_chain_q8(const moe_config *cfg, const moe_weights_q8 *layers, int n_layers,
                               const moe_bf16 *x0, const moe_bf16 *resid, moe_bf16 *out,
                               moe_bf16 *x_last, void *ws, size_t ws_bytes, void *stream);

/* moe_decode_chain for layers with 4-bit expert weights (moe_weights_q4): every expert row
 * streamed as its codes (a quarter of the bytes of bf16) and block scales, each block's codes
 * dotted in fp32 and scaled; otherwise the same steps, rounding points, barriers and errors. */
moe_status moe_decode_chain_q4(const moe_config *cfg, const moe_weights_q4 *layers, int n_layers,
                               const moe_bf16 *x0, const moe_bf16 *resid, moe_bf16 *out,
                               moe_bf16 *x_last, void *ws, size_t ws_bytes, void *stream);

/* Block-wise 4-bit quantisation of a bf16 matrix w [rows, cols] (device pointers; cols a multiple
 * of 32): per block of 32 columns, scale = max |w| / 7 (1 for an all-zero block) and code =
 * round-half-even(w / scale) clamped to [-7, 7], in fp32 with IEEE division (a function of the
 * block alone).  q [rows, cols/2] packed nibbles (column 2j low, 2j+1 high), scale [rows, cols/32]
 * fp32.  Blocks holding an infinity or a NaN give unspecified codes.  Asynchronous on `stream`;
 * rows or cols of 0 do nothing; a negative size, cols not a multiple of 32 or a NULL pointer is
 * MOE_ERR_INVALID_ARG. */
moe_status moe_quantize_q4(const moe_bf16 *w, int rows, int cols, uint8_t *q, float *scale, void *stream);

/* Row-wise E4M3 quantisation of a bf16 matrix w [rows, cols] (device pointers): scale[r] =
 * max_c |w[r,c]| / 448 (1 for an all-zero row) and q[r,c] = the E4M3 code nearest to
 * w[r,c] / scale[r] (ties to even; magnitudes past 448 saturate), in fp32 with IEEE division,
 * so the result is a function of the row alone.  q [rows, cols] bytes, scale [rows] fp32.
 * Rows holding an infinity or a NaN give unspecified codes.  Asynchronous on `stream`; rows or
 * cols of 0 do nothing; a negative size or a NULL pointer is MOE_ERR_INVALID_ARG. */
moe_status moe_quantize_e4m3(const moe_bf16 *w, int rows, int cols, uint8_t *q, float *scale,
                             void *stream);

/* Reads and clears the device status word in `ws` (synchronises `stream`).  *device_status
 * receives MOE_OK or the first error recorded by a kernel (MOE_ERR_TIMEOUT for a wait that
 * ran out, MOE_ERR_INVALID_ARG for an out-of-range expert id).  Returns MOE_ERR_CUDA if the
 * copy fails. */
moe_status moe_check_status(void *ws, size_t ws_bytes, int *device_status, void *stream);

/* Diagnostics, not a step of the layer: one device thread waits on a barrier with the same
 * bounded wait every pipeline of this library uses.  With arrive != 0 the barrier completes
 * first and the wait returns at once; with arrive == 0 nothing arrives, the wait gives up after
 * limit_ns nanoseconds (at most 1e9) and records MOE_ERR_TIMEOUT in the workspace status word,
 * which moe_check_status then reports.  No fault, trap or hang: the kernel returns, and the
 * stream and context stay usable.  ws: at least the 256-byte status area of a workspace
 * (256-byte aligned).  Returns MOE_ERR_INVALID_ARG for a bad workspace or limit. */
moe_status moe_selftest_wait(void *ws, size_t ws_bytes, unsigned long long limit_ns, int arrive,
                             void *stream);

/* Sizes of the pieces moe_forward splits T into: writes up to max_pieces sizes to `pieces`
 * and returns the number of pieces (host only, no device work); -1 if T < 0. */
int moe_plan_pieces(int T, int *pieces, int max_pieces);

/* Number of kernels this library has launched in this process (host counter). */
uint64_t moe_launch_count(void);

/* Optional per-kernel timing.  While enabled, every kernel launch is bracketed by CUDA events
 * on its stream; moe_timing_read() synchronises them and returns, for kernel class `name`
 * (see moe_timing_name()), the number of launches and their total device time in ms, then
 * forgets them.  Returns MOE_ERR_INVALID_ARG for an unknown name.  Not for use inside CUDA
 * graph capture. */
moe_status moe_timing_enable(int enable);
moe_status moe_timing_read(const char *name, int *launches, double *total_ms);
/* 1 when this library was built with MOE_DEBUG: every kernel then checks each index it reads from
 * device data (permutation rows, caller-given expert offsets, combine rows, GEMM output rows)
 * before using it, records MOE_ERR_INVALID_ARG in the workspace status word (moe_combine has
 * none) and skips the access.  0 for the ordinary build, which does not check them. */
int moe_debug_build(void);

/* Name of kernel class i (0 <= i < moe_timing_classes()), or NULL. */
const char *moe_timing_name(int i);
int moe_timing_classes(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
