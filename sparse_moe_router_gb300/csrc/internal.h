// internal.h -- declarations shared by the translation units of libmoe.so (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Kernel classes for launch counting and optional per-kernel timing.
enum KernelClass {
    KC_ROUTER_GEMM = 0,   // router logits on tensor cores
    KC_TOPK,              // softmax + top-k + renormalise
    KC_PERMUTE,           // histogram + scan + stable scatter
    KC_TILE_PREFIX,       // token-tile prefix from given offsets
    KC_GATEUP_GEMM,       // routed grouped gate/up GEMM + SwiGLU
    KC_DOWN_GEMM,         // routed grouped down GEMM (+ weighted combine)
    KC_SHARED_GATEUP,     // shared expert gate/up + SwiGLU
    KC_SHARED_DOWN,       // shared expert down
    KC_FINALIZE,          // fp32 accumulator -> bf16 out (+ residual)
    KC_COMBINE,           // unfused weighted combine
    KC_ZERO,              // accumulator clear
    KC_DECODE_ROUTER,     // decode: router GEMV
    KC_DECODE_EXPERTS,    // decode: top-k, expert gate/up slices, split-K down, combine
    KC_GATHER_X,          // token rows copied into expert-sorted order
    KC_DECODE_CHAIN,      // decode: a chain of layers in one cooperative launch
    KC_QUANTIZE,          // row-wise E4M3 quantisation of weights
    KC_COUNT
};

const char *kernel_class_name(int kc);

// Launch bookkeeping: counts the launch and, when timing is on, records events around it.
struct LaunchScope {
    LaunchScope(int kc, cudaStream_t s);
    ~LaunchScope();
    int kc;
    cudaStream_t stream;
    cudaEvent_t ev0, ev1;
    bool timed;
};

struct DeviceInfo {
    int sm_count;
};
const DeviceInfo &device_info();

// cuTensorMapEncodeTiled obtained through the runtime's driver entry point: a 2-D bf16 map
// over [rows, cols] (cols contiguous) with a box_rows x box_cols box, 128-byte swizzle (or
// none: plain row-major boxes).
bool encode_tmap_2d_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows, uint32_t box_cols, bool swizzle128 = true);

// ---- GEMM (tcgen05, swap-AB: weight rows on M, tokens on N) ---------------------------

constexpr int kTileN = 256;   // tokens per GEMM tile (MMA N upper bound)
constexpr int kTileM = 128;   // weight rows per GEMM tile (MMA M)
// token rows per TMA box of a GEMM's token operand: each CTA of a pair holds half a tile
constexpr int kTokenBoxRows = kTileN / 2;
// The token operand's maps: m[i] has a box of 16 (i + 1) rows x 64 columns, so that each CTA
// loads, in one TMA instruction a K block, the smallest box that holds its half of a tile.
// `shared` (box kTokenBoxRows rows) is the shared expert's token rows when they live in a
// buffer of their own (GemmArgs::shared_b_own).
constexpr int kTokenBoxes = kTokenBoxRows / 16;
struct TokenMaps {
    CUtensorMap m[kTokenBoxes];
    CUtensorMap shared;
};
// m[] over [rows, cols] bf16 at base; `shared` set to m[kTokenBoxes - 1]
bool encode_token_maps(TokenMaps *tm, const void *base, uint64_t rows, uint64_t cols);

// EPI_F32: out[r, f] = D + bias[f] (fp32).  EPI_SWIGLU: h = bf16(silu(gate) * up).
// EPI_COMBINE: out[epi_tok[r], f] = bf16(epi_w[r] * D) -- the weighted expert rows, stored in
// pair order for the combine that follows.
enum GemmEpi { EPI_F32 = 0, EPI_SWIGLU = 1, EPI_COMBINE = 2 };

#ifdef __CUDACC__
// MOE_DEBUG builds check every index a kernel reads from device data (permutation rows,
// caller-given offsets, combine rows, GEMM output rows) before using it: an index outside its
// buffer records MOE_ERR_INVALID_ARG in the status word (when the kernel has one) and the access
// is skipped.  Ordinary builds compile the checks away.
#ifdef MOE_DEBUG
__device__ __forceinline__ bool moe_debug_ok(bool ok, int *status) {
    if (!ok && status) atomicCAS(status, 0, (int)MOE_ERR_INVALID_ARG);
    return ok;
}
#define MOE_DEBUG_OK(cond, status) moe_debug_ok((cond), (status))
#else
#define MOE_DEBUG_OK(cond, status) true
#endif

// Order-preserving map of fp32 onto uint32 (-0 folded onto +0, so equal values get equal keys)
// and its inverse: top-k rounds compare logits with one integer warp reduction.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
#endif

struct GemmArgs {
    // token side (B operand): row r of the group row space is row r of b_src ([*, K] bf16),
    // loaded through the B tensor map
    const void *b_src;
    int K;
    // groups: group_rows [G+1] row offsets and group_tiles [G+1] token-tile prefix, both on the
    // device; or NULL for one group of M_single rows.
    int n_groups;
    const int32_t *group_rows;
    const int32_t *group_tiles;
    int M_single;
    // weight side (A operand): F rows per group, group g starts at row g*F of the tensor maps
    int F;
    // epilogue
    void *out;
    int ld;
    const float *bias;
    // EPI_COMBINE: row r stores bf16(epi_w[r] * D) into out row epi_tok[r] (NULL: row r, weight 1)
    const int32_t *epi_tok;
    const float *epi_w;
    int *status;
    // token tile cap (a multiple of 16, <= 256; 0 = 256).  Each CTA of a pair loads half a
    // tile: N/2 rows, N = the tile's rows rounded up to 16
    int tile_cap;
    // the last group is the shared expert: its weight rows come from the tm_s* maps (row
    // ftile*kFT of the shared matrix), its tiles are interleaved evenly among the routed ones,
    // and the combine epilogue stores its rows in place with weight 1
    bool shared_last;
    // with shared_last: the last group's token rows are rows 0.. of the TokenMaps' `shared` map
    // (the tokens in order, e.g. x itself) instead of rows group_rows[G-1].. of the m[] maps
    bool shared_b_own;
    // tile schedule: pair p takes tiles p, p + pairs, ... except the last dyn_tail tiles, which
    // pairs claim from tile_counter (a device counter, zero at launch) as they come free.
    // tile_counter NULL or dyn_tail 0: every tile round-robin.
    int *tile_counter;
    int dyn_tail;
    // E4M3 weights: the weight maps are over byte codes (row-major, no swizzle, 64-byte boxes of
    // 64 or 128 rows) and the accumulator of weight row f of group g is multiplied by
    // w_scale0[g * F + f] (SwiGLU: gate rows; w_scale1: up rows); the shared expert's group by
    // ws_scale0 / ws_scale1 [f]
    bool q8;
    const float *w_scale0, *w_scale1, *ws_scale0, *ws_scale1;
    // MOE_DEBUG: rows of `out` and of the group row space (epi_tok / epi_w), 0 = unknown
    int out_rows, src_rows;
    // ints to zero before the GEMM's own work (the next kernels' count table), or NULL
    int32_t *zero_ptr;
    int zero_n;
};

// Launch the persistent grouped GEMM.  tm_a0 (and tm_a1 for EPI_SWIGLU: the up projection)
// are 2-D tensor maps over the weight rows (64- or 128-row box, 64 columns); tm_b holds the maps
// over the B rows ([rows, K], see TokenMaps).  tm_s0 / tm_s1 are the shared expert's
// weight maps, read for the last group when a.shared_last (pass any map otherwise).
cudaError_t launch_gemm(GemmEpi epi, const GemmArgs &a, const CUtensorMap &tm_a0, const CUtensorMap &tm_a1,
                        const TokenMaps &tm_b, const CUtensorMap &tm_s0, const CUtensorMap &tm_s1, int kc,
                        cudaStream_t s);

// ---- routing / permutation / elementwise ---------------------------------------------

cudaError_t launch_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                        cudaStream_t s);
// The same selection, and each chunk's expert counts added into chunk_tab (which must hold
// zeros: permute_scratch_ints(T, E, k) of them), for launch_scan_scatter.
cudaError_t launch_topk_hist(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                             int32_t *chunk_tab, cudaStream_t s);
// The permutation from the counts launch_topk_hist left in chunk_tab, in one launch: every block
// derives its chunk's first row per expert from the whole table (the offsets and the token-tile
// prefix are written by block 0), then scatters its chunk as launch_permute does.  The table is
// read only.
cudaError_t launch_scan_scatter(const int32_t *ids, int T, int E, int k, int32_t *offsets, int32_t *perm,
                                int32_t *inv, int32_t *tile_prefix, const int32_t *chunk_tab,
                                const float *topk_w, int32_t *row_tok, float *row_w, int *status,
                                cudaStream_t s, int extra_rows, int *sched);
// chunk_tab: device scratch of permute_scratch_ints(T, E, k) ints.  When row_tok / row_w are
// not NULL the scatter also writes, per row of the sorted order, the token (pair / k) and the
// routing weight topk_w[pair] (what the expert GEMMs read per row).  extra_rows > 0 appends one
// more group of that many rows after the experts (offsets[E+1], tile_prefix[E+1]): the shared
// expert's rows when it runs inside the routed GEMMs.
// The permutation works on chunks of whole tokens: chunk c holds tokens [c*CT, (c+1)*CT) and so
// pairs [c*CT*k, (c+1)*CT*k), with CT = perm_chunk_tokens(k) a multiple of 8 (the top-k kernel's
// 8-token blocks each fall in one chunk) and CT*k <= kPermChunk pairs (one block of the scatter).
// The chunk table holds one row of E counts per chunk.
constexpr int kPermChunk = 2048;
__host__ __device__ __forceinline__ int perm_chunk_tokens(int k) {
    const int ct = (kPermChunk / k) & ~7;
    return ct < 8 ? 8 : ct;
}
// Tile counters of the grouped GEMMs that follow a permutation (gate/up, down): `sched` (or
// NULL) receives kSchedCounters zeros from the permutation's scan kernel.
constexpr int kSchedCounters = 2;
size_t permute_scratch_ints(int T, int E, int k);
cudaError_t launch_permute(const int32_t *ids, int T, int E, int k, int32_t *offsets,
                           int32_t *perm, int32_t *inv, int32_t *tile_prefix, int tile_n,
                           int32_t *chunk_tab, const float *topk_w, int32_t *row_tok,
                           float *row_w, int *status, cudaStream_t s, int extra_rows = 0,
                           int *sched = nullptr);
// Token-tile prefix from given offsets, and row_tok[r] = perm[r] / k for the P rows (and the
// zeroed tile counters, as launch_permute).
cudaError_t launch_tile_prefix(const int32_t *offsets, int E, int32_t *tile_prefix, int tile_n,
                               const int32_t *perm, int P, int k, int32_t *row_tok,
                               cudaStream_t s, int *sched = nullptr, int *status = nullptr);
// out[t] = bf16( sum_j y[t*k + j] + acc[t] ) with y bf16 [T*k, H] (the weighted expert rows in
// pair order) and acc fp32 [T, H] (the shared expert, or NULL); when x_next != NULL also
// x_next = bf16(resid + out).  The sum runs in fp32, slots in order, then the shared term.
// xp[r] = x[row_tok[r]] for the P expert-sorted rows (H bf16 each); a row whose token index is
// outside [0, T) is written as zeros.
// n_tail > 0: rows P .. P+n_tail-1 of xp are x's rows 0 .. n_tail-1 in order (the shared
// expert's group).
cudaError_t launch_gather_rows(const uint16_t *x, int T, int H, const int32_t *row_tok, int P,
                               uint16_t *xp, cudaStream_t s, int n_tail = 0);
// y_tail (bf16 [T, H], or NULL) is added like one more expert row of weight 1.
cudaError_t launch_finalize(const uint16_t *y, int k, const float *acc, const uint16_t *resid, int T,
                            int H, uint16_t *out, uint16_t *x_next, cudaStream_t s,
                            const uint16_t *y_tail = nullptr);
cudaError_t launch_combine(const float *y_rows, const int32_t *inv, const float *topk_w,
                           const float *shared_y, int T, int H, int k, uint16_t *out,
                           cudaStream_t s);
// true when the library was compiled with MOE_DEBUG (device index checks)
bool debug_build();
cudaError_t launch_zero(float *p, size_t n, cudaStream_t s);

// ---- decode (T = 1) ------------------------------------------------------------------

// Decode path: 1 <= T <= kMaxDecodeT tokens with T * H <= kMaxDecodeTH (their x in shared memory).
// Above 4 tokens the expert weights the tokens share no longer outweigh the decode kernels'
// per-block costs, and the prefill path is faster (measured: 8 tokens 162 vs 138 us per layer).
constexpr int kMaxDecodeT = 4;
constexpr int kMaxDecodeTH = 32768;
inline bool decode_fits(int T, int H) { return T >= 1 && T <= kMaxDecodeT && (long)T * H <= kMaxDecodeTH; }

struct DecodeArgs {
    int T;  // tokens (1 .. kMaxDecodeT); x, out, resid, x_next are [T, H], logits [T, E], acc [T, H]
    int H, E, k, I, Is;
    const uint16_t *x;
    const uint16_t *w_router;
    const float *b_router;
    const uint16_t *w_gate, *w_up, *w_down;
    const uint16_t *ws_gate, *ws_up, *ws_down;
    float *logits;     // [E]
    int32_t *ids;      // [k]
    float *topw;       // [k]
    uint16_t *h;       // [k, I]
    uint16_t *h_s;     // [Is]
    uint16_t *out;     // [H]
    const uint16_t *resid;  // [H] residual added into x_next
    uint16_t *x_next;  // [H] or NULL
    float *acc;        // [H] fp32 accumulator (cleared by the first kernel)
    int *counter;      // ticket counter, zero between calls (the last block resets it)
    int *status;       // device status word or NULL
};
// tm_down: map over w_down as [E*H, I], tm_sdown: over ws_down as [H, Is] (or any map when
// Is == 0); both unswizzled with a 128-row x decode_slice()-column box.
cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &tm_down, const CUtensorMap &tm_sdown,
                          cudaStream_t s);
int decode_slice();
int decode_box_rows();
// Router logits of one token with the decode GEMV (the logits the decode path selects on).
cudaError_t launch_decode_router(const DecodeArgs &a, cudaStream_t s);

// One token through a chain of L layers in one cooperative launch (moe_decode_chain): per layer
// out_l = layer_l(x_l), x_{l+1} = bf16(r + out_l) with r = resid, or x_l when resid is NULL.
constexpr int kChainMaxLayers = 64;
struct ChainLayer {
    const uint16_t *w_router;
    const float *b_router;
    // bf16 expert rows, or (the code formats) their codes
    const void *w_gate, *w_up, *ws_gate, *ws_up;
    // E4M3: fp32 scales per output row (gate/up [E, I], down [E, H]; shared [Is], [H]);
    // 4-bit codes: per block of 32 columns (gate/up [E, I, H/32], down [E, H, I/32]; shared
    // [Is, H/32], [H, Is/32])
    const float *s_gate, *s_up, *s_down, *ss_gate, *ss_up, *ss_down;
};
struct ChainParams {
    CUtensorMap tm_down[kChainMaxLayers];   // w_down as [E*H, I] (bf16 or bytes), decode box
    CUtensorMap tm_sdown[kChainMaxLayers];  // ws_down as [H, Is]
    ChainLayer lay[kChainMaxLayers];
    int H, E, k, I, Is, L;
    const uint16_t *x0;     // [H]
    const uint16_t *resid;  // [H] or NULL
    uint16_t *out;          // [H] the last layer's output
    uint16_t *x_last;       // [H] or NULL: bf16(r + out) after the last layer
    // [E] tagged logits: (layer + 1) << 32 | fp32 bits, zero at launch
    unsigned long long *logits;
    float *acc0, *acc1, *acc2;  // [H] each; layer l adds into acc(l % 3)
    unsigned *bar;          // grid-barrier counter, zero at launch
    int *abort;             // zero at launch; set by a block that gives up
    int *status;            // device status word
};
// The chain's expert weight formats: bf16; E4M3 codes with fp32 row scales (ChainLayer's s_*);
// 4-bit codes with fp32 scales per block of 32 columns.  The code formats' W_d maps are over bytes.
constexpr int kChainBf16 = 0, kChainE4m3 = 1, kChainQ4 = 2;
cudaError_t launch_decode_chain(const ChainParams &p, int wf, cudaStream_t s);
// Row-wise E4M3 quantisation: scale[r] = max_c |w[r,c]| / 448 (1 for a zero row),
// q[r,c] = E4M3(w[r,c] / scale[r]), fp32 arithmetic, round to nearest even, saturating.
cudaError_t launch_quantize_e4m3(const uint16_t *w, int rows, int cols, uint8_t *q, float *scale,
                                 cudaStream_t s);
// Block-wise 4-bit quantisation (cols % 32 == 0): per block of 32 columns scale = max |w| / 7 (1 for
// an all-zero block), code = round-half-even(w / scale) clamped to [-7, 7] (fp32, IEEE division),
// packed two's-complement nibbles (column 2j low, 2j+1 high); q [rows, cols/2], scale [rows, cols/32].
cudaError_t launch_quantize_q4(const uint16_t *w, int rows, int cols, uint8_t *q, float *scale, cudaStream_t s);

// Token tiles of a group of c rows: ceil(c / 256) tiles of equal size rounded up to 16 (the
// MMA's N granularity); the last tile takes the remainder.  Shared by the permutation (tile
// prefix) and the GEMM (tile decode), so both agree on every tile.
// (A launch may lower the cap below 256 for more, smaller tiles: the router GEMM.)
__host__ __device__ __forceinline__ int token_tile_size(int c, int cap = kTileN) {
    if (c <= 0) return cap;
    const int n = (c + cap - 1) / cap;
    const int sz = (c + n - 1) / n;
    return (sz + 15) & ~15;
}
__host__ __device__ __forceinline__ int token_tile_count(int c, int cap = kTileN) {
    if (c <= 0) return 0;
    const int sz = token_tile_size(c, cap);
    return (c + sz - 1) / sz;
}

}  // namespace moe
