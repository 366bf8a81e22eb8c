// moe_abi.cu -- the extern "C" entry points of include/moe.h: argument validation,
// workspace carving, tensor-map encoding, and the order of kernel launches for each call.
//
// moe_forward composes a prompt of any length from pieces of 8192, 4096, 2048 and 1024
// tokens and an exact tail ("AIMA AMD395 Qwen3.6 35B Windows Engine", "性能优化做了什么":
// any prompt split into a q8192 tile, q1024 and a tail; "AIMA AMD395 Qwen3.6 35B Linux
// Engine", "Read this boundary first": resident q1024/q2048/q4096/q8192 buckets).  The pages
// pad the last bucket; here the tail runs at its exact length, because the layer treats every
// token independently and the kernels take any token count (padding would only add work).
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include "internal.h"

namespace moe {

// ------------------------------------------------------------------ bookkeeping --

namespace {
std::atomic<uint64_t> g_launches{0};
std::atomic<bool> g_timing{false};
std::mutex g_timing_mu;
struct TimedPair {
    cudaEvent_t a, b;
};
std::vector<TimedPair> g_timed[KC_COUNT];

const char *const kClassNames[KC_COUNT] = {
    "router_gemm", "topk",          "permute",     "tile_prefix",   "gateup_gemm",
    "down_gemm",   "shared_gateup", "shared_down", "finalize",      "combine",
    "zero",        "decode_router", "decode_experts", "gather_x",
    "decode_chain", "quantize"};
}  // namespace

const char *kernel_class_name(int kc) { return (kc >= 0 && kc < KC_COUNT) ? kClassNames[kc] : nullptr; }

// set while this thread captures a graph: launches are counted when the graph is replayed,
// and no timing events are recorded into it
thread_local bool t_capturing = false;

LaunchScope::LaunchScope(int kc_, cudaStream_t s) : kc(kc_), stream(s), ev0(nullptr), ev1(nullptr), timed(false) {
    if (t_capturing) return;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (g_timing.load(std::memory_order_relaxed)) {
        if (cudaEventCreate(&ev0) == cudaSuccess && cudaEventCreate(&ev1) == cudaSuccess) {
            timed = cudaEventRecord(ev0, s) == cudaSuccess;
        }
    }
}

LaunchScope::~LaunchScope() {
    if (timed && cudaEventRecord(ev1, stream) == cudaSuccess) {
        std::lock_guard<std::mutex> lk(g_timing_mu);
        g_timed[kc].push_back({ev0, ev1});
        return;
    }
    if (ev0) cudaEventDestroy(ev0);
    if (ev1) cudaEventDestroy(ev1);
}

const DeviceInfo &device_info() {
    static DeviceInfo infos[64];
    static bool have[64] = {false};
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!have[dev]) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        infos[dev].sm_count = sms > 0 ? sms : 1;
        have[dev] = true;
    }
    return infos[dev];
}

// ------------------------------------------------------------------ tensor maps --

namespace {
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

namespace {
bool encode_tmap_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_cols, bool swizzle128, CUtensorMapDataType dtype, uint64_t esize) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
}  // namespace

bool encode_tmap_2d_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows, uint32_t box_cols, bool swizzle128) {
    return encode_tmap_2d(map, base, rows, cols, box_rows, box_cols, swizzle128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2);
}

bool encode_token_maps(TokenMaps *tm, const void *base, uint64_t rows, uint64_t cols) {
    for (int i = 0; i < kTokenBoxes; ++i)
        if (!encode_tmap_2d_bf16(&tm->m[i], base, rows, cols, (uint32_t)(16 * (i + 1)), 64)) return false;
    tm->shared = tm->m[kTokenBoxes - 1];
    return true;
}

// E4M3 weight codes [rows, cols] as a plain row-major byte map with box_rows x 64-byte boxes
// (the raw slot layout the GEMM's converter warps read).
bool encode_tmap_2d_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    return encode_tmap_2d(map, base, rows, cols, box_rows, 64, false, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1);
}

// -------------------------------------------------------------- workspace layout --

namespace {

// NVTX range around an entry point (visible in profilers that record NVTX; a few ns otherwise).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

constexpr int kMaxPiece = 8192;

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

struct Layout {
    size_t status, sched, logits, ids, topw, offsets, tiles, chunks, perm, inv, row_tok, row_w, h, h_s, acc, y, total;
};

Layout layout(const moe_config &c, int T) {
    Layout L;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t r = o;
        o += align256(bytes);
        return r;
    };
    const size_t Tt = (size_t)(T > 0 ? T : 1);
    L.status = take(256);
    L.sched = take(256);  // the grouped GEMMs' tile counters
    // fp32 [T, E]; the decode chain's tagged logits take 8 bytes an expert
    L.logits = take(Tt * c.n_experts * 4 > (size_t)c.n_experts * 8 ? Tt * c.n_experts * 4 : (size_t)c.n_experts * 8);
    L.ids = take(Tt * c.top_k * 4);
    L.topw = take(Tt * c.top_k * 4);
    // E + 2 entries: the experts and, when it runs inside the routed GEMMs, the shared expert
    L.offsets = take((size_t)(c.n_experts + 2) * 4);
    L.tiles = take((size_t)(c.n_experts + 2) * 4);
    L.chunks = take(permute_scratch_ints((int)Tt, c.n_experts, c.top_k) * 4);
    L.perm = take(Tt * c.top_k * 4);
    L.inv = take(Tt * c.top_k * 4);
    L.row_tok = take(Tt * c.top_k * 4);
    L.row_w = take(Tt * c.top_k * 4);
    L.h = take(Tt * (c.top_k + 1) * c.inter * 2);  // + the shared expert's rows
    L.h_s = take(Tt * (size_t)c.shared_inter * 2);
    L.acc = take((Tt > 3 ? Tt : 3) * c.hidden * 4);  // >= 3 rows: the decode chain's accumulators
    L.y = take(Tt * (c.top_k + 1) * c.hidden * 2);
    L.total = o;
    return L;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_config(const moe_config *c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->hidden <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->inter <= 0 || c->shared_inter < 0)
        return MOE_ERR_INVALID_ARG;
    if (c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
    if (c->top_k > 32 || c->n_experts > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->hidden % 128 || c->inter % 128 || c->shared_inter % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->hidden > 16384 || c->inter > 8192 || c->shared_inter > 8192) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

moe_status check_weights(const moe_config *c, const moe_weights *w, bool router, bool experts) {
    if (!w) return MOE_ERR_INVALID_ARG;
    if (router && (!w->w_router || !aligned16(w->w_router))) return MOE_ERR_INVALID_ARG;
    if (experts) {
        if (!w->w_gate || !w->w_up || !w->w_down) return MOE_ERR_INVALID_ARG;
        if (!aligned16(w->w_gate) || !aligned16(w->w_up) || !aligned16(w->w_down)) return MOE_ERR_INVALID_ARG;
        if (c->shared_inter > 0) {
            if (!w->ws_gate || !w->ws_up || !w->ws_down) return MOE_ERR_INVALID_ARG;
            if (!aligned16(w->ws_gate) || !aligned16(w->ws_up) || !aligned16(w->ws_down))
                return MOE_ERR_INVALID_ARG;
        }
    }
    return MOE_OK;
}

moe_status check_weights_q8(const moe_config *c, const moe_weights_q8 *w) {
    if (!w) return MOE_ERR_INVALID_ARG;
    if (!w->w_router || !aligned16(w->w_router) || !w->q_gate || !w->q_up || !w->q_down || !w->s_gate ||
        !w->s_up || !w->s_down || !aligned16(w->q_gate) || !aligned16(w->q_up) || !aligned16(w->q_down))
        return MOE_ERR_INVALID_ARG;
    if (c->shared_inter > 0 &&
        (!w->qs_gate || !w->qs_up || !w->qs_down || !w->ss_gate || !w->ss_up || !w->ss_down ||
         !aligned16(w->qs_gate) || !aligned16(w->qs_up) || !aligned16(w->qs_down)))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status check_weights_q4(const moe_config *c, const moe_weights_q4 *w) {
    if (!w) return MOE_ERR_INVALID_ARG;
    if (!w->w_router || !aligned16(w->w_router) || !w->q_gate || !w->q_up || !w->q_down || !w->s_gate ||
        !w->s_up || !w->s_down || !aligned16(w->q_gate) || !aligned16(w->q_up) || !aligned16(w->q_down))
        return MOE_ERR_INVALID_ARG;
    if (c->shared_inter > 0 &&
        (!w->qs_gate || !w->qs_up || !w->qs_down || !w->ss_gate || !w->ss_up || !w->ss_down ||
         !aligned16(w->qs_gate) || !aligned16(w->qs_up) || !aligned16(w->qs_down)))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status check_ws(const moe_config *c, void *ws, size_t ws_bytes, int T) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < layout(*c, T).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return MOE_OK;
}

moe_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    return MOE_ERR_CUDA;
}

#define MOE_TRY(expr)                          \
    do {                                       \
        moe_status _st = (expr);               \
        if (_st != MOE_OK) return _st;         \
    } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

// Router logits on tensor cores: logits[T,E] = x Wr^T + b.  The router has few weight tiles
// (E/128), so its token tiles are capped lower than the experts' to occupy more SMs.
#ifndef MOE_ROUTER_TILE_N
#define MOE_ROUTER_TILE_N 128
#endif
constexpr int kRouterTileN = MOE_ROUTER_TILE_N;
// zero_ptr (or NULL): zero_n ints the GEMM's CTAs clear before their work (the count table the
// top-k kernel that follows adds into).
moe_status run_router_gemm(const moe_config &c, const moe_weights &w, const uint16_t *x, int T,
                           float *logits, int *status, cudaStream_t s, int32_t *zero_ptr = nullptr,
                           int zero_n = 0) {
    CUtensorMap tm;
    TokenMaps tb;
    if (!encode_tmap_2d_bf16(&tm, w.w_router, (uint64_t)c.n_experts, (uint64_t)c.hidden, kTileM, 64) ||
        !encode_token_maps(&tb, x, (uint64_t)T, (uint64_t)c.hidden))
        return MOE_ERR_CUDA;
    GemmArgs a{};
    a.b_src = x;
    a.K = c.hidden;
    a.n_groups = 1;
    a.M_single = T;
    a.tile_cap = kRouterTileN;
    a.F = c.n_experts;
    a.out = logits;
    a.ld = c.n_experts;
    a.bias = w.b_router;
    a.status = status;
    a.zero_ptr = zero_ptr;
    a.zero_n = zero_n;
    MOE_CUDA(launch_gemm(EPI_F32, a, tm, tm, tb, tm, tm, KC_ROUTER_GEMM, s));
    return MOE_OK;
}

// Shared expert over T tokens: h_s = SwiGLU(x), then Ws_down h_s stored (not added) into
// out (fp32 [T,H]).  Gate/up maps use 64-row boxes: a SwiGLU tile holds 64 features' gate
// rows and the same features' up rows.
// wq != NULL: the shared expert's E4M3 codes and row scales instead of w's bf16 matrices.
moe_status run_shared(const moe_config &c, const moe_weights &w, const uint16_t *x, int T,
                      uint16_t *h_s, float *out, int *status, cudaStream_t s, const moe_weights_q8 *wq = nullptr) {
    CUtensorMap tg, tu, td;
    TokenMaps tx, th;
    const bool q8 = wq != nullptr;
    if (q8 ? (!encode_tmap_2d_u8(&tg, wq->qs_gate, c.shared_inter, c.hidden, kTileM / 2) ||
              !encode_tmap_2d_u8(&tu, wq->qs_up, c.shared_inter, c.hidden, kTileM / 2) ||
              !encode_tmap_2d_u8(&td, wq->qs_down, c.hidden, c.shared_inter, kTileM))
           : (!encode_tmap_2d_bf16(&tg, w.ws_gate, c.shared_inter, c.hidden, kTileM / 2, 64) ||
              !encode_tmap_2d_bf16(&tu, w.ws_up, c.shared_inter, c.hidden, kTileM / 2, 64) ||
              !encode_tmap_2d_bf16(&td, w.ws_down, c.hidden, c.shared_inter, kTileM, 64)))
        return MOE_ERR_CUDA;
    if (!encode_token_maps(&tx, x, (uint64_t)T, c.hidden) ||
        !encode_token_maps(&th, h_s, (uint64_t)T, c.shared_inter))
        return MOE_ERR_CUDA;
    GemmArgs a{};
    a.b_src = x;
    a.K = c.hidden;
    a.n_groups = 1;
    a.M_single = T;
    a.F = c.shared_inter;
    a.out = h_s;
    a.ld = c.shared_inter;
    a.status = status;
    if (q8) {
        a.q8 = true;
        a.w_scale0 = wq->ss_gate;
        a.w_scale1 = wq->ss_up;
    }
    MOE_CUDA(launch_gemm(EPI_SWIGLU, a, tg, tu, tx, tg, tu, KC_SHARED_GATEUP, s));
    GemmArgs d{};
    d.b_src = h_s;
    d.K = c.shared_inter;
    d.n_groups = 1;
    d.M_single = T;
    d.F = c.hidden;
    d.out = out;
    d.ld = c.hidden;
    d.status = status;
    if (q8) {
        d.q8 = true;
        d.w_scale0 = wq->ss_down;
    }
    MOE_CUDA(launch_gemm(EPI_F32, d, td, td, th, td, td, KC_SHARED_DOWN, s));
    return MOE_OK;
}

// Tiles at the end of a grouped GEMM that CTA pairs claim dynamically, in waves of one tile
// per pair (the rest run round-robin).
#ifndef MOE_DYN_TAIL_WAVES
#define MOE_DYN_TAIL_WAVES 1
#endif
int dyn_tail_tiles() { return MOE_DYN_TAIL_WAVES * (device_info().sm_count / 2); }

// Routed experts, grouped: h rows (expert-sorted order) from the expert-sorted copy of x
// (xp), then the down projection either stored per row in fp32 (y_rows, unfused) or weighted
// and stored as bf16 rows in pair order (y_pairs[perm[r]] = bf16(row_w[r] * y)) for the
// combine.  with_shared: the shared expert (I_s == I) runs as one more group of the T tokens
// in order, read straight from x, into rows P .. P+T-1 of h and y_pairs (weight 1);
// offsets/tiles then hold E + 2 entries.
moe_status run_routed(const moe_config &c, const moe_weights &w, const uint16_t *x, int T,
                      const int32_t *offsets, const int32_t *tiles, const int32_t *row_tok,
                      const int32_t *perm, const float *row_w, uint16_t *xp, uint16_t *h, float *y_rows,
                      uint16_t *y_pairs, int *status, int *sched, cudaStream_t s, bool with_shared = false,
                      const moe_weights_q8 *wq = nullptr) {
    const uint64_t EI = (uint64_t)c.n_experts * c.inter;
    const uint64_t P = (uint64_t)T * c.top_k;
    const uint64_t rows = P + (with_shared ? (uint64_t)T : 0);
    CUtensorMap tg, tu, td, tsg, tsu, tsd;
    TokenMaps tx, th;
    const bool q8 = wq != nullptr;
    const uint64_t EH = (uint64_t)c.n_experts * c.hidden;
    if (q8 ? (!encode_tmap_2d_u8(&tg, wq->q_gate, EI, c.hidden, kTileM / 2) ||
              !encode_tmap_2d_u8(&tu, wq->q_up, EI, c.hidden, kTileM / 2) ||
              !encode_tmap_2d_u8(&td, wq->q_down, EH, c.inter, kTileM))
           : (!encode_tmap_2d_bf16(&tg, w.w_gate, EI, c.hidden, kTileM / 2, 64) ||
              !encode_tmap_2d_bf16(&tu, w.w_up, EI, c.hidden, kTileM / 2, 64) ||
              !encode_tmap_2d_bf16(&td, w.w_down, EH, c.inter, kTileM, 64)))
        return MOE_ERR_CUDA;
    if (!encode_token_maps(&tx, xp, P, c.hidden) || !encode_token_maps(&th, h, rows, c.inter))
        return MOE_ERR_CUDA;
    // the shared expert's token rows are x itself, in order
    if (with_shared && !encode_tmap_2d_bf16(&tx.shared, x, (uint64_t)T, c.hidden, kTokenBoxRows, 64))
        return MOE_ERR_CUDA;
    if (with_shared) {
        if (q8 ? (!encode_tmap_2d_u8(&tsg, wq->qs_gate, c.shared_inter, c.hidden, kTileM / 2) ||
                  !encode_tmap_2d_u8(&tsu, wq->qs_up, c.shared_inter, c.hidden, kTileM / 2) ||
                  !encode_tmap_2d_u8(&tsd, wq->qs_down, c.hidden, c.shared_inter, kTileM))
               : (!encode_tmap_2d_bf16(&tsg, w.ws_gate, c.shared_inter, c.hidden, kTileM / 2, 64) ||
                  !encode_tmap_2d_bf16(&tsu, w.ws_up, c.shared_inter, c.hidden, kTileM / 2, 64) ||
                  !encode_tmap_2d_bf16(&tsd, w.ws_down, c.hidden, c.shared_inter, kTileM, 64)))
            return MOE_ERR_CUDA;
    } else {
        tsg = tg;
        tsu = tu;
        tsd = td;
    }
    // the token rows in expert-sorted order, so that both GEMM operands load as TMA tiles
    MOE_CUDA(launch_gather_rows(x, T, c.hidden, row_tok, (int)P, xp, s, 0));
    GemmArgs a{};
    a.b_src = xp;
    a.K = c.hidden;
    a.n_groups = c.n_experts + (with_shared ? 1 : 0);
    a.group_rows = offsets;
    a.group_tiles = tiles;
    a.F = c.inter;
    a.out = h;
    a.ld = c.inter;
    a.out_rows = (int)rows;
    a.status = status;
    a.shared_last = with_shared;
    a.shared_b_own = with_shared;
    a.tile_counter = sched;
    a.dyn_tail = dyn_tail_tiles();
    if (q8) {
        a.q8 = true;
        a.w_scale0 = wq->s_gate;
        a.w_scale1 = wq->s_up;
        a.ws_scale0 = wq->ss_gate;
        a.ws_scale1 = wq->ss_up;
    }
    MOE_CUDA(launch_gemm(EPI_SWIGLU, a, tg, tu, tx, tsg, tsu, KC_GATEUP_GEMM, s));
    GemmArgs d{};
    d.b_src = h;
    d.K = c.inter;
    d.n_groups = a.n_groups;
    d.group_rows = offsets;
    d.group_tiles = tiles;
    d.F = c.hidden;
    d.ld = c.hidden;
    d.status = status;
    d.shared_last = with_shared;
    d.tile_counter = sched ? sched + 1 : nullptr;
    d.dyn_tail = dyn_tail_tiles();
    if (q8) {
        d.q8 = true;
        d.w_scale0 = wq->s_down;
        d.ws_scale0 = wq->ss_down;
    }
    d.src_rows = (int)rows;
    d.out_rows = (int)rows;  // y_rows [P, H] or the weighted rows [P + T, H]
    if (y_rows) {
        if (with_shared) return MOE_ERR_INVALID_ARG;
        d.out = y_rows;
        MOE_CUDA(launch_gemm(EPI_F32, d, td, td, th, td, td, KC_DOWN_GEMM, s));
    } else {
        d.out = y_pairs;
        d.epi_tok = perm;
        d.epi_w = row_w;
        MOE_CUDA(launch_gemm(EPI_COMBINE, d, td, td, th, tsd, tsd, KC_DOWN_GEMM, s));
    }
    return MOE_OK;
}

// One prefill piece of T tokens (T >= 2), the whole layer.
moe_status forward_piece(const moe_config &c, const moe_weights &w, const uint16_t *x, int T,
                         uint16_t *out, const uint16_t *resid, uint16_t *x_next, void *ws,
                         cudaStream_t s, const moe_weights_q8 *wq = nullptr) {
    const Layout L = layout(c, T);
    int *status = at<int>(ws, L.status);
    float *logits = at<float>(ws, L.logits);
    int32_t *ids = at<int32_t>(ws, L.ids);
    float *topw = at<float>(ws, L.topw);
    int32_t *offsets = at<int32_t>(ws, L.offsets);
    int32_t *tiles = at<int32_t>(ws, L.tiles);
    int32_t *perm = at<int32_t>(ws, L.perm);
    int32_t *inv = at<int32_t>(ws, L.inv);
    uint16_t *h = at<uint16_t>(ws, L.h);
    uint16_t *h_s = at<uint16_t>(ws, L.h_s);
    float *acc = at<float>(ws, L.acc);
    // routing in three launches: the router GEMM (which also zeroes the chunk count table), the
    // top-k (which adds each chunk's expert counts into it), and the permutation's scan + scatter
    int32_t *chunks = at<int32_t>(ws, L.chunks);
    MOE_TRY(run_router_gemm(c, w, x, T, logits, status, s, chunks,
                            (int)permute_scratch_ints(T, c.n_experts, c.top_k)));
    MOE_CUDA(launch_topk_hist(logits, T, c.n_experts, c.top_k, ids, topw, chunks, s));
    int32_t *row_tok = at<int32_t>(ws, L.row_tok);
    float *row_w = at<float>(ws, L.row_w);
    // a shared expert as wide as the routed ones runs inside the routed GEMMs, as group E
    const bool merged = c.shared_inter > 0 && c.shared_inter == c.inter;
    int *sched = at<int>(ws, L.sched);
    MOE_CUDA(launch_scan_scatter(ids, T, c.n_experts, c.top_k, offsets, perm, inv, tiles, chunks, topw, row_tok,
                                 row_w, status, s, merged ? T : 0, sched));
    uint16_t *y = at<uint16_t>(ws, L.y);
    if (c.shared_inter > 0 && !merged) MOE_TRY(run_shared(c, w, x, T, h_s, acc, status, s, wq));
    // y doubles as the expert-sorted copy of x: the gate/up GEMM is done reading it before the
    // down GEMM writes y (same stream)
    MOE_TRY(run_routed(c, w, x, T, offsets, tiles, row_tok, perm, row_w, y, h, nullptr, y, status, sched, s, merged,
                       wq));
    const size_t P = (size_t)T * c.top_k;
    MOE_CUDA(launch_finalize(y, c.top_k, (c.shared_inter > 0 && !merged) ? acc : nullptr, resid, T, c.hidden, out,
                             x_next, s, merged ? y + P * c.hidden : nullptr));
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_NOT_IMPLEMENTED: return "not implemented";
    }
    return "unknown status";
}

size_t moe_workspace_size(const moe_config *cfg, int max_T) {
    if (check_config(cfg) != MOE_OK || max_T < 0) return 0;
    return layout(*cfg, max_T).total;
}

moe_status moe_route(const moe_config *cfg, const moe_weights *w, const moe_bf16 *x, int T,
                     float *logits_out, int32_t *topk_ids, float *topk_w, void *ws,
                     size_t ws_bytes, void *stream) {
    NvtxRange nvtx_range("moe_route");
    MOE_TRY(check_config(cfg));
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights(cfg, w, true, false));
    if (!x || !topk_ids || !topk_w || !aligned16(x)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ws(cfg, ws, ws_bytes, T));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Layout L = layout(*cfg, T);
    float *logits = logits_out ? logits_out : at<float>(ws, L.logits);
    if (decode_fits(T, cfg->hidden)) {
        // a few tokens: the decode path's GEMV, so the reported logits are the ones moe_forward
        // selects on for such T
        DecodeArgs a{};
        a.T = T;
        a.H = cfg->hidden;
        a.E = cfg->n_experts;
        a.x = x;
        a.w_router = w->w_router;
        a.b_router = w->b_router;
        a.logits = logits;
        MOE_CUDA(launch_decode_router(a, s));
    } else {
        MOE_TRY(run_router_gemm(*cfg, *w, x, T, logits, at<int>(ws, L.status), s));
    }
    MOE_CUDA(launch_topk(logits, T, cfg->n_experts, cfg->top_k, topk_ids, topk_w, s));
    return MOE_OK;
}

moe_status moe_route_from_logits(const moe_config *cfg, const float *logits, int T,
                                 int32_t *topk_ids, float *topk_w, void *stream) {
    NvtxRange nvtx_range("moe_route_from_logits");
    MOE_TRY(check_config(cfg));
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_topk(logits, T, cfg->n_experts, cfg->top_k, topk_ids, topk_w,
                         static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status moe_permute(const moe_config *cfg, const int32_t *topk_ids, int T,
                       int32_t *expert_offsets, int32_t *perm, int32_t *inv, void *ws,
                       size_t ws_bytes, void *stream) {
    NvtxRange nvtx_range("moe_permute");
    MOE_TRY(check_config(cfg));
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!topk_ids || !expert_offsets || !perm || !inv) return MOE_ERR_INVALID_ARG;
    if ((long long)T * cfg->top_k > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED_SHAPE;
    MOE_TRY(check_ws(cfg, ws, ws_bytes, T));
    const Layout L = layout(*cfg, T);
    MOE_CUDA(launch_permute(topk_ids, T, cfg->n_experts, cfg->top_k, expert_offsets, perm, inv,
                            at<int32_t>(ws, L.tiles), kTileN, at<int32_t>(ws, L.chunks), nullptr,
                            at<int32_t>(ws, L.row_tok), nullptr, at<int>(ws, L.status),
                            static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status moe_expert_ffn(const moe_config *cfg, const moe_weights *w, const moe_bf16 *x, int T,
                          const int32_t *expert_offsets, const int32_t *perm, moe_bf16 *h_rows,
                          float *y_rows, float *shared_y, void *ws, size_t ws_bytes,
                          void *stream) {
    NvtxRange nvtx_range("moe_expert_ffn");
    MOE_TRY(check_config(cfg));
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights(cfg, w, false, true));
    if (!x || !expert_offsets || !perm || !h_rows || !y_rows) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(h_rows) || !aligned16(y_rows)) return MOE_ERR_INVALID_ARG;
    if (shared_y && !aligned16(shared_y)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ws(cfg, ws, ws_bytes, T));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Layout L = layout(*cfg, T);
    int *status = at<int>(ws, L.status);
    int32_t *tiles = at<int32_t>(ws, L.tiles);
    int32_t *row_tok = at<int32_t>(ws, L.row_tok);
    int *sched = at<int>(ws, L.sched);
    MOE_CUDA(launch_tile_prefix(expert_offsets, cfg->n_experts, tiles, kTileN, perm, T * cfg->top_k,
                                cfg->top_k, row_tok, s, sched, status));
    MOE_TRY(run_routed(*cfg, *w, x, T, expert_offsets, tiles, row_tok, perm, nullptr, at<uint16_t>(ws, L.y), h_rows,
                       y_rows, nullptr, status, sched, s));
    if (shared_y && cfg->shared_inter > 0)
        MOE_TRY(run_shared(*cfg, *w, x, T, at<uint16_t>(ws, L.h_s), shared_y, status, s));
    return MOE_OK;
}

moe_status moe_combine(const moe_config *cfg, const float *y_rows, const int32_t *inv,
                       const float *topk_w, const float *shared_y, int T, moe_bf16 *out,
                       void *stream) {
    NvtxRange nvtx_range("moe_combine");
    MOE_TRY(check_config(cfg));
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y_rows || !inv || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_rows) || !aligned16(out) || (shared_y && !aligned16(shared_y))) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_combine(y_rows, inv, topk_w, shared_y, T, cfg->hidden, cfg->top_k, out,
                            static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

int moe_plan_pieces(int T, int *pieces, int max_pieces) {
    if (T < 0) return -1;
    static const int kBuckets[4] = {8192, 4096, 2048, 1024};
    int n = 0, rem = T;
    for (int b = 0; b < 4; ++b) {
        while (rem >= kBuckets[b]) {
            if (pieces && n < max_pieces) pieces[n] = kBuckets[b];
            ++n;
            rem -= kBuckets[b];
        }
    }
    if (rem > 0) {
        if (pieces && n < max_pieces) pieces[n] = rem;
        ++n;
    }
    return n;
}

moe_status moe_forward(const moe_config *cfg, const moe_weights *w, const moe_bf16 *x, int T,
                       moe_bf16 *out, const moe_bf16 *resid, moe_bf16 *x_next, void *ws,
                       size_t ws_bytes, void *stream) {
    NvtxRange nvtx_range("moe_forward");
    MOE_TRY(check_config(cfg));
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights(cfg, w, true, true));
    if (!x || !out || !aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if (x_next && !aligned16(x_next)) return MOE_ERR_INVALID_ARG;
    if (resid && !aligned16(resid)) return MOE_ERR_INVALID_ARG;
    if (!resid) resid = x;
    const int Tmax = T < kMaxPiece ? T : kMaxPiece;
    MOE_TRY(check_ws(cfg, ws, ws_bytes, Tmax));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int H = cfg->hidden;
    if (decode_fits(T, H)) {
        // up to kMaxDecodeT tokens: router GEMV, then each selected expert's weights streamed once
        // for all tokens that chose it
        const Layout L = layout(*cfg, T);
        DecodeArgs a{};
        a.T = T;
        a.H = H;
        a.E = cfg->n_experts;
        a.k = cfg->top_k;
        a.I = cfg->inter;
        a.Is = cfg->shared_inter;
        a.x = x;
        a.w_router = w->w_router;
        a.b_router = w->b_router;
        a.w_gate = w->w_gate;
        a.w_up = w->w_up;
        a.w_down = w->w_down;
        a.ws_gate = w->ws_gate;
        a.ws_up = w->ws_up;
        a.ws_down = w->ws_down;
        a.logits = at<float>(ws, L.logits);
        a.ids = at<int32_t>(ws, L.ids);
        a.topw = at<float>(ws, L.topw);
        a.h = at<uint16_t>(ws, L.h);
        a.h_s = at<uint16_t>(ws, L.h_s);
        a.out = out;
        a.resid = resid;
        a.x_next = x_next;
        a.acc = at<float>(ws, L.acc);
        a.counter = at<int>(ws, L.status) + 1;  // in the status area: zero between calls
        a.status = at<int>(ws, L.status);
        CUtensorMap td, tsd;
        const uint32_t sl = (uint32_t)decode_slice(), br = (uint32_t)decode_box_rows();
        if (!encode_tmap_2d_bf16(&td, w->w_down, (uint64_t)cfg->n_experts * H, cfg->inter, br, sl, false))
            return MOE_ERR_CUDA;
        if (cfg->shared_inter > 0) {
            if (!encode_tmap_2d_bf16(&tsd, w->ws_down, H, cfg->shared_inter, br, sl, false)) return MOE_ERR_CUDA;
        } else {
            tsd = td;
        }
        MOE_CUDA(launch_decode(a, td, tsd, s));
        return MOE_OK;
    }
    // the pieces in moe_plan_pieces order: the largest bucket that fits, then the exact tail
    static const int kBuckets[4] = {8192, 4096, 2048, 1024};
    size_t t0 = 0;
    for (int rem = T; rem > 0;) {
        int Tp = rem;
        for (int b = 0; b < 4; ++b)
            if (rem >= kBuckets[b]) {
                Tp = kBuckets[b];
                break;
            }
        rem -= Tp;
        uint16_t *xn = x_next ? x_next + t0 * H : nullptr;
        if (decode_fits(Tp, H)) {
            // a tail of a few tokens takes the decode path of the same layer
            MOE_TRY(moe_forward(cfg, w, x + t0 * H, Tp, out + t0 * H, resid + t0 * H, xn, ws, ws_bytes,
                                stream));
        } else {
            MOE_TRY(forward_piece(*cfg, *w, x + t0 * H, Tp, out + t0 * H, resid + t0 * H, xn, ws, s));
        }
        t0 += Tp;
    }
    return MOE_OK;
}

moe_status moe_forward_q8(const moe_config *cfg, const moe_weights_q8 *w, const moe_bf16 *x, int T,
                          moe_bf16 *out, const moe_bf16 *resid, moe_bf16 *x_next, void *ws, size_t ws_bytes,
                          void *stream) {
    NvtxRange nvtx_range("moe_forward_q8");
    MOE_TRY(check_config(cfg));
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights_q8(cfg, w));
    if (!x || !out || !aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if ((x_next && !aligned16(x_next)) || (resid && !aligned16(resid))) return MOE_ERR_INVALID_ARG;
    if (!resid) resid = x;
    const int Tmax = T < kMaxPiece ? T : kMaxPiece;
    MOE_TRY(check_ws(cfg, ws, ws_bytes, Tmax));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int H = cfg->hidden;
    // the bf16 router (the selection stays on bf16 weights)
    moe_weights wr{};
    wr.w_router = w->w_router;
    wr.b_router = w->b_router;
    static const int kBuckets[4] = {8192, 4096, 2048, 1024};
    size_t t0 = 0;
    for (int rem = T; rem > 0;) {
        int Tp = rem;
        for (int b = 0; b < 4; ++b)
            if (rem >= kBuckets[b]) {
                Tp = kBuckets[b];
                break;
            }
        rem -= Tp;
        MOE_TRY(forward_piece(*cfg, wr, x + t0 * H, Tp, out + t0 * H, resid + t0 * H,
                              x_next ? x_next + t0 * H : nullptr, ws, s, w));
        t0 += Tp;
    }
    return MOE_OK;
}

namespace {
// The part of a chain launch both weight formats share: shape, token and workspace pointers.
moe_status chain_common(const moe_config *cfg, int n_layers, const moe_bf16 *x0, const moe_bf16 *resid,
                        moe_bf16 *out, moe_bf16 *x_last, void *ws, size_t ws_bytes, ChainParams &p) {
    MOE_TRY(check_config(cfg));
    if (n_layers < 1) return MOE_ERR_INVALID_ARG;
    if (n_layers > kChainMaxLayers) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!decode_fits(1, cfg->hidden)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!x0 || !out || !aligned16(x0) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if ((resid && !aligned16(resid)) || (x_last && !aligned16(x_last))) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ws(cfg, ws, ws_bytes, 1));
    const Layout L = layout(*cfg, 1);
    p.H = cfg->hidden;
    p.E = cfg->n_experts;
    p.k = cfg->top_k;
    p.I = cfg->inter;
    p.Is = cfg->shared_inter;
    p.L = n_layers;
    p.x0 = x0;
    p.resid = resid;
    p.out = out;
    p.x_last = x_last;
    p.logits = at<unsigned long long>(ws, L.logits);
    p.acc0 = at<float>(ws, L.acc);
    p.acc1 = p.acc0 + cfg->hidden;
    p.acc2 = p.acc1 + cfg->hidden;
    int *st = at<int>(ws, L.status);
    p.status = st;
    // st[1] is the one-layer path's ticket counter; the chain's barrier count and abort flag follow
    p.bar = reinterpret_cast<unsigned *>(st + 2);
    p.abort = st + 3;
    return MOE_OK;
}
}  // namespace

moe_status moe_decode_chain(const moe_config *cfg, const moe_weights *layers, int n_layers, const moe_bf16 *x0,
                            const moe_bf16 *resid, moe_bf16 *out, moe_bf16 *x_last, void *ws, size_t ws_bytes,
                            void *stream) {
    NvtxRange nvtx_range("moe_decode_chain");
    if (!layers) return MOE_ERR_INVALID_ARG;
    // about 20 KB: the per-layer pointers and down-projection tensor maps travel as the kernel's
    // parameter block
    static thread_local ChainParams p;
    MOE_TRY(chain_common(cfg, n_layers, x0, resid, out, x_last, ws, ws_bytes, p));
    for (int l = 0; l < n_layers; ++l) MOE_TRY(check_weights(cfg, &layers[l], true, true));
    const int H = cfg->hidden;
    const uint32_t sl = (uint32_t)decode_slice(), br = (uint32_t)decode_box_rows();
    for (int l = 0; l < n_layers; ++l) {
        const moe_weights &w = layers[l];
        p.lay[l] = ChainLayer{w.w_router, w.b_router, w.w_gate, w.w_up, w.ws_gate, w.ws_up};
        if (!encode_tmap_2d_bf16(&p.tm_down[l], w.w_down, (uint64_t)cfg->n_experts * H, cfg->inter, br, sl, false))
            return MOE_ERR_CUDA;
        if (cfg->shared_inter > 0) {
            if (!encode_tmap_2d_bf16(&p.tm_sdown[l], w.ws_down, H, cfg->shared_inter, br, sl, false))
                return MOE_ERR_CUDA;
        } else {
            p.tm_sdown[l] = p.tm_down[l];
        }
    }
    MOE_CUDA(launch_decode_chain(p, kChainBf16, static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status moe_decode_chain_q8(const moe_config *cfg, const moe_weights_q8 *layers, int n_layers,
                               const moe_bf16 *x0, const moe_bf16 *resid, moe_bf16 *out, moe_bf16 *x_last,
                               void *ws, size_t ws_bytes, void *stream) {
    NvtxRange nvtx_range("moe_decode_chain_q8");
    if (!layers) return MOE_ERR_INVALID_ARG;
    static thread_local ChainParams p;
    MOE_TRY(chain_common(cfg, n_layers, x0, resid, out, x_last, ws, ws_bytes, p));
    const bool shared = cfg->shared_inter > 0;
    for (int l = 0; l < n_layers; ++l) MOE_TRY(check_weights_q8(cfg, &layers[l]));
    const int H = cfg->hidden;
    const uint32_t sl = (uint32_t)decode_slice(), br = (uint32_t)decode_box_rows();
    for (int l = 0; l < n_layers; ++l) {
        const moe_weights_q8 &w = layers[l];
        p.lay[l] = ChainLayer{w.w_router, w.b_router, w.q_gate, w.q_up, w.qs_gate, w.qs_up,
                              w.s_gate, w.s_up, w.s_down, w.ss_gate, w.ss_up, w.ss_down};
        if (!encode_tmap_2d(&p.tm_down[l], w.q_down, (uint64_t)cfg->n_experts * H, cfg->inter, br, sl, false,
                            CU_TENSOR_MAP_DATA_TYPE_UINT8, 1))
            return MOE_ERR_CUDA;
        if (shared) {
            if (!encode_tmap_2d(&p.tm_sdown[l], w.qs_down, H, cfg->shared_inter, br, sl, false,
                                CU_TENSOR_MAP_DATA_TYPE_UINT8, 1))
                return MOE_ERR_CUDA;
        } else {
            p.tm_sdown[l] = p.tm_down[l];
        }
    }
    MOE_CUDA(launch_decode_chain(p, kChainE4m3, static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status moe_decode_chain_q4(const moe_config *cfg, const moe_weights_q4 *layers, int n_layers,
                               const moe_bf16 *x0, const moe_bf16 *resid, moe_bf16 *out, moe_bf16 *x_last,
                               void *ws, size_t ws_bytes, void *stream) {
    NvtxRange nvtx_range("moe_decode_chain_q4");
    if (!layers) return MOE_ERR_INVALID_ARG;
    static thread_local ChainParams p;
    MOE_TRY(chain_common(cfg, n_layers, x0, resid, out, x_last, ws, ws_bytes, p));
    const bool shared = cfg->shared_inter > 0;
    for (int l = 0; l < n_layers; ++l) MOE_TRY(check_weights_q4(cfg, &layers[l]));
    const int H = cfg->hidden;
    const uint32_t sl = (uint32_t)decode_slice(), br = (uint32_t)decode_box_rows();
    for (int l = 0; l < n_layers; ++l) {
        const moe_weights_q4 &w = layers[l];
        p.lay[l] = ChainLayer{w.w_router, w.b_router, w.q_gate, w.q_up, w.qs_gate, w.qs_up,
                              w.s_gate, w.s_up, w.s_down, w.ss_gate, w.ss_up, w.ss_down};
        // W_d as byte rows of I/2 codes; a box is a slice's 16 bytes of kBoxRows rows
        if (!encode_tmap_2d(&p.tm_down[l], w.q_down, (uint64_t)cfg->n_experts * H, cfg->inter / 2, br, sl / 2, false,
                            CU_TENSOR_MAP_DATA_TYPE_UINT8, 1))
            return MOE_ERR_CUDA;
        if (shared) {
            if (!encode_tmap_2d(&p.tm_sdown[l], w.qs_down, H, cfg->shared_inter / 2, br, sl / 2, false,
                                CU_TENSOR_MAP_DATA_TYPE_UINT8, 1))
                return MOE_ERR_CUDA;
        } else {
            p.tm_sdown[l] = p.tm_down[l];
        }
    }
    MOE_CUDA(launch_decode_chain(p, kChainQ4, static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status moe_quantize_q4(const moe_bf16 *w, int rows, int cols, uint8_t *q, float *scale, void *stream) {
    NvtxRange nvtx_range("moe_quantize_q4");
    if (rows < 0 || cols < 0 || cols % 32 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MOE_OK;
    if (!w || !q || !scale) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_quantize_q4(w, rows, cols, q, scale, static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status moe_quantize_e4m3(const moe_bf16 *w, int rows, int cols, uint8_t *q, float *scale, void *stream) {
    NvtxRange nvtx_range("moe_quantize_e4m3");
    if (rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MOE_OK;
    if (!w || !q || !scale) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(launch_quantize_e4m3(w, rows, cols, q, scale, static_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status moe_check_status(void *ws, size_t ws_bytes, int *device_status, void *stream) {
    if (!ws || !device_status || ws_bytes < 256) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    *device_status = v;
    if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

struct moe_graph_s {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int kernels = 0;
};

namespace {
// The stack of moe_graph_create: layer l reads x_l and writes x_{l+1} into x_last or scratch,
// alternating so that the last layer writes x_last.
moe_status run_stack(const moe_config *cfg, const moe_weights *layers, int n, int T, const moe_bf16 *x0,
                     const moe_bf16 *resid, moe_bf16 *out, moe_bf16 *x_last, moe_bf16 *scratch, void *ws,
                     size_t ws_bytes, void *stream) {
    const moe_bf16 *x = x0;
    for (int l = 0; l < n; ++l) {
        moe_bf16 *nxt = ((n - 1 - l) & 1) ? scratch : x_last;
        MOE_TRY(moe_forward(cfg, &layers[l], x, T, out, resid, nxt, ws, ws_bytes, stream));
        x = nxt;
    }
    return MOE_OK;
}
}  // namespace

moe_status moe_graph_create(const moe_config *cfg, const moe_weights *layers, int n_layers, int T,
                            const moe_bf16 *x0, const moe_bf16 *resid, moe_bf16 *out, moe_bf16 *x_last,
                            moe_bf16 *scratch, void *ws, size_t ws_bytes, void *stream, moe_graph *graph) {
    NvtxRange nvtx_range("moe_graph_create");
    if (!graph) return MOE_ERR_INVALID_ARG;
    *graph = nullptr;
    if (!layers || n_layers < 1 || T < 1) return MOE_ERR_INVALID_ARG;
    if (n_layers > kChainMaxLayers) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (n_layers > 1) {
        if (!x_last || !scratch || x_last == scratch) return MOE_ERR_INVALID_ARG;
        for (const moe_bf16 *b : {(const moe_bf16 *)x_last, (const moe_bf16 *)scratch})
            if (b == x0 || b == resid || b == out) return MOE_ERR_INVALID_ARG;
    }
    // one eager run: validates every argument and fills the per-device launch caches (function
    // attributes, occupancy), which must not be queried inside the capture
    MOE_TRY(run_stack(cfg, layers, n_layers, T, x0, resid, out, x_last, scratch, ws, ws_bytes, stream));
    // captured on a private stream: nothing runs until a launch, which the caller orders on
    // its own stream
    cudaStream_t cs = nullptr;
    MOE_CUDA(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
    moe_graph g = new moe_graph_s();
    moe_status st = MOE_OK;
    cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
        t_capturing = true;
        st = run_stack(cfg, layers, n_layers, T, x0, resid, out, x_last, scratch, ws, ws_bytes, cs);
        t_capturing = false;
        const cudaError_t e2 = cudaStreamEndCapture(cs, &g->graph);
        if (st == MOE_OK && e2 != cudaSuccess) st = MOE_ERR_CUDA;
    } else {
        st = MOE_ERR_CUDA;
    }
    if (st == MOE_OK && cudaGraphInstantiate(&g->exec, g->graph, 0) != cudaSuccess) st = MOE_ERR_CUDA;
    if (st == MOE_OK) {
        size_t n = 0;
        if (cudaGraphGetNodes(g->graph, nullptr, &n) != cudaSuccess) st = MOE_ERR_CUDA;
        std::vector<cudaGraphNode_t> nodes(n);
        if (st == MOE_OK && n > 0 && cudaGraphGetNodes(g->graph, nodes.data(), &n) != cudaSuccess) st = MOE_ERR_CUDA;
        for (size_t i = 0; st == MOE_OK && i < n; ++i) {
            cudaGraphNodeType ty;
            if (cudaGraphNodeGetType(nodes[i], &ty) == cudaSuccess && ty == cudaGraphNodeTypeKernel) ++g->kernels;
        }
    }
    cudaStreamDestroy(cs);
    if (st != MOE_OK) {
        moe_graph_destroy(g);
        return st;
    }
    *graph = g;
    return MOE_OK;
}

moe_status moe_graph_launch(moe_graph graph, void *stream) {
    if (!graph || !graph->exec) return MOE_ERR_INVALID_ARG;
    MOE_CUDA(cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)));
    g_launches.fetch_add((uint64_t)graph->kernels, std::memory_order_relaxed);
    return MOE_OK;
}

int moe_graph_kernel_count(moe_graph graph) { return graph ? graph->kernels : -1; }

moe_status moe_graph_destroy(moe_graph graph) {
    if (!graph) return MOE_OK;
    if (graph->exec) cudaGraphExecDestroy(graph->exec);
    if (graph->graph) cudaGraphDestroy(graph->graph);
    delete graph;
    return MOE_OK;
}

uint64_t moe_launch_count(void) { return g_launches.load(); }

moe_status moe_timing_enable(int enable) {
    g_timing.store(enable != 0);
    return MOE_OK;
}

moe_status moe_timing_read(const char *name, int *launches, double *total_ms) {
    if (!name || !launches || !total_ms) return MOE_ERR_INVALID_ARG;
    int kc = -1;
    for (int i = 0; i < KC_COUNT; ++i)
        if (std::strcmp(name, kClassNames[i]) == 0) kc = i;
    if (kc < 0) return MOE_ERR_INVALID_ARG;
    std::vector<TimedPair> v;
    {
        std::lock_guard<std::mutex> lk(g_timing_mu);
        v.swap(g_timed[kc]);
    }
    double tot = 0.0;
    int n = 0;
    moe_status st = MOE_OK;
    for (auto &p : v) {
        float ms = 0.f;
        if (cudaEventSynchronize(p.b) == cudaSuccess && cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
            tot += ms;
            ++n;
        } else {
            st = MOE_ERR_CUDA;
        }
        cudaEventDestroy(p.a);
        cudaEventDestroy(p.b);
    }
    *launches = n;
    *total_ms = tot;
    return st;
}

const char *moe_timing_name(int i) { return kernel_class_name(i); }

int moe_timing_classes(void) { return KC_COUNT; }

int moe_debug_build(void) { return debug_build() ? 1 : 0; }

}  // extern "C"
