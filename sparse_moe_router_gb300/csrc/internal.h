// internal.h -- declarations shared by the translation units of libmoe.so (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

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
    KC_DECODE_ROUTER,     // decode: router GEMV + shared gate/up GEMV
    KC_DECODE_GATEUP,     // decode: top-k + routed gate/up GEMV
    KC_DECODE_DOWN,       // decode: down GEMVs + combine + residual
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
// over [rows, cols] (cols contiguous) with a box_rows x box_cols box, 128-byte swizzle.
bool encode_tmap_2d_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows, uint32_t box_cols);

// ---- GEMM (tcgen05, swap-AB: weight rows on M, tokens on N) ---------------------------

enum GemmEpi { EPI_F32 = 0, EPI_SWIGLU = 1, EPI_COMBINE = 2 };

struct GemmArgs {
    // token side (B operand): row r of the group row space reads source row
    // gather_perm ? gather_perm[r] / gather_k : r of b_src ([*, K] bf16)
    const void *b_src;
    const int32_t *gather_perm;
    int gather_k;
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
    const int32_t *epi_perm;
    const float *epi_w;
    int epi_k;
    int *status;
};

// Launches the persistent grouped GEMM.  tm_a0 (and tm_a1 for EPI_SWIGLU: the up
// projection) are 2-D tensor maps over the weight rows with a 128 x 64 box.
cudaError_t launch_gemm(GemmEpi epi, const GemmArgs &a, const CUtensorMap &tm_a0,
                        const CUtensorMap &tm_a1, int kc, cudaStream_t s);

// ---- routing / permutation / elementwise ---------------------------------------------

cudaError_t launch_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                        cudaStream_t s);
cudaError_t launch_permute(const int32_t *ids, int T, int E, int k, int32_t *offsets,
                           int32_t *perm, int32_t *inv, int32_t *tile_prefix, int tile_n,
                           int *status, cudaStream_t s);
cudaError_t launch_tile_prefix(const int32_t *offsets, int E, int32_t *tile_prefix, int tile_n,
                               cudaStream_t s);
cudaError_t launch_finalize(const float *acc, const uint16_t *x, int T, int H, uint16_t *out,
                            uint16_t *x_next, cudaStream_t s);
cudaError_t launch_combine(const float *y_rows, const int32_t *inv, const float *topk_w,
                           const float *shared_y, int T, int H, int k, uint16_t *out,
                           cudaStream_t s);
cudaError_t launch_zero(float *p, size_t n, cudaStream_t s);

// ---- decode (T = 1) ------------------------------------------------------------------

struct DecodeArgs {
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
    uint16_t *x_next;  // [H] or NULL
};
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);
// Router logits of one token with the decode GEMV (the logits the decode path selects on).
cudaError_t launch_decode_router(const DecodeArgs &a, cudaStream_t s);

constexpr int kTileN = 128;   // tokens per GEMM tile (MMA N upper bound)
constexpr int kTileM = 128;   // weight rows per GEMM tile (MMA M)

}  // namespace moe
