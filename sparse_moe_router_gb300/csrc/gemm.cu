// gemm.cu -- persistent grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// with the MoE epilogues fused: fp32 store (+bias), SwiGLU -> bf16, weighted row scatter.
//
// The layer's expert projections ("AI MAX+ 395部署Qwen3大模型：GFX1151引擎实测优化解析",
// "MOE 内核优化": the MoE kernel bounds prefill) are, per expert e, products of the expert's
// weight rows with the rows of the tokens routed to e.  The kernel computes them "swap-AB":
//   D[f, j] = sum_k W[g*F + f, k] * B[row0 + j, k]
// with weight rows on the MMA's M side and up to 256 of the group's token rows on the N side.
// A group of c rows is cut into ceil(c/256) token tiles of equal size (rounded up to 16), so an
// expert with 270 tokens costs two 144/126-wide tiles that each read the weight tile once, not
// three tiles of 128/128/14.
//
// CTA pairs (clusters of two, tcgen05 cta_group::2).  A pair computes a 256 x N tile with one
// MMA stream issued by its even CTA: each CTA loads its own 128 weight rows and HALF of the N
// token rows, the tensor cores of both SMs read both halves, and each CTA's TMEM receives its
// own 128 rows of the accumulator.  Per SM that is 32 KB of operands per 64-wide K step instead
// of 48 KB for a one-CTA 128 x 256 tile, which matters because the operand traffic of all SMs
// together runs into the L2 -> SM limit (about 20 TB/s measured on this part).
//   SwiGLU: each CTA's 128 weight rows are 64 gate rows and the same 64 features' up rows,
//           so gate and up land in TMEM lanes i and 64 + i of its accumulator.
//
// Roles (one CTA per SM, two per pair):
//   warps 0..P-1  epilogue (P = 16 for the weighted row scatter, else 8): warp w reads TMEM
//               lanes 32*(w%4)..+31 (the hardware's lane quarters), and the P/4 warps of a
//               quarter take every (P/4)-th 16-token chunk;
//   warps P..P+3 producers: one thread issues the TMA loads of its CTA's weight rows and token
//               rows (the token rows with the smallest of eight boxes, 16..128 rows, that holds
//               the CTA's half of the tile); both CTAs' loads complete on the even CTA's stage
//               barrier;
//   warp P+4    allocates TMEM (both CTAs, pair form); in the even CTA lane 0 issues
//               tcgen05.mma (kind::f16, M = 256, bf16 -> fp32) and tcgen05.commit, whose
//               arrivals go to both CTAs' barriers.
// Pipelines: 192 KB of shared-memory stages (full/empty mbarriers): 3 stages of two 64-wide K
// blocks for the fp32-output GEMMs (router), 6 stages of one block for the routed gate/up and down
// GEMMs; and two
// TMEM accumulators of 256 columns (acc_full/acc_empty; the odd CTA's epilogue releases an
// accumulator with a remote arrive), so the epilogue of one tile overlaps the next main loop.
// Pair tiles are walked statically (tile = pair + i*pairs), ordered (group, weight tile, token
// tile) with the token tile fastest, so pairs sharing a weight tile run together; a shared-expert
// group's tiles are spread evenly among the routed ones.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = kTileM;   // weight rows per CTA tile (the pair's MMA has M = 2 * BM)
constexpr int BN = kTileN;   // token rows per tile (max MMA N)
constexpr int BK = 64;       // K elements per block: one 128-byte swizzle row
constexpr int kBHalf = BN / 2;              // token rows each CTA of the pair holds
constexpr int kABytes = BM * BK * 2;        // 16 KB
constexpr int kBBytes = kBHalf * BK * 2;    // 16 KB
constexpr int kStepBytes = kABytes + kBBytes;  // one K block's operands in one CTA: 32 KB
constexpr int kPipeBytes = 6 * kStepBytes;      // 192 KB of stages
constexpr int kAccCols = BN;                // fp32 accumulator columns per TMEM buffer
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr int kMaxGroups = 1026;                  // E <= 1024 experts, the shared expert, a spare
constexpr int kStgStride = BM + 4;                // SwiGLU staging row (floats), padded for banks
// combine transpose: a row of 32 words (features) per token pair, padded to 36 so that the
// 16-byte reads of 8 lanes fall in distinct banks
constexpr int kPairStride = 36;
// Dynamic schedule: slots of the ring through which the even CTA's producer hands each claimed
// pair tile to the other roles of both CTAs (more than the tiles any role can run ahead).
constexpr int kSchedDepth = 8;

// Q8: the weight operand arrives as E4M3 codes (one byte a weight, 8 KB per 128-row K block)
// in a raw slot of the stage; converter warps widen the codes exactly to bf16 into the stage's
// weight slot (the layout TMA would have written), and the epilogue multiplies each weight
// row's accumulator by the row's fp32 scale.
constexpr int kRawBytes = BM * BK;  // 8 KB
constexpr int kConvBar = 8;         // named barrier of the converter warps

template <int EPI, bool Q8 = false>
struct Cfg {
    // K blocks per pipeline stage.  The router GEMM (K = H, a single wave of small tiles) takes two,
    // so the MMA thread waits and commits once per 8 MMAs (each handshake costs the tensor pipe time
    // it does not hide); the routed GEMMs keep one and the deeper ring (gate/up measured 275.3 us with
    // six one-block stages against 276.1 with three two-block ones), and so does the E4M3 variant
    // (its stages carry the raw codes too).
    static constexpr int kKB = (EPI == EPI_F32 && !Q8) ? 2 : 1;
    static constexpr int kStep = kStepBytes + (Q8 ? kRawBytes : 0);  // one K block in one CTA
    static constexpr int kStages = kPipeBytes / (kKB * kStep);
    static constexpr int kStageBytes = kKB * kStep;
    // epilogue warps: the weighted row scatter keeps many warps storing; the others need 8
    static constexpr int kEpiWarps = (EPI == EPI_COMBINE) ? 16 : 8;
    static constexpr int kProdWarp0 = kEpiWarps;      // 4 producer warps (lane 0 of the first: TMA)
    static constexpr int kConvWarp0 = kEpiWarps + 1;  // Q8: 4 converter warps
    static constexpr int kConvWarps = Q8 ? 4 : 0;
    // TMEM allocation; lane 0 of the even CTA: MMA
    static constexpr int kMmaWarp = Q8 ? kConvWarp0 + kConvWarps : kEpiWarps + 4;
    static constexpr int kThreads = (kMmaWarp + 1) * 32;
    static constexpr int kFT = (EPI == EPI_SWIGLU) ? 64 : BM;    // output features per CTA tile
    // SwiGLU: gate/up exchange, fp32 [2 sub-groups][16 rows][kStgStride];
    // combine: per-warp transpose buffers [warps][8 token pairs][kPairStride words]
    static constexpr int kStagingBytes =
        (EPI == EPI_SWIGLU) ? 2 * 16 * kStgStride * 4 : (EPI == EPI_COMBINE ? kEpiWarps * 8 * kPairStride * 4 : 0);
    // combine: per-tile (output row, weight) of the BN tile rows, double-buffered
    static constexpr int kMetaBytes = (EPI == EPI_COMBINE) ? 2 * BN * 8 : 0;
    // full, empty, raw_full per stage; acc_full, acc_empty per accumulator; drain; sched_full,
    // sched_empty per slot of the tile ring
    static constexpr int kBarBytes = (3 * kStages + 5 + 2 * kSchedDepth) * 8;
    static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kPipeBytes + kStagingBytes +
                                      kMetaBytes + kBarBytes + 32 + 2 * (kMaxGroups + 1) * 4 +
                                      kSchedDepth * 4;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory over the per-CTA limit");
};

struct TileInfo {
    int g, ftile, row0, nvalid;
};

__device__ __forceinline__ TileInfo decode_tile(int tau, int nft, const int *g_tiles,
                                                const int *g_rows, int G, int cap, bool shared_last) {
    if (shared_last) {
        // S shared-expert tiles (group G-1, L2-resident weights) spread evenly among the R
        // routed ones: position iQ holds shared tile i, the others the routed tiles in order
        const int R = nft * g_tiles[G - 1];
        const int S = nft * (g_tiles[G] - g_tiles[G - 1]);
        if (S > 0) {
            const int Q = (R + S) / S;
            const int q = tau / Q;
            if (tau % Q == 0 && q < S) tau = R + q;
            else tau -= (q + 1 < S ? q + 1 : S);
        }
    }
    // Largest group g with nft*g_tiles[g] <= tau (empty groups share their successor's base,
    // and the largest index picks the non-empty one).
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (nft * g_tiles[mid] <= tau) lo = mid; else hi = mid - 1;
    }
    TileInfo t;
    t.g = lo;
    const int local = tau - nft * g_tiles[lo];
    const int ntt = g_tiles[lo + 1] - g_tiles[lo];
    int tt;
    if (shared_last && lo == G - 1) {
        // shared expert: its weights (a few MB) stay in L2 anyway, so walk the weight tiles
        // fastest and let the nft tiles that read one token tile run close together
        tt = local / nft;
        t.ftile = local - tt * nft;
    } else {
        t.ftile = local / ntt;
        tt = local - t.ftile * ntt;
    }
    const int c = g_rows[lo + 1] - g_rows[lo];
    const int tsz = token_tile_size(c, cap);
    t.row0 = g_rows[lo] + tt * tsz;
    const int rem = c - tt * tsz;
    t.nvalid = rem < tsz ? rem : tsz;
    return t;
}

__device__ __forceinline__ void set_error(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// silu(g) * u = g * u / (1 + e^-g), with the fast exponential and an IEEE reciprocal: its error
// (a few fp32 ulp) is far below the bf16 rounding of h that follows.  g -> -inf gives
// 1 / inf = 0, so the product stays 0.
__device__ __forceinline__ float silu_mul(float g, float u) { return g * u * __frcp_rn(1.0f + __expf(-g)); }

// bf16(a) in the low half, bf16(b) in the high half (round to nearest even)
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int EPI, bool Q8>
__global__ void __launch_bounds__(Cfg<EPI, Q8>::kThreads, 1)
    gemm_kernel(const GemmArgs p, const __grid_constant__ CUtensorMap tm_a0,
                const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ TokenMaps tm_b,
                const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_s1) {
    using C = Cfg<EPI, Q8>;
    constexpr int kStep = C::kStep;
    constexpr int kStages = C::kStages;
    constexpr int kStageBytes = C::kStageBytes;
    constexpr int kKB = C::kKB;
    constexpr int kEpiWarps = C::kEpiWarps;
    constexpr int kProdWarp0 = C::kProdWarp0;
    constexpr int kMmaWarp = C::kMmaWarp;
    constexpr int kThreads = C::kThreads;
    constexpr int kSubs = kEpiWarps / 4;  // warps per TMEM lane quarter
    extern __shared__ uint8_t smem_raw[];
    // aligned by an offset from the shared array itself (not through an integer address), so that
    // every access derived from it compiles to a shared-memory access rather than a generic one
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    float *staging = reinterpret_cast<float *>(smem + kStages * kStageBytes);
    int32_t *meta_row = reinterpret_cast<int32_t *>(smem + kStages * kStageBytes + C::kStagingBytes);
    float *meta_w = reinterpret_cast<float *>(meta_row + 2 * BN);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes + C::kStagingBytes + C::kMetaBytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + kStages;
    uint64_t *acc_full = bars + 2 * kStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint64_t *sched_full = drain + 1;                // [kSchedDepth], one arrival (the claimer)
    uint64_t *sched_empty = sched_full + kSchedDepth;  // [kSchedDepth], even CTA: every reader
    uint64_t *raw_full = sched_empty + kSchedDepth;    // [kStages] Q8: this CTA's raw codes landed
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(raw_full + kStages);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    volatile int *epi_vote = reinterpret_cast<volatile int *>(tmem_holder + 2);  // 2 slots
    // stage fills issued by the producer / consumed by the MMA (read on abort), a zero flag
    volatile int *fills = reinterpret_cast<volatile int *>(tmem_holder + 4);
    int *g_tiles = reinterpret_cast<int *>(tmem_holder + 8);
    int *g_rows = g_tiles + (kMaxGroups + 1);
    volatile int *sched_tile = g_rows + (kMaxGroups + 1);  // [kSchedDepth] claimed tile ids

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // the next kernels' count table, zeroed by every CTA (also those with no tile) before its work
    if (p.zero_ptr)
        for (int i = (int)blockIdx.x * kThreads + tid; i < p.zero_n; i += (int)gridDim.x * kThreads) p.zero_ptr[i] = 0;
    const int cap = p.tile_cap > 0 ? p.tile_cap : BN;  // token tile cap
    // CTA pair: rank 0 issues the pair's MMAs (M = 256: its 128 weight rows, then the peer's);
    // each CTA holds half of the tile's token rows and its own rows of the accumulator
    const uint32_t rank = ptx::cluster_ctarank();

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            // Q8: the even producer's expect_tx (token rows) and every converter warp of both CTAs
            ptx::mbar_init(&full[s], 1 + 2 * C::kConvWarps);
            ptx::mbar_init(&empty[s], 1);
            ptx::mbar_init(&raw_full[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], 2 * kEpiWarps);  // one arrival per epilogue warp of the pair
        }
        ptx::mbar_init(drain, 1);
        for (int i = 0; i < kSchedDepth; ++i) {
            ptx::mbar_init(&sched_full[i], 1);
            // readers of a slot: the even CTA's MMA thread, the odd CTA's producer, and every
            // epilogue (and Q8: converter) warp of both CTAs
            ptx::mbar_init(&sched_empty[i], 2 + 2 * kEpiWarps + 2 * C::kConvWarps);
        }
        *abort_flag = 0;
        epi_vote[0] = 0;
        epi_vote[1] = 0;
        fills[0] = fills[1] = fills[2] = 0;
        ptx::fence_mbar_init();
    }
    int G;
    if (p.group_rows == nullptr) {
        G = 1;
        if (tid == 0) {
            g_rows[0] = 0;
            g_rows[1] = p.M_single;
            g_tiles[0] = 0;
            g_tiles[1] = token_tile_count(p.M_single, cap);
        }
    } else {
        G = p.n_groups;
        for (int i = tid; i <= G; i += kThreads) {
            g_rows[i] = p.group_rows[i];
            g_tiles[i] = p.group_tiles[i];
        }
    }
    __syncthreads();
    const int nft = (p.F + C::kFT - 1) / C::kFT;  // CTA tiles along the features
    const int nfp = (nft + 1) >> 1;               // pair tiles along the features
    const int total = nfp * g_tiles[G];
    const int pid = (int)(blockIdx.x >> 1), npair = (int)(gridDim.x >> 1);
    if (pid >= total) return;  // the same for both CTAs of the pair; nothing allocated yet
    auto tile_of = [&](int u) { return decode_tile(u, nfp, g_tiles, g_rows, G, cap, p.shared_last); };

    // The pair's n-th tile.  The first S = max(npair, total - dyn_tail) tiles are walked
    // round-robin (pair p takes p, p + npair, ...: its first ns of them), which keeps the pairs in
    // step over neighbouring tiles, so that pairs sharing a weight tile stream it together.  The
    // last tiles go to whichever pair is free: the even CTA's producer claims each (S + the launch
    // counter's next value; `total` once all are handed out) and publishes it through ring slot
    // (n - ns) % kSchedDepth of both CTAs, which every other role reads in the same order and
    // then releases on the even CTA's sched_empty.
    const bool dyn = p.tile_counter != nullptr && p.dyn_tail > 0;
    const int S = dyn ? max(npair, total - p.dyn_tail) : total;
    const int ns = (S - pid + npair - 1) / npair;  // >= 1: pid < npair <= S
    auto ring_get = [&](int n, int &tau) -> bool {
        if (!dyn || n < ns) {
            tau = pid + n * npair;
            return true;
        }
        const int u = n - ns, slot = u % kSchedDepth;
        if (!ptx::mbar_wait_cluster(&sched_full[slot], (uint32_t)(u / kSchedDepth) & 1u, kWaitLimitNs, abort_flag))
            return false;
        tau = sched_tile[slot];
        return true;
    };
    auto ring_release = [&](int n) {
        if (!dyn || n < ns) return;
        const int slot = (n - ns) % kSchedDepth;
        if (rank == 0) ptx::mbar_arrive(&sched_empty[slot]);
        else ptx::mbar_arrive_remote(ptx::mapa_shared(ptx::smem_u32(&sched_empty[slot]), 0));
    };

    if (warp == kMmaWarp) ptx::tmem_alloc_pair(tmem_holder, kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();  // the peer's barriers are initialised before anyone signals them
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int nks = p.K / (BK * kKB);  // stages per tile

    if (warp >= kProdWarp0 && warp < kMmaWarp) {
        // ------------------------------------------------------------ producers --
        bool ok = true;
        if (tid == kProdWarp0 * 32) {
            ptx::tma_prefetch_desc(&tm_a0);
            if (EPI == EPI_SWIGLU) ptx::tma_prefetch_desc(&tm_a1);
#pragma unroll
            for (int i = 0; i < kTokenBoxes; ++i) ptx::tma_prefetch_desc(&tm_b.m[i]);
            if (p.shared_b_own) ptx::tma_prefetch_desc(&tm_b.shared);
            if (p.shared_last) {
                ptx::tma_prefetch_desc(&tm_s0);
                if (EPI == EPI_SWIGLU) ptx::tma_prefetch_desc(&tm_s1);
            }
            // stage s of both CTAs completes on the even CTA's full[s], which expects both
            // CTAs' bytes; the odd CTA's loads signal it across the pair
            const uint32_t full_even = ptx::mapa_shared(ptx::smem_u32(full), 0);
            int it = 0, s = 0;
            uint32_t ph = 0;
            // dynamic tail, even CTA: tile n + 1 is published when tile n starts (so no role ever
            // waits on the claim), and it was claimed one tile before that (so the atomic's round
            // trip never stalls this thread)
            const bool claimer = dyn && rank == 0;
            int pend = (claimer && ns <= 1) ? atomicAdd(p.tile_counter, 1) : 0;
            bool more = true;  // the counter may still hand out tiles
            int tau = pid;
            for (int n = 0;; ++n) {
                if (n > 0 && !claimer) {
                    if (!ring_get(n, tau)) {
                        ok = false;
                        break;
                    }
                    ring_release(n);
                }
                if (tau >= total) break;
                int tau_next = pid + (n + 1) * npair;
                if (claimer && n + 1 >= ns) {
                    // publish tile n + 1 in both CTAs' ring slot (n + 1 - ns) % kSchedDepth
                    const int u = n + 1 - ns, slot = u % kSchedDepth;
                    if (u >= kSchedDepth &&
                        !ptx::mbar_wait_cluster(&sched_empty[slot], (uint32_t)(u / kSchedDepth - 1) & 1u, kWaitLimitNs,
                                                abort_flag)) {
                        ok = false;
                        break;
                    }
                    tau_next = S + pend < total ? S + pend : total;
                    more = tau_next < total;
                    sched_tile[slot] = tau_next;
                    ptx::st_cluster_u32(ptx::mapa_shared(ptx::smem_u32((const void *)&sched_tile[slot]), 1),
                                        (uint32_t)tau_next);
                    ptx::mbar_arrive(&sched_full[slot]);
                    ptx::mbar_arrive_remote(ptx::mapa_shared(ptx::smem_u32(&sched_full[slot]), 1));
                }
                if (claimer && more && n + 2 >= ns) pend = atomicAdd(p.tile_counter, 1);  // tile n + 2
                const TileInfo t = tile_of(tau);
                const bool shg = p.shared_last && t.g == G - 1;
                const int ftile = 2 * t.ftile + (int)rank;
                // a pair tile past the last feature tile (odd count) reads rows it never stores
                const int arow = (shg ? 0 : t.g * p.F) + ftile * C::kFT;
                const void *ma0 = shg ? (const void *)&tm_s0 : (const void *)&tm_a0;
                const void *ma1 = shg ? (const void *)&tm_s1 : (const void *)&tm_a1;
                // token rows: this CTA holds columns [rank * N/2, (rank + 1) * N/2) of the MMA, loaded
                // with the smallest box that holds N/2 rows (both CTAs use the same box)
                const int half = ((t.nvalid + 15) & ~15) >> 1;
                const bool own = shg && p.shared_b_own;
                const int nbox = own ? kTokenBoxes : (half + 15) >> 4;  // box rows / 16, 1..kTokenBoxes
                const void *mb = own ? (const void *)&tm_b.shared : (const void *)&tm_b.m[nbox - 1];
                const int brow = (own ? t.row0 - g_rows[G - 1] : t.row0) + (int)rank * half;
                // bytes the even CTA's full barrier counts: both CTAs' token rows, and (bf16 weights)
                // both CTAs' weight rows; Q8 weight codes complete on each CTA's raw_full instead
                const uint32_t stage_tx = 2u * (uint32_t)kKB * (uint32_t)((Q8 ? 0 : kABytes) + nbox * 16 * BK * 2);
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    if (!ptx::mbar_wait(&empty[s], ph ^ 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
                    const uint32_t bar = full_even + (uint32_t)(s * 8);
                    if (rank == 0) ptx::mbar_arrive_expect_tx(&full[s], stage_tx);
                    if (Q8) ptx::mbar_arrive_expect_tx(&raw_full[s], (uint32_t)(kKB * kRawBytes));
#pragma unroll
                    for (int j = 0; j < kKB; ++j) {
                        uint8_t *st = smem + s * kStageBytes + j * kStep;
                        const int kc = (ks * kKB + j) * BK;
                        if (Q8) {
                            // the codes of this CTA's weight rows, row-major 64 bytes a row
                            uint8_t *raw = st + kStepBytes;
                            if (EPI == EPI_SWIGLU) {
                                ptx::tma_load_2d(raw, ma0, kc, arow, &raw_full[s]);
                                ptx::tma_load_2d(raw + kRawBytes / 2, ma1, kc, arow, &raw_full[s]);
                            } else {
                                ptx::tma_load_2d(raw, ma0, kc, arow, &raw_full[s]);
                            }
                        } else if (EPI == EPI_SWIGLU) {
                            ptx::tma_load_2d_pair(st, ma0, kc, arow, bar);
                            ptx::tma_load_2d_pair(st + kABytes / 2, ma1, kc, arow, bar);
                        } else {
                            ptx::tma_load_2d_pair(st, ma0, kc, arow, bar);
                        }
                        ptx::tma_load_2d_pair(st + kABytes, mb, kc, brow, bar);
                    }
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (claimer) tau = tau_next;
            }
            fills[0] = it;
        } else if (Q8 && warp >= C::kConvWarp0) {
            // ------------------------------------------------------- converters (Q8) --
            // 16-byte chunk idx = ci + 128 i (i < 4) of a K block's raw codes holds codes
            // 16 (idx % 4) .. +15 of weight row idx / 4.  They are widened exactly (E4M3 -> f16 ->
            // f32 -> bf16: every E4M3 value is a bf16 value) into bf16 chunks 2 (idx % 4) and
            // 2 (idx % 4) + 1 of that row, at their 128-byte-swizzled places (chunk c of row r at
            // r * 128 + (c ^ r % 8) * 16, as TMA would write bf16 weights).  Each lane fences its
            // writes for the async proxy; the warp then adds one arrival to the even CTA's full
            // barrier of the stage (so no named barrier: a warp that gives up leaves alone).
            const int ci = tid - C::kConvWarp0 * 32;
            const uint32_t full_even = ptx::mapa_shared(ptx::smem_u32(full), 0);
            int s = 0;
            uint32_t ph = 0;
            for (int n = 0; ok; ++n) {
                int tau = total, okr = 1;
                if (lane == 0) {
                    okr = ring_get(n, tau) ? 1 : 0;
                    if (okr) ring_release(n);
                }
                okr = __shfl_sync(0xffffffffu, okr, 0);
                tau = __shfl_sync(0xffffffffu, tau, 0);
                if (!okr) {
                    ok = false;
                    break;
                }
                if (tau >= total) break;
                for (int ks = 0; ks < nks; ++ks) {
                    const bool w_ok = __all_sync(0xffffffffu, ptx::mbar_wait(&raw_full[s], ph, kWaitLimitNs, abort_flag));
                    if (!w_ok) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int jb = 0; jb < kKB; ++jb) {
                        uint8_t *a = smem + s * kStageBytes + jb * kStep;
                        const uint8_t *raw = a + kStepBytes;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int idx = ci + 128 * i, r = idx >> 2, q = idx & 3;
                            const uint4 cw = *reinterpret_cast<const uint4 *>(raw + idx * 16);
                            const __nv_fp8x2_storage_t *c2 = reinterpret_cast<const __nv_fp8x2_storage_t *>(&cw);
                            uint32_t o[8];
#pragma unroll
                            for (int m = 0; m < 8; ++m) {
                                const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(c2[m], __NV_E4M3);
                                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
                                o[m] = pack_bf16x2(f.x, f.y);
                            }
                            *reinterpret_cast<uint4 *>(a + r * 128 + (((2 * q) ^ (r & 7)) << 4)) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                            *reinterpret_cast<uint4 *>(a + r * 128 + (((2 * q + 1) ^ (r & 7)) << 4)) =
                                make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (rank == 0) ptx::mbar_arrive(&full[s]);
                        else ptx::mbar_arrive_remote(full_even + (uint32_t)(s * 8));
                    }
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
            }
        }
        if (!ok) {
            set_error(p.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------- MMA (even CTA of the pair) --
            // The tensor core runs only a few instructions ahead of this one thread, so the issue
            // loop is kept to a handful of instructions per stage: stage and phase are counters,
            // and the operand descriptors are stage 0's plus constant steps.
            int it = 0, tc = 0, s = 0;
            uint32_t ph = 0;
            const uint64_t desc0 = ptx::sw128_desc(ptx::smem_u32(smem));
            bool ok = true;
            for (int n = 0;; ++n, ++tc) {
                int tau;
                if (!ring_get(n, tau)) {
                    ok = false;
                    break;
                }
                ring_release(n);
                if (tau >= total) break;
                const TileInfo t = tile_of(tau);
                const uint32_t nmma = (uint32_t)((t.nvalid + 15) & ~15);
                const int buf = tc & 1;
                const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
                // both CTAs' epilogues have drained this accumulator
                if (!ptx::mbar_wait_cluster(&acc_empty[buf], aph ^ 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d_base = tmem_base + (uint32_t)(buf * kAccCols);
                const uint32_t idesc = ptx::idesc_bf16_f32(2 * BM, nmma);
                for (int ks = 0; ks < nks; ++ks, ++it) {
                    if (!ptx::mbar_wait_cluster(&full[s], ph, kWaitLimitNs, abort_flag)) { ok = false; break; }
                    ptx::tc_fence_after();
                    // descriptors of stage s, block j: the start-address field steps by bytes / 16,
                    // and one K=16 slice is 32 bytes further along the swizzled 128-byte row
#pragma unroll
                    for (int j = 0; j < kKB; ++j) {
                        const uint64_t da = desc0 + (uint64_t)((s * kStageBytes + j * kStep) >> 4);
                        const uint64_t db = da + (uint64_t)(kABytes >> 4);
                        ptx::mma_bf16_pair(d_base, da, db, idesc, (ks | j) != 0 ? 1u : 0u);
#pragma unroll
                        for (int kk = 1; kk < BK / 16; ++kk)
                            ptx::mma_bf16_pair(d_base, da + (uint64_t)(2 * kk), db + (uint64_t)(2 * kk), idesc, 1u);
                    }
                    ptx::mma_commit_pair(&empty[s], (uint16_t)3);  // frees stage s in both CTAs
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit_pair(&acc_full[buf], (uint16_t)3);
            }
            fills[1] = it;
            // Wait for every MMA of the pair before TMEM is released.
            ptx::mma_commit_pair(drain, (uint16_t)1);
            if (!ptx::mbar_wait(drain, 0, kWaitLimitNs, abort_flag)) ok = false;
            if (!ok) {
                set_error(p.status, MOE_ERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue --
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        const int sub = warp >> 2;     // this warp takes chunks cidx with cidx % kSubs == sub
        const int frow = quarter * 32 + lane;
        float *stg = staging + sub * 16 * kStgStride;  // SwiGLU exchange buffer of this sub-group
        const uint32_t acc_empty_remote = ptx::mapa_shared(ptx::smem_u32(acc_empty), 0);
        int tc = 0;
        bool ok = true;
        for (int n = 0;; ++n, ++tc) {
            // lane 0 takes the tile from the ring and hands it to the warp; every warp then
            // passes the vote below even on the last (end) round, so they leave together
            int tau = total;
            int ok_t = 1;
            if (lane == 0) {
                ok_t = ring_get(n, tau) ? 1 : 0;
                if (ok_t) ring_release(n);
            }
            ok_t = __shfl_sync(0xffffffffu, ok_t, 0);
            tau = __shfl_sync(0xffffffffu, tau, 0);
            const bool end = ok_t && tau >= total;
            const bool live = ok_t && !end;
            const TileInfo t = live ? tile_of(tau) : TileInfo{0, 0, 0, 0};
            const int buf = tc & 1;
            const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
            const int ftile = 2 * t.ftile + (int)rank;
            const bool store = ftile < nft;  // false only for the odd half of a last pair tile
            // combine: the 16 warps fetch (output row, weight) of the tile's rows into shared
            // memory before the accumulator is ready (the loads overlap the main loop); the
            // vote barrier below publishes them to all epilogue warps
            if (EPI == EPI_COMBINE && live && lane < BN / kEpiWarps) {
                const int j = warp * (BN / kEpiWarps) + lane;
                int orow = 0;
                float w = 0.f;
                if (j < t.nvalid) {
                    const int row = t.row0 + j;
                    if (p.shared_last && t.g == G - 1) {  // shared expert: in place, weight 1
                        orow = row;
                        w = 1.f;
                    } else if (MOE_DEBUG_OK(p.src_rows == 0 || (row >= 0 && row < p.src_rows), p.status)) {
                        orow = p.epi_tok ? __ldg(&p.epi_tok[row]) : row;
                        w = p.epi_w ? __ldg(&p.epi_w[row]) : 1.f;
                    } else {
                        orow = -1;
                    }
                    // -1: the row is not stored
                    if (orow >= 0 && !MOE_DEBUG_OK(p.out_rows == 0 || orow < p.out_rows, p.status)) orow = -1;
                }
                meta_row[buf * BN + j] = orow;
                meta_w[buf * BN + j] = w;
            }
            // The epilogue warps share named barriers, so they give up together: lane 0 of
            // each warp votes, and the vote is read by all after the barrier.
            const bool got = live ? ptx::mbar_wait(&acc_full[buf], aph, kWaitLimitNs, abort_flag) : true;
            if (lane == 0 && (!ok_t || !got)) epi_vote[tc & 1] = 1;
            ptx::named_bar(1, kEpiWarps * 32);
            const bool fail = epi_vote[tc & 1] != 0;
            ptx::named_bar(1, kEpiWarps * 32);
            if (fail) { ok = false; break; }
            if (end) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * kAccCols);
            float bias_f = 0.f;
            if (EPI == EPI_F32) {
                const int f = ftile * BM + frow;
                if (p.bias != nullptr && f < p.F) bias_f = __ldg(&p.bias[f]);
            }
            // Q8: this lane's weight row scale (SwiGLU: lanes 0..63 gate rows, 64..127 the same
            // features' up rows; the shared expert's group reads its own scale arrays)
            float sc = 1.f;
            if (Q8 && store) {
                const bool shg = p.shared_last && t.g == G - 1;
                const size_t gofs = shg ? 0 : (size_t)t.g * p.F;
                if (EPI == EPI_SWIGLU) {
                    const float *sp = frow < 64 ? (shg ? p.ws_scale0 : p.w_scale0) : (shg ? p.ws_scale1 : p.w_scale1);
                    sc = __ldg(sp + gofs + ftile * 64 + (frow & 63));
                } else {
                    const int f = ftile * BM + frow;
                    if (f < p.F) sc = __ldg((shg ? p.ws_scale0 : p.w_scale0) + gofs + f);
                }
            }
            // this warp's chunks are cidx = sub, sub + kSubs, ...; the TMEM load of the next
            // chunk is issued before the current one is processed, hiding its latency
            const int n_chunks = store ? (t.nvalid + 15) >> 4 : 0;
            uint32_t rn[16];
            if (sub < n_chunks) ptx::tmem_ld_16(taddr + (uint32_t)(16 * sub), rn);
            for (int cidx = sub; cidx < n_chunks; cidx += kSubs) {
                const int j0 = 16 * cidx;
                uint32_t r[16];
                ptx::tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 16; ++q) r[q] = rn[q];
                if (cidx + kSubs < n_chunks) ptx::tmem_ld_16(taddr + (uint32_t)(j0 + 16 * kSubs), rn);
                if (EPI == EPI_SWIGLU) {
                    // lanes 0..63 hold gate, 64..127 the same features' up: exchange through
                    // shared memory, then thread q computes token q/8, features 8*(q%8)..+7
                    // and writes them as one 16-byte store.
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) stg[jj * kStgStride + frow] = sc * __uint_as_float(r[jj]);
                    ptx::named_bar(2 + sub, 128);
                    const int q = frow;
                    const int jj = q >> 3, fg = (q & 7) * 8;
                    if (j0 + jj < t.nvalid &&
                        MOE_DEBUG_OK(p.out_rows == 0 || t.row0 + j0 + jj < p.out_rows, p.status)) {
                        const float4 g0 = *reinterpret_cast<const float4 *>(&stg[jj * kStgStride + fg]);
                        const float4 g1 = *reinterpret_cast<const float4 *>(&stg[jj * kStgStride + fg + 4]);
                        const float4 u0 = *reinterpret_cast<const float4 *>(&stg[jj * kStgStride + 64 + fg]);
                        const float4 u1 = *reinterpret_cast<const float4 *>(&stg[jj * kStgStride + 64 + fg + 4]);
                        __align__(16) __nv_bfloat16 h[8] = {
                            __float2bfloat16_rn(silu_mul(g0.x, u0.x)), __float2bfloat16_rn(silu_mul(g0.y, u0.y)),
                            __float2bfloat16_rn(silu_mul(g0.z, u0.z)), __float2bfloat16_rn(silu_mul(g0.w, u0.w)),
                            __float2bfloat16_rn(silu_mul(g1.x, u1.x)), __float2bfloat16_rn(silu_mul(g1.y, u1.y)),
                            __float2bfloat16_rn(silu_mul(g1.z, u1.z)), __float2bfloat16_rn(silu_mul(g1.w, u1.w))};
                        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out);
                        *reinterpret_cast<uint4 *>(&o[(size_t)(t.row0 + j0 + jj) * p.ld + ftile * 64 + fg]) =
                            *reinterpret_cast<const uint4 *>(h);
                    }
                    ptx::named_bar(2 + sub, 128);
                } else if (EPI == EPI_F32) {
                    const int f = ftile * BM + frow;
                    float *o = static_cast<float *>(p.out);
                    if (f < p.F) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            if (j0 + jj < t.nvalid &&
                                MOE_DEBUG_OK(p.out_rows == 0 || t.row0 + j0 + jj < p.out_rows, p.status))
                                o[(size_t)(t.row0 + j0 + jj) * p.ld + f] = sc * __uint_as_float(r[jj]) + bias_f;
                    }
                } else {
                    // Weighted row scatter: tile row r is stored as bf16(w_r * D[:, r]) into
                    // output row meta_row[r] (the pair index, so the k rows of a token end up
                    // adjacent).  The lane (one feature) packs tokens 2m and 2m+1 into one word;
                    // the warp's 32 features x 16 tokens go through its own buffer, transposed,
                    // and lane (m, seg) splits the words of features 8*seg.. into the two
                    // tokens' 16-byte rows.
                    uint32_t *tb = reinterpret_cast<uint32_t *>(staging) + warp * (8 * kPairStride);
                    const int mb = buf * BN + j0;
                    const float4 *wv = reinterpret_cast<const float4 *>(meta_w + mb);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 w4 = wv[q];
                        const uint32_t lo = pack_bf16x2(w4.x * (sc * __uint_as_float(r[4 * q])),
                                                        w4.y * (sc * __uint_as_float(r[4 * q + 1])));
                        const uint32_t hi = pack_bf16x2(w4.z * (sc * __uint_as_float(r[4 * q + 2])),
                                                        w4.w * (sc * __uint_as_float(r[4 * q + 3])));
                        tb[(2 * q) * kPairStride + lane] = lo;
                        tb[(2 * q + 1) * kPairStride + lane] = hi;
                    }
                    __syncwarp();
                    uint16_t *o = static_cast<uint16_t *>(p.out);
                    const int seg = lane & 3, m = lane >> 2;
                    const uint4 a = *reinterpret_cast<const uint4 *>(&tb[m * kPairStride + seg * 8]);
                    const uint4 c = *reinterpret_cast<const uint4 *>(&tb[m * kPairStride + seg * 8 + 4]);
                    // words hold (token 2m in the low half, token 2m+1 in the high half)
                    const uint4 e0 = make_uint4(__byte_perm(a.x, a.y, 0x5410), __byte_perm(a.z, a.w, 0x5410),
                                                __byte_perm(c.x, c.y, 0x5410), __byte_perm(c.z, c.w, 0x5410));
                    const uint4 e1 = make_uint4(__byte_perm(a.x, a.y, 0x7632), __byte_perm(a.z, a.w, 0x7632),
                                                __byte_perm(c.x, c.y, 0x7632), __byte_perm(c.z, c.w, 0x7632));
                    const size_t col = (size_t)ftile * BM + quarter * 32 + seg * 8;
                    const int or0 = meta_row[mb + 2 * m], or1 = meta_row[mb + 2 * m + 1];
                    // y is read once, by the finalise: streaming stores leave L2 to the weight and
                    // h tiles that the next tiles read again
                    if (j0 + 2 * m < t.nvalid && or0 >= 0)
                        __stcs(reinterpret_cast<uint4 *>(&o[(size_t)or0 * p.ld + col]), e0);
                    if (j0 + 2 * m + 1 < t.nvalid && or1 >= 0)
                        __stcs(reinterpret_cast<uint4 *>(&o[(size_t)or1 * p.ld + col]), e1);
                    __syncwarp();
                }
            }
            // release the accumulator to the even CTA's MMA: one arrival per warp, after the
            // warp's TMEM loads are complete
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) ptx::mbar_arrive(&acc_empty[buf]);
                else ptx::mbar_arrive_remote(acc_empty_remote + (uint32_t)(buf * 8));
            }
        }
        if (!ok) {
            set_error(p.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // a wait gave up: the stage fills issued but not consumed may still be landing in shared
        // memory; let them finish (bounded) before the pair's shared memory is released.  The
        // even CTA's full barriers count both CTAs' bytes; the odd CTA cannot wait on them and
        // gives its own copies a fixed 100 us instead (a TMA load lands within microseconds).
        if (tid == kProdWarp0 * 32) {
            if (rank == 0) {
                for (int i = fills[1]; i < fills[0]; ++i)
                    ptx::mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u, kWaitLimitNs, fills + 2);
            } else {
                const uint64_t t0 = ptx::globaltimer();
                while (ptx::globaltimer() - t0 < 100000ull) {}
            }
        }
        __syncthreads();
    }
    // neither CTA of the pair leaves (or frees TMEM) while the other may still signal it
    ptx::cluster_sync();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <int EPI, bool Q8>
cudaError_t launch_impl(const GemmArgs &a, const CUtensorMap &m0, const CUtensorMap &m1,
                        const TokenMaps &mb, const CUtensorMap &s0, const CUtensorMap &s1, int kc,
                        cudaStream_t s) {
    using C = Cfg<EPI, Q8>;
    // per device: the shared-memory opt-in and how many CTA pairs fit on the GPU at once (set
    // once under a lock, so that two host threads' first launches do not race)
    static int max_pairs[64] = {0};
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::unique_lock<std::mutex> lk(mu);
    if (max_pairs[dev] == 0) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<EPI, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(device_info().sm_count & ~1, 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, gemm_kernel<EPI, Q8>, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        max_pairs[dev] = n;
    }
    int pairs = max_pairs[dev];
    lk.unlock();
    if (a.group_rows == nullptr) {
        const int nft = (a.F + C::kFT - 1) / C::kFT;
        const int ptiles = ((nft + 1) / 2) * token_tile_count(a.M_single, a.tile_cap > 0 ? a.tile_cap : BN);
        if (ptiles < pairs) pairs = ptiles;
    }
    if (pairs <= 0) return cudaSuccess;
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    LaunchScope scope(kc, s);
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_kernel<EPI, Q8>, a, m0, m1, mb, s0, s1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(GemmEpi epi, const GemmArgs &a, const CUtensorMap &tm_a0, const CUtensorMap &tm_a1,
                        const TokenMaps &tm_b, const CUtensorMap &tm_s0, const CUtensorMap &tm_s1, int kc,
                        cudaStream_t s) {
    if (a.n_groups > kMaxGroups - 1) return cudaErrorInvalidValue;
    if (a.K % (2 * BK) != 0 || a.K <= 0) return cudaErrorInvalidValue;
    if (a.tile_cap < 0 || a.tile_cap > BN || a.tile_cap % 16 != 0) return cudaErrorInvalidValue;
    if (a.tile_cap != 0 && a.group_rows != nullptr) return cudaErrorInvalidValue;  // groups use 256
    if (a.shared_last && (a.group_rows == nullptr || a.n_groups < 2))
        return cudaErrorInvalidValue;
    if (a.shared_b_own && !a.shared_last) return cudaErrorInvalidValue;
    if (epi == EPI_SWIGLU && (a.F % 64 != 0 || a.ld % 8 != 0)) return cudaErrorInvalidValue;
    if (epi == EPI_COMBINE && (a.F % BM != 0 || a.ld % 8 != 0)) return cudaErrorInvalidValue;
    if (a.q8) {
        if (!a.w_scale0 || (epi == EPI_SWIGLU && !a.w_scale1)) return cudaErrorInvalidValue;
        if (a.shared_last && (!a.ws_scale0 || (epi == EPI_SWIGLU && !a.ws_scale1))) return cudaErrorInvalidValue;
        switch (epi) {
            case EPI_F32: return launch_impl<EPI_F32, true>(a, tm_a0, tm_a1, tm_b, tm_s0, tm_s1, kc, s);
            case EPI_SWIGLU: return launch_impl<EPI_SWIGLU, true>(a, tm_a0, tm_a1, tm_b, tm_s0, tm_s1, kc, s);
            case EPI_COMBINE: return launch_impl<EPI_COMBINE, true>(a, tm_a0, tm_a1, tm_b, tm_s0, tm_s1, kc, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (epi) {
        case EPI_F32: return launch_impl<EPI_F32, false>(a, tm_a0, tm_a1, tm_b, tm_s0, tm_s1, kc, s);
        case EPI_SWIGLU: return launch_impl<EPI_SWIGLU, false>(a, tm_a0, tm_a1, tm_b, tm_s0, tm_s1, kc, s);
        case EPI_COMBINE: return launch_impl<EPI_COMBINE, false>(a, tm_a0, tm_a1, tm_b, tm_s0, tm_s1, kc, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
