// gemm.cu -- persistent grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// with the MoE epilogues fused: fp32 store (+bias), SwiGLU -> bf16, weighted scatter-add.
//
// The layer's expert projections ("AI MAX+ 395部署Qwen3大模型：GFX1151引擎实测优化解析",
// "MOE 内核优化": the MoE kernel bounds prefill) are, per expert e, products of the expert's
// weight rows with the rows of the tokens routed to e.  The kernel computes them "swap-AB":
//   D[f, j] = sum_k W[g*F + f, k] * B[row0 + j, k]
// with the weight rows f on the MMA's M side (128 per tile) and the group's token rows j on
// the N side (up to 128 per tile, N rounded up to 16).  A ragged expert with 257 rows thus
// costs one extra 16-wide column block, not a second 128-row tile.
//
// Roles (288 threads):
//   warps 0-3  epilogue: tcgen05.ld of the fp32 accumulator (warp w reads TMEM lanes
//              32w..32w+31 = weight rows), fused epilogue, global stores / atomics;
//   warps 4-7  producers: the B operand (token rows, optionally gathered through the expert
//              permutation) with 16-byte cp.async into the 128-byte-swizzled K-major layout;
//              thread 128 also issues the TMA loads of the weight tile(s);
//   warp 8     allocates TMEM; lane 0 issues tcgen05.mma (kind::f16, bf16 -> fp32) and
//              tcgen05.commit.
// Pipelines: S shared-memory stages (full/empty mbarriers) and two TMEM accumulator buffers
// (acc_full/acc_empty), so the epilogue of one tile overlaps the main loop of the next.
// Tiles are walked statically (tile = blockIdx.x + i*gridDim.x), ordered (group, weight
// tile, token tile) with the token tile fastest, so the CTAs that share a weight tile run
// at the same time and the weight tile is fetched from HBM once.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = kTileM;   // weight rows per tile (MMA M)
constexpr int BN = kTileN;   // token rows per tile (max MMA N)
constexpr int BK = 64;       // K elements per stage: one 128-byte swizzle row
constexpr int kThreads = 288;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr int kMaxGroups = 1025;                  // E <= 1024 experts (+1 spare)

template <int EPI>
struct Cfg {
    static constexpr int kAParts = (EPI == EPI_SWIGLU) ? 2 : 1;
    static constexpr int kABytes = kAParts * BM * BK * 2;
    static constexpr int kBBytes = BN * BK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStages = (EPI == EPI_SWIGLU) ? 4 : 6;
    static constexpr int kLag = kStages - 1;
    static constexpr int kAccCols = kAParts * BN;
    static constexpr uint32_t kTmemCols = 2 * kAccCols;
    static constexpr int kBarBytes = (2 * kStages + 5) * 8;
    static constexpr int kSmemBytes =
        1024 /*alignment slack*/ + kStages * kStageBytes + kBarBytes + 16 + 2 * (kMaxGroups + 1) * 4;
};

struct TileInfo {
    int g, ftile, row0, nvalid;
};

__device__ __forceinline__ TileInfo decode_tile(int tau, int nft, const int *g_tiles,
                                                const int *g_rows, int G) {
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
    t.ftile = local / ntt;
    const int tt = local - t.ftile * ntt;
    t.row0 = g_rows[lo] + tt * BN;
    const int rem = g_rows[lo + 1] - t.row0;
    t.nvalid = rem < BN ? rem : BN;
    return t;
}

__device__ __forceinline__ void set_error(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const GemmArgs p, const __grid_constant__ CUtensorMap tm_a0,
                const __grid_constant__ CUtensorMap tm_a1) {
    using C = Cfg<EPI>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStageBytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + C::kStages;
    uint64_t *acc_full = bars + 2 * C::kStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *g_tiles = reinterpret_cast<int *>(tmem_holder + 4);
    int *g_rows = g_tiles + (kMaxGroups + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&full[s], 128 + 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], 128);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    int G;
    if (p.group_rows == nullptr) {
        G = 1;
        if (tid == 0) {
            g_rows[0] = 0;
            g_rows[1] = p.M_single;
            g_tiles[0] = 0;
            g_tiles[1] = (p.M_single + BN - 1) / BN;
        }
    } else {
        G = p.n_groups;
        for (int i = tid; i <= G; i += kThreads) {
            g_rows[i] = p.group_rows[i];
            g_tiles[i] = p.group_tiles[i];
        }
    }
    __syncthreads();
    const int nft = (p.F + BM - 1) / BM;
    const int total = nft * g_tiles[G];
    if ((int)blockIdx.x >= total) return;  // CTA-uniform; nothing allocated yet

    if (warp == 8) ptx::tmem_alloc(tmem_holder, C::kTmemCols);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int nkb = p.K / BK;

    if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ producers --
        const int q = tid - 128;
        const int c = q & 7;        // 16-byte chunk within the 128-byte row segment
        const int rbase = q >> 3;   // rows rbase + 16*i
        const uint16_t *bsrc = static_cast<const uint16_t *>(p.b_src);
        if (q == 0) {
            ptx::tma_prefetch_desc(&tm_a0);
            if (EPI == EPI_SWIGLU) ptx::tma_prefetch_desc(&tm_a1);
        }
        int it = 0;
        bool ok = true;
        for (int tau = blockIdx.x; tau < total && ok; tau += gridDim.x) {
            const TileInfo t = decode_tile(tau, nft, g_tiles, g_rows, G);
            const int nmma = (t.nvalid + 15) & ~15;
            const uint16_t *src[8];
            uint32_t nbytes[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = rbase + 16 * i;
                if (j < t.nvalid) {
                    const int r = t.row0 + j;
                    const int srow = p.gather_perm ? (__ldg(&p.gather_perm[r]) / p.gather_k) : r;
                    src[i] = bsrc + (size_t)srow * p.K + c * 8;
                    nbytes[i] = 16;
                } else if (j < nmma) {
                    src[i] = bsrc;
                    nbytes[i] = 0;  // zero fill: read by the MMA, ignored by the epilogue
                } else {
                    src[i] = nullptr;
                    nbytes[i] = 0;
                }
            }
            const int arow = t.g * p.F + t.ftile * BM;
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int s = it % C::kStages;
                const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
                if (!ptx::mbar_wait(&empty[s], ph ^ 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
                uint8_t *st = smem + s * C::kStageBytes;
                if (q == 0) {
                    ptx::mbar_arrive_expect_tx(&full[s], C::kABytes);
                    ptx::tma_load_2d(st, &tm_a0, kb * BK, arow, &full[s]);
                    if (EPI == EPI_SWIGLU) ptx::tma_load_2d(st + BM * BK * 2, &tm_a1, kb * BK, arow, &full[s]);
                }
                const uint32_t bst = ptx::smem_u32(st + C::kABytes);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (src[i] != nullptr) {
                        const int j = rbase + 16 * i;
                        const uint32_t dst = bst + j * 128 + ((c ^ (j & 7)) << 4);
                        const uint16_t *sp = nbytes[i] ? src[i] + kb * BK : src[i];
                        ptx::cp_async_16(dst, sp, nbytes[i]);
                    }
                }
                ptx::cp_async_commit();
                if (it >= C::kLag) {
                    ptx::cp_async_wait<C::kLag>();
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(&full[(it - C::kLag) % C::kStages]);
                }
            }
        }
        ptx::cp_async_wait<0>();
        ptx::fence_proxy_async_smem();
        for (int d = (it > C::kLag ? it - C::kLag : 0); d < it; ++d) ptx::mbar_arrive(&full[d % C::kStages]);
        if (!ok) {
            set_error(p.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp == 8) {
        // ---------------------------------------------------------------- MMA --
        if (lane == 0) {
            int it = 0, tc = 0;
            bool ok = true;
            for (int tau = blockIdx.x; tau < total && ok; tau += gridDim.x, ++tc) {
                const TileInfo t = decode_tile(tau, nft, g_tiles, g_rows, G);
                const uint32_t nmma = (uint32_t)((t.nvalid + 15) & ~15);
                const int buf = tc & 1;
                const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
                if (!ptx::mbar_wait(&acc_empty[buf], aph ^ 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d_base = tmem_base + (uint32_t)(buf * C::kAccCols);
                const uint32_t idesc = ptx::idesc_bf16_f32(BM, nmma);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % C::kStages;
                    const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
                    if (!ptx::mbar_wait(&full[s], ph, kWaitLimitNs, abort_flag)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t a_addr = ptx::smem_u32(smem + s * C::kStageBytes);
                    const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t bd = ptx::sw128_desc(b_addr + kk * 32);
                        const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                        ptx::mma_bf16(d_base, ptx::sw128_desc(a_addr + kk * 32), bd, idesc, acc);
                        if (EPI == EPI_SWIGLU)
                            ptx::mma_bf16(d_base + BN, ptx::sw128_desc(a_addr + BM * BK * 2 + kk * 32), bd,
                                          idesc, acc);
                    }
                    ptx::mma_commit(&empty[s]);
                }
                if (!ok) break;
                ptx::mma_commit(&acc_full[buf]);
            }
            // Wait for every MMA of this CTA before TMEM is released.
            ptx::mma_commit(drain);
            if (!ptx::mbar_wait(drain, 0, kWaitLimitNs, abort_flag)) ok = false;
            if (!ok) {
                set_error(p.status, MOE_ERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue --
        const int quarter = warp;  // warps 0..3 own TMEM lanes 32*warp .. 32*warp+31
        const int frow = quarter * 32 + lane;
        int tc = 0;
        bool ok = true;
        for (int tau = blockIdx.x; tau < total; tau += gridDim.x, ++tc) {
            const TileInfo t = decode_tile(tau, nft, g_tiles, g_rows, G);
            const int buf = tc & 1;
            const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
            if (!ptx::mbar_wait(&acc_full[buf], aph, kWaitLimitNs, abort_flag)) { ok = false; break; }
            ptx::tc_fence_after();
            const int f = t.ftile * BM + frow;
            const bool fvalid = f < p.F;
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * C::kAccCols);
            float bias_f = 0.f;
            if (EPI == EPI_F32 && p.bias != nullptr && fvalid) bias_f = __ldg(&p.bias[f]);
            for (int j0 = 0; j0 < t.nvalid; j0 += 16) {
                uint32_t r[16];
                ptx::tmem_ld_16(taddr + (uint32_t)j0, r);
                if (EPI == EPI_SWIGLU) {
                    uint32_t u[16];
                    ptx::tmem_ld_16(taddr + BN + (uint32_t)j0, u);
                    ptx::tmem_ld_wait();
                    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        if (j < t.nvalid && fvalid) {
                            const float g = __uint_as_float(r[jj]);
                            const float uu = __uint_as_float(u[jj]);
                            const float h = g / (1.0f + expf(-g)) * uu;
                            o[(size_t)(t.row0 + j) * p.ld + f] = __float2bfloat16_rn(h);
                        }
                    }
                } else if (EPI == EPI_F32) {
                    ptx::tmem_ld_wait();
                    float *o = static_cast<float *>(p.out);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        if (j < t.nvalid && fvalid)
                            o[(size_t)(t.row0 + j) * p.ld + f] = __uint_as_float(r[jj]) + bias_f;
                    }
                } else {
                    ptx::tmem_ld_wait();
                    // token and routing weight of the 16 rows, spread over lanes 0..15
                    int my_tok = 0;
                    float my_w = 1.f;
                    if (lane < 16 && j0 + lane < t.nvalid) {
                        const int row = t.row0 + j0 + lane;
                        if (p.epi_perm != nullptr) {
                            const int pair = __ldg(&p.epi_perm[row]);
                            my_tok = pair / p.epi_k;
                            my_w = __ldg(&p.epi_w[pair]);
                        } else {
                            my_tok = row;
                        }
                    }
                    float *o = static_cast<float *>(p.out);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int tok = __shfl_sync(0xffffffffu, my_tok, jj);
                        const float w = __shfl_sync(0xffffffffu, my_w, jj);
                        if (j0 + jj < t.nvalid && fvalid)
                            atomicAdd(&o[(size_t)tok * p.ld + f], w * __uint_as_float(r[jj]));
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&acc_empty[buf]);
        }
        if (!ok) {
            set_error(p.status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int EPI>
cudaError_t launch_impl(const GemmArgs &a, const CUtensorMap &m0, const CUtensorMap &m1, int kc,
                        cudaStream_t s) {
    using C = Cfg<EPI>;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const DeviceInfo &di = device_info();
    int grid = di.sm_count;
    if (a.group_rows == nullptr) {
        const int nft = (a.F + BM - 1) / BM;
        const int tiles = nft * ((a.M_single + BN - 1) / BN);
        if (tiles < grid) grid = tiles;
    }
    if (grid <= 0) return cudaSuccess;
    LaunchScope scope(kc, s);
    gemm_kernel<EPI><<<grid, kThreads, C::kSmemBytes, s>>>(a, m0, m1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(GemmEpi epi, const GemmArgs &a, const CUtensorMap &tm_a0,
                        const CUtensorMap &tm_a1, int kc, cudaStream_t s) {
    if (a.n_groups > kMaxGroups - 1) return cudaErrorInvalidValue;
    if (a.K % BK != 0 || a.K <= 0) return cudaErrorInvalidValue;
    switch (epi) {
        case EPI_F32: return launch_impl<EPI_F32>(a, tm_a0, tm_a1, kc, s);
        case EPI_SWIGLU: return launch_impl<EPI_SWIGLU>(a, tm_a0, tm_a1, kc, s);
        case EPI_COMBINE: return launch_impl<EPI_COMBINE>(a, tm_a0, tm_a1, kc, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
