// decode.cu -- the single-token (T = 1) layer: every weight byte the token needs is streamed
// from HBM once with 128-bit loads (or TMA), fp32 accumulation.
//
// Batch-1 decode is the pages' execution mode ("AIMA AMD395 Qwen3.6 35B Windows Engine",
// "产品定位": batch size 1, greedy decode).  At T = 1 each selected expert is a matrix-vector
// product bound by HBM bandwidth.  Two kernels per layer, chained with programmatic
// dependent launch so that each kernel is resident and prefetching before its predecessor
// ends:
//   K1  router logits (E rows), one warp per row.  Before waiting on the previous kernel it
//       prefetches its weight rows into L2 (they do not depend on x), so the next layer's
//       router weights stream while the current layer's experts do.  It also clears the fp32
//       output accumulator K2 adds into.
//   K2  one block per (routed slot j, 32-wide slice of I) and per 32-wide slice of the shared
//       expert's Is.  A routed block computes the softmax/top-k/renormalisation from the E
//       logits itself (no block waits on another: each lane sorts its logits once, then k
//       rounds compare list heads); then every block
//         - starts a TMA copy of the down-projection columns of its slice (H x 32, in chunks
//           of 2048 rows) into shared memory (a shared-expert block before it even waits for
//           K1: its weights do not depend on the routing),
//         - computes its 32 features of h = bf16(silu(Wg x) * (Wu x)),
//         - adds w_j * Wd[:, slice] h_slice into the fp32 accumulator (split-K over I).
//       The last block to finish (a ticket counter that resets itself) writes out = bf16(acc)
//       and x_next = bf16(resid + out).
// The accumulator adds are fp32 atomics: the summation order, hence the last bit of out,
// can differ from run to run at T = 1.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kK1Warps = 8;
constexpr int kK1Block = kK1Warps * 32;
constexpr int kK2Threads = 512;
constexpr int kK2Warps = kK2Threads / 32;
constexpr int kSlice = 32;           // features of I (or Is) per K2 block
constexpr int kBoxRows = 128;        // TMA box rows of the down-projection slice
constexpr int kChunkRows = 2048;     // rows of the slice held in shared memory at once
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float dot8(const uint4 &w, const uint4 &x) {
    const __nv_bfloat162 *wp = reinterpret_cast<const __nv_bfloat162 *>(&w);
    const __nv_bfloat162 *xp = reinterpret_cast<const __nv_bfloat162 *>(&x);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(wp[i]);
        const float2 b = __bfloat1622float2(xp[i]);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
    }
    return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Lane-partial dot products of two weight rows with the shared-memory vector xs (len bf16,
// len % 8 == 0), eight 16-byte loads per row in flight per lane.
__device__ __forceinline__ void dot2_rows(const uint16_t *r0, const uint16_t *r1, const uint4 *xs,
                                          int len, int lane, float &a0, float &a1) {
    const int n16 = len / 8;
    const uint4 *p0 = reinterpret_cast<const uint4 *>(r0);
    const uint4 *p1 = reinterpret_cast<const uint4 *>(r1);
    int c = lane;
    for (; c + 32 * 7 < n16; c += 32 * 8) {
        uint4 w0[8], w1[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            w0[u] = ld_stream(p0 + c + 32 * u);
            w1[u] = ld_stream(p1 + c + 32 * u);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint4 xv = xs[c + 32 * u];
            a0 += dot8(w0[u], xv);
            a1 += dot8(w1[u], xv);
        }
    }
    for (; c < n16; c += 32) {
        const uint4 xv = xs[c];
        a0 += dot8(ld_stream(p0 + c), xv);
        a1 += dot8(ld_stream(p1 + c), xv);
    }
}

__device__ __forceinline__ void dot1_row(const uint16_t *r0, const uint4 *xs, int len, int lane, float &a0) {
    const int n16 = len / 8;
    const uint4 *p0 = reinterpret_cast<const uint4 *>(r0);
    int c = lane;
    for (; c + 32 * 7 < n16; c += 32 * 8) {
        uint4 w0[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) w0[u] = ld_stream(p0 + c + 32 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u) a0 += dot8(w0[u], xs[c + 32 * u]);
    }
    for (; c < n16; c += 32) a0 += dot8(ld_stream(p0 + c), xs[c]);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ uint16_t bf16_bits(float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t *>(&h);
}

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// ---------------------------------------------------------------------- kernel 1 --
__global__ void __launch_bounds__(kK1Block) decode_k1_kernel(DecodeArgs a) {
    extern __shared__ uint4 xs[];  // H bf16
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int task = blockIdx.x * kK1Warps + warp;
    // The weights do not depend on the previous kernel: start them towards L2 right away.
    const int row_bytes = a.H * 2;
    if (task < a.E) {
        const char *r = reinterpret_cast<const char *>(a.w_router + (size_t)task * a.H);
        for (int o = lane * 128; o < row_bytes; o += 32 * 128) prefetch_l2(r + o);
    }
    pdl_launch_dependents();
    pdl_wait();  // x (and the accumulator's last reader) come from the previous kernels
    if (a.acc) {
        // clear the fp32 accumulator K2 adds into
        for (int n = blockIdx.x * kK1Block + tid; n < a.H; n += gridDim.x * kK1Block) a.acc[n] = 0.f;
    }
    const uint4 *xg = reinterpret_cast<const uint4 *>(a.x);
    for (int i = tid; i < a.H / 8; i += kK1Block) xs[i] = xg[i];
    __syncthreads();
    if (task < a.E) {
        float s0 = 0.f;
        dot1_row(a.w_router + (size_t)task * a.H, xs, a.H, lane, s0);
        s0 = warp_sum(s0);
        if (lane == 0) a.logits[task] = s0 + (a.b_router ? a.b_router[task] : 0.f);
    }
}

// ---------------------------------------------------------------------- kernel 2 --
// Warp-level top-k over the E logits (value descending, index ascending on ties) and the
// renormalised softmax weights of the chosen k, into shared memory.  Lane L holds the logits
// e = L + 32*i (i < PER) in registers and sorts them once; each of the k rounds is a warp
// arg-max over the lanes' list heads, and the winner pops its head.  Ids are clamped into
// [0, E) so that a corrupted logit vector can never make the block read outside the weights.
template <int PER>
__device__ __forceinline__ void warp_topk_t(const float *logits, int E, int k, int *s_ids, float *s_w) {
    const int lane = threadIdx.x & 31;
    float v[PER];
    int id[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        id[i] = lane + 32 * i;
        v[i] = id[i] < E ? logits[id[i]] : -INFINITY;
    }
#pragma unroll
    for (int kk = 2; kk <= PER; kk <<= 1) {
#pragma unroll
        for (int j = kk >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    const bool l_first = v[l] > v[i] || (v[l] == v[i] && id[l] < id[i]);
                    if (((i & kk) == 0) ? l_first : !l_first) {
                        const float tv = v[i]; v[i] = v[l]; v[l] = tv;
                        const int ti = id[i]; id[i] = id[l]; id[l] = ti;
                    }
                }
            }
        }
    }
    float top = 0.f, my_val = 0.f;
    int my_id = 0;
    for (int r = 0; r < k; ++r) {
        // two warp reductions a round: the largest head, then the lowest expert index among
        // the lanes whose head equals it
        const uint32_t key = order_key(v[0]);
        const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
        const uint32_t cand = (key == mk && id[0] < E) ? (uint32_t)id[0] : 0xffffffffu;
        const uint32_t sel = __reduce_min_sync(0xffffffffu, cand);
        const float bv = key_value(mk);
        const int bi = (int)sel;
        if (sel != 0xffffffffu && (int)(sel & 31u) == lane) {
#pragma unroll
            for (int i = 0; i + 1 < PER; ++i) { v[i] = v[i + 1]; id[i] = id[i + 1]; }
            v[PER - 1] = -INFINITY;
            id[PER - 1] = 0x7fffffff;
        }
        if (r == 0) top = bv;
        if (lane == r) { my_val = bv; my_id = bi; }
    }
    const float ej = lane < k ? expf(my_val - top) : 0.f;
    const float s = warp_sum(ej);
    if (lane < k) {
        s_ids[lane] = (my_id >= 0 && my_id < E) ? my_id : 0;
        s_w[lane] = ej / s;
    }
}

// The same selection for E > 256 without holding the logits in registers: they are staged in
// shared memory (lg, E <= 1024) with a bitmask of the experts already chosen; each of the k
// rounds is a warp arg-max over the unchosen ones.
__device__ __noinline__ void warp_topk_smem(const float *logits, int E, int k, int *s_ids, float *s_w, float *lg,
                                            unsigned *chosen) {
    const int lane = threadIdx.x & 31;
    for (int e = lane; e < E; e += 32) lg[e] = logits[e];
    chosen[lane] = 0u;  // 32 words: 1024 experts
    __syncwarp();
    float top = 0.f, my_val = 0.f;
    int my_id = 0;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int e = lane; e < E; e += 32) {
            if ((chosen[e >> 5] >> (e & 31)) & 1u) continue;
            const float v = lg[e];
            if (v > bv || (v == bv && e < bi)) { bv = v; bi = e; }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0 && bi >= 0 && bi < E) chosen[bi >> 5] |= 1u << (bi & 31);
        __syncwarp();
        if (r == 0) top = bv;
        if (lane == r) { my_val = bv; my_id = bi; }
    }
    const float ej = lane < k ? expf(my_val - top) : 0.f;
    const float sum = warp_sum(ej);
    if (lane < k) {
        s_ids[lane] = (my_id >= 0 && my_id < E) ? my_id : 0;
        s_w[lane] = ej / sum;
    }
}

__device__ __forceinline__ void warp_topk(const float *logits, int E, int k, int *s_ids, float *s_w, float *lg,
                                          unsigned *chosen) {
    const int per = (E + 31) / 32;
    if (per <= 1) warp_topk_t<1>(logits, E, k, s_ids, s_w);
    else if (per <= 2) warp_topk_t<2>(logits, E, k, s_ids, s_w);
    else if (per <= 4) warp_topk_t<4>(logits, E, k, s_ids, s_w);
    else if (per <= 8) warp_topk_t<8>(logits, E, k, s_ids, s_w);
    else warp_topk_smem(logits, E, k, s_ids, s_w, lg, chosen);
}

// 96 registers a thread (512 threads: 48K of the SM's 64K) leave room for a K1 block of the next
// layer on the same SM, so the router spreads over the GPU instead of the few SMs K2 leaves idle.
__global__ void __maxnreg__(96)
    decode_k2_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap tm_down,
                     const __grid_constant__ CUtensorMap tm_sdown, int n_routed_blocks) {
    extern __shared__ uint8_t smem_raw[];
    // TMA destinations: align the dynamic shared memory up to 1024 bytes (the launch adds slack)
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint16_t *wd = reinterpret_cast<uint16_t *>(smem);                           // [kChunkRows][kSlice]
    uint4 *xs = reinterpret_cast<uint4 *>(smem + (size_t)kChunkRows * kSlice * 2);  // [H] bf16
    float *hsl = reinterpret_cast<float *>(xs + a.H / 8);                        // [kSlice] fp32
    __shared__ int s_ids[32];
    __shared__ float s_w[32];
    __shared__ float s_lg[1024];       // logits staging for E > 256
    __shared__ unsigned s_chosen[32];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_last;
    __shared__ int s_ok;
    __shared__ int s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool shared_task = (int)blockIdx.x >= n_routed_blocks;
    const int slices = a.I / kSlice;
    const int slot = shared_task ? 0 : (int)blockIdx.x / slices;
    const int i0 = shared_task ? ((int)blockIdx.x - n_routed_blocks) * kSlice : ((int)blockIdx.x % slices) * kSlice;
    const CUtensorMap *tm = shared_task ? &tm_sdown : &tm_down;
    if (tid == 0) {
        ptx::mbar_init(&bar, 1);
        s_ok = 1;
        s_abort = 0;
        ptx::fence_mbar_init();
        ptx::tma_prefetch_desc(tm);
    }
    pdl_launch_dependents();
    __syncthreads();
    // TMA of rows [r0, r0 + rows) of the slice's columns into shared memory, on `bar`; run by a
    // whole warp: lane 0 posts the byte count, then lane b issues box b (at most 16 boxes)
    constexpr int kLoadWarp = kK2Warps - 1;
    auto load_chunk = [&](int base_row, int r0, int rows) {
        if (lane == 0) ptx::mbar_arrive_expect_tx(&bar, (uint32_t)(rows * kSlice * 2));
        __syncwarp();
        if (lane < rows / kBoxRows)
            ptx::tma_load_2d(wd + (size_t)lane * kBoxRows * kSlice, tm, i0, base_row + r0 + lane * kBoxRows, &bar);
    };
    const int rows0 = a.H < kChunkRows ? a.H : kChunkRows;
    if (shared_task) {
        // the shared expert's weights do not depend on the routing: start its down columns
        // into shared memory and its gate/up rows into L2 before waiting for K1
        if (warp == kLoadWarp) load_chunk(0, 0, rows0);
        const int row_bytes = a.H * 2;
        for (int f = warp; f < kSlice; f += kK2Warps) {
            const char *g = reinterpret_cast<const char *>(a.ws_gate + (size_t)(i0 + f) * a.H);
            const char *u = reinterpret_cast<const char *>(a.ws_up + (size_t)(i0 + f) * a.H);
            for (int o = lane * 128; o < row_bytes; o += 32 * 128) {
                prefetch_l2(g + o);
                prefetch_l2(u + o);
            }
        }
    }
    pdl_wait();  // x, the logits and the cleared accumulator come after K1
    if (warp == 0 && !shared_task) warp_topk(a.logits, a.E, a.k, s_ids, s_w, s_lg, s_chosen);
    const uint4 *xg = reinterpret_cast<const uint4 *>(a.x);
    for (int i = tid; i < a.H / 8; i += kK2Threads) xs[i] = xg[i];
    __syncthreads();
    float wj = 1.f;
    int base_row = 0;  // first row of this block's weight matrix in the tensor map
    const uint16_t *wg = a.ws_gate, *wu = a.ws_up;  // shared expert: rows i0.. of [Is, H]
    if (!shared_task) {
        const int e = s_ids[slot];
        wj = s_w[slot];
        base_row = e * a.H;
        if (warp == kLoadWarp) load_chunk(base_row, 0, rows0);
        wg = a.w_gate + (size_t)e * a.I * a.H;
        wu = a.w_up + (size_t)e * a.I * a.H;
    }
    // h for features i0 .. i0+31: 16 warps x 2 features (gate and up rows)
    for (int f = warp; f < kSlice; f += kK2Warps) {
        const size_t row = (size_t)(i0 + f);
        float g = 0.f, u = 0.f;
        dot2_rows(wg + row * a.H, wu + row * a.H, xs, a.H, lane, g, u);
        g = warp_sum(g);
        u = warp_sum(u);
        if (lane == 0) hsl[f] = __bfloat162float(__float2bfloat16_rn(silu_mul(g, u)));
    }
    // split-K partial of the down projection, chunk by chunk: rows n of the chunk, 32 columns
    // each from shared memory (chunk order rotated per row against bank conflicts)
    for (int r0 = 0, ph = 0; r0 < a.H; r0 += kChunkRows, ph ^= 1) {
        const int rows = (a.H - r0) < kChunkRows ? (a.H - r0) : kChunkRows;
        if (tid == 0 && !ptx::mbar_wait(&bar, (uint32_t)ph, kWaitLimitNs, (volatile int *)&s_abort)) s_ok = 0;
        __syncthreads();
        if (!s_ok) break;
        // rows is a multiple of 128, so every warp runs the same number of iterations
        for (int n = tid; n < rows; n += kK2Threads) {
            const uint4 *rw = reinterpret_cast<const uint4 *>(wd + (size_t)n * kSlice);
            float acc = 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int c = (cc + (n >> 1)) & 3;
                const uint4 q = rw[c];
                const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float2 f = __bfloat1622float2(b[m]);
                    acc = fmaf(f.x, hsl[c * 8 + 2 * m], acc);
                    acc = fmaf(f.y, hsl[c * 8 + 2 * m + 1], acc);
                }
            }
            // lanes 4q..4q+3 hold rows n..n+3: one 16-byte reduction per four rows
            const float v1 = __shfl_down_sync(0xffffffffu, acc, 1);
            const float v2 = __shfl_down_sync(0xffffffffu, acc, 2);
            const float v3 = __shfl_down_sync(0xffffffffu, acc, 3);
            if ((lane & 3) == 0) ptx::red_add_v4(&a.acc[r0 + n], wj * acc, wj * v1, wj * v2, wj * v3);
        }
        __syncthreads();  // the chunk buffer is free again
        if (r0 + kChunkRows < a.H && warp == kLoadWarp) {
            const int next = (a.H - r0 - kChunkRows) < kChunkRows ? (a.H - r0 - kChunkRows) : kChunkRows;
            load_chunk(base_row, r0 + kChunkRows, next);
        }
    }
    if (!s_ok && tid == 0 && a.status) atomicCAS(a.status, 0, (int)MOE_ERR_TIMEOUT);
    // last block: every other block's adds are in the accumulator
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int ticket = atomicAdd(a.counter, 1);
        s_last = (ticket == (int)gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // four outputs a thread: one 16-byte accumulator load, 8-byte bf16 loads and stores
    for (int n4 = tid; n4 < a.H / 4; n4 += kK2Threads) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.acc) + n4);
        const float vv[4] = {v.x, v.y, v.z, v.w};
        uint16_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = bf16_bits(vv[q]);
        *reinterpret_cast<uint2 *>(a.out + 4 * n4) =
            make_uint2((uint32_t)o[0] | ((uint32_t)o[1] << 16), (uint32_t)o[2] | ((uint32_t)o[3] << 16));
        if (a.x_next) {
            const uint2 r = *reinterpret_cast<const uint2 *>(a.resid + 4 * n4);
            const uint16_t rr[4] = {(uint16_t)(r.x & 0xffffu), (uint16_t)(r.x >> 16), (uint16_t)(r.y & 0xffffu),
                                    (uint16_t)(r.y >> 16)};
            uint16_t xn[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) xn[q] = bf16_bits(bf16_to_f(rr[q]) + bf16_to_f(o[q]));
            *reinterpret_cast<uint2 *>(a.x_next + 4 * n4) =
                make_uint2((uint32_t)xn[0] | ((uint32_t)xn[1] << 16), (uint32_t)xn[2] | ((uint32_t)xn[3] << 16));
        }
    }
    if (tid == 0) atomicExch(a.counter, 0);
}

cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void **args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

size_t k2_smem(int H) { return 1024 + (size_t)kChunkRows * kSlice * 2 + (size_t)H * 2 + kSlice * 4; }

}  // namespace

int decode_slice() { return kSlice; }
int decode_box_rows() { return kBoxRows; }

cudaError_t launch_decode_router(const DecodeArgs &a, cudaStream_t s) {
    DecodeArgs r = a;
    r.acc = nullptr;  // router rows only, no accumulator to clear
    LaunchScope scope(KC_DECODE_ROUTER, s);
    decode_k1_kernel<<<(r.E + kK1Warps - 1) / kK1Warps, kK1Block, (size_t)r.H * 2, s>>>(r);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &tm_down, const CUtensorMap &tm_sdown,
                          cudaStream_t s) {
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        // largest supported H (16384): 128 KB of slice columns + 32 KB of x
        cudaError_t e = cudaFuncSetAttribute(decode_k2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)k2_smem(16384));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(decode_k1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 32 * 1024);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    {
        DecodeArgs k1 = a;
        const int tasks = a.E;
        void *args[] = {&k1};
        LaunchScope scope(KC_DECODE_ROUTER, s);
        const cudaError_t e = launch_pdl(reinterpret_cast<const void *>(decode_k1_kernel),
                                         dim3((tasks + kK1Warps - 1) / kK1Warps), dim3(kK1Block),
                                         (size_t)a.H * 2, s, args);
        if (e != cudaSuccess) return e;
    }
    {
        DecodeArgs k2 = a;
        int n_routed = a.k * (a.I / kSlice);
        const int blocks = n_routed + a.Is / kSlice;
        CUtensorMap m0 = tm_down, m1 = tm_sdown;
        void *args[] = {&k2, &m0, &m1, &n_routed};
        LaunchScope scope(KC_DECODE_EXPERTS, s);
        return launch_pdl(reinterpret_cast<const void *>(decode_k2_kernel), dim3(blocks), dim3(kK2Threads),
                          k2_smem(a.H), s, args);
    }
}

}  // namespace moe
