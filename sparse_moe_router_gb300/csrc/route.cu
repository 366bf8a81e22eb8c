// route.cu -- router softmax/top-k/renormalise, the stable expert permutation, and the
// elementwise kernels (finalise, unfused combine, clear).
//
// Top-k routing ("AI MAX+ 395部署Qwen3大模型：GFX1151引擎实测优化解析", explanatory MoE
// paragraph under "MOE 内核优化": each token activates only a few of many experts) is taken
// on the fp32 logits: the k largest, lower expert index first on equal values, in descending
// order; the weights are the softmax over all E logits renormalised over the k chosen, which
// equals exp(l_j - m) / sum_i exp(l_i - m) over the chosen.
#include <cuda_bf16.h>
#include <float.h>

#include <mutex>

#include "internal.h"

namespace moe {
namespace {

// ------------------------------------------------------------------------ top-k --
// One warp per token.  Lane L holds the logits e = L + 32*i (i < PER_LANE) and first sorts
// them (bitonic network on the total order: value descending, index ascending).  Each of the
// k rounds is then a warp arg-max over the lanes' list heads only; the winning lane pops its
// head.  The order makes ties go to the lower expert index.
template <int N>
__device__ __forceinline__ void sort_desc(float (&v)[N], int (&e)[N]) {
#pragma unroll
    for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    const bool l_first = v[l] > v[i] || (v[l] == v[i] && e[l] < e[i]);
                    const bool swap = ((i & k) == 0) ? l_first : !l_first;
                    if (swap) {
                        const float tv = v[i]; v[i] = v[l]; v[l] = tv;
                        const int te = e[i]; e[i] = e[l]; e[l] = te;
                    }
                }
            }
        }
    }
}

// One token's selection (the warp's): sort, k rounds, the renormalised weights.
template <int PER_LANE, bool HIST>
__device__ __forceinline__ void topk_one(const float *__restrict__ l, int E, int k, int32_t *__restrict__ ids_t,
                                         float *__restrict__ w_t, int lane, int *s_hist) {
    float v[PER_LANE];
    int e[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        e[i] = lane + 32 * i;
        v[i] = e[i] < E ? __ldg(&l[e[i]]) : -INFINITY;
    }
    sort_desc<PER_LANE>(v, e);
    float my_val = 0.f, top = 0.f;
    int my_id = 0;
    for (int r = 0; r < k; ++r) {
        // the largest head, then the lowest expert index among the lanes holding it (padding,
        // e >= E, never wins)
        const uint32_t key = order_key(v[0]);
        const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
        const uint32_t cand = (key == mk && e[0] < E) ? (uint32_t)e[0] : 0xffffffffu;
        const uint32_t sel = __reduce_min_sync(0xffffffffu, cand);
        const float bv = key_value(mk);
        const int bi = (int)sel;
        if (sel != 0xffffffffu && (int)(sel & 31u) == lane) {  // pop the head of the winner's list
#pragma unroll
            for (int i = 0; i + 1 < PER_LANE; ++i) {
                v[i] = v[i + 1];
                e[i] = e[i + 1];
            }
            v[PER_LANE - 1] = -INFINITY;
            e[PER_LANE - 1] = 0x7fffffff;
        }
        if (r == 0) top = bv;
        if (lane == r) {
            my_val = bv;
            my_id = bi;
        }
    }
    const float ej = lane < k ? expf(my_val - top) : 0.f;
    float s = ej;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane < k) {
        ids_t[lane] = my_id;
        w_t[lane] = ej / s;
        if (HIST && my_id >= 0 && my_id < E) atomicAdd(&s_hist[my_id], 1);
    }
}

// HIST: the block's 8 tokens' expert counts are also added into row (8 * block) / CT of chunk_tab
// (a table of zeros before the launch), the chunk counts the permutation starts from.
template <int PER_LANE, bool HIST>
__global__ void __launch_bounds__(256) topk_kernel(const float *__restrict__ logits, int T, int E,
                                                   int k, int32_t *__restrict__ ids,
                                                   float *__restrict__ w, int32_t *__restrict__ chunk_tab,
                                                   int CT) {
    extern __shared__ int s_hist[];  // HIST: [E]
    const int warp = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (HIST) {
        for (int i = threadIdx.x; i < E; i += blockDim.x) s_hist[i] = 0;
        __syncthreads();
    }
    if (warp < T) topk_one<PER_LANE, HIST>(logits + (size_t)warp * E, E, k, ids + (size_t)warp * k,
                                           w + (size_t)warp * k, lane, s_hist);
    if (HIST) {
        __syncthreads();
        const int chunk = (int)(blockIdx.x * (blockDim.x >> 5)) / CT;
        for (int i = threadIdx.x; i < E; i += blockDim.x) {
            const int c = s_hist[i];
            if (c) atomicAdd(&chunk_tab[(size_t)chunk * E + i], c);
        }
    }
}


// --------------------------------------------------------------------- permute --
// Stable counting sort of the P = T*k pairs by expert, with no block ever waiting on another.
// Chunk c is the pairs of tokens [c*CT, (c+1)*CT) (CT = perm_chunk_tokens(k), CP = CT*k pairs).
// In three launches (moe_permute):
//   1. perm_hist:    block c counts the experts of its chunk;
//   2. perm_scan:    one block: per expert (a group of adjacent lanes, each summing a range
//                    of chunks), the exclusive prefix over chunks, then the exclusive prefix
//                    over experts (the offsets) and the token-tile prefix;
//                    the chunk table now holds each chunk's first row per expert;
//   3. perm_scatter: block c walks its chunk again; warp w owns pairs [64w, 64w+64) of the
//                    chunk, per-warp counts give each warp its first row per expert, and a
//                    pair's rank among equal ids earlier in its 32-pair batch (match_any)
//                    finishes its row.
// Inside a layer (moe_forward) the counts come from the top-k kernel itself (its 8-token blocks
// add them into a table the router GEMM zeroed), and one launch, perm_scan_scatter, does the
// rest: each block derives its own chunk's first rows from the whole table (a few KB) instead
// of waiting for a separate scan.
// Pairs of one expert therefore keep increasing pair order: the result is bit-exact.
constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;
static_assert(kPermChunk == 64 * kPermWarps, "the scatter gives each warp two 32-pair batches");

__device__ __forceinline__ int block_excl_scan(int v, int *sh_warp, int *total) {
    // exclusive scan of one value per thread across the 1024-thread block
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) sh_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = sh_warp[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        sh_warp[lane] = s;  // inclusive
    }
    __syncthreads();
    const int base = wid > 0 ? sh_warp[wid - 1] : 0;
    const int incl = base + x;
    *total = sh_warp[31];
    __syncthreads();
    return incl - v;
}

__global__ void __launch_bounds__(kPermThreads) perm_hist_kernel(const int32_t *__restrict__ ids, int P,
                                                                  int E, int CP, int32_t *__restrict__ chunk_tab,
                                                                  int *status) {
    extern __shared__ int cnt[];  // [E]
    const int tid = threadIdx.x;
    for (int i = tid; i < E; i += kPermThreads) cnt[i] = 0;
    __syncthreads();
    const int beg = blockIdx.x * CP;
    for (int p = beg + tid; p < min(P, beg + CP); p += kPermThreads) {
        const int e = __ldg(&ids[p]);
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else if (status) atomicCAS(status, 0, (int)MOE_ERR_INVALID_ARG);
    }
    __syncthreads();
    for (int i = tid; i < E; i += kPermThreads) chunk_tab[(size_t)blockIdx.x * E + i] = cnt[i];
}

__global__ void __launch_bounds__(kPermThreads, 1)
    perm_scan_kernel(int32_t *__restrict__ chunk_tab, int n_chunks, int E, int32_t *__restrict__ offsets,
                     int32_t *__restrict__ tile_prefix, int tile_n, int extra_rows, int *__restrict__ sched) {
    __shared__ int sh_warp[32];
    const int tid = threadIdx.x;
    // the grouped GEMMs' tile counters (gate/up, down) start at zero for the launches that follow
    if (sched && tid < kSchedCounters) sched[tid] = 0;
    // tpe adjacent lanes per expert (a power of two <= 32 with E * tpe <= 1024); lane `sub` of
    // expert e owns chunks [c0, c1) of e's column of the table
    int tpe = 1;
    while (tpe < 32 && E * tpe * 2 <= kPermThreads) tpe *= 2;
    const int e = tid / tpe, sub = tid % tpe;
    const bool live = e < E;
    const int cpt = (n_chunks + tpe - 1) / tpe;
    const int c0 = sub * cpt, c1 = min(n_chunks, c0 + cpt);
    // pass 1: this lane's share of expert e's count, eight loads in flight
    int part = 0;
    if (live)
        for (int c = c0; c < c1; c += 8) {
            int h[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) h[u] = (c + u < c1) ? chunk_tab[(size_t)(c + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) part += h[u];
        }
    // the lanes' exclusive prefix within the expert, and the expert's total
    int incl = part;
    for (int d = 1; d < tpe; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d, tpe);
        if (sub >= d) incl += y;
    }
    const int excl = incl - part;
    const int cnt = __shfl_sync(0xffffffffu, incl, tpe - 1, tpe);
    // offsets over experts (the first lane of each group carries its expert's count)
    int total = 0;
    const int off_first = block_excl_scan((live && sub == 0) ? cnt : 0, sh_warp, &total);
    const int off = __shfl_sync(0xffffffffu, off_first, 0, tpe);
    const int tiles = (live && sub == 0) ? token_tile_count(cnt) : 0;
    int total_tiles = 0;
    const int toff = block_excl_scan(tiles, sh_warp, &total_tiles);
    if (live && sub == 0) {
        offsets[e] = off;
        if (tile_prefix) tile_prefix[e] = toff;
    }
    if (tid == 0) {
        offsets[E] = total;
        if (tile_prefix) tile_prefix[E] = total_tiles;
        if (extra_rows > 0) {  // one more group after the experts
            offsets[E + 1] = total + extra_rows;
            if (tile_prefix) tile_prefix[E + 1] = total_tiles + token_tile_count(extra_rows);
        }
    }
    // pass 2: each chunk's first row for expert e
    if (live) {
        int run = off + excl;
        for (int c = c0; c < c1; c += 8) {
            int h[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) h[u] = (c + u < c1) ? chunk_tab[(size_t)(c + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c + u < c1) {
                    chunk_tab[(size_t)(c + u) * E + e] = run;
                    run += h[u];
                }
        }
    }
}

// Block-wide scatter of chunk c's pairs [beg, end): base_e[e] is the first row of the chunk's
// pairs of expert e; wh is shared memory for kPermWarps * E ints.  Warp w owns pairs
// beg + [64w, 64w + 64); per-warp counts give each warp its first row per expert, and a pair's
// rank among equal ids earlier in its 32-pair batch (match_any) finishes its row.
__device__ __forceinline__ void scatter_chunk(const int32_t *__restrict__ ids, int P, int E, int k, int beg,
                                              int end, const int32_t *base_e, int *wh,
                                              int32_t *__restrict__ perm, int32_t *__restrict__ inv,
                                              const float *__restrict__ topk_w, int32_t *__restrict__ row_tok,
                                              float *__restrict__ row_w, int *status) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    for (int i = tid; i < kPermWarps * E; i += kPermThreads) wh[i] = 0;
    const int base = beg + wid * (kPermChunk / kPermWarps);
    const uint32_t lt_mask = (1u << lane) - 1u;
    int e2[2];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int p = base + 32 * b + lane;
        int e = p < end ? __ldg(&ids[p]) : -1;
        if (e >= E) e = -1;
        e2[b] = e;
    }
    __syncthreads();
    int *my = wh + wid * E;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const uint32_t grp = __match_any_sync(0xffffffffu, e2[b]);
        if (e2[b] >= 0 && (grp & lt_mask) == 0) my[e2[b]] += __popc(grp);
        __syncwarp();
    }
    __syncthreads();
    // per expert: first row of each warp's pairs = chunk's first row + earlier warps' counts
    for (int e = tid; e < E; e += kPermThreads) {
        int run = base_e[e];
        for (int w2 = 0; w2 < kPermWarps; ++w2) {
            const int c = wh[w2 * E + e];
            wh[w2 * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int p = base + 32 * b + lane;
        const int e = e2[b];
        const uint32_t grp = __match_any_sync(0xffffffffu, e);
        int row = -1;
        if (e >= 0) row = my[e] + __popc(grp & lt_mask);
        __syncwarp();
        if (e >= 0 && (grp & lt_mask) == 0) my[e] += __popc(grp);
        __syncwarp();
        if (p < end) {
            if (row >= 0 && !MOE_DEBUG_OK(row < P, status)) row = -1;  // a corrupt count table
            inv[p] = row;
            if (row >= 0) {
                perm[row] = p;
                if (row_tok) row_tok[row] = p / k;
                if (row_w) row_w[row] = __ldg(&topk_w[p]);
            }
        }
    }
}

__global__ void __launch_bounds__(kPermThreads) perm_scatter_kernel(const int32_t *__restrict__ ids, int P,
                                                                     int E, int k, int CP,
                                                                     const int32_t *__restrict__ chunk_tab,
                                                                     int32_t *__restrict__ perm,
                                                                     int32_t *__restrict__ inv,
                                                                     const float *__restrict__ topk_w,
                                                                     int32_t *__restrict__ row_tok,
                                                                     float *__restrict__ row_w, int *status) {
    extern __shared__ int wh[];  // [kPermWarps][E]
    const int beg = blockIdx.x * CP;
    scatter_chunk(ids, P, E, k, beg, min(P, beg + CP), chunk_tab + (size_t)blockIdx.x * E, wh, perm, inv, topk_w,
                  row_tok, row_w, status);
}

// The scan and the scatter in one launch, from the chunk table of counts (read only).  Block c:
// per expert e (a group of tpe adjacent lanes, each summing a range of chunks) the total and the
// count in chunks before c; the exclusive prefix over experts of the totals (the offsets); then
// the first row of chunk c for e is offset_e + the count before c, and the chunk is scattered.
// Block 0 also writes the offsets, the token-tile prefix (with one more group of extra_rows
// after the experts, when asked) and zeroes the grouped GEMMs' tile counters.
__global__ void __launch_bounds__(kPermThreads, 1)
    perm_scan_scatter_kernel(const int32_t *__restrict__ chunk_tab, int n_chunks, const int32_t *__restrict__ ids,
                             int P, int E, int k, int CP, int32_t *__restrict__ offsets,
                             int32_t *__restrict__ tile_prefix, int extra_rows, int *__restrict__ sched,
                             int32_t *__restrict__ perm, int32_t *__restrict__ inv,
                             const float *__restrict__ topk_w, int32_t *__restrict__ row_tok,
                             float *__restrict__ row_w, int *status) {
    extern __shared__ int sm[];  // wh [kPermWarps][E], then the chunk's first rows [E]
    int *wh = sm, *sbase = sm + kPermWarps * E;
    __shared__ int sh_warp[32];
    const int tid = threadIdx.x, c = (int)blockIdx.x;
    if (c == 0 && sched && tid < kSchedCounters) sched[tid] = 0;
    int tpe = 1;
    while (tpe < 32 && E * tpe * 2 <= kPermThreads) tpe *= 2;
    const int e = tid / tpe, sub = tid % tpe;
    const bool live = e < E;
    const int cpt = (n_chunks + tpe - 1) / tpe;
    const int c0 = sub * cpt, c1 = min(n_chunks, c0 + cpt);
    int part = 0, before = 0;
    if (live)
        for (int cc = c0; cc < c1; cc += 8) {
            int h[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) h[u] = (cc + u < c1) ? chunk_tab[(size_t)(cc + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                part += h[u];
                if (cc + u < c) before += h[u];
            }
        }
    for (int d = 1; d < tpe; d <<= 1) {
        part += __shfl_xor_sync(0xffffffffu, part, d, tpe);
        before += __shfl_xor_sync(0xffffffffu, before, d, tpe);
    }
    int total = 0;
    const int off_first = block_excl_scan((live && sub == 0) ? part : 0, sh_warp, &total);
    if (live && sub == 0) sbase[e] = off_first + before;
    if (c == 0) {
        const int tiles = (live && sub == 0) ? token_tile_count(part) : 0;
        int total_tiles = 0;
        const int toff = block_excl_scan(tiles, sh_warp, &total_tiles);
        if (live && sub == 0) {
            offsets[e] = off_first;
            if (tile_prefix) tile_prefix[e] = toff;
        }
        if (tid == 0) {
            offsets[E] = total;
            if (tile_prefix) tile_prefix[E] = total_tiles;
            if (extra_rows > 0) {
                offsets[E + 1] = total + extra_rows;
                if (tile_prefix) tile_prefix[E + 1] = total_tiles + token_tile_count(extra_rows);
            }
        }
    }
    __syncthreads();
    const int beg = c * CP;
    scatter_chunk(ids, P, E, k, beg, min(P, beg + CP), sbase, wh, perm, inv, topk_w, row_tok, row_w, status);
}

// Token-tile prefix from given offsets (for the unfused expert entry point).
__global__ void __launch_bounds__(kPermThreads, 1)
    tile_prefix_kernel(const int32_t *__restrict__ offsets, int E, int32_t *__restrict__ tile_prefix,
                       int tile_n, const int32_t *__restrict__ perm, int P, int k,
                       int32_t *__restrict__ row_tok, int *__restrict__ sched, int *status) {
    __shared__ int sh_warp[32];
    const int tid = threadIdx.x;
    if (sched && tid < kSchedCounters) sched[tid] = 0;
    for (int r = tid; r < P; r += kPermThreads) {
        const int pr = perm[r];
        row_tok[r] = MOE_DEBUG_OK(pr >= 0 && pr < P, status) ? pr / k : -1;  // -1: a zero row
    }
    int cnt = tid < E ? offsets[tid + 1] - offsets[tid] : 0;
    // the caller's offsets: non-decreasing, from 0 to at most P (else no rows for this expert)
    if (tid < E && !MOE_DEBUG_OK(cnt >= 0 && offsets[tid] >= 0 && offsets[tid + 1] <= P, status)) cnt = 0;
    const int tiles = tid < E ? token_tile_count(cnt) : 0;
    int total = 0;
    const int toff = block_excl_scan(tiles, sh_warp, &total);
    if (tid < E) tile_prefix[tid] = toff;
    if (tid == 0) tile_prefix[E] = total;
}

// ------------------------------------------------------------------- finalise --
// out[t] = bf16( sum_j y[t*k+j] + acc[t] ) in fp32 (slots in order, then the shared term);
// x_next = bf16(resid + out).  8 features per thread (H % 8 == 0): the k bf16 rows of a
// token are adjacent, so every load is a 16-byte coalesced read.
__global__ void __launch_bounds__(256) finalize_kernel(const uint16_t *__restrict__ y, int k,
                                                       const uint16_t *__restrict__ y_tail,
                                                       const float *__restrict__ acc,
                                                       const uint16_t *resid, int H8, size_t n8,
                                                       uint16_t *__restrict__ out,
                                                       uint16_t *x_next) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        const size_t t = i / H8, c = i % H8;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint4 *yr = reinterpret_cast<const uint4 *>(y) + (t * k) * H8 + c;
        // the weighted rows are read once: evict-first loads leave L2 to the data read again
        for (int j = 0; j < k; ++j) {
            const uint4 q = __ldcs(yr + (size_t)j * H8);
            const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 f = __bfloat1622float2(b[m]);
                v[2 * m] += f.x;
                v[2 * m + 1] += f.y;
            }
        }
        if (y_tail) {
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(y_tail) + i);
            const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 f = __bfloat1622float2(b[m]);
                v[2 * m] += f.x;
                v[2 * m + 1] += f.y;
            }
        }
        if (acc) {
            const float4 a0 = __ldg(reinterpret_cast<const float4 *>(acc) + 2 * i);
            const float4 a1 = __ldg(reinterpret_cast<const float4 *>(acc) + 2 * i + 1);
            v[0] += a0.x; v[1] += a0.y; v[2] += a0.z; v[3] += a0.w;
            v[4] += a1.x; v[5] += a1.y; v[6] += a1.z; v[7] += a1.w;
        }
        __align__(16) __nv_bfloat16 o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = __float2bfloat16_rn(v[j]);
        // out is not read again in a layer stack (x_next is): a streaming store
        __stcs(reinterpret_cast<uint4 *>(out) + i, *reinterpret_cast<const uint4 *>(o));
        if (x_next) {
            const uint4 xr = reinterpret_cast<const uint4 *>(resid)[i];
            const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(&xr);
            __align__(16) __nv_bfloat16 n[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                n[j] = __float2bfloat16_rn(__bfloat162float(xb[j]) + __bfloat162float(o[j]));
            reinterpret_cast<uint4 *>(x_next)[i] = *reinterpret_cast<const uint4 *>(n);
        }
    }
}

// ---------------------------------------------------------------- unfused combine --
// out[t, n] = bf16( sum_j w[t,j] * y_rows[inv[t*k+j], n] + shared_y[t, n] ), slot order.
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ y_rows,
                                                      const int32_t *__restrict__ inv,
                                                      const float *__restrict__ topk_w,
                                                      const float *__restrict__ shared_y, int T,
                                                      int H, int k, uint16_t *__restrict__ out) {
    const int H4 = H / 4;
    const size_t n = (size_t)T * H4;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / H4), c = (int)(i % H4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int row = __ldg(&inv[(size_t)t * k + j]);
            if (row < 0 || !MOE_DEBUG_OK(row < T * k, nullptr)) continue;
            const float wj = __ldg(&topk_w[(size_t)t * k + j]);
            const float4 y = __ldg(reinterpret_cast<const float4 *>(y_rows + (size_t)row * H) + c);
            acc.x += wj * y.x;
            acc.y += wj * y.y;
            acc.z += wj * y.z;
            acc.w += wj * y.w;
        }
        if (shared_y) {
            const float4 s = __ldg(reinterpret_cast<const float4 *>(shared_y + (size_t)t * H) + c);
            acc.x += s.x;
            acc.y += s.y;
            acc.z += s.z;
            acc.w += s.w;
        }
        __align__(8) __nv_bfloat16 o[4] = {__float2bfloat16_rn(acc.x), __float2bfloat16_rn(acc.y),
                                           __float2bfloat16_rn(acc.z), __float2bfloat16_rn(acc.w)};
        reinterpret_cast<uint2 *>(out + (size_t)t * H)[c] = *reinterpret_cast<const uint2 *>(o);
    }
}

__global__ void __launch_bounds__(256) zero_kernel(float4 *__restrict__ p, size_t n4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

int grid_for(size_t work, int per_block) {
    const DeviceInfo &di = device_info();
    size_t b = (work + per_block - 1) / per_block;
    const size_t cap = (size_t)di.sm_count * 8;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return (int)b;
}

}  // namespace

namespace {
template <bool HIST>
cudaError_t topk_launch(const float *logits, int T, int E, int k, int32_t *ids, float *w, int32_t *chunk_tab,
                        cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int blocks = (T + 7) / 8;  // 8 warps (tokens) per block
    const size_t smem = HIST ? (size_t)E * sizeof(int) : 0;
    const int ct = perm_chunk_tokens(k);
    LaunchScope scope(KC_TOPK, s);
    const int per = (E + 31) / 32;
    if (per <= 1) topk_kernel<1, HIST><<<blocks, 256, smem, s>>>(logits, T, E, k, ids, w, chunk_tab, ct);
    else if (per <= 2) topk_kernel<2, HIST><<<blocks, 256, smem, s>>>(logits, T, E, k, ids, w, chunk_tab, ct);
    else if (per <= 4) topk_kernel<4, HIST><<<blocks, 256, smem, s>>>(logits, T, E, k, ids, w, chunk_tab, ct);
    else if (per <= 8) topk_kernel<8, HIST><<<blocks, 256, smem, s>>>(logits, T, E, k, ids, w, chunk_tab, ct);
    else if (per <= 16) topk_kernel<16, HIST><<<blocks, 256, smem, s>>>(logits, T, E, k, ids, w, chunk_tab, ct);
    else topk_kernel<32, HIST><<<blocks, 256, smem, s>>>(logits, T, E, k, ids, w, chunk_tab, ct);
    return cudaGetLastError();
}

// the permutation kernels' shared-memory opt-in, once per device (under a lock: two host threads'
// first calls would otherwise race on the flag)
cudaError_t perm_attrs() {
    static bool attr_done[64] = {false};
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(kPermWarps * 1024 * sizeof(int)));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(perm_scan_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)((kPermWarps + 1) * 1024 * sizeof(int)));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w, cudaStream_t s) {
    return topk_launch<false>(logits, T, E, k, ids, w, nullptr, s);
}

cudaError_t launch_topk_hist(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                             int32_t *chunk_tab, cudaStream_t s) {
    return topk_launch<true>(logits, T, E, k, ids, w, chunk_tab, s);
}

size_t permute_scratch_ints(int T, int E, int k) {
    const int ct = perm_chunk_tokens(k);
    return (size_t)(((long)T + ct - 1) / ct) * E;
}

cudaError_t launch_permute(const int32_t *ids, int T, int E, int k, int32_t *offsets,
                           int32_t *perm, int32_t *inv, int32_t *tile_prefix, int tile_n,
                           int32_t *chunk_tab, const float *topk_w, int32_t *row_tok,
                           float *row_w, int *status, cudaStream_t s, int extra_rows, int *sched) {
    const int P = T * k;
    const int ct = perm_chunk_tokens(k), cp = ct * k;
    const int n_chunks = (T + ct - 1) / ct;
    cudaError_t e = perm_attrs();
    if (e != cudaSuccess) return e;
    {
        LaunchScope scope(KC_PERMUTE, s);
        perm_hist_kernel<<<n_chunks, kPermThreads, E * sizeof(int), s>>>(ids, P, E, cp, chunk_tab, status);
    }
    {
        LaunchScope scope(KC_PERMUTE, s);
        perm_scan_kernel<<<1, kPermThreads, 0, s>>>(chunk_tab, n_chunks, E, offsets, tile_prefix, tile_n,
                                                    extra_rows, sched);
    }
    LaunchScope scope(KC_PERMUTE, s);
    perm_scatter_kernel<<<n_chunks, kPermThreads, kPermWarps * E * sizeof(int), s>>>(
        ids, P, E, k, cp, chunk_tab, perm, inv, topk_w, row_tok, row_w, status);
    return cudaGetLastError();
}

cudaError_t launch_scan_scatter(const int32_t *ids, int T, int E, int k, int32_t *offsets, int32_t *perm,
                                int32_t *inv, int32_t *tile_prefix, const int32_t *chunk_tab,
                                const float *topk_w, int32_t *row_tok, float *row_w, int *status,
                                cudaStream_t s, int extra_rows, int *sched) {
    const int P = T * k;
    const int ct = perm_chunk_tokens(k), cp = ct * k;
    const int n_chunks = (T + ct - 1) / ct;
    cudaError_t e = perm_attrs();
    if (e != cudaSuccess) return e;
    LaunchScope scope(KC_PERMUTE, s);
    perm_scan_scatter_kernel<<<n_chunks, kPermThreads, (kPermWarps + 1) * E * sizeof(int), s>>>(
        chunk_tab, n_chunks, ids, P, E, k, cp, offsets, tile_prefix, extra_rows, sched, perm, inv, topk_w, row_tok,
        row_w, status);
    return cudaGetLastError();
}

cudaError_t launch_tile_prefix(const int32_t *offsets, int E, int32_t *tile_prefix, int tile_n,
                               const int32_t *perm, int P, int k, int32_t *row_tok,
                               cudaStream_t s, int *sched, int *status) {
    LaunchScope scope(KC_TILE_PREFIX, s);
    tile_prefix_kernel<<<1, kPermThreads, 0, s>>>(offsets, E, tile_prefix, tile_n, perm, P, k, row_tok, sched,
                                                  status);
    return cudaGetLastError();
}

// One warp per expert-sorted row: 16-byte loads of the token's row, four in flight per lane.
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const uint4 *__restrict__ x, int T, const int32_t *__restrict__ row_tok, int P,
                       int n_tail, int H8, uint4 *__restrict__ xp) {
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < P + n_tail; r += gridDim.x * wpb) {
        const int t = r < P ? __ldg(&row_tok[r]) : r - P;
        uint4 *dst = xp + (size_t)r * H8;
        if (t < 0 || t >= T) {
            for (int i = lane; i < H8; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
            continue;
        }
        const uint4 *src = x + (size_t)t * H8;
        int i = lane;
        // x is read k times and stays in L2; the copies (k times its size) are written with
        // streaming stores so that they do not push it out
        for (; i + 224 < H8; i += 256) {  // eight 16-byte loads a lane in flight (a 4 KB row per warp)
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldg(&src[i + 32 * u]);
#pragma unroll
            for (int u = 0; u < 8; ++u) __stcs(&dst[i + 32 * u], v[u]);
        }
        for (; i < H8; i += 32) __stcs(&dst[i], __ldg(&src[i]));
    }
}

cudaError_t launch_gather_rows(const uint16_t *x, int T, int H, const int32_t *row_tok, int P,
                               uint16_t *xp, cudaStream_t s, int n_tail) {
    if (P + n_tail <= 0) return cudaSuccess;
    LaunchScope scope(KC_GATHER_X, s);
    gather_rows_kernel<<<grid_for((size_t)(P + n_tail), 8), 256, 0, s>>>(
        reinterpret_cast<const uint4 *>(x), T, row_tok, P, n_tail, H / 8, reinterpret_cast<uint4 *>(xp));
    return cudaGetLastError();
}

cudaError_t launch_finalize(const uint16_t *y, int k, const float *acc, const uint16_t *resid, int T,
                            int H, uint16_t *out, uint16_t *x_next, cudaStream_t s, const uint16_t *y_tail) {
    const size_t n8 = (size_t)T * H / 8;
    if (n8 == 0) return cudaSuccess;
    LaunchScope scope(KC_FINALIZE, s);
    finalize_kernel<<<grid_for(n8, 256), 256, 0, s>>>(y, k, y_tail, acc, resid, H / 8, n8, out, x_next);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float *y_rows, const int32_t *inv, const float *topk_w,
                           const float *shared_y, int T, int H, int k, uint16_t *out,
                           cudaStream_t s) {
    const size_t n = (size_t)T * (H / 4);
    if (n == 0) return cudaSuccess;
    LaunchScope scope(KC_COMBINE, s);
    combine_kernel<<<grid_for(n, 256), 256, 0, s>>>(y_rows, inv, topk_w, shared_y, T, H, k, out);
    return cudaGetLastError();
}

bool debug_build() {
#ifdef MOE_DEBUG
    return true;
#else
    return false;
#endif
}

cudaError_t launch_zero(float *p, size_t n, cudaStream_t s) {
    const size_t n4 = n / 4;
    if (n4 == 0) return cudaSuccess;
    LaunchScope scope(KC_ZERO, s);
    zero_kernel<<<grid_for(n4, 256), 256, 0, s>>>(reinterpret_cast<float4 *>(p), n4);
    return cudaGetLastError();
}

}  // namespace moe
