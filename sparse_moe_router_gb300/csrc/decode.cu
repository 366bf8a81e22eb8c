// decode.cu -- the single-token (T = 1) layer: every weight byte the token needs is streamed
// from HBM once with 128-bit loads (or TMA), fp32 accumulation.  A bf16 product is taken by the
// mixed-precision FMA (bf16 x bf16 into an fp32 sum), with no widening of the operands first.
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
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

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

// c + a * b for bf16 halves of two 32-bit words (HA, HB: 0 low, 1 high), in fp32 with one
// rounding.  A product of two bf16 values is exact in fp32, so this is fmaf on the widened values.
template <int HA, int HB>
__device__ __forceinline__ float fma_bf16h(uint32_t a2, uint32_t b2, float c) {
    float d;
    if constexpr (HA == 0 && HB == 0)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a0, b0, %3;\n\t}" : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    else if constexpr (HA == 0)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a0, b1, %3;\n\t}" : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    else if constexpr (HB == 0)
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a1, b0, %3;\n\t}" : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    else
        asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
            "fma.rn.f32.bf16 %0, a1, b1, %3;\n\t}" : "=f"(d) : "r"(a2), "r"(b2), "f"(c));
    return d;
}

// 8 bf16 weights against 8 bf16 values, in order, fp32 sums
__device__ __forceinline__ float dot8(const uint4 &w, const uint4 &x) {
    float acc = 0.f;
    acc = fma_bf16h<0, 0>(w.x, x.x, acc);
    acc = fma_bf16h<1, 1>(w.x, x.x, acc);
    acc = fma_bf16h<0, 0>(w.y, x.y, acc);
    acc = fma_bf16h<1, 1>(w.y, x.y, acc);
    acc = fma_bf16h<0, 0>(w.z, x.z, acc);
    acc = fma_bf16h<1, 1>(w.z, x.z, acc);
    acc = fma_bf16h<0, 0>(w.w, x.w, acc);
    acc = fma_bf16h<1, 1>(w.w, x.w, acc);
    return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// The same for up to NT token vectors: token i of the list is xs + tl[i] * n16 (n of them).
// One row load feeds every token; U loads per row stay in flight.
template <int NT>
__device__ __forceinline__ void dot2_rows_t(const uint16_t *r0, const uint16_t *r1, const uint4 *xs, int n16,
                                            int lane, const int *tl, int n, float (&a0)[NT], float (&a1)[NT]) {
    constexpr int U = 8;
    const uint4 *p0 = reinterpret_cast<const uint4 *>(r0);
    const uint4 *p1 = reinterpret_cast<const uint4 *>(r1);
    int c = lane;
    for (; c + 32 * (U - 1) < n16; c += 32 * U) {
        uint4 w0[U], w1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            w0[u] = ld_stream(p0 + c + 32 * u);
            w1[u] = ld_stream(p1 + c + 32 * u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int t = 0; t < NT; ++t)
                if (t < n) {
                    const uint4 xv = xs[tl[t] * n16 + c + 32 * u];
                    a0[t] += dot8(w0[u], xv);
                    a1[t] += dot8(w1[u], xv);
                }
    }
    for (; c < n16; c += 32) {
        const uint4 w0 = ld_stream(p0 + c), w1 = ld_stream(p1 + c);
#pragma unroll
        for (int t = 0; t < NT; ++t)
            if (t < n) {
                const uint4 xv = xs[tl[t] * n16 + c];
                a0[t] += dot8(w0, xv);
                a1[t] += dot8(w1, xv);
            }
    }
}

// One row against the first n (<= NT) token vectors of xs (token t at xs + t * n16).
template <int NT>
__device__ __forceinline__ void dot1_row_t(const uint16_t *r0, const uint4 *xs, int n16, int lane, int n,
                                           float (&a0)[NT]) {
    constexpr int U = NT == 1 ? 8 : 4;
    const uint4 *p0 = reinterpret_cast<const uint4 *>(r0);
    int c = lane;
    for (; c + 32 * (U - 1) < n16; c += 32 * U) {
        uint4 w0[U];
#pragma unroll
        for (int u = 0; u < U; ++u) w0[u] = ld_stream(p0 + c + 32 * u);
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int t = 0; t < NT; ++t)
                if (t < n) a0[t] += dot8(w0[u], xs[t * n16 + c + 32 * u]);
    }
    for (; c < n16; c += 32) {
        const uint4 w0 = ld_stream(p0 + c);
#pragma unroll
        for (int t = 0; t < NT; ++t)
            if (t < n) a0[t] += dot8(w0, xs[t * n16 + c]);
    }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ uint16_t bf16_bits(float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t *>(&h);
}

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// ---------------------------------------------------------------------- kernel 1 --
template <int NT>
__global__ void __launch_bounds__(kK1Block) decode_k1_kernel(DecodeArgs a) {
    extern __shared__ uint4 xs[];  // [T][H] bf16
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
    const int n16 = a.H / 8;
    if (a.acc) {
        // clear the fp32 accumulator K2 adds into
        for (int n = blockIdx.x * kK1Block + tid; n < a.T * a.H; n += gridDim.x * kK1Block) a.acc[n] = 0.f;
    }
    const uint4 *xg = reinterpret_cast<const uint4 *>(a.x);
    for (int i = tid; i < a.T * n16; i += kK1Block) xs[i] = xg[i];
    __syncthreads();
    if (task < a.E) {
        // one pass over the router row for all T tokens
        float sc[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) sc[t] = 0.f;
        dot1_row_t<NT>(a.w_router + (size_t)task * a.H, xs, n16, lane, a.T, sc);
        const float b = a.b_router ? a.b_router[task] : 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t)
            if (t < a.T) {  // the same for the whole warp
                const float v = warp_sum(sc[t]);
                if (lane == 0) a.logits[(size_t)t * a.E + task] = v + b;
            }
    }
}

// Warp-wide top-k over one token's E logits: value descending, lower expert index first on
// equal values.  Lane L holds v[i] = logit of e = L + 32 i (i < PER; entries with e >= E are
// ignored).  Each logit becomes one 64-bit key, its order bits above the complement of its
// index, so that a single unsigned comparison orders value and index together (e >= E: key 0,
// below every real key).  Every lane sorts its PER keys once with a bitonic network of selects
// (no branches: a lone warp pays for divergence on every compare-exchange), then each of the k
// rounds takes the largest list head with two warp reductions (the order bits, then the index
// bits among the lanes whose head carries them) and the winning lane pops its head.  (The
// prefill top-k kernel, one warp per token and thousands of warps, keeps float compares with
// per-lane swaps: there throughput counts, and that form issues fewer instructions.)  Lane r < k
// returns the r-th choice (*val its logit, *id its index); every lane returns the largest
// logit in *top.
__device__ __forceinline__ void topk_cx(unsigned long long &a, unsigned long long &b) {
    const bool sw = b > a;
    const unsigned long long hi = sw ? b : a, lo = sw ? a : b;
    a = hi;
    b = lo;
}

template <int PER>
__device__ __forceinline__ void warp_topk_select(const float (&v)[PER], int E, int k, int lane, float *val,
                                                 int *id, float *top) {
    unsigned long long q[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = lane + 32 * i;
        q[i] = e < E ? ((unsigned long long)order_key(v[i]) << 32) | (uint32_t)~(uint32_t)e : 0ull;
    }
#pragma unroll
    for (int kk = 2; kk <= PER; kk <<= 1) {
#pragma unroll
        for (int j = kk >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    if ((i & kk) == 0) topk_cx(q[i], q[l]);
                    else topk_cx(q[l], q[i]);
                }
            }
        }
    }
    float my_val = 0.f, t = 0.f;
    int my_id = 0;
    for (int r = 0; r < k; ++r) {
        const uint32_t hi = (uint32_t)(q[0] >> 32), lo = (uint32_t)q[0];
        const uint32_t mk = __reduce_max_sync(0xffffffffu, hi);
        const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mk ? lo : 0u);
        const bool win = hi == mk && lo == ml;
#pragma unroll
        for (int i = 0; i + 1 < PER; ++i) q[i] = win ? q[i + 1] : q[i];
        q[PER - 1] = win ? 0ull : q[PER - 1];
        const float bv = key_value(mk);
        if (r == 0) t = bv;
        if (lane == r) {
            my_val = bv;
            my_id = (int)~ml;
        }
    }
    *val = my_val;
    *id = my_id;
    *top = t;
}

// ---------------------------------------------------------------------- kernel 2 --
// Warp-level top-k over the E logits (value descending, index ascending on ties: the rounds of
// warp_topk_select) and the renormalised softmax weights of the chosen k, into shared memory.
// Ids are clamped into [0, E) so that a corrupted logit vector can never make the block read
// outside the weights.
template <int PER>
__device__ __forceinline__ void warp_topk_regs(const float (&v)[PER], int E, int k, int *s_ids, float *s_w) {
    const int lane = threadIdx.x & 31;
    float my_val, top;
    int my_id;
    warp_topk_select<PER>(v, E, k, lane, &my_val, &my_id, &top);
    const float ej = lane < k ? expf(my_val - top) : 0.f;
    const float s = warp_sum(ej);
    if (lane < k) {
        s_ids[lane] = (my_id >= 0 && my_id < E) ? my_id : 0;
        s_w[lane] = ej / s;
    }
}

template <int PER>
__device__ __forceinline__ void warp_topk_t(const float *logits, int E, int k, int *s_ids, float *s_w) {
    const int lane = threadIdx.x & 31;
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) v[i] = lane + 32 * i < E ? logits[lane + 32 * i] : 0.f;
    warp_topk_regs<PER>(v, E, k, s_ids, s_w);
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

// 104 registers a thread (512 threads: 52K of the SM's 64K) leave room for a K1 block of the next
// layer on the same SM, so the router spreads over the GPU instead of the few SMs K2 leaves idle
// (with several tokens the gate/up accumulators need 128).
//
// T tokens (NT = 1, or kMaxDecodeT = 4 for 2 <= T <= 4).  Work items: the shared expert's 32-feature slices
// first (a block whose first item is one starts its loads before K1 finishes), then one item per
// (token t, slot j, slice).  A routed item works only for the first (token, slot) in token order
// that selected its expert e, and then serves every token that selected e: the expert's
// weights leave HBM once however many of the T tokens chose it; its other items are skipped.
// Blocks walk items w = blockIdx.x + i * gridDim.x; the launch gives every item its own block.
template <int NT>
__global__ void __maxnreg__(NT == 1 ? 104 : 128)
    decode_k2_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap tm_down,
                     const __grid_constant__ CUtensorMap tm_sdown, int n_shared_blocks) {
    extern __shared__ uint8_t smem_raw[];
    // TMA destinations: align the dynamic shared memory up to 1024 bytes (the launch adds slack)
    // aligned by an offset from the shared array itself (not through an integer address), so that
    // every access derived from it compiles to a shared-memory access rather than a generic one
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint16_t *wd = reinterpret_cast<uint16_t *>(smem);                           // [kChunkRows][kSlice]
    uint4 *xs = reinterpret_cast<uint4 *>(smem + (size_t)kChunkRows * kSlice * 2);  // [T][H] bf16
    float *hsl = reinterpret_cast<float *>(xs + (size_t)a.T * (a.H / 8));          // [NT][kSlice] fp32
    __shared__ int s_ids[kMaxDecodeT][32];
    __shared__ float s_w[kMaxDecodeT][32];
    __shared__ float s_lg[1024];       // logits staging for E > 256
    __shared__ unsigned s_chosen[32];
    __shared__ int s_tl[kMaxDecodeT];  // tokens this block serves, and their routing weights
    __shared__ float s_tw[kMaxDecodeT];
    __shared__ int s_n;
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_last;
    __shared__ int s_ok;
    __shared__ int s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T;
    const int n16 = a.H / 8;
    const int slices = a.I / kSlice;
    const int n_items = n_shared_blocks + T * a.k * slices;  // shared slices, then routed
    // item w: shared slice w, or routed (token, slot, slice) w - n_shared_blocks
    auto item_shared = [&](int w) { return w < n_shared_blocks; };
    auto item_i0 = [&](int w) { return w < n_shared_blocks ? w * kSlice : ((w - n_shared_blocks) % slices) * kSlice; };
    const int w0 = (int)blockIdx.x;  // this block's first item (blocks <= items)
    if (tid == 0) {
        ptx::mbar_init(&bar, 1);
        s_ok = 1;
        s_abort = 0;
        ptx::fence_mbar_init();
        ptx::tma_prefetch_desc(&tm_down);
        ptx::tma_prefetch_desc(&tm_sdown);
    }
    pdl_launch_dependents();
    __syncthreads();
    // TMA of rows [r0, r0 + rows) of a slice's columns into shared memory, on `bar`; run by a
    // whole warp: lane 0 posts the byte count, then lane b issues box b (at most 16 boxes)
    constexpr int kLoadWarp = kK2Warps - 1;
    auto load_chunk = [&](const CUtensorMap *tm, int i0, int base_row, int r0, int rows) {
        if (lane == 0) ptx::mbar_arrive_expect_tx(&bar, (uint32_t)(rows * kSlice * 2));
        __syncwarp();
        if (lane < rows / kBoxRows)
            ptx::tma_load_2d(wd + (size_t)lane * kBoxRows * kSlice, tm, i0, base_row + r0 + lane * kBoxRows, &bar);
    };
    const int rows0 = a.H < kChunkRows ? a.H : kChunkRows;
    const bool first_shared = item_shared(w0);
    if (first_shared) {
        // the shared expert's weights do not depend on the routing: start the first item's down
        // columns into shared memory and its gate/up rows into L2 before waiting for K1
        const int i0 = item_i0(w0);
        if (warp == kLoadWarp) load_chunk(&tm_sdown, i0, 0, 0, rows0);
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
    if (n_items > n_shared_blocks) {
        // every token's top-k: one warp per token (warp 0 for all of them above 256 experts,
        // whose selection stages the logits in shared memory)
        if (a.E <= 256) {
            if (warp < T) warp_topk(a.logits + (size_t)warp * a.E, a.E, a.k, s_ids[warp], s_w[warp], s_lg, s_chosen);
        } else if (warp == 0) {
            for (int t = 0; t < T; ++t) warp_topk(a.logits + (size_t)t * a.E, a.E, a.k, s_ids[t], s_w[t], s_lg, s_chosen);
        }
    }
    if (NT == 1 && warp == 0) {
        // one token (one item per block): the item serves that token, with no duplicates to skip
        __syncwarp();  // s_w of the top-k above, written by other lanes
        if (lane == 0) {
            s_tl[0] = 0;
            s_tw[0] = item_shared(w0) ? 1.f : s_w[0][((w0 - n_shared_blocks) / slices) % a.k];
            s_n = 1;
        }
    }
    const uint4 *xg = reinterpret_cast<const uint4 *>(a.x);
    for (int i = tid; i < T * n16; i += kK2Threads) xs[i] = xg[i];
    __syncthreads();
    uint32_t ph = 0;  // parity of the next chunk load on `bar`
    for (int w = w0; w < n_items && s_ok; w += (int)gridDim.x) {
        const bool shared_task = item_shared(w);
        const int i0 = item_i0(w);
        const int rb = w - n_shared_blocks;  // routed item index
        const int tok = shared_task ? 0 : rb / (a.k * slices);
        const int slot = shared_task ? 0 : (rb / slices) % a.k;
        if (NT > 1 && warp == 0) {
            // the tokens this item serves: pair p = t*k + j (32 per round, T*k <= 4*32) holds token
            // t's slot-j expert; the item works when (tok, slot) is the expert's first pair
            if (shared_task) {
                if (lane < T) {
                    s_tl[lane] = lane;
                    s_tw[lane] = 1.f;
                }
                if (lane == 0) s_n = T;
            } else {
                const int e = s_ids[tok][slot];
                const int pme = tok * a.k + slot;  // this item's pair
                int base = 0;
                bool first = true;  // no earlier pair selected e (the same for the whole warp)
                for (int half = 0; 32 * half < T * a.k; ++half) {
                    const int pp = lane + 32 * half;
                    const bool hit = pp < T * a.k && s_ids[pp / a.k][pp % a.k] == e;
                    const unsigned m = __ballot_sync(0xffffffffu, hit);
                    const int lo = pme - 32 * half;  // this round's pairs before pme: bits [0, lo)
                    const unsigned before = lo <= 0 ? 0u : (lo >= 32 ? 0xffffffffu : ((1u << lo) - 1u));
                    if (m & before) first = false;
                    const unsigned later = m & ~before;  // pairs from pme on: one per token at most
                    if ((later >> lane) & 1u) {
                        const int rank = base + __popc(later & ((1u << lane) - 1u));
                        s_tl[rank] = pp / a.k;
                        s_tw[rank] = s_w[pp / a.k][pp % a.k];
                    }
                    base += __popc(later);
                }
                if (lane == 0) s_n = first ? base : 0;
            }
        }
        if (NT > 1) __syncthreads();
        const int nt = s_n;  // 0: another item serves this expert
        if (nt == 0) {
            __syncthreads();  // s_n is rewritten by the next item
            continue;
        }
        const CUtensorMap *tm = shared_task ? &tm_sdown : &tm_down;
        int base_row = 0;  // first row of this item's weight matrix in its tensor map
        const uint16_t *wg = a.ws_gate, *wu = a.ws_up;  // shared expert: rows i0.. of [Is, H]
        if (!shared_task) {
            const int e = s_ids[tok][slot];
            base_row = e * a.H;
            wg = a.w_gate + (size_t)e * a.I * a.H;
            wu = a.w_up + (size_t)e * a.I * a.H;
        }
        if (!(w == w0 && first_shared) && warp == kLoadWarp) load_chunk(tm, i0, base_row, 0, rows0);
        // h for features i0 .. i0+31 and each served token: 16 warps x 2 features
        for (int f = warp; f < kSlice; f += kK2Warps) {
            const size_t row = (size_t)(i0 + f);
            float g[NT], u[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) g[t] = u[t] = 0.f;
            dot2_rows_t<NT>(wg + row * a.H, wu + row * a.H, xs, n16, lane, s_tl, nt, g, u);
#pragma unroll
            for (int t = 0; t < NT; ++t)
                if (t < nt) {  // the same for the whole warp
                    const float gs = warp_sum(g[t]), us = warp_sum(u[t]);
                    if (lane == 0) hsl[t * kSlice + f] = __bfloat162float(__float2bfloat16_rn(silu_mul(gs, us)));
                }
        }
        // split-K partial of the down projection, chunk by chunk: rows n of the chunk, 32 columns
        // each from shared memory (chunk order rotated per row against bank conflicts)
        for (int r0 = 0; r0 < a.H; r0 += kChunkRows, ph ^= 1u) {
            const int rows = (a.H - r0) < kChunkRows ? (a.H - r0) : kChunkRows;
            if (tid == 0 && !ptx::mbar_wait(&bar, ph, kWaitLimitNs, (volatile int *)&s_abort)) s_ok = 0;
            __syncthreads();
            if (!s_ok) break;
            // rows is a multiple of 128, so every warp runs the same number of iterations.  The row's
            // chunk order (cc + n/2) % 4 is the same for every row of this thread (rows tid + 512 i):
            // with one token its h is read into registers once, in that order.
            const int rot = (tid >> 1) & 3;
            // one token: h (bf16-rounded, so its fp32 words' high halves are its bf16 bits) packed
            // two features a word
            uint32_t hr[NT == 1 ? 16 : 1];
            if constexpr (NT == 1) {
                const float4 *h4 = reinterpret_cast<const float4 *>(hsl);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float4 u = h4[((cc + rot) & 3) * 2 + j];
                        hr[cc * 4 + 2 * j] = __byte_perm(__float_as_uint(u.x), __float_as_uint(u.y), 0x7632);
                        hr[cc * 4 + 2 * j + 1] = __byte_perm(__float_as_uint(u.z), __float_as_uint(u.w), 0x7632);
                    }
            }
            for (int n = tid; n < rows; n += kK2Threads) {
                const uint4 *rw = reinterpret_cast<const uint4 *>(wd + (size_t)n * kSlice);
                // the row's four 16-byte chunks, read in an order rotated per row (against bank
                // conflicts); chunk cc of q holds features 8*((cc + n/2) % 4) ..
                uint4 q[4];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) q[cc] = rw[(cc + rot) & 3];
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (t >= nt) break;  // the same for the whole block
                    float acc = 0.f;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        if constexpr (NT == 1) {
                            const uint32_t qw[4] = {q[cc].x, q[cc].y, q[cc].z, q[cc].w};
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                acc = fma_bf16h<0, 0>(qw[m], hr[cc * 4 + m], acc);
                                acc = fma_bf16h<1, 1>(qw[m], hr[cc * 4 + m], acc);
                            }
                        } else {
                            const int c = (cc + rot) & 3;
                            const __nv_bfloat162 *bq = reinterpret_cast<const __nv_bfloat162 *>(&q[cc]);
                            const float *hf = hsl + t * kSlice + c * 8;
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const float2 fv = __bfloat1622float2(bq[m]);
                                acc = fmaf(fv.x, hf[2 * m], acc);
                                acc = fmaf(fv.y, hf[2 * m + 1], acc);
                            }
                        }
                    }
                    // lanes 4q..4q+3 hold rows n..n+3: one 16-byte reduction per four rows
                    const float v1 = __shfl_down_sync(0xffffffffu, acc, 1);
                    const float v2 = __shfl_down_sync(0xffffffffu, acc, 2);
                    const float v3 = __shfl_down_sync(0xffffffffu, acc, 3);
                    const float wt = s_tw[t];
                    if ((lane & 3) == 0)
                        ptx::red_add_v4(&a.acc[(size_t)s_tl[t] * a.H + r0 + n], wt * acc, wt * v1, wt * v2, wt * v3);
                }
            }
            __syncthreads();  // the chunk buffer, hsl and the token list are free again
            if (r0 + kChunkRows < a.H && warp == kLoadWarp) {
                const int next = (a.H - r0 - kChunkRows) < kChunkRows ? (a.H - r0 - kChunkRows) : kChunkRows;
                load_chunk(tm, i0, base_row, r0 + kChunkRows, next);
            }
        }
    }
    if (!s_ok && tid == 0 && a.status) atomicCAS(a.status, 0, (int)MOE_ERR_TIMEOUT);
    // last block: every other block's adds are in the accumulator.  The block's reductions are
    // ordered before thread 0's ticket by the barrier and the ticket's release; the last block
    // sees all of them through the ticket's acquire.
    __syncthreads();
    if (tid == 0) {
        int ticket;
        asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(ticket) : "l"(a.counter) : "memory");
        s_last = (ticket == (int)gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    // four outputs a thread: one 16-byte accumulator load, 8-byte bf16 loads and stores
    for (int n4 = tid; n4 < T * a.H / 4; n4 += kK2Threads) {
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

size_t k2_smem(int T, int H, int nt) {
    return 1024 + (size_t)kChunkRows * kSlice * 2 + (size_t)T * H * 2 + (size_t)nt * kSlice * 4;
}

// Shared-memory limits of both instantiations (T = 1 up to H = 16384; T <= 8 with T*H <= 32768).
cudaError_t decode_attrs() {
    static bool done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && done[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(decode_k2_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)k2_smem(1, 16384, 1));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_k2_kernel<kMaxDecodeT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)k2_smem(1, kMaxDecodeTH, kMaxDecodeT));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_k1_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 32 * 1024);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_k1_kernel<kMaxDecodeT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMaxDecodeTH * 2);
    if (e == cudaSuccess && dev < 64) done[dev] = true;
    return e;
}

// ------------------------------------------------------------ chain of layers --
// One token through L layers in one cooperative launch.  Each block keeps one work item of the
// one-token layer (a 32-feature slice of a routed slot or of the shared expert, as in K2) and
// the layers are separated by two grid barriers instead of kernel boundaries:
//   A  every block: x_l into shared memory (from the previous layer's accumulator), up to
//      ceil(E / blocks) router rows (one warp each, the same dot as K1, so the logits are the
//      same bits).  Each logit is stored as one 64-bit word with its layer's tag (l + 1) above
//      the value bits, so a reader that sees the tag sees the value: no barrier between the
//      router rows and the selection.  A shared-expert block goes straight on to stream its
//      slice: it needs only x_l.
//   B  a routed block reads the logits until all carry this layer's tag, selects the top-k and
//      streams its expert slice; every block adds its split-K down partial into the
//      accumulator, then B2.
// Three accumulators rotate: the one cleared during layer l (for layer l + 1) last held layer
// l - 2's sums, which every block read before B2 of layer l - 1, so no barrier is needed between
// reading one and clearing another.  Layer 0 keeps one barrier, B1, after the blocks clear its
// accumulator and before the first partial is added.
// Barriers count arrivals on one word (release by the arriving block, acquire by the waiting
// one); every spin is bounded and a block that gives up raises a flag the others see.
constexpr uint64_t kBarLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// All threads of the block: the block's earlier writes are visible GPU-wide before its arrival
// (a release reduction: no round trip for the arriving thread).
__device__ __forceinline__ void grid_arrive(unsigned *bar) {
    __syncthreads();
    if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
}

// Tagged logits: the tag (the layer + 1) in the high word, the fp32 bits in the low one.  One
// 64-bit access each way, so that the pair is written and read whole.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Warp-wide: v[i] = logit e0 + lane + 32 i (i < 8, e < E; 0 past E) once every one of them
// carries `tag`.  Bounded like grid_wait: false (for the whole warp) when the wait runs out or
// another block gave up.
__device__ __forceinline__ bool wait_logits(const unsigned long long *lgt, int e0, int E, uint32_t tag, float (&v)[8],
                                            int *abort, int *status) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (uint32_t n = 0;; ++n) {
        unsigned long long u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = e0 + lane + 32 * i;
            u[i] = e < E ? ld_relaxed_u64(lgt + e) : (unsigned long long)tag << 32;
        }
        bool got = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) got = got && (uint32_t)(u[i] >> 32) == tag;
        if (__all_sync(0xffffffffu, got)) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __uint_as_float((uint32_t)u[i]);
            return true;
        }
        if (n == 0) {
            t0 = ptx::globaltimer();
        } else if ((n & 31u) == 0u) {  // the rest every 32 polls, decided by lane 0
            int stop = 0;
            if (lane == 0) {
                if (*reinterpret_cast<volatile int *>(abort)) {
                    stop = 1;
                } else if (ptx::globaltimer() - t0 > kBarLimitNs) {
                    stop = 1;
                    atomicExch(abort, 1);
                    if (status) atomicCAS(status, 0, (int)MOE_ERR_TIMEOUT);
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) return false;
        }
    }
}

__device__ __forceinline__ float *chain_acc(const ChainParams &p, int i) {
    return i == 0 ? p.acc0 : (i == 1 ? p.acc1 : p.acc2);
}

// All threads of the block: true once `target` arrivals are counted; false (for the whole
// block) when the wait runs out or another block gave up.
__device__ __forceinline__ bool grid_wait(unsigned *bar, unsigned target, int *abort, int *status,
                                          volatile int *s_flag) {
    if (threadIdx.x == 0) {
        int ok = 1;
        if (ld_acquire_u32(bar) < target) {
            const uint64_t t0 = ptx::globaltimer();
            for (uint32_t n = 1; ld_acquire_u32(bar) < target; ++n) {
                if ((n & 31u) != 0u) continue;  // poll the count alone; the rest every 32 polls
                if (*reinterpret_cast<volatile int *>(abort)) { ok = 0; break; }
                if (ptx::globaltimer() - t0 > kBarLimitNs) {
                    ok = 0;
                    atomicExch(abort, 1);
                    if (status) atomicCAS(status, 0, (int)MOE_ERR_TIMEOUT);
                    break;
                }
            }
        }
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

// r = bf16 residual bits, a = fp32 accumulator: out = bf16(a), x = bf16(r + out) (the rounding
// of the single-layer finish)
__device__ __forceinline__ void finish4(const float4 &a, uint2 r, uint2 *o, uint2 *xn) {
    const float vv[4] = {a.x, a.y, a.z, a.w};
    const uint16_t rr[4] = {(uint16_t)(r.x & 0xffffu), (uint16_t)(r.x >> 16), (uint16_t)(r.y & 0xffffu),
                            (uint16_t)(r.y >> 16)};
    uint16_t ob[4], xb[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        ob[q] = bf16_bits(vv[q]);
        xb[q] = bf16_bits(bf16_to_f(rr[q]) + bf16_to_f(ob[q]));
    }
    *o = make_uint2((uint32_t)ob[0] | ((uint32_t)ob[1] << 16), (uint32_t)ob[2] | ((uint32_t)ob[3] << 16));
    *xn = make_uint2((uint32_t)xb[0] | ((uint32_t)xb[1] << 16), (uint32_t)xb[2] | ((uint32_t)xb[3] << 16));
}

// 16 E4M3 codes (one 16-byte load) against 16 bf16 values of x (two 16-byte chunks): each code
// pair is widened exactly to two halves, then to fp32
__device__ __forceinline__ float dot16_q8(const uint4 &w, const uint4 &xa, const uint4 &xb) {
    const __nv_fp8x2_storage_t *wp = reinterpret_cast<const __nv_fp8x2_storage_t *>(&w);
    const __nv_bfloat162 *x0 = reinterpret_cast<const __nv_bfloat162 *>(&xa);
    const __nv_bfloat162 *x1 = reinterpret_cast<const __nv_bfloat162 *>(&xb);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(wp[i], __NV_E4M3);
        const float2 wf = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
        const float2 xf = __bfloat1622float2(i < 4 ? x0[i] : x1[i - 4]);
        acc = fmaf(wf.x, xf.x, acc);
        acc = fmaf(wf.y, xf.y, acc);
    }
    return acc;
}

// Two rows of H E4M3 codes (gate and up of one feature) against x in shared memory (bf16, n16
// chunks of 8): 16 codes per load, four loads a row in flight per lane.
__device__ __forceinline__ void dot2_rows_q8(const uint8_t *r0, const uint8_t *r1, const uint4 *xs, int n16,
                                             int lane, float &a0, float &a1) {
    constexpr int U = 4;
    const int nq = n16 >> 1;  // 16-byte chunks of a code row
    const uint4 *p0 = reinterpret_cast<const uint4 *>(r0);
    const uint4 *p1 = reinterpret_cast<const uint4 *>(r1);
    int c = lane;
    for (; c + 32 * (U - 1) < nq; c += 32 * U) {
        uint4 w0[U], w1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            w0[u] = ld_stream(p0 + c + 32 * u);
            w1[u] = ld_stream(p1 + c + 32 * u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint4 xa = xs[2 * (c + 32 * u)], xb = xs[2 * (c + 32 * u) + 1];
            a0 += dot16_q8(w0[u], xa, xb);
            a1 += dot16_q8(w1[u], xa, xb);
        }
    }
    for (; c < nq; c += 32) {
        const uint4 w0 = ld_stream(p0 + c), w1 = ld_stream(p1 + c);
        const uint4 xa = xs[2 * c], xb = xs[2 * c + 1];
        a0 += dot16_q8(w0, xa, xb);
        a1 += dot16_q8(w1, xa, xb);
    }
}

// dot1_row_t<1> with the row already in shared memory: the same per-lane order, the same bits
__device__ __forceinline__ float dot1_row_smem(const uint4 *w, const uint4 *xs, int n16, int lane) {
    constexpr int U = 8;
    float a = 0.f;
    int c = lane;
    for (; c + 32 * (U - 1) < n16; c += 32 * U) {
        uint4 w0[U];
#pragma unroll
        for (int u = 0; u < U; ++u) w0[u] = w[c + 32 * u];
#pragma unroll
        for (int u = 0; u < U; ++u) a += dot8(w0[u], xs[c + 32 * u]);
    }
    for (; c < n16; c += 32) a += dot8(w[c], xs[c]);
    return a;
}

// Rows of the router staged in shared memory a layer ahead: at most kStageRows rows a block, of
// at most kStageH elements.
constexpr int kStageRows = 2;
constexpr int kStageH = 4096;

// 4-bit codes: a word holds 8 nibbles, columns 8k .. 8k+7 with the lowest nibble first.  Flipping
// bit 3 of every nibble turns the two's-complement code into code + 8.

// Nibbles s and s + 4 of an offset-8 code word (two's-complement nibble ^ 8) as two bf16 codes:
// 0x4300 | u is the bf16 value 128 + u (u < 16 fits its 7 fraction bits), and subtracting 136
// leaves u - 8, the code, exactly.
__device__ __forceinline__ uint32_t q4_pair_bf16(uint32_t w, int s) {
    const uint32_t t = ((w >> (4 * s)) & 0x000F000Fu) | 0x43004300u;
    uint32_t c;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(t), "r"(0x43084308u));
    return c;
}

// the 32 codes of one block (16 bytes) against 32 bf16 values (16 words, column 2m in the low
// half of word m), in column order, fp32 sums: the products and sums of fmaf on the widened
// codes and values, bit for bit
__device__ __forceinline__ float q4_dot32(const uint4 &q, const uint32_t (&v)[16]) {
    const uint32_t w[4] = {q.x ^ 0x88888888u, q.y ^ 0x88888888u, q.z ^ 0x88888888u, q.w ^ 0x88888888u};
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        // c_s holds columns 8k + s (low) and 8k + s + 4 (high)
        const uint32_t c0 = q4_pair_bf16(w[k], 0), c1 = q4_pair_bf16(w[k], 1);
        const uint32_t c2 = q4_pair_bf16(w[k], 2), c3 = q4_pair_bf16(w[k], 3);
        a = fma_bf16h<0, 0>(c0, v[4 * k], a);
        a = fma_bf16h<0, 1>(c1, v[4 * k], a);
        a = fma_bf16h<0, 0>(c2, v[4 * k + 1], a);
        a = fma_bf16h<0, 1>(c3, v[4 * k + 1], a);
        a = fma_bf16h<1, 0>(c0, v[4 * k + 2], a);
        a = fma_bf16h<1, 1>(c1, v[4 * k + 2], a);
        a = fma_bf16h<1, 0>(c2, v[4 * k + 3], a);
        a = fma_bf16h<1, 1>(c3, v[4 * k + 3], a);
    }
    return a;
}

// Four rows of H 4-bit codes (nblk = H / 32 blocks of 16 bytes, fp32 scale per block) against x
// in shared memory (bf16): lane L takes blocks L, L + 32, ..., one at a time (the four rows' codes
// of a block in flight together); acc[r] += scale * (the block's codes . x).
__device__ __forceinline__ void dot4_rows_q4(const uint8_t *const (&rows)[4], const float *const (&sc)[4],
                                             const uint4 *xs, int nblk, int lane, float (&acc)[4]) {
    for (int c = lane; c < nblk; c += 32) {
        uint4 w[4];
        float s[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            w[r] = ld_stream(reinterpret_cast<const uint4 *>(rows[r]) + c);
            s[r] = __ldg(sc[r] + c);
        }
        uint32_t xw[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 xv = xs[4 * c + i];
            xw[4 * i] = xv.x, xw[4 * i + 1] = xv.y, xw[4 * i + 2] = xv.z, xw[4 * i + 3] = xv.w;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] = fmaf(q4_dot32(w[r], xw), s[r], acc[r]);
    }
}

__host__ __device__ __forceinline__ size_t chain_stage_off(int H, int E) {
    return ((size_t)kChunkRows * kSlice * 2 + (size_t)H * 2 + (size_t)kSlice * 4 + (size_t)E * 4 + 15) & ~(size_t)15;
}

// The expert weight format WF: kChainBf16; kChainE4m3: E4M3 codes with fp32 scales per output
// row (gate/up rows of H bytes, the down slice 32 bytes a row); kChainQ4: 4-bit codes with one
// fp32 scale per block of 32 columns (gate/up rows of H/2 bytes, the down slice 16 bytes a row,
// which is one block).  The router stays bf16.
template <int WF>
__global__ void __launch_bounds__(kK2Threads, 1) decode_chain_kernel(const __grid_constant__ ChainParams p) {
    constexpr bool Q8 = WF == kChainE4m3, Q4 = WF == kChainQ4;
    // bytes of an expert row of n weights, and of a row of the down slice (kSlice weights)
    auto row_bytes = [](int n) { return Q4 ? n / 2 : (Q8 ? n : 2 * n); };
    constexpr int kSliceBytes = Q4 ? kSlice / 2 : (Q8 ? kSlice : 2 * kSlice);
    extern __shared__ uint8_t smem_raw[];
    // aligned by an offset from the shared array itself (not through an integer address), so that
    // every access derived from it compiles to a shared-memory access rather than a generic one
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *wd = smem;                                                          // [kChunkRows][kSlice] weights
    uint4 *xs = reinterpret_cast<uint4 *>(smem + (size_t)kChunkRows * kSlice * 2);  // [H] bf16: x_l
    float *hsl = reinterpret_cast<float *>(xs + p.H / 8);                          // [kSlice]
    float *lg = hsl + kSlice;                                                      // [E] logits copy
    uint4 *wr_s = reinterpret_cast<uint4 *>(smem + chain_stage_off(p.H, p.E));     // [kStageRows][H]
    __shared__ int s_ids[32];
    __shared__ float s_w[32];
    __shared__ float s_lg[1024];
    __shared__ unsigned s_chosen[32];
    __shared__ __align__(8) uint64_t tbar;
    __shared__ int s_ok, s_abort, s_flag, s_lgok;
    __shared__ int s_zero[1];  // the token list of one token: token 0
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = p.H, E = p.E, n16 = H / 8;
    const int slices = p.I / kSlice, n_shared = p.Is / kSlice;
    const int n_items = n_shared + p.k * slices;
    const int nb = (int)gridDim.x, b = (int)blockIdx.x;
    const int rows0 = H < kChunkRows ? H : kChunkRows;
    constexpr int kLoadWarp = kK2Warps - 1;
    if (tid == 0) {
        ptx::mbar_init(&tbar, 1);
        s_ok = 1;
        s_abort = 0;
        s_zero[0] = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // TMA of rows [r0, r0 + rows) of a slice's columns into shared memory (as in K2)
    // (the map's columns are bytes for the code formats: the slice starts at byte row_bytes(i0))
    auto load_chunk = [&](const CUtensorMap *tm, int i0, int base_row, int r0, int rows) {
        if (lane == 0) ptx::mbar_arrive_expect_tx(&tbar, (uint32_t)(rows * kSliceBytes));
        __syncwarp();
        if (lane < rows / kBoxRows)
            ptx::tma_load_2d(wd + (size_t)lane * kBoxRows * kSliceBytes, tm, WF == kChainBf16 ? i0 : row_bytes(i0),
                             base_row + r0 + lane * kBoxRows, &tbar);
    };
    // the router rows of warps 0..1 (e = b + nb * warp) and their biases are staged in shared
    // memory and registers while the previous layer's barrier completes, when every block has at
    // most two rows of moderate length.  (Rows on warps 1..2, which leaves warp 0 free to poll
    // for the logits at once, measured 2 us a layer slower: its polls crowd the lines the other
    // blocks are writing.)
    const bool stage = E <= kStageRows * nb && H <= kStageH;
    const int rw = warp;  // this warp's first router row is b + nb * rw
    float sbias = 0.f;
    auto stage_rows = [&](int l) {
        const int e = b + nb * rw;
        if (rw >= 0 && rw < kStageRows && e < E) {
            sbias = p.lay[l].b_router ? p.lay[l].b_router[e] : 0.f;
            const uint4 *src = reinterpret_cast<const uint4 *>(p.lay[l].w_router + (size_t)e * H);
            uint4 *dst = wr_s + (size_t)rw * n16;
            for (int c0 = lane; c0 < n16; c0 += 32 * 8) {
                uint4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (c0 + 32 * u < n16) v[u] = ld_stream(src + c0 + 32 * u);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (c0 + 32 * u < n16) dst[c0 + 32 * u] = v[u];
            }
        }
    };
    if (stage) stage_rows(0);
    uint32_t ph = 0;        // parity of the next chunk on tbar
    bool pending = false;   // a chunk was issued and not yet waited for
    unsigned nbar = 0;      // barriers passed
    bool ok = true;
    for (int l = 0; l < p.L && ok; ++l) {
        const ChainLayer &ly = p.lay[l];
        float *acc = chain_acc(p, l % 3);
        const float *acc_prev = chain_acc(p, (l + 2) % 3);
        // ---------------------------------------------------------------- phase A --
        if (l == 0) {
            const uint4 *xg = reinterpret_cast<const uint4 *>(p.x0);
            for (int i = tid; i < n16; i += kK2Threads) xs[i] = xg[i];
        } else {
            // x_l = bf16(r + bf16(acc_prev)), r = resid or x_{l-1} (in place: xs holds x_{l-1})
            uint2 *x2 = reinterpret_cast<uint2 *>(xs);
            for (int i = tid; i < H / 4; i += kK2Threads) {
                const float4 a = __ldcg(reinterpret_cast<const float4 *>(acc_prev) + i);
                const uint2 r = p.resid ? reinterpret_cast<const uint2 *>(p.resid)[i] : x2[i];
                uint2 o, xn;
                finish4(a, r, &o, &xn);
                x2[i] = xn;
            }
        }
        if (l == 0)  // the first layer's accumulator; later ones are cleared a layer ahead
            for (int i = b * kK2Threads + tid; i < H / 4; i += nb * kK2Threads)
                reinterpret_cast<float4 *>(acc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncthreads();
        for (int e = b + nb * rw; rw >= 0 && e < E; e += nb * kK2Warps) {
            float sc[1] = {0.f};
            if (stage) sc[0] = dot1_row_smem(wr_s + (size_t)rw * n16, xs, n16, lane);
            else dot1_row_t<1>(ly.w_router + (size_t)e * H, xs, n16, lane, 1, sc);
            const float bias = stage ? sbias : (ly.b_router ? ly.b_router[e] : 0.f);
            const float v = warp_sum(sc[0]);
            if (lane == 0)
                st_relaxed_u64(p.logits + e, (unsigned long long)(l + 1) << 32 | __float_as_uint(v + bias));
        }
        unsigned t_b1 = 0;
        if (l == 0) {
            grid_arrive(p.bar);  // B1: the cleared first accumulator
            t_b1 = (++nbar) * (unsigned)nb;
        }
        if (l + 1 < p.L) {  // the next layer's router rows towards L2 while this layer streams
            const char *wr = reinterpret_cast<const char *>(p.lay[l + 1].w_router);
            for (int e = b + nb * warp; e < E; e += nb * kK2Warps)
                for (int o = lane * 128; o < H * 2; o += 32 * 128) prefetch_l2(wr + (size_t)e * H * 2 + o);
        }
        // ---------------------------------------------------------------- phase B --
        bool b1 = l > 0, topk_done = false;
        for (int w = b; w < n_items && ok; w += nb) {
            const bool shared_task = w < n_shared;
            const int i0 = shared_task ? w * kSlice : ((w - n_shared) % slices) * kSlice;
            float wt = 1.f;
            const CUtensorMap *tm = shared_task ? &p.tm_sdown[l] : &p.tm_down[l];
            int base_row = 0;
            const uint8_t *wg = static_cast<const uint8_t *>(ly.ws_gate), *wu = static_cast<const uint8_t *>(ly.ws_up);
            // Q8: the row scales of this item's gate/up rows and down rows
            const float *sgr = ly.ss_gate, *sur = ly.ss_up, *sdr = ly.ss_down;
            if (!shared_task) {
                if (!topk_done) {
                    if (warp == 0) {
                        // the logits other blocks wrote, once all carry this layer's tag
                        const uint32_t tag = (uint32_t)(l + 1);
                        bool got = true;
                        if (E <= 256) {
                            float v[8];
                            got = wait_logits(p.logits, 0, E, tag, v, p.abort, p.status);
                            if (got) warp_topk_regs<8>(v, E, p.k, s_ids, s_w);
                        } else {
                            for (int e0 = 0; e0 < E && got; e0 += 256) {
                                float v[8];
                                got = wait_logits(p.logits, e0, E, tag, v, p.abort, p.status);
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    if (got && e0 + lane + 32 * i < E) lg[e0 + lane + 32 * i] = v[i];
                            }
                            __syncwarp();
                            if (got) warp_topk(lg, E, p.k, s_ids, s_w, s_lg, s_chosen);
                        }
                        if (lane == 0) s_lgok = got ? 1 : 0;
                    }
                    __syncthreads();
                    if (!s_lgok) {
                        ok = false;
                        break;
                    }
                    topk_done = true;
                }
                const int slot = (w - n_shared) / slices;
                const int e = s_ids[slot];
                wt = s_w[slot];
                base_row = e * H;
                wg = static_cast<const uint8_t *>(ly.w_gate) + (size_t)e * p.I * row_bytes(H);
                wu = static_cast<const uint8_t *>(ly.w_up) + (size_t)e * p.I * row_bytes(H);
                if (Q8) {
                    sgr = ly.s_gate + (size_t)e * p.I;
                    sur = ly.s_up + (size_t)e * p.I;
                    sdr = ly.s_down + (size_t)e * H;
                }
                if (Q4) {  // block scales: gate/up [I, H/32], down [H, I/32]
                    sgr = ly.s_gate + (size_t)e * p.I * (H / 32);
                    sur = ly.s_up + (size_t)e * p.I * (H / 32);
                    sdr = ly.s_down + (size_t)e * H * (p.I / 32);
                }
            }
            if (warp == kLoadWarp) load_chunk(tm, i0, base_row, 0, rows0);
            pending = true;
            if constexpr (Q4) {
                // h for features i0 + warp and i0 + warp + 16: both features' gate and up rows in
                // flight at once (the rows are a quarter of the bf16 bytes)
                const int nblk = H / 32;
                const size_t r0w = (size_t)(i0 + warp), r1w = r0w + kK2Warps;
                const uint8_t *rows4[4] = {wg + r0w * (H / 2), wu + r0w * (H / 2), wg + r1w * (H / 2),
                                           wu + r1w * (H / 2)};
                const float *sc4[4] = {sgr + r0w * nblk, sur + r0w * nblk, sgr + r1w * nblk, sur + r1w * nblk};
                float a4[4] = {0.f, 0.f, 0.f, 0.f};
                dot4_rows_q4(rows4, sc4, xs, nblk, lane, a4);
#pragma unroll
                for (int r = 0; r < 4; ++r) a4[r] = warp_sum(a4[r]);
                if (lane == 0) {
                    hsl[warp] = __bfloat162float(__float2bfloat16_rn(silu_mul(a4[0], a4[1])));
                    hsl[warp + kK2Warps] = __bfloat162float(__float2bfloat16_rn(silu_mul(a4[2], a4[3])));
                }
            }
            // h for features i0 .. i0+31: 16 warps x 2 features
            for (int f = warp; f < (Q4 ? 0 : kSlice); f += kK2Warps) {
                const size_t row = (size_t)(i0 + f);
                float gs, us;
                if constexpr (Q8) {
                    const float sg = __ldg(sgr + row), su = __ldg(sur + row);  // in flight with the rows
                    float g = 0.f, u = 0.f;
                    dot2_rows_q8(wg + row * H, wu + row * H, xs, n16, lane, g, u);
                    gs = sg * warp_sum(g);
                    us = su * warp_sum(u);
                } else {
                    float g[1] = {0.f}, u[1] = {0.f};
                    dot2_rows_t<1>(reinterpret_cast<const uint16_t *>(wg) + row * H,
                                   reinterpret_cast<const uint16_t *>(wu) + row * H, xs, n16, lane, s_zero, 1, g, u);
                    gs = warp_sum(g[0]);
                    us = warp_sum(u[0]);
                }
                if (lane == 0) hsl[f] = __bfloat162float(__float2bfloat16_rn(silu_mul(gs, us)));
            }
            if (!b1) {  // layer 0: the accumulator is cleared once B1 completes
                if (!grid_wait(p.bar, t_b1, p.abort, p.status, (volatile int *)&s_flag)) { ok = false; break; }
                b1 = true;
            }
            for (int r0 = 0; r0 < H; r0 += kChunkRows, ph ^= 1u) {
                const int rows = (H - r0) < kChunkRows ? (H - r0) : kChunkRows;
                // Q8: this thread's down-row scales (rows tid + 512 i), in flight across the wait
                float sdn[kChunkRows / kK2Threads];
                if constexpr (Q8) {
#pragma unroll
                    for (int i = 0; i < kChunkRows / kK2Threads; ++i) {
                        const int n = tid + i * kK2Threads;
                        sdn[i] = n < rows ? __ldg(sdr + r0 + n) : 0.f;
                    }
                }
                if constexpr (Q4) {  // row r0 + n's scale of the block this slice is: [rows, I/32]
                    const int nb_row = (shared_task ? p.Is : p.I) / 32, blk = i0 / 32;
#pragma unroll
                    for (int i = 0; i < kChunkRows / kK2Threads; ++i) {
                        const int n = tid + i * kK2Threads;
                        sdn[i] = n < rows ? __ldg(sdr + (size_t)(r0 + n) * nb_row + blk) : 0.f;
                    }
                }
                if (tid == 0 && !ptx::mbar_wait(&tbar, ph, kWaitLimitNs, (volatile int *)&s_abort)) s_ok = 0;
                __syncthreads();
                if (!s_ok) {
                    ok = false;
                    break;
                }
                pending = false;
                if constexpr (Q4) {
                    // row n of the chunk: 16 bytes, the 32 codes of this slice's block (a warp's 32
                    // consecutive rows: conflict-free 16-byte reads); h into registers once
                    // (h is bf16-rounded: its fp32 words' high halves are its bf16 bits)
                    uint32_t hq[16];
                    const float4 *h4 = reinterpret_cast<const float4 *>(hsl);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 u = h4[j];
                        hq[2 * j] = __byte_perm(__float_as_uint(u.x), __float_as_uint(u.y), 0x7632);
                        hq[2 * j + 1] = __byte_perm(__float_as_uint(u.z), __float_as_uint(u.w), 0x7632);
                    }
#pragma unroll
                    for (int i = 0; i < kChunkRows / kK2Threads; ++i) {
                        const int n = tid + i * kK2Threads;
                        if (n >= rows) break;  // rows is a multiple of 128: whole warps leave together
                        const uint4 q = *reinterpret_cast<const uint4 *>(wd + (size_t)n * kSliceBytes);
                        const float a = q4_dot32(q, hq) * sdn[i];
                        atomicAdd(&acc[r0 + n], wt * a);  // the warp's 32 rows: one 128-byte reduction
                    }
                } else if constexpr (Q8) {
                    // the row's halves are read in the order n % 2, (n % 2) ^ 1 (against bank conflicts);
                    // n % 2 = tid % 2 for every row of this thread, so h is read into registers once
                    const int hb = tid & 1;
                    float hq[32];
                    const float4 *h4 = reinterpret_cast<const float4 *>(hsl);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 u0 = h4[hb * 4 + j], u1 = h4[(hb ^ 1) * 4 + j];
                        hq[4 * j] = u0.x, hq[4 * j + 1] = u0.y, hq[4 * j + 2] = u0.z, hq[4 * j + 3] = u0.w;
                        hq[16 + 4 * j] = u1.x, hq[17 + 4 * j] = u1.y, hq[18 + 4 * j] = u1.z, hq[19 + 4 * j] = u1.w;
                    }
                    const float *h0 = hq, *h1 = hq + 16;
#pragma unroll
                    for (int i = 0; i < kChunkRows / kK2Threads; ++i) {
                        const int n = tid + i * kK2Threads;
                        if (n >= rows) break;  // rows is a multiple of 128: whole warps leave together
                        const uint4 *rw = reinterpret_cast<const uint4 *>(wd + (size_t)n * kSlice);
                        const uint4 q0 = rw[hb], q1 = rw[hb ^ 1];  // alternate halves against bank conflicts
                        const __nv_fp8x2_storage_t *c0 = reinterpret_cast<const __nv_fp8x2_storage_t *>(&q0);
                        const __nv_fp8x2_storage_t *c1 = reinterpret_cast<const __nv_fp8x2_storage_t *>(&q1);
                        float a = 0.f;
#pragma unroll
                        for (int m = 0; m < 8; ++m) {
                            const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(c0[m], __NV_E4M3);
                            const float2 fv = __half22float2(*reinterpret_cast<const __half2 *>(&r));
                            a = fmaf(fv.x, h0[2 * m], a);
                            a = fmaf(fv.y, h0[2 * m + 1], a);
                        }
#pragma unroll
                        for (int m = 0; m < 8; ++m) {
                            const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(c1[m], __NV_E4M3);
                            const float2 fv = __half22float2(*reinterpret_cast<const __half2 *>(&r));
                            a = fmaf(fv.x, h1[2 * m], a);
                            a = fmaf(fv.y, h1[2 * m + 1], a);
                        }
                        a *= sdn[i];
                        atomicAdd(&acc[r0 + n], wt * a);  // the warp's 32 rows: one 128-byte reduction
                    }
                } else {
                // row n's 16-byte chunks are read in the order (cc + n/2) % 4 (no bank conflicts);
                // n/2 % 4 is the same for every row of this thread (rows tid + 512 i), so h is read
                // into registers once, in that order.  (This phase is bound by the shared-memory
                // pipe, which also carries shuffles and narrow loads: h comes in 16-byte loads and
                // each row is added on its own, the warp's 32 rows in one reduction.)
                const int rot = (tid >> 1) & 3;
                // h is bf16-rounded: its fp32 words' high halves are its bf16 bits, two a word
                uint32_t hr[16];
                const float4 *h4 = reinterpret_cast<const float4 *>(hsl);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float4 u = h4[((cc + rot) & 3) * 2 + j];
                        hr[cc * 4 + 2 * j] = __byte_perm(__float_as_uint(u.x), __float_as_uint(u.y), 0x7632);
                        hr[cc * 4 + 2 * j + 1] = __byte_perm(__float_as_uint(u.z), __float_as_uint(u.w), 0x7632);
                    }
                for (int n = tid; n < rows; n += kK2Threads) {
                    const uint4 *rw = reinterpret_cast<const uint4 *>(wd + (size_t)n * kSlice * 2);
                    uint4 q[4];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) q[cc] = rw[(cc + rot) & 3];
                    float a = 0.f;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint32_t qw[4] = {q[cc].x, q[cc].y, q[cc].z, q[cc].w};
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            a = fma_bf16h<0, 0>(qw[m], hr[cc * 4 + m], a);
                            a = fma_bf16h<1, 1>(qw[m], hr[cc * 4 + m], a);
                        }
                    }
                    atomicAdd(&acc[r0 + n], wt * a);  // the warp's 32 rows: one 128-byte reduction
                }
                }
                __syncthreads();  // the chunk buffer and hsl are free again
                if (r0 + kChunkRows < H && warp == kLoadWarp) {
                    const int next = (H - r0 - kChunkRows) < kChunkRows ? (H - r0 - kChunkRows) : kChunkRows;
                    load_chunk(tm, i0, base_row, r0 + kChunkRows, next);
                }
                if (r0 + kChunkRows < H) pending = true;
            }
        }
        if (!ok) break;
        if (!b1 && !grid_wait(p.bar, t_b1, p.abort, p.status, (volatile int *)&s_flag)) {  // a block with no item
            ok = false;
            break;
        }
        // the next layer's accumulator held layer l-2's sums, which every block read into x_{l-1}
        // before B2 of layer l-1: clear it here; it is added into only after this layer's B2
        if (l + 1 < p.L) {
            float *acc_next = chain_acc(p, (l + 1) % 3);
            for (int i = b * kK2Threads + tid; i < H / 4; i += nb * kK2Threads)
                reinterpret_cast<float4 *>(acc_next)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        grid_arrive(p.bar);  // B2: this layer's partials (and the next layer's cleared sums)
        const unsigned t_b2 = (++nbar) * (unsigned)nb;
        if (stage && l + 1 < p.L) stage_rows(l + 1);  // lands while the barrier completes
        if (!grid_wait(p.bar, t_b2, p.abort, p.status, (volatile int *)&s_flag)) ok = false;
    }
    if (!ok || !s_ok) {
        if (tid == 0) {
            atomicExch(p.abort, 1);
            if (p.status) atomicCAS(p.status, 0, (int)MOE_ERR_TIMEOUT);
            // a chunk still landing in shared memory finishes before the block leaves (bounded)
            if (pending) {
                volatile int zero = 0;
                ptx::mbar_wait(&tbar, ph, kWaitLimitNs, &zero);
            }
        }
        return;
    }
    // after the last B2: out = bf16(acc), x_last = bf16(r + out); the first block writes them
    if (b == 0) {
        const float *acc = chain_acc(p, (p.L - 1) % 3);
        const uint2 *x2 = reinterpret_cast<const uint2 *>(xs);
        for (int i = tid; i < H / 4; i += kK2Threads) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(acc) + i);
            const uint2 r = p.resid ? reinterpret_cast<const uint2 *>(p.resid)[i] : x2[i];
            uint2 o, xn;
            finish4(a, r, &o, &xn);
            reinterpret_cast<uint2 *>(p.out)[i] = o;
            if (p.x_last) reinterpret_cast<uint2 *>(p.x_last)[i] = xn;
        }
    }
}

size_t chain_smem(int H, int E) {
    return 1024 + chain_stage_off(H, E) + (size_t)kStageRows * (H < kStageH ? H : kStageH) * 2;
}

}  // namespace

int decode_slice() { return kSlice; }
int decode_box_rows() { return kBoxRows; }

cudaError_t launch_decode_router(const DecodeArgs &a, cudaStream_t s) {
    if (!decode_fits(a.T, a.H)) return cudaErrorInvalidValue;
    const cudaError_t e = decode_attrs();
    if (e != cudaSuccess) return e;
    DecodeArgs r = a;
    r.acc = nullptr;  // router rows only, no accumulator to clear
    LaunchScope scope(KC_DECODE_ROUTER, s);
    const dim3 grid((r.E + kK1Warps - 1) / kK1Warps);
    const size_t smem = (size_t)r.T * r.H * 2;
    if (r.T == 1) decode_k1_kernel<1><<<grid, kK1Block, smem, s>>>(r);
    else decode_k1_kernel<kMaxDecodeT><<<grid, kK1Block, smem, s>>>(r);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &tm_down, const CUtensorMap &tm_sdown,
                          cudaStream_t s) {
    if (!decode_fits(a.T, a.H)) return cudaErrorInvalidValue;
    cudaError_t e = decode_attrs();
    if (e != cudaSuccess) return e;
    const bool one = a.T == 1;
    {
        DecodeArgs k1 = a;
        void *args[] = {&k1};
        LaunchScope scope(KC_DECODE_ROUTER, s);
        e = launch_pdl(one ? reinterpret_cast<const void *>(decode_k1_kernel<1>)
                           : reinterpret_cast<const void *>(decode_k1_kernel<kMaxDecodeT>),
                       dim3((a.E + kK1Warps - 1) / kK1Warps), dim3(kK1Block), (size_t)a.T * a.H * 2, s, args);
        if (e != cudaSuccess) return e;
    }
    {
        DecodeArgs k2 = a;
        int n_shared = a.Is / kSlice;
        // one block per item: with one block per SM resident, a finished item's SM takes the next
        // item at once (measured faster than blocks that walk several items)
        const int blocks = a.T * a.k * (a.I / kSlice) + n_shared;
        CUtensorMap m0 = tm_down, m1 = tm_sdown;
        void *args[] = {&k2, &m0, &m1, &n_shared};
        LaunchScope scope(KC_DECODE_EXPERTS, s);
        return launch_pdl(one ? reinterpret_cast<const void *>(decode_k2_kernel<1>)
                              : reinterpret_cast<const void *>(decode_k2_kernel<kMaxDecodeT>),
                          dim3(blocks), dim3(kK2Threads), k2_smem(a.T, a.H, one ? 1 : kMaxDecodeT), s, args);
    }
}

cudaError_t launch_decode_chain(const ChainParams &p, int wf, cudaStream_t s) {
    if (p.L < 1 || p.L > kChainMaxLayers || p.H % kBoxRows != 0 || p.H > 16384 || p.E < 1 || p.E > 1024 ||
        p.k < 1 || p.k > p.E || p.k > 32 || p.I % kSlice != 0 || p.Is % kSlice != 0 || wf < 0 || wf > 2)
        return cudaErrorInvalidValue;
    const void *fn = wf == kChainE4m3 ? reinterpret_cast<const void *>(decode_chain_kernel<kChainE4m3>)
                     : wf == kChainQ4 ? reinterpret_cast<const void *>(decode_chain_kernel<kChainQ4>)
                                      : reinterpret_cast<const void *>(decode_chain_kernel<kChainBf16>);
    const size_t smem = chain_smem(p.H, p.E);
    // per device and format: the shared-memory opt-in and the resident blocks per SM (set once,
    // under a lock: two host threads' first launches would otherwise race)
    static int per_sm[3][64] = {{0}};
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::unique_lock<std::mutex> lk(mu);
    if (per_sm[wf][dev] == 0) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chain_smem(16384, 1024));
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kK2Threads, chain_smem(16384, 1024));
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        per_sm[wf][dev] = n;
    }
    const int resident = per_sm[wf][dev];
    lk.unlock();
    // every block must be resident at once (the layers are separated by grid barriers): at most
    // the blocks the GPU holds, each walking items blockIdx.x + i * gridDim.x
    const int n_items = p.Is / kSlice + p.k * (p.I / kSlice);
    int grid = resident * device_info().sm_count;
    if (n_items < grid) grid = n_items;
    // the barrier count and abort flag (adjacent words), and the logits' tags
    cudaError_t e = reinterpret_cast<void *>(p.abort) == reinterpret_cast<void *>(p.bar + 1)
                        ? cudaMemsetAsync(p.bar, 0, 2 * sizeof(unsigned), s)
                        : cudaMemsetAsync(p.bar, 0, sizeof(unsigned), s);
    if (e == cudaSuccess && reinterpret_cast<void *>(p.abort) != reinterpret_cast<void *>(p.bar + 1))
        e = cudaMemsetAsync(p.abort, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p.logits, 0, (size_t)p.E * sizeof(unsigned long long), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kK2Threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    LaunchScope scope(KC_DECODE_CHAIN, s);
    ChainParams pc = p;
    void *args[] = {&pc};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

namespace {
// One block per row: the row's largest magnitude, then its codes.  fp32 arithmetic with IEEE
// division, so that the scale and every code follow from the row's values alone.
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const uint16_t *__restrict__ w, int cols,
                                                            uint8_t *__restrict__ q, float *__restrict__ scale) {
    __shared__ float red[8];
    __shared__ float s_scale;
    const int r = blockIdx.x, tid = threadIdx.x;
    const uint16_t *row = w + (size_t)r * cols;
    float amax = 0.f;
    for (int c = tid; c < cols; c += 256) amax = fmaxf(amax, fabsf(bf16_to_f(row[c])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    if (tid == 0) {
        float m = red[0];
        for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
        const float sc = m > 0.f ? __fdiv_rn(m, 448.0f) : 1.0f;
        s_scale = sc;
        scale[r] = sc;
    }
    __syncthreads();
    const float sc = s_scale;
    for (int c = tid; c < cols; c += 256)
        q[(size_t)r * cols + c] =
            (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(bf16_to_f(row[c]), sc), __NV_SATFINITE, __NV_E4M3);
}
}  // namespace

cudaError_t launch_quantize_e4m3(const uint16_t *w, int rows, int cols, uint8_t *q, float *scale, cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    LaunchScope scope(KC_QUANTIZE, s);
    quantize_e4m3_kernel<<<rows, 256, 0, s>>>(w, cols, q, scale);
    return cudaGetLastError();
}

namespace {
// One warp per block of 32 columns: lane j holds column 32 b + j.  The block's largest magnitude
// (a warp maximum), its scale, each lane's code, and the lanes' nibbles packed in pairs (column
// 2m in the low nibble of byte m).  fp32 arithmetic with IEEE division, so the scale and every
// code follow from the block's values alone.
__global__ void __launch_bounds__(256) quantize_q4_kernel(const uint16_t *__restrict__ w, int rows, int cols,
                                                          uint8_t *__restrict__ q, float *__restrict__ scale) {
    const int nblk = cols / 32;
    const size_t blk = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (blk >= (size_t)rows * nblk) return;  // the same for the whole warp
    const int lane = threadIdx.x & 31;
    const size_t r = blk / nblk, b = blk % nblk;
    const float v = bf16_to_f(w[r * cols + 32 * b + lane]);
    float amax = fabsf(v);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 7.0f) : 1.0f;
    float c = rintf(__fdiv_rn(v, sc));
    c = fminf(fmaxf(c, -7.0f), 7.0f);
    const uint32_t nib = (uint32_t)(int)c & 15u;
    const uint32_t hi = __shfl_down_sync(0xffffffffu, nib, 1);
    if ((lane & 1) == 0) q[r * (cols / 2) + 16 * b + lane / 2] = (uint8_t)(nib | (hi << 4));
    if (lane == 0) scale[r * nblk + b] = sc;
}
}  // namespace

cudaError_t launch_quantize_q4(const uint16_t *w, int rows, int cols, uint8_t *q, float *scale, cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (cols % 32 != 0) return cudaErrorInvalidValue;
    const size_t nblocks = (size_t)rows * (cols / 32);
    LaunchScope scope(KC_QUANTIZE, s);
    quantize_q4_kernel<<<(unsigned)((nblocks + 7) / 8), 256, 0, s>>>(w, rows, cols, q, scale);
    return cudaGetLastError();
}

}  // namespace moe
