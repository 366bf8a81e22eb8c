// decode.cu -- the single-token (T = 1) layer: every weight byte the token needs is streamed
// from HBM exactly once with 128-bit loads, fp32 accumulation.
//
// Batch-1 decode is the pages' execution mode ("AIMA AMD395 Qwen3.6 35B Windows Engine",
// "产品定位": batch size 1, greedy decode).  At T = 1 each selected expert is a matrix-vector
// product, bound by HBM bandwidth, not by tensor cores:
//   kernel 1  router logits (E rows) and the shared expert's gate/up rows: one warp per row
//             (pair), x staged in shared memory;
//   kernel 2  softmax/top-k/renormalise (redone by every block from the E logits, so no block
//             waits on another), then the k experts' gate/up row pairs -> h (bf16);
//   kernel 3  for each output n: sum_j w_j * Wd[e_j][n,:].h_j + Ws_down[n,:].h_s, one warp
//             per output, all k+1 rows of the output streamed together; bf16 out and the
//             residual update resid + out.
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kBlock = kWarps * 32;

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    // weights are read once: bypass L1
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
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

// Lane-partial dot products of two weight rows with the same shared-memory vector of `len`
// bf16 elements (len % 8 == 0), four 16-byte loads per row in flight per lane.
__device__ __forceinline__ void dot2_rows(const uint16_t *r0, const uint16_t *r1, const uint4 *xs,
                                          int len, int lane, float &a0, float &a1) {
    const int n16 = len / 8;
    const uint4 *p0 = reinterpret_cast<const uint4 *>(r0);
    const uint4 *p1 = reinterpret_cast<const uint4 *>(r1);
    int c = lane;
    for (; c + 32 * 3 < n16; c += 32 * 4) {
        uint4 w0[4], w1[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            w0[u] = ld_stream(p0 + c + 32 * u);
            w1[u] = ld_stream(p1 + c + 32 * u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
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

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ uint16_t bf16_bits(float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t *>(&h);
}

// ---------------------------------------------------------------------- kernel 1 --
__global__ void __launch_bounds__(kBlock) decode_router_kernel(DecodeArgs a) {
    extern __shared__ uint4 xs[];  // H bf16
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4 *xg = reinterpret_cast<const uint4 *>(a.x);
    for (int i = tid; i < a.H / 8; i += kBlock) xs[i] = xg[i];
    __syncthreads();
    const int task = blockIdx.x * kWarps + warp;
    if (task < a.E) {
        const uint16_t *r = a.w_router + (size_t)task * a.H;
        float s0 = 0.f, s1 = 0.f;
        // the second row of the pair is the same row; its loads hit L1-bypassed L2 lines
        // already in flight, so only one row is fetched from HBM
        dot2_rows(r, r, xs, a.H, lane, s0, s1);
        s0 = warp_sum(s0);
        if (lane == 0) a.logits[task] = s0 + (a.b_router ? a.b_router[task] : 0.f);
    } else if (task < a.E + a.Is) {
        const int i = task - a.E;
        float g = 0.f, u = 0.f;
        dot2_rows(a.ws_gate + (size_t)i * a.H, a.ws_up + (size_t)i * a.H, xs, a.H, lane, g, u);
        g = warp_sum(g);
        u = warp_sum(u);
        if (lane == 0) a.h_s[i] = bf16_bits(silu_mul(g, u));
    }
}

// ---------------------------------------------------------------------- kernel 2 --
// Warp-level top-k over the E logits (value descending, index ascending on ties) and the
// renormalised softmax weights of the chosen k, into shared memory.
__device__ __forceinline__ void warp_topk(const DecodeArgs &a, int *s_ids, float *s_w) {
    const int lane = threadIdx.x & 31;
    const int per = (a.E + 31) / 32;
    float top = 0.f, my_val = 0.f;
    int my_id = 0;
    uint32_t taken = 0;  // bit i: logit lane + 32*i already chosen (per <= 32)
    for (int r = 0; r < a.k; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = 0; i < per; ++i) {
            const int e = lane + 32 * i;
            if (e < a.E && !((taken >> i) & 1u)) {
                const float v = a.logits[e];
                if (v > bv || bi == 0x7fffffff) { bv = v; bi = e; }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (r == 0) top = bv;
        if (lane == r) { my_val = bv; my_id = bi; }
    }
    const float ej = lane < a.k ? expf(my_val - top) : 0.f;
    const float s = warp_sum(ej);
    if (lane < a.k) {
        s_ids[lane] = my_id;
        s_w[lane] = ej / s;
    }
}

__global__ void __launch_bounds__(kBlock) decode_gateup_kernel(DecodeArgs a) {
    extern __shared__ uint4 xs[];  // H bf16
    __shared__ int s_ids[32];
    __shared__ float s_w[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4 *xg = reinterpret_cast<const uint4 *>(a.x);
    for (int i = tid; i < a.H / 8; i += kBlock) xs[i] = xg[i];
    if (warp == 0) warp_topk(a, s_ids, s_w);
    __syncthreads();
    if (blockIdx.x == 0 && tid < a.k) {
        a.ids[tid] = s_ids[tid];
        a.topw[tid] = s_w[tid];
    }
    const int task = blockIdx.x * kWarps + warp;
    if (task >= a.k * a.I) return;
    const int j = task / a.I, i = task - j * a.I;
    const size_t row = (size_t)s_ids[j] * a.I + i;
    float g = 0.f, u = 0.f;
    dot2_rows(a.w_gate + row * a.H, a.w_up + row * a.H, xs, a.H, lane, g, u);
    g = warp_sum(g);
    u = warp_sum(u);
    if (lane == 0) a.h[(size_t)j * a.I + i] = bf16_bits(silu_mul(g, u));
}

// ---------------------------------------------------------------------- kernel 3 --
__global__ void __launch_bounds__(kBlock) decode_down_kernel(DecodeArgs a) {
    extern __shared__ uint4 hs[];  // [k*I] routed h, then [Is] shared h (bf16)
    __shared__ int s_ids[32];
    __shared__ float s_w[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nh = (a.k * a.I) / 8, ns = a.Is / 8;
    for (int i = tid; i < nh; i += kBlock) hs[i] = reinterpret_cast<const uint4 *>(a.h)[i];
    for (int i = tid; i < ns; i += kBlock) hs[nh + i] = reinterpret_cast<const uint4 *>(a.h_s)[i];
    if (tid < a.k) {
        s_ids[tid] = a.ids[tid];
        s_w[tid] = a.topw[tid];
    }
    __syncthreads();
    const int n = blockIdx.x * kWarps + warp;
    if (n >= a.H) return;
    const int nI = a.I / 8;
    float acc = 0.f;
    // routed experts: rows Wd[e_j][n, :] of I elements, two slots per pass for load overlap
    for (int j = 0; j < a.k; j += 2) {
        const bool two = j + 1 < a.k;
        const uint4 *r0 = reinterpret_cast<const uint4 *>(a.w_down + ((size_t)s_ids[j] * a.H + n) * a.I);
        const uint4 *r1 = two ? reinterpret_cast<const uint4 *>(a.w_down + ((size_t)s_ids[j + 1] * a.H + n) * a.I) : r0;
        float p0 = 0.f, p1 = 0.f;
        for (int c = lane; c < nI; c += 32) {
            const uint4 w0 = ld_stream(r0 + c);
            const uint4 w1 = two ? ld_stream(r1 + c) : make_uint4(0, 0, 0, 0);
            p0 += dot8(w0, hs[j * nI + c]);
            if (two) p1 += dot8(w1, hs[(j + 1) * nI + c]);
        }
        acc += s_w[j] * p0;
        if (two) acc += s_w[j + 1] * p1;
    }
    if (a.Is > 0) {
        const uint4 *rs = reinterpret_cast<const uint4 *>(a.ws_down + (size_t)n * a.Is);
        float ps = 0.f;
        for (int c = lane; c < ns; c += 32) ps += dot8(ld_stream(rs + c), hs[nh + c]);
        acc += ps;
    }
    acc = warp_sum(acc);
    if (lane == 0) {
        const __nv_bfloat16 o = __float2bfloat16_rn(acc);
        a.out[n] = *reinterpret_cast<const uint16_t *>(&o);
        if (a.x_next) {
            const __nv_bfloat16 xv = *reinterpret_cast<const __nv_bfloat16 *>(&a.resid[n]);
            a.x_next[n] = bf16_bits(__bfloat162float(xv) + __bfloat162float(o));
        }
    }
}

}  // namespace

cudaError_t launch_decode_router(const DecodeArgs &a, cudaStream_t s) {
    DecodeArgs r = a;
    r.Is = 0;  // router rows only
    LaunchScope scope(KC_DECODE_ROUTER, s);
    decode_router_kernel<<<(r.E + kWarps - 1) / kWarps, kBlock, (size_t)r.H * 2, s>>>(r);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        // kernel 3 stages k*I + Is bf16 of h: up to 32 x 8192 + 8192 elements
        cudaError_t e = cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             200 * 1024);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const size_t xs_bytes = (size_t)a.H * 2;
    {
        const int tasks = a.E + a.Is;
        LaunchScope scope(KC_DECODE_ROUTER, s);
        decode_router_kernel<<<(tasks + kWarps - 1) / kWarps, kBlock, xs_bytes, s>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const int tasks = a.k * a.I;
        LaunchScope scope(KC_DECODE_GATEUP, s);
        decode_gateup_kernel<<<(tasks + kWarps - 1) / kWarps, kBlock, xs_bytes, s>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const size_t hs_bytes = ((size_t)a.k * a.I + a.Is) * 2;
        LaunchScope scope(KC_DECODE_DOWN, s);
        decode_down_kernel<<<(a.H + kWarps - 1) / kWarps, kBlock, hs_bytes, s>>>(a);
        return cudaGetLastError();
    }
}

}  // namespace moe
