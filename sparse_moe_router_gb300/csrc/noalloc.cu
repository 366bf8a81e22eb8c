// noalloc.cu -- moe_permute_noalloc: the expert permutation without any caller-provided or
// library-allocated workspace.
//
// Who needs it: callers that may not allocate device memory at the point where they route
// tokens -- a serving process that reserves all device memory once at start-up and hands out
// fixed arenas, or host code that simply has no allocator at hand.  moe_permute needs a
// workspace for its per-chunk count table; this variant keeps that table in a fixed-size
// array compiled into the library instead, so the caller passes only inputs and outputs.
//
// The scratch array lives in device memory of every GPU that loads the library, for as long
// as the process runs.  Host code cannot use the array's name as a device address (it is a
// host-side stand-in), so on the first call on each device, with that device current, the
// entry point looks the address up with cudaGetSymbolAddress and remembers it; later calls on
// that device reuse it.  Every call shares the one array, so calls that overlap on the GPU
// (two streams, or two threads) race on it and must be serialised by the caller.
#include <mutex>

#include "internal.h"

namespace moe {
namespace {

// Largest problem the fixed table serves: T*k <= 65536 pairs and E <= 1024 experts.  The
// permutation cuts the pairs into chunks of whole tokens (at most kPermChunk pairs each, 8-token
// granularity), which for T*k <= 65536 and any k <= 32 makes at most 36 chunks.
constexpr int kNoAllocMaxPairs = 65536;
constexpr int kNoAllocMaxExperts = 1024;
constexpr int kNoAllocChunks = 40;
constexpr size_t kNoAllocTableInts = (size_t)kNoAllocChunks * kNoAllocMaxExperts;

// The chunk count table: every entry a call reads is first written by that same call, so
// nothing in it has to start at zero.
static __device__ __align__(256) int32_t g_noalloc_chunk_tab[kNoAllocTableInts];

std::mutex g_noalloc_mu;
void *g_noalloc_addr[64] = {nullptr};

// Device address of the table on the current device (looked up once per device).
cudaError_t noalloc_table(int32_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_chunk_tab);
        if (e != cudaSuccess) return e;
        g_noalloc_addr[dev] = p;
    }
    *out = static_cast<int32_t *>(g_noalloc_addr[dev]);
    return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_noalloc(const moe_config *cfg, const int32_t *topk_ids, int T,
                                          int32_t *expert_offsets, int32_t *perm, int32_t *inv,
                                          void *stream) {
    if (!cfg || T < 0) return MOE_ERR_INVALID_ARG;
    if (cfg->n_experts <= 0 || cfg->top_k <= 0 || cfg->top_k > cfg->n_experts) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!topk_ids || !expert_offsets || !perm || !inv) return MOE_ERR_INVALID_ARG;
    if (cfg->n_experts > kNoAllocMaxExperts || cfg->top_k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)T * cfg->top_k > kNoAllocMaxPairs) return MOE_ERR_UNSUPPORTED_SHAPE;
    // the table the permutation will index: one row of E counts per chunk of pairs
    if (permute_scratch_ints(T, cfg->n_experts, cfg->top_k) > kNoAllocTableInts) return MOE_ERR_UNSUPPORTED_SHAPE;
    int32_t *table = nullptr;
    if (noalloc_table(&table) != cudaSuccess) return MOE_ERR_CUDA;
    // No tile prefix, per-row token/weight arrays or status word: outputs only.
    const cudaError_t e = launch_permute(topk_ids, T, cfg->n_experts, cfg->top_k, expert_offsets, perm, inv,
                                         nullptr, kTileN, table, nullptr, nullptr, nullptr, nullptr,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
