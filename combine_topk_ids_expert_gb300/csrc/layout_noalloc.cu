// layout_noalloc.cu - the dispatch layout for callers that cannot allocate
// device memory.
//
// Some callers have no way to call cudaMalloc or to keep a workspace: a
// plugin or custom op inside a host framework that owns every device
// allocation and only hands the op its input and output tensors, or code
// running under an allocator policy that forbids new device allocations.
// ep_dispatch_layout_noalloc serves them: the caller passes the ids and the
// layout outputs; the only other global memory the layout kernels need (the
// per-tile count tables) lives in g_layout_scratch below, a file-scope
// device array that every GPU which loads this library holds until the
// process exits.
//
// g_layout_scratch is a host-side stand-in in host code, not a device
// address: host code must never pass it to a kernel. The first call on each
// device (with that device current) asks the runtime for the array's device
// address with cudaGetSymbolAddress and caches it; kernels receive that
// address. Make that first call before any stream capture. The cache is keyed
// by the device's current context as well (its driver context id), so after a
// cudaDeviceReset, or under another context of the same device, the next call
// looks the address up again instead of using one that is no longer mapped.
//
// Every call shares the one array, which keeps the last call's contents.
// Nothing in it needs to start at zero (each word a call reads was written
// earlier in the same call), but calls whose GPU work overlaps (two streams,
// or two threads) race on it: serialize them.
#include <cuda.h>            // driver types only: the entry points are looked up at run time
#include <cuda_runtime.h>

#include <mutex>

#include "ep.h"
#include "ep_kernels.cuh"

namespace {

constexpr size_t kScratchBytes = EP_NOALLOC_SCRATCH_BYTES;   // 4 MiB per device
constexpr size_t kSegAlign = 256;
constexpr int kCachedDevices = 64;

static __device__ __align__(256) uint8_t g_layout_scratch[kScratchBytes];

std::mutex g_scratch_mu;
struct ScratchSlot {
    unsigned long long ctx;   // driver id of the context the address belongs to (0: unknown)
    void* addr;               // device address of g_layout_scratch in that context
};
ScratchSlot g_scratch[kCachedDevices];   // per device

// The current context's driver id, or 0 when there is none yet or the driver
// entry points cannot be had (then the cache is keyed by device alone). The
// entry points come from the runtime, so the library does not link libcuda.
unsigned long long current_context_id()
{
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
    });
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
    if (get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

size_t seg(size_t bytes) { return (bytes + kSegAlign - 1) / kSegAlign * kSegAlign; }

// Tiles of max(1, 2048/K) tokens: a fixed tiling, so the scratch bound
// depends on the call's sizes only.
int64_t noalloc_tokens_per_tile(int K) { return 2048 / K > 0 ? 2048 / K : 1; }

// Bytes of scratch the layout of T tokens needs (tile tables plus one word).
size_t scratch_needed(int64_t T, int K, int E, int R)
{
    const size_t tiles = (size_t)ep::tile_count(T, noalloc_tokens_per_tile(K));
    const size_t Ep = (size_t)ep::round_up4(E);
    return 2 * seg(tiles * Ep * 4) + seg(tiles * (size_t)R * 4) + seg(4);
}

// Device address of g_layout_scratch on the current device, looked up once per
// device (and again when the device's current context has changed).
cudaError_t scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kCachedDevices;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cached && g_scratch[dev].addr && g_scratch[dev].ctx == current_context_id()) {
        *out = g_scratch[dev].addr;
        return cudaSuccess;
    }
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_layout_scratch);
    if (e != cudaSuccess) return e;
    // The lookup has made the runtime's context current: key the entry by it.
    if (cached) g_scratch[dev] = ScratchSlot{current_context_id(), ptr};
    *out = ptr;
    return cudaSuccess;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" size_t ep_dispatch_layout_noalloc_scratch_bytes(int64_t num_tokens, int32_t topk,
                                                          int32_t num_experts, int32_t num_ranks)
{
    if (num_tokens < 0 || topk < 1 || num_experts < 1 || num_ranks < 1) return 0;
    return scratch_needed(num_tokens, topk, num_experts, num_ranks);
}

extern "C" ep_status ep_dispatch_layout_noalloc(
    const int32_t* topk_expert_ids_TK, int64_t num_tokens, int64_t num_tokens_per_rank,
    int32_t topk, int32_t num_experts, int32_t num_ranks, int32_t* tokens_per_expert,
    int32_t* expert_offset, int32_t* rows_per_rank, int32_t* rank_prefix,
    int32_t* tokens_in_rank, int32_t* pos, uint32_t* error_flags, ep_stream_t stream)
{
    const int64_t T = num_tokens, N = num_tokens_per_rank;
    const int K = topk, E = num_experts, R = num_ranks;
    if (T < 0 || N < T) return EP_ERR_INVALID_ARG;
    if (E < 1 || E > ep::kMaxExperts || R < 1 || R > ep::kMaxRanks || E % R != 0)
        return EP_ERR_INVALID_ARG;
    if (K < 1 || K > E || K > ep::kMaxTopk) return EP_ERR_INVALID_ARG;
    if (!tokens_per_expert || !expert_offset || !rows_per_rank || !rank_prefix ||
        !tokens_in_rank || (T > 0 && (!topk_expert_ids_TK || !pos)))
        return EP_ERR_INVALID_ARG;
    if (!aligned4(topk_expert_ids_TK) || !aligned4(tokens_per_expert) ||
        !aligned4(expert_offset) || !aligned4(rows_per_rank) || !aligned4(rank_prefix) ||
        !aligned4(tokens_in_rank) || !aligned4(pos) || !aligned4(error_flags))
        return EP_ERR_ALIGNMENT;
    const int64_t S = (N + 3) / 4 * 4 * K;
    if (S > INT32_MAX / R || T * K > INT32_MAX) return EP_ERR_CAPACITY;
    if (scratch_needed(T, K, E, R) > kScratchBytes) return EP_ERR_CAPACITY;

    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return EP_ERR_CUDA;
    uint8_t* p = static_cast<uint8_t*>(base);
    ep::LayoutArgs a;
    a.ids = topk_expert_ids_TK;
    a.T = T;
    a.S = S;
    a.tpt = noalloc_tokens_per_tile(K);
    a.ntiles = (int)ep::tile_count(T, a.tpt);
    a.K = K;
    a.E = E;
    a.R = R;
    a.Ep = ep::round_up4(E);
    const size_t tiles = (size_t)a.ntiles;
    a.tile_cnt = reinterpret_cast<int32_t*>(p);
    p += seg(tiles * (size_t)a.Ep * 4);
    a.tile_pre = reinterpret_cast<int32_t*>(p);
    p += seg(tiles * (size_t)a.Ep * 4);
    a.tile_tok = reinterpret_cast<int32_t*>(p);
    a.tile_tok_pre = nullptr;
    p += seg(tiles * (size_t)R * 4);
    a.cnt = tokens_per_expert;
    a.expert_offset = expert_offset;
    a.rows_per_rank = rows_per_rank;
    a.rank_prefix = rank_prefix;
    a.tokens_in_rank = tokens_in_rank;
    a.pos = pos;
    // Without a caller word, bad-id reports land in a scratch word nobody reads.
    a.err = error_flags ? error_flags : reinterpret_cast<uint32_t*>(p);
    a.gbar = nullptr;
    a.tile_ready = nullptr;
    a.packed = false;
    int64_t launches = 0;
    const ep::LaunchOpts o{static_cast<cudaStream_t>(stream), true, &launches};
    if (ep::launch_layout(a, o) != cudaSuccess) return EP_ERR_CUDA;
    return EP_OK;
}
