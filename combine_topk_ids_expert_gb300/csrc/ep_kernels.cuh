// ep_kernels.cuh - internal interface between the C ABI (ep_api.cu,
// layout_noalloc.cu) and the sm_103a kernels of the dispatch + combine step
// (layout.cu, permute.cu, combine.cu); ep_next.cuh extends it for the dedupe,
// the expert GEMM and the debug checks. Not installed.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ep {

// Limits the kernels are written for (checked on the host).
constexpr int kMaxExperts = 1024;   // one scan column per thread of a 1024-thread block
constexpr int kMaxRanks = 64;       // per-token rank sets are 64-bit masks
constexpr int kMaxTopk = 64;        // per-token positions staged in shared memory

// Layout tiles: CTA `tile` of the count and position kernels owns tokens
// [tile*tpt, min(T, (tile+1)*tpt)). Tile tables have rows of Ep = roundup4(E)
// ints so the scan can read them as 16-byte vectors.
constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kMaxTilePairs = 8192;   // pairs one tile may hold (fused kernel's shared table)
constexpr int kTileBaseCap = 1024;    // tiles per call before large calls add more

inline int round_up4(int e) { return (e + 3) / 4 * 4; }

// Tokens per tile for a call of T tokens: about one tile per SM, more tiles
// when a tile would exceed kMaxTilePairs pairs.
inline int64_t tokens_per_tile(int64_t T, int K, int num_sms)
{
    if (T <= 0) return 1;
    int64_t tiles = num_sms < kTileBaseCap ? num_sms : kTileBaseCap;
    const int64_t need = (T * K + kMaxTilePairs - 1) / kMaxTilePairs;
    if (need > tiles) tiles = need;
    if (tiles > T) tiles = T;
    if (tiles < 1) tiles = 1;
    return (T + tiles - 1) / tiles;
}

inline int64_t tile_count(int64_t T, int64_t tpt) { return T <= 0 ? 0 : (T + tpt - 1) / tpt; }

// Upper bound of tile_count over every T <= n_max (any SM count), for sizing.
inline int64_t max_tiles(int64_t n_max, int K)
{
    int64_t t = kTileBaseCap;
    const int64_t need = (n_max * K + kMaxTilePairs - 1) / kMaxTilePairs;
    if (need > t) t = need;
    if (t > n_max) t = n_max;
    return t < 1 ? 1 : t;
}

// Device error word bits (same values as EP_DEVERR_* in ep.h).
constexpr uint32_t kErrBadId = 0x1u;
constexpr uint32_t kErrRowOob = 0x2u;
constexpr uint32_t kErrTimeout = 0x4u;

struct LayoutArgs {
    const int32_t* ids;        // [T][K]
    int64_t T;
    int64_t S;                 // rows per rank for this call
    int64_t tpt;               // tokens per tile
    int ntiles;
    int K, E, R, Ep;
    int32_t* tile_cnt;         // [tiles][Ep] per-tile expert counts (scratch)
    int32_t* tile_pre;         // [tiles][Ep] exclusive prefix over tiles (scratch)
    int32_t* tile_tok;         // [tiles][R] per-tile distinct-token counts (scratch)
    int32_t* tile_tok_pre;     // [tiles][R] their exclusive prefix over tiles, or null
    int32_t* cnt;              // [E]
    int32_t* expert_offset;    // [E]
    int32_t* rows_per_rank;    // [R]
    int32_t* rank_prefix;      // [R]
    int32_t* tokens_in_rank;   // [R]
    int32_t* pos;              // [T][K]
    uint32_t* err;
    uint32_t* gbar;            // [4] one-pass dispatch: even-generation arrivals,
                               // generation, the counter of its shared token pool,
                               // odd-generation arrivals; or null
    uint32_t* tile_ready;      // [tiles] one-pass dispatch: the generation in which each
                               // tile's positions were published; or null
    bool packed;               // ranks back to back instead of r*S
};

// Launch options shared by every kernel: programmatic dependent launch lets a
// kernel start while its predecessor in the stream drains.
struct LaunchOpts {
    cudaStream_t stream;
    bool pdl;
    int64_t* launches;         // incremented per kernel launched
};

// count + scan: fills cnt, expert_offset, rows_per_rank, rank_prefix,
// tokens_in_rank and the tile tables.
cudaError_t launch_layout_counts(const LayoutArgs& a, const LaunchOpts& o);
// positions of every pair (after launch_layout_counts).
cudaError_t launch_layout_positions(const LayoutArgs& a, const LaunchOpts& o);
// all three.
cudaError_t launch_layout(const LayoutArgs& a, const LaunchOpts& o);

struct PermuteArgs {
    const void* x;             // [T][row_bytes]
    const float* scores;       // [T][K]
    const int32_t* pos;        // [T][K]
    void* recv_x;              // [R*S][row_bytes]
    float* recv_scores;        // [R*S]
    int32_t* recv_src;         // [R*S]
    int64_t T;
    int K;
    int64_t row_bytes;         // multiple of 16
    uint32_t* err;
    // Test hook for the bounded-wait path: CTA 0 of the bulk kernels never
    // issues the load of its local token with this index, so that token's wait
    // runs out (EP_DEVERR_TIMEOUT). -1 (the default) disables it.
    int64_t skip_load;
};
struct PermutePlan {
    int impl;                  // 1 = vec, 2 = bulk
    int grid;                  // standalone permute kernels
    int stages;                // bulk: shared-memory row slots per CTA (standalone)
    int smem_bytes;            // bulk: dynamic shared memory per CTA (standalone)
    int fused_smem_cap;        // fused layout+permute: max dynamic shared memory per CTA
};
// Chooses grids and staging for a row size on the current device.
// tiles_per_sm: fused-dispatch CTAs sharing an SM (each gets that share of
// shared memory for its ring).
cudaError_t plan_permute(int impl, int64_t row_bytes, int K, int E, int num_sms, int tiles_per_sm,
                         PermutePlan* plan);
cudaError_t launch_permute(const PermuteArgs& a, const PermutePlan& plan, const LaunchOpts& o);

// Positions + bulk permute in one kernel, one CTA per layout tile, after
// launch_layout_counts. Returns cudaErrorNotSupported when the call does not
// fit the fused kernel (then the caller runs positions + permute separately).
cudaError_t launch_dispatch_fused(const LayoutArgs& l, const PermuteArgs& p,
                                  const PermutePlan& plan, const LaunchOpts& o);
// Layout + positions + permute in one cooperative kernel (count, grid
// barrier, prefix, positions, copies); cudaErrorNotSupported where a tile does
// not fit or the tiles cannot all be resident. pdl_ok: cooperative launches
// accept the programmatic-serialization attribute (probe_cooperative_pdl).
// pool_pct: the share (percent) of each tile's tokens whose rows go to a pool
// that any CTA may copy once its own share is done (needs l.tile_ready).
// small_pairs: calls of at most this many (token, k) pairs skip the grid
// barrier: every CTA counts all of the call's ids itself.
cudaError_t launch_dispatch_onepass(const LayoutArgs& l, const PermuteArgs& p,
                                    const PermutePlan& plan, const LaunchOpts& o, bool pdl_ok,
                                    int pool_pct, int64_t small_pairs);
// Synchronous: whether a cooperative launch with programmatic serialization runs.
bool probe_cooperative_pdl();

struct CombineArgs {
    const void* y;             // [R*S][D] of in_dtype
    const float* scores;       // [T][K]
    const int32_t* pos;        // [T][K]
    const int32_t* rank_prefix;// [R]
    void* out;                 // [T][D] of out_dtype
    int64_t T;
    int K, R;
    int64_t S;
    int64_t D;
    int in_dtype, out_dtype;   // 0 = bf16, 1 = fp32
    uint32_t* err;
    bool packed;               // row validity: p < total instead of per-rank ranges
    // Dispatch backward reuses the combine gather: weights of 1 (scores unused),
    // and gather_out[t][k] = gather_in[pos[t][k]] (0 without a valid row).
    bool unit_weights;
    const float* gather_in;    // [R*S] or null
    float* gather_out;         // [T][K] or null
    // Set by launch_combine: CTAs (vector chunks) per token, 1 unless the call
    // has fewer tokens than the grid has CTAs.
    int vsplit;
};
// grid: num_sms times the CTAs per SM that fit, at most per_sm_cap (0: no cap).
cudaError_t plan_combine(int in_dtype, int num_sms, int per_sm_cap, int* grid);
cudaError_t launch_combine(const CombineArgs& a, int grid, const LaunchOpts& o);

struct CombineBwdArgs {
    const void* grad_out;      // [T][D] of dtype
    const void* y;             // [R*S][D] of dtype (read only when grad_scores is set)
    const float* scores;       // [T][K]
    const int32_t* pos;        // [T][K]
    const int32_t* rank_prefix;// [R]
    void* grad_y;              // [R*S][D] of dtype
    float* grad_scores;        // [T][K] or null
    int64_t T;
    int K, R;
    int64_t S;
    int64_t D;
    int dtype;                 // 0 = bf16, 1 = fp32
    uint32_t* err;
    bool packed;
};
cudaError_t launch_combine_backward(const CombineBwdArgs& a, int grid, const LaunchOpts& o);

// Launches kernel with an optional programmatic-dependent-launch attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          const LaunchOpts& o, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = o.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = o.pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
    if (e == cudaSuccess && o.launches) ++*o.launches;
    return e;
}

}  // namespace ep
