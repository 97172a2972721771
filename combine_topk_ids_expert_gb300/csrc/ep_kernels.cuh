// ep_kernels.cuh - internal interface between the C ABI (ep_api.cu) and the
// sm_103a kernels (layout.cu, permute.cu, combine.cu). Not installed.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ep {

// Limits the kernels are written for (checked by ep_buffer_init).
constexpr int kMaxExperts = 1024;   // one scan element per thread of a 1024-thread block
constexpr int kMaxRanks = 64;       // per-token rank sets are 64-bit masks
constexpr int kMaxTopk = 64;        // per-token positions staged in shared memory

// Layout tiles: each CTA of the count and position kernels owns a contiguous
// run of tokens holding about kLayoutPairs (token, k) pairs.
constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kLayoutPairs = 2048;
inline int64_t layout_tokens_per_tile(int K) {
    int64_t t = kLayoutPairs / K;
    return t > 0 ? t : 1;
}
inline int64_t layout_tiles(int64_t T, int K) {
    const int64_t tpt = layout_tokens_per_tile(K);
    return (T + tpt - 1) / tpt;
}

// Device error word bits (same values as EP_DEVERR_* in ep.h).
constexpr uint32_t kErrBadId = 0x1u;
constexpr uint32_t kErrRowOob = 0x2u;
constexpr uint32_t kErrTimeout = 0x4u;

struct LayoutArgs {
    const int32_t* ids;        // [T][K]
    int64_t T;
    int64_t S;                 // rows per rank for this call
    int K, E, R;
    int32_t* tile_cnt;         // [tiles][E] per-tile expert counts (scratch)
    int32_t* tile_pre;         // [tiles][E] exclusive prefix over tiles (scratch)
    int32_t* tile_tok;         // [tiles][R] per-tile distinct-token counts (scratch)
    int32_t* cnt;              // [E]
    int32_t* expert_offset;    // [E]
    int32_t* rows_per_rank;    // [R]
    int32_t* rank_prefix;      // [R]
    int32_t* tokens_in_rank;   // [R]
    int32_t* pos;              // [T][K]
    uint32_t* err;
};
// Enqueues the layout kernels; adds the number of kernels launched to *launches.
cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t s, int64_t* launches);

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
};
struct PermutePlan {
    int impl;                  // 1 = vec, 2 = bulk
    int grid;
    int stages;                // bulk: shared-memory row slots per CTA
    int smem_bytes;            // bulk: dynamic shared memory per CTA
};
// Chooses grid and staging for a row size on the current device.
cudaError_t plan_permute(int impl, int64_t row_bytes, int K, int num_sms, PermutePlan* plan);
cudaError_t launch_permute(const PermuteArgs& a, const PermutePlan& plan, cudaStream_t s,
                           int64_t* launches);

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
};
cudaError_t plan_combine(int in_dtype, int num_sms, int* grid);
cudaError_t launch_combine(const CombineArgs& a, int grid, cudaStream_t s, int64_t* launches);

}  // namespace ep
