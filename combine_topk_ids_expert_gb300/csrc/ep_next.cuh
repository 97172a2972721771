// ep_next.cuh - declarations of the kernels beyond one dispatch + combine
// step: the per-rank dedupe dispatch and its expansion (dedup.cu) and the
// expert grouped GEMM (expert_gemm.cu). Kept apart from ep_kernels.cuh so that
// work on these leaves the step's kernel sources untouched.
#pragma once

#include "ep_kernels.cuh"

namespace ep {

// Per-rank dedupe (dedup.cu): one receive row per distinct (token, rank).
struct DedupArgs {
    const void* x;             // [T][row_bytes]
    const float* scores;       // [T][K]
    const int32_t* ids;        // [T][K]
    int64_t T;
    int K, E, R;
    int64_t P;                 // rows reserved per rank
    int64_t row_bytes;
    void* recv_x;              // [R*P][row_bytes]
    int32_t* recv_tok_src;     // [R*P]
    int32_t* recv_topk_idx;    // [R*P][K]
    float* recv_topk_w;        // [R*P][K]
    int32_t* tok_pos;          // [T][R]
    uint32_t* err;
};
// positions (per layout tile, after launch_layout) + copies.
cudaError_t launch_dedup(const LayoutArgs& l, const DedupArgs& a, const LaunchOpts& o);
// per-expert positions + dedupe rows + copies in one kernel (after
// launch_layout_counts); cudaErrorNotSupported if a tile's tables do not fit.
cudaError_t launch_dedup_fused(const LayoutArgs& l, const DedupArgs& a, const LaunchOpts& o);
// The dedupe dispatch as one cooperative kernel (layout with a grid barrier,
// positions, dedupe rows, copies); needs l.gbar. cudaErrorNotSupported where
// the rows do not fit its ring or the tiles cannot all be resident. pdl_ok as
// for launch_dispatch_onepass.
cudaError_t launch_dedup_onepass(const LayoutArgs& l, const DedupArgs& a, const LaunchOpts& o,
                                 bool pdl_ok);
// y[pos[t][k]] = recv_x[tok_pos[t][r(e)]] for every routed pair.
cudaError_t launch_dedup_expand(const DedupArgs& a, const int32_t* pos, void* y,
                                const LaunchOpts& o);

// Expert consumer: grouped GEMM y[p] = x[p] * W_e^T over each expert's rows,
// driven by the device counts and offsets (expert_gemm.cu).
struct GemmArgs {
    const int32_t* cnt;            // [E] rows per expert
    const int32_t* expert_offset;  // [E] first receive row of each expert
    void* y;                       // [rows][dout] bf16
    int64_t din, dout;             // din % 64 == 0, dout % 128 == 0
    int E;
    int kind;                      // 1 single-CTA 128-row tiles, 2 two-SM 256-row tiles
                                   // (needs dout % 256 == 0, else falls back to 1)
    int bk;                        // K per ring stage: 64 or 32
    int light_rows;                // experts with at most this many rows are scheduled as
                                   // light (interleaved with the rest); 0: none is
    uint32_t* err;
};
// x: [rows][din] bf16 receive rows; w: [E][dout][din] bf16.
// kernel_used: the kind that ran (see GemmArgs::kind); grid_used: its CTAs.
cudaError_t launch_expert_gemm(const GemmArgs& a, const void* x, int64_t rows, const void* w,
                               int grid, const LaunchOpts& o, int* kernel_used, int* grid_used);

// Sentinel checks of the receive buffer (debug.cu, EP_DEBUG=1).
constexpr uint32_t kErrDebugUnwritten = 0x8u;   // a row inside a rank's total kept the sentinel
constexpr uint32_t kErrDebugStray = 0x10u;      // a row past a rank's total was written
struct SentinelArgs {
    const uint8_t* recv_x;          // [R*S][row_bytes]
    int64_t S, row_bytes;
    int R;
    bool packed;
    const int32_t* rows_per_rank;   // [R]
    const int32_t* rank_prefix;     // [R]
    uint32_t* err;
};
cudaError_t launch_sentinel_check(const SentinelArgs& a, int num_sms, const LaunchOpts& o);

}  // namespace ep
