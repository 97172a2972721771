// layout.cu - dispatch layout on the device: per-expert and per-rank counts,
// their prefix sums, and the receive row of every (token, k) pair.
//
// Follows "Unify expert parallel token dispatcher API" (section "API design":
// num_local_tokens_per_expert_E; "Backend behavior": the current capacity is
// the per-rank layout stride) and "ep: graph-safe worst-token HT
// dispatch+combine" (section "Internode", items 2 and 3: per-expert counts
// written to device memory, and a device prefix sum holding the true
// received total). Nothing is copied to the host and nothing waits on it.
//
// Kernels, sized from T and K only:
//   count : one CTA per tile of tokens (about one tile per SM); warp-
//           aggregated shared-memory histogram (__match_any_sync groups equal
//           expert ids so one lane per group adds the group size), plus the
//           distinct tokens per rank.
//   scan  : one CTA of 1024 threads; column prefix of the tile histograms read
//           as 16-byte vectors by row groups, per-expert totals, expert offsets
//           within each rank, per-rank totals and their inclusive prefix.
//   pos   : one CTA per tile; stable rank of each pair among the pairs of the
//           same expert in flat order t*K+k (tile_positions).
// The default bulk dispatch does all three inside its one-pass kernel
// (permute.cu); these kernels serve the layout-only call, the vector permute,
// the dedupe dispatch and the bulk dispatch where a tile does not fit.
#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kScanRows = 10;   // tile rows a scan thread holds in registers

__global__ void __launch_bounds__(kLayoutThreads)
layout_count_kernel(LayoutArgs a)
{
    __shared__ int s_hist[kMaxExperts];
    __shared__ int s_tok[kMaxRanks];
    griddep_wait();
    griddep_launch_dependents();
    const int tile = blockIdx.x;
    tile_histogram(a, tile, s_hist, s_tok);
    for (int e = threadIdx.x; e < a.Ep; e += blockDim.x)
        a.tile_cnt[(int64_t)tile * a.Ep + e] = s_hist[e];
    if (threadIdx.x < a.R) a.tile_tok[(int64_t)tile * a.R + threadIdx.x] = s_tok[threadIdx.x];
}

__device__ __forceinline__ int4 add4(int4 a, int4 b)
{
    return make_int4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// One CTA of 1024 threads. Thread (g, q) owns columns 4q..4q+3 of the rows of
// row group g; the groups' sums are scanned per column in shared memory.
__global__ void __launch_bounds__(1024)
layout_scan_kernel(LayoutArgs a)
{
    __shared__ int s_grp[4096];          // [groups][Ep], groups * Ep <= 4096
    __shared__ int s_tok[1024];          // [groups2][R]
    __shared__ int s_incl[kMaxExperts];
    __shared__ int s_warp[32];
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int G = a.ntiles, Ep = a.Ep, Q = Ep / 4;
    int NG = 1024 / Q;
    if (NG > 64) NG = 64;
    const int g = tid / Q, q = tid % Q;
    const bool active = g < NG;
    const int RG = (G + NG - 1) / NG;
    const int r0 = min(G, g * RG), r1 = min(G, r0 + RG);
    const int4* tc = reinterpret_cast<const int4*>(a.tile_cnt);
    int4* tp = reinterpret_cast<int4*>(a.tile_pre);

    // Row-group sums of the tile histograms. The group's rows are loaded into
    // registers in one round (kScanRows at a time) and kept for the prefix pass.
    int4 rows[kScanRows];
    int4 acc = make_int4(0, 0, 0, 0);
    if (active) {
        for (int c0 = r0; c0 < r1; c0 += kScanRows) {
#pragma unroll
            for (int j = 0; j < kScanRows; ++j) {
                const int r = c0 + j;
                rows[j] = (r < r1) ? ld_cg_v4(tc + (int64_t)r * Q + q) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < kScanRows; ++j) acc = add4(acc, rows[j]);
        }
        s_grp[g * Ep + 4 * q + 0] = acc.x;
        s_grp[g * Ep + 4 * q + 1] = acc.y;
        s_grp[g * Ep + 4 * q + 2] = acc.z;
        s_grp[g * Ep + 4 * q + 3] = acc.w;
    }
    // Distinct tokens per rank: thread (g2, r) sums the contiguous rows of row
    // group g2 of column r.
    const int NG2 = 1024 / a.R;
    const int RG2 = (G + NG2 - 1) / NG2;
    const int g2 = tid / a.R, rr = tid % a.R;
    const int q0 = min(G, g2 * RG2), q1 = min(G, q0 + RG2);
    if (tid < NG2 * a.R) {
        int s = 0;
#pragma unroll 4
        for (int row = q0; row < q1; ++row) s += __ldcg(a.tile_tok + (int64_t)row * a.R + rr);
        s_tok[tid] = s;
    }
    __syncthreads();

    // Exclusive scan of the group sums down each column; the column total is
    // the expert's count.
    int total = 0;
    if (tid < Ep) {
        for (int gg = 0; gg < NG; ++gg) {
            const int v = s_grp[gg * Ep + tid];
            s_grp[gg * Ep + tid] = total;
            total += v;
        }
    }
    if (tid < a.R) {   // exclusive scan of the group sums down column tid
        int s = 0;
        for (int gg = 0; gg < NG2; ++gg) {
            const int v = s_tok[gg * a.R + tid];
            s_tok[gg * a.R + tid] = s;
            s += v;
        }
        a.tokens_in_rank[tid] = s;
    }
    __syncthreads();
    if (a.tile_tok_pre && tid < NG2 * a.R) {   // each tile's exclusive prefix per rank
        int run = s_tok[tid];
        for (int row = q0; row < q1; ++row) {
            const int v = __ldcg(a.tile_tok + (int64_t)row * a.R + rr);
            a.tile_tok_pre[(int64_t)row * a.R + rr] = run;
            run += v;
        }
    }

    // Exclusive prefix of every tile row: the group's base plus its earlier rows
    // (from registers when the group fits one chunk, else reloaded).
    if (active) {
        int4 run = make_int4(s_grp[g * Ep + 4 * q + 0], s_grp[g * Ep + 4 * q + 1],
                             s_grp[g * Ep + 4 * q + 2], s_grp[g * Ep + 4 * q + 3]);
        if (r1 - r0 <= kScanRows) {
#pragma unroll
            for (int j = 0; j < kScanRows; ++j) {
                const int r = r0 + j;
                if (r < r1) {
                    tp[(int64_t)r * Q + q] = run;
                    run = add4(run, rows[j]);
                }
            }
        } else {
            for (int r = r0; r < r1; ++r) {
                const int4 v = ld_cg_v4(tc + (int64_t)r * Q + q);
                tp[(int64_t)r * Q + q] = run;
                run = add4(run, v);
            }
        }
    }
    if (tid < a.E) a.cnt[tid] = total;

    // Inclusive scan of the per-expert totals over e (warp shuffles, then warp sums).
    int v = (tid < a.E) ? total : 0;
    const int own = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += n;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += n;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += s_warp[warp - 1];
    if (tid < a.E) s_incl[tid] = v;
    __syncthreads();

    // Ranks own contiguous expert blocks, so a rank's rows start where the
    // inclusive prefix of its first expert's predecessor ends.
    const int eloc = a.E / a.R;
    if (tid < a.E) {
        if (a.packed) {
            a.expert_offset[tid] = v - own;              // after every lower expert
        } else {
            const int r = tid / eloc;
            const int base = (r > 0) ? s_incl[r * eloc - 1] : 0;
            a.expert_offset[tid] = (int32_t)((int64_t)r * a.S + (v - own - base));
        }
    }
    if (tid < a.R) {
        const int hi = s_incl[(tid + 1) * eloc - 1];
        const int lo = (tid > 0) ? s_incl[tid * eloc - 1] : 0;
        a.rows_per_rank[tid] = hi - lo;
        a.rank_prefix[tid] = hi;
    }
}

__global__ void __launch_bounds__(kLayoutThreads)
layout_pos_kernel(LayoutArgs a)
{
    __shared__ int s_base[kLayoutWarps * kMaxExperts];
    griddep_wait();
    griddep_launch_dependents();
    tile_positions(a, blockIdx.x, s_base, a.pos, nullptr);
}

}  // namespace

cudaError_t launch_layout_counts(const LayoutArgs& a, const LaunchOpts& o)
{
    cudaError_t e = cudaSuccess;
    if (a.ntiles > 0)
        e = launch_kernel(layout_count_kernel, dim3(a.ntiles), dim3(kLayoutThreads), 0, o, a);
    if (e != cudaSuccess) return e;
    return launch_kernel(layout_scan_kernel, dim3(1), dim3(1024), 0, o, a);
}

cudaError_t launch_layout_positions(const LayoutArgs& a, const LaunchOpts& o)
{
    if (a.ntiles <= 0) return cudaSuccess;
    return launch_kernel(layout_pos_kernel, dim3(a.ntiles), dim3(kLayoutThreads), 0, o, a);
}

cudaError_t launch_layout(const LayoutArgs& a, const LaunchOpts& o)
{
    cudaError_t e = launch_layout_counts(a, o);
    return e != cudaSuccess ? e : launch_layout_positions(a, o);
}

}  // namespace ep
