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
// Three kernels, all sized from T and K only:
//   count : one CTA per tile of tokens; warp-aggregated shared-memory
//           histogram (__match_any_sync groups equal expert ids so one lane
//           per group adds the group size), plus distinct tokens per rank.
//   scan  : one CTA; column prefix of the tile histograms, per-expert totals,
//           expert offsets within each rank, per-rank totals and their
//           inclusive prefix.
//   pos   : one CTA per tile; stable rank of each pair among the pairs of the
//           same expert (flat order t*K+k), from per-warp histograms, their
//           prefix over warps, the tile prefix and the expert offset.
#include "ep_kernels.cuh"

namespace ep {
namespace {

__device__ __forceinline__ int valid_id(int e, int E) { return (e >= -1 && e < E) ? e : -1; }

__device__ __forceinline__ unsigned lanemask_lt(int lane) { return (1u << lane) - 1u; }

__global__ void __launch_bounds__(kLayoutThreads)
layout_count_kernel(LayoutArgs a, int64_t tpt)
{
    __shared__ int s_hist[kMaxExperts];
    __shared__ int s_tok[kMaxRanks];
    const int tile = blockIdx.x;
    const int64_t t0 = (int64_t)tile * tpt;
    const int64_t t1 = min(a.T, t0 + tpt);
    const int64_t p0 = t0 * a.K;
    const int np = (int)((t1 - t0) * a.K);
    const int lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < a.E; i += blockDim.x) s_hist[i] = 0;
    if (threadIdx.x < a.R) s_tok[threadIdx.x] = 0;
    __syncthreads();

    // Full warps walk the tile so every lane takes part in __match_any_sync.
    const int np32 = (np + 31) & ~31;
    bool bad = false;
    for (int i = threadIdx.x; i < np32; i += blockDim.x) {
        int e = -1;
        if (i < np) {
            const int raw = __ldg(a.ids + p0 + i);
            e = valid_id(raw, a.E);
            bad |= (e != raw);
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[e], __popc(peers));
    }
    if (bad) atomicOr(a.err, kErrBadId);

    // Distinct tokens per logical rank: one 64-bit rank set per token.
    const int eloc = a.E / a.R;
    for (int64_t t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
        unsigned long long mask = 0ull;
        for (int k = 0; k < a.K; ++k) {
            const int e = valid_id(__ldg(a.ids + t * a.K + k), a.E);
            if (e >= 0) mask |= 1ull << (e / eloc);
        }
        while (mask) {
            atomicAdd(&s_tok[__ffsll((long long)mask) - 1], 1);
            mask &= mask - 1ull;
        }
    }
    __syncthreads();

    for (int e = threadIdx.x; e < a.E; e += blockDim.x)
        a.tile_cnt[(int64_t)tile * a.E + e] = s_hist[e];
    if (threadIdx.x < a.R) a.tile_tok[(int64_t)tile * a.R + threadIdx.x] = s_tok[threadIdx.x];
}

// One CTA of 1024 threads: thread e owns expert e (E <= 1024).
__global__ void __launch_bounds__(1024)
layout_scan_kernel(LayoutArgs a, int ntiles)
{
    __shared__ int s_incl[kMaxExperts];
    __shared__ int s_warp[32];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int32_t* __restrict__ tc = a.tile_cnt;
    int32_t* __restrict__ tp = a.tile_pre;

    // Column prefix over tiles (exclusive) and the expert's total.
    int total = 0;
    if (tid < a.E) {
        int64_t idx = tid;
#pragma unroll 8
        for (int tile = 0; tile < ntiles; ++tile, idx += a.E) {
            const int c = tc[idx];
            tp[idx] = total;
            total += c;
        }
        a.cnt[tid] = total;
    }
    if (tid < a.R) {
        int s = 0;
        for (int tile = 0; tile < ntiles; ++tile) s += a.tile_tok[(int64_t)tile * a.R + tid];
        a.tokens_in_rank[tid] = s;
    }

    // Inclusive scan of the per-expert totals over e (warp shuffles, then warp sums).
    int v = total;
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
        const int r = tid / eloc;
        const int base = (r > 0) ? s_incl[r * eloc - 1] : 0;
        a.expert_offset[tid] = (int32_t)((int64_t)r * a.S + (v - total - base));
    }
    if (tid < a.R) {
        const int hi = s_incl[(tid + 1) * eloc - 1];
        const int lo = (tid > 0) ? s_incl[tid * eloc - 1] : 0;
        a.rows_per_rank[tid] = hi - lo;
        a.rank_prefix[tid] = hi;
    }
}

__global__ void __launch_bounds__(kLayoutThreads)
layout_pos_kernel(LayoutArgs a, int64_t tpt)
{
    __shared__ int s_base[kLayoutWarps * kMaxExperts];   // [warp][expert]
    const int tile = blockIdx.x;
    const int64_t t0 = (int64_t)tile * tpt;
    const int64_t t1 = min(a.T, t0 + tpt);
    const int64_t p0 = t0 * a.K;
    const int np = (int)((t1 - t0) * a.K);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int E = a.E;

    // Warp w owns the flat pairs [w*seg, w*seg + seg) of the tile; seg is a
    // multiple of 32 so every chunk is a full warp.
    const int seg = (((np + kLayoutWarps - 1) / kLayoutWarps) + 31) & ~31;
    const int w_begin = warp * seg;
    const int w_end = min(np, w_begin + seg);
    int* mine = s_base + warp * E;

    for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) s_base[i] = 0;
    __syncthreads();

    // Pass 1: per-warp histogram (one writer per row; no atomics).
    for (int c = w_begin; c < w_begin + seg; c += 32) {
        const int i = c + lane;
        const int e = (i < w_end) ? valid_id(__ldg(a.ids + p0 + i), E) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // Exclusive prefix over warps, seeded with the expert offset and the
    // counts of all earlier tiles.
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int base = a.expert_offset[e] + a.tile_pre[(int64_t)tile * E + e];
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int c = s_base[w * E + e];
            s_base[w * E + e] = base;
            base += c;
        }
    }
    __syncthreads();

    // Pass 2: row = running base of the expert + rank among equal ids in lower lanes.
    for (int c = w_begin; c < w_begin + seg; c += 32) {
        const int i = c + lane;
        const bool in = i < w_end;
        const int e = in ? valid_id(__ldg(a.ids + p0 + i), E) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int b = (e >= 0) ? mine[e] : 0;
        if (in) a.pos[p0 + i] = (e >= 0) ? b + __popc(peers & lanemask_lt(lane)) : -1;
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] = b + __popc(peers);
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t s, int64_t* launches)
{
    const int64_t tpt = layout_tokens_per_tile(a.K);
    const int64_t ntiles = layout_tiles(a.T, a.K);
    if (ntiles > 0) {
        layout_count_kernel<<<(unsigned)ntiles, kLayoutThreads, 0, s>>>(a, tpt);
        ++*launches;
    }
    layout_scan_kernel<<<1, 1024, 0, s>>>(a, (int)ntiles);
    ++*launches;
    if (ntiles > 0) {
        layout_pos_kernel<<<(unsigned)ntiles, kLayoutThreads, 0, s>>>(a, tpt);
        ++*launches;
    }
    return cudaGetLastError();
}

}  // namespace ep
