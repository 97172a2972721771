// ep_device.cuh - device helpers shared by the layout, permute, combine,
// dedupe and GEMM kernels: programmatic-dependent-launch controls, id checks,
// mbarrier and bulk-async-copy wrappers (hand-written PTX), the per-tile
// expert histogram, the stable per-tile position pass and the grid barrier
// of the one-pass dispatch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ep_kernels.cuh"

namespace ep {

// ---- programmatic dependent launch -----------------------------------------
// Kernels are launched so that they may start while their predecessor in the
// stream finishes (the combine is the exception: in captured graphs an early
// combine measured slower). A kernel calls griddep_wait() before touching
// memory its predecessor may write or read, and griddep_launch_dependents()
// once its own successor may start its prologue. Both are no-ops for a normal
// launch.

__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- loads of data another kernel wrote ----------------------------------
// Kernels may start before their predecessor finishes (above), so data written
// by an earlier kernel is read with L2-coherent loads (ld.global.cg), never
// through the non-coherent L1 path.

__device__ __forceinline__ int4 ld_cg_v4(const void* p)
{
    int4 v;
    asm volatile("ld.global.cg.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Whether receive row p holds data: inside its rank's true total, read from
// the device prefix sum ("ep: graph-safe worst-token HT dispatch+combine",
// "Internode" item 3): p - r*S < rank_prefix[r] - rank_prefix[r-1] for
// r = p / S (strided), or p < rank_prefix[R-1] (packed).
__device__ __forceinline__ bool row_valid(int p, int64_t S, int R, const int32_t* rank_prefix,
                                          bool packed)
{
    if (p < 0) return false;
    if (packed) return p < __ldcg(rank_prefix + R - 1);
    const int64_t r = (int64_t)p / S;
    if (r >= R) return false;
    const int lo = (r > 0) ? __ldcg(rank_prefix + r - 1) : 0;
    return ((int64_t)p - r * S) < (int64_t)(__ldcg(rank_prefix + r) - lo);
}

// ---- ids ---------------------------------------------------------------------

__device__ __forceinline__ int valid_id(int e, int E) { return (e >= -1 && e < E) ? e : -1; }

__device__ __forceinline__ unsigned lanemask_lt(int lane) { return (1u << lane) - 1u; }

// ---- mbarrier and bulk async copies ------------------------------------------

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // bounded waits (then kErrTimeout)

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0u;
}

// False if the phase has not completed by the deadline (%globaltimer ns).
__device__ __forceinline__ bool mbar_wait_until(uint32_t bar, uint32_t parity, uint64_t deadline)
{
    while (true) {
        for (int it = 0; it < 64; ++it)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() > deadline) return false;
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_until(bar, parity, globaltimer_ns() + kWaitLimitNs);
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---- stable positions of one layout tile ------------------------------------
//
// Receive row of each pair of tile `tile` (tokens [t0, t1), flat pairs
// [p0, p0 + np)): expert_offset[e] + tile_pre[tile][e] + (pairs with the same
// expert in the earlier warps' segments) + (peers in lower lanes of the same
// 32-pair chunk). Warp w owns the flat pairs [w*seg, w*seg + seg) of the tile,
// so the order is the flat pair order t*K + k. Called by all kLayoutThreads
// threads of the block; s_base holds kLayoutWarps * Ep ints. Writes the rows
// to pos_out (global) and, if s_pos is given, to s_pos[i] (shared). If s_seed
// is given, s_seed[e] replaces expert_offset[e] + tile_pre[tile][e]. If s_ids
// is given, it holds the tile's ids as tile_histogram kept them, and they are
// read from there instead of from global memory (s_ids may be s_pos: each
// entry is read before its position is written over it).
__device__ __forceinline__ void tile_positions(const LayoutArgs& a, int tile, int* s_base,
                                               int32_t* pos_out, int* s_pos,
                                               const int* s_seed = nullptr,
                                               const int* s_ids = nullptr)
{
    const int64_t t0 = (int64_t)tile * a.tpt;
    const int64_t t1 = min(a.T, t0 + a.tpt);
    const int64_t p0 = t0 * a.K;
    const int np = (int)((t1 - t0) * a.K);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int E = a.E, Ep = a.Ep;
    const int seg = (((np + kLayoutWarps - 1) / kLayoutWarps) + 31) & ~31;
    const int w_begin = warp * seg;
    const int w_end = min(np, w_begin + seg);
    int* mine = s_base + warp * Ep;

    for (int i = threadIdx.x; i < kLayoutWarps * Ep; i += blockDim.x) s_base[i] = 0;
    __syncthreads();

    // Pass 1: per-warp histogram (one writer per row, one add per peer group).
    for (int c = w_begin; c < w_begin + seg; c += 32) {
        const int i = c + lane;
        const int e = (i >= w_end) ? -1 : s_ids ? s_ids[i] : valid_id(__ldcg(a.ids + p0 + i), E);
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // Exclusive prefix over warps, seeded with the expert's first row and the
    // counts of all earlier tiles (from s_seed when the caller has them).
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int base = s_seed ? s_seed[e]
                          : __ldcg(a.expert_offset + e) + __ldcg(a.tile_pre + (int64_t)tile * Ep + e);
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int c = s_base[w * Ep + e];
            s_base[w * Ep + e] = base;
            base += c;
        }
    }
    __syncthreads();

    // Pass 2: running base of the expert + rank among equal ids in lower lanes.
    for (int c = w_begin; c < w_begin + seg; c += 32) {
        const int i = c + lane;
        const bool in = i < w_end;
        const int e = !in ? -1 : s_ids ? s_ids[i] : valid_id(__ldcg(a.ids + p0 + i), E);
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int b = (e >= 0) ? mine[e] : 0;
        if (in) {
            const int p = (e >= 0) ? b + __popc(peers & lanemask_lt(lane)) : -1;
            pos_out[p0 + i] = p;
            if (s_pos) s_pos[i] = p;
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] = b + __popc(peers);
        __syncwarp();
    }
    __syncthreads();
}

// ---- per-tile expert histogram -----------------------------------------------
//
// s_hist[e] = pairs of tile `tile` with expert e (e < Ep; zeroed here), s_tok[r]
// = tokens of the tile with at least one expert on rank r. Full warps walk the
// tile so every lane takes part in __match_any_sync (equal ids are grouped and
// one lane per group adds the group size); each thread loads kHistUnroll ids
// before matching them. Invalid ids count as none and set kErrBadId. If s_ids
// is given, the tile's ids (invalid ones as -1) are also kept there, s_ids[i]
// for the tile's pair i, and the rank sets are taken from them. Ends with
// __syncthreads.
constexpr int kHistUnroll = 4;

__device__ __forceinline__ void tile_histogram(const LayoutArgs& a, int tile, int* s_hist,
                                               int* s_tok, int* s_ids = nullptr)
{
    const int64_t t0 = (int64_t)tile * a.tpt;
    const int64_t t1 = min(a.T, t0 + a.tpt);
    const int64_t p0 = t0 * a.K;
    const int np = (int)((t1 - t0) * a.K);
    const int lane = threadIdx.x & 31;
    const int nthr = (int)blockDim.x;

    for (int i = threadIdx.x; i < a.Ep; i += nthr) s_hist[i] = 0;
    if (threadIdx.x < a.R) s_tok[threadIdx.x] = 0;
    __syncthreads();

    const int np32 = (np + 31) & ~31;
    bool bad = false;
    for (int base = 0; base < np32; base += kHistUnroll * nthr) {
        int e[kHistUnroll];
#pragma unroll
        for (int j = 0; j < kHistUnroll; ++j) {
            const int i = base + j * nthr + (int)threadIdx.x;
            const int raw = (i < np) ? __ldcg(a.ids + p0 + i) : -1;
            e[j] = valid_id(raw, a.E);
            bad |= (e[j] != raw);
            if (s_ids && i < np) s_ids[i] = e[j];
        }
#pragma unroll
        for (int j = 0; j < kHistUnroll; ++j) {
            const int warp_first = base + j * nthr + ((int)threadIdx.x & ~31);
            if (warp_first < np32) {
                const unsigned peers = __match_any_sync(0xffffffffu, e[j]);
                if (e[j] >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[e[j]], __popc(peers));
            }
        }
    }
    if (bad) atomicOr(a.err, kErrBadId);
    if (s_ids) __syncthreads();

    // Distinct tokens per logical rank: one 64-bit rank set per token.
    const int eloc = a.E / a.R;
    for (int64_t t = t0 + threadIdx.x; t < t1; t += nthr) {
        unsigned long long mask = 0ull;
#pragma unroll 8
        for (int k = 0; k < a.K; ++k) {
            const int e = s_ids ? s_ids[(t - t0) * a.K + k]
                                : valid_id(__ldcg(a.ids + t * a.K + k), a.E);
            if (e >= 0) mask |= 1ull << (e / eloc);
        }
        while (mask) {
            atomicAdd(&s_tok[__ffsll((long long)mask) - 1], 1);
            mask &= mask - 1ull;
        }
    }
    __syncthreads();
}

// ---- grid barrier ----------------------------------------------------------
//
// For a cooperative launch (every CTA resident). bar[1] is the generation of
// the next barrier; bar[0] and bar[3] count the arrivals of even and odd
// generations. A barrier of generation g is complete once its counter holds
// n: the last arrival's own atomic completes it, and the waiters poll the
// counter itself (one round trip after the last arrival). The last arrival
// also sets the other counter to zero for the next barrier (nothing uses it
// during this one: the kernel that used it has completed) and advances bar[1].
// A waiter tests for exactly n, so a counter left above n never opens.
//
// gen: bar[1] as read by this CTA at the kernel's start (grid_generation),
// which stays unchanged until every CTA of this launch has arrived. Called by
// one thread per CTA after the CTA's writes are fenced; false if the others
// have not arrived within the wait limit (the counters are then inconsistent:
// the host resets every word when it reads the timeout bit). *epoch receives
// gen + 1, the generation this barrier opens.
__device__ __forceinline__ uint32_t grid_generation(const uint32_t* bar)
{
    uint32_t g;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(g) : "l"(bar + 1) : "memory");
    return g;
}

__device__ __forceinline__ bool grid_barrier(uint32_t* bar, uint32_t n, uint32_t gen,
                                             uint32_t* epoch)
{
    *epoch = gen + 1u;
    uint32_t* cnt = bar + ((gen & 1u) ? 3 : 0);
    uint32_t* next = bar + ((gen & 1u) ? 0 : 3);
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(cnt) : "memory");
    if (old + 1u == n) {
        asm volatile("st.relaxed.gpu.global.u32 [%0], 0;" ::"l"(next) : "memory");
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(bar + 1) : "memory");
        return true;
    }
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    while (true) {
        uint32_t c;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(c) : "l"(cnt) : "memory");
        if (c == n) return true;
        if (globaltimer_ns() > deadline) return false;
        __nanosleep(64);
    }
}

// ---- one-pass layout ----------------------------------------------------------

// Second half of the layout, from the call's per-expert totals s_tot[e] and
// this tile's counts of earlier pairs s_seed[e]: s_off[e] = expert_offset[e],
// s_rank[0][r] = rows_per_rank[r], s_rank[1][r] = rank_prefix[r] (inclusive),
// and s_seed[e] += expert_offset[e] (this tile's first receive row of e).
// s_work: at least E ints. Ends with __syncthreads.
__device__ __forceinline__ void layout_offsets(const LayoutArgs& L, int* s_work, int* s_seed,
                                               const int* s_tot, int* s_off,
                                               int (*s_rank)[kMaxRanks], int* s_wsum)
{
    const int Ep = L.Ep, E = L.E, R = L.R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Inclusive prefix of the totals over experts (C consecutive experts per
    // thread, then warps, then the block) into s_off.
    const int C = (Ep + kLayoutThreads - 1) / kLayoutThreads;
    const int e0 = threadIdx.x * C;
    int run = 0;
    for (int j = 0; j < C; ++j) {
        const int e = e0 + j;
        if (e < E) run += s_tot[e];
    }
    int v = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += n;
    }
    if (lane == 31) s_wsum[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int c = s_wsum[w];
            s_wsum[w] = acc;
            acc += c;
        }
    }
    __syncthreads();
    int incl = v - run + s_wsum[warp];   // exclusive prefix of this thread's first expert
    for (int j = 0; j < C; ++j) {
        const int e = e0 + j;
        if (e < E) {
            incl += s_tot[e];
            s_off[e] = incl;
        }
    }
    __syncthreads();

    // Offsets: ranks own contiguous expert blocks (packed: back to back).
    const int eloc = E / R;
    if (threadIdx.x < R) {
        const int r = threadIdx.x;
        const int hi = s_off[(r + 1) * eloc - 1];
        const int lo = (r > 0) ? s_off[r * eloc - 1] : 0;
        s_rank[0][r] = hi - lo;
        s_rank[1][r] = hi;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int excl = s_off[e] - s_tot[e];
        int off;
        if (L.packed) {
            off = excl;
        } else {
            const int r = e / eloc;
            const int lo = (r > 0) ? s_off[r * eloc - 1] : 0;
            off = (int)((int64_t)r * L.S + (excl - lo));
        }
        s_work[e] = off;   // s_off still holds the inclusive prefix other threads read
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        s_off[e] = s_work[e];
        s_seed[e] += s_work[e];
    }
    __syncthreads();
}

// One-pass layout of tile `tile` (the one-pass dispatch and dedupe): this tile's counts, a
// grid barrier, then every tile's counts summed per expert (before this tile,
// and in all) and scanned over experts. Leaves s_seed[e] = this tile's first
// receive row of expert e, s_tot[e] = cnt[e], s_off[e] = expert_offset[e],
// s_rank[0][r] = rows_per_rank[r], s_rank[1][r] = rank_prefix[r],
// s_rank[2][r] = tokens_in_rank[r]. Global writes: this tile's rows of the
// count tables and the barrier words only. False if the barrier timed out.
// s_work: kLayoutWarps * Ep ints. s_ids: the tile's pairs' ids are kept there
// (tile_histogram) for the positions, or null. s_tokpre, if given, receives
// each rank's distinct tokens in the tiles before this one (kMaxRanks ints).
// issue_rows runs on thread 0 right after the histogram.
template <typename IssueRows>
__device__ __forceinline__ bool onepass_layout(const LayoutArgs& L, int tile, int* s_work,
                                               int* s_seed, int* s_tot, int* s_off,
                                               int (*s_rank)[kMaxRanks], int* s_tok,
                                               int* s_wsum, int* s_flag, uint32_t* s_epoch,
                                               int* s_ids, int* s_tokpre, IssueRows issue_rows)
{
    const int Ep = L.Ep, R = L.R, G = (int)gridDim.x;
    // The barrier's generation, read now so that its latency hides behind the
    // histogram (it cannot change before every CTA of this launch arrives).
    const uint32_t gen = threadIdx.x == 0 ? grid_generation(L.gbar) : 0u;
    // The ids first: issued behind the tile's row loads they would wait for
    // those; the rows are started right after the histogram instead (they are
    // in by the time the positions are known).
    tile_histogram(L, tile, s_tot, s_tok, s_ids);   // ends with __syncthreads
    if (threadIdx.x == 0) issue_rows();
    for (int e = threadIdx.x; e < Ep; e += blockDim.x) L.tile_cnt[(int64_t)tile * Ep + e] = s_tot[e];
    if (threadIdx.x < R) L.tile_tok[(int64_t)tile * R + threadIdx.x] = s_tok[threadIdx.x];
    // The token pool's counter starts over for this call: the previous kernel
    // in the stream has completed (the kernel waited for it on entry), and no
    // CTA of this call takes from the pool before the barrier.
    if (tile == 0 && threadIdx.x == 0) L.gbar[2] = 0u;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_flag = grid_barrier(L.gbar, (uint32_t)G, gen, s_epoch) ? 1 : 0;
    __syncthreads();
    if (!*s_flag) return false;

    // Column sums of all tiles' counts: thread (g, q) adds the 4-expert column
    // q over tiles g, g + NG, ... into s_work[2g][.] (tiles before this one)
    // and s_work[2g + 1][.] (all tiles).
    const int Q = Ep / 4;
    int NG = kLayoutThreads / Q;
    if (NG > kLayoutWarps / 2) NG = kLayoutWarps / 2;
    if (NG < 1) NG = 1;
    const int g = threadIdx.x / Q, q = threadIdx.x % Q;
    if (g < NG && q < Q) {
        // Loads in batches of kSumBatch rows, all in flight before the adds.
        constexpr int kSumBatch = 20;
        const int4* tc = reinterpret_cast<const int4*>(L.tile_cnt);
        int4 bef = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
        for (int tb = g; tb < G; tb += kSumBatch * NG) {
            int4 v[kSumBatch];
#pragma unroll
            for (int u = 0; u < kSumBatch; ++u) {
                const int t = tb + u * NG;
                v[u] = (t < G) ? ld_cg_v4(tc + (int64_t)t * Q + q) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kSumBatch; ++u) {
                tot.x += v[u].x; tot.y += v[u].y; tot.z += v[u].z; tot.w += v[u].w;
                if (tb + u * NG < tile) {
                    bef.x += v[u].x; bef.y += v[u].y; bef.z += v[u].z; bef.w += v[u].w;
                }
            }
        }
        int* b = s_work + (2 * g) * Ep + 4 * q;
        int* a = s_work + (2 * g + 1) * Ep + 4 * q;
        b[0] = bef.x; b[1] = bef.y; b[2] = bef.z; b[3] = bef.w;
        a[0] = tot.x; a[1] = tot.y; a[2] = tot.z; a[3] = tot.w;
    }
    // Distinct tokens per rank over all tiles (and over the tiles before this
    // one): thread (g2, r) adds rows g2, g2 + NG2, ...
    const int NG2 = kLayoutThreads / R;
    const int g2 = threadIdx.x / R, r2 = threadIdx.x % R;
    int tsum = 0, tbef = 0;
    if (g2 < NG2)
        for (int t = g2; t < G; t += NG2) {
            const int c = __ldcg(L.tile_tok + (int64_t)t * R + r2);
            tsum += c;
            if (t < tile) tbef += c;
        }
    __syncthreads();
    for (int e = threadIdx.x; e < Ep; e += blockDim.x) {
        int b = 0, a = 0;
        for (int gg = 0; gg < NG; ++gg) {
            b += s_work[(2 * gg) * Ep + e];
            a += s_work[(2 * gg + 1) * Ep + e];
        }
        s_seed[e] = b;
        s_tot[e] = a;
    }
    if (threadIdx.x < R) {
        s_rank[2][threadIdx.x] = 0;
        if (s_tokpre) s_tokpre[threadIdx.x] = 0;
    }
    __syncthreads();
    if (g2 < NG2 && tsum) atomicAdd(&s_rank[2][r2], tsum);
    if (s_tokpre && g2 < NG2 && tbef) atomicAdd(&s_tokpre[r2], tbef);

    layout_offsets(L, s_work, s_seed, s_tot, s_off, s_rank, s_wsum);
    return true;
}

}  // namespace ep
