// permute.cu - dispatch permute: copy each token row into the receive rows
// of its experts, with the row's score and source pair index.
//
// Follows "Unify expert parallel token dispatcher API", section "Backend
// behavior" (HybridEP: non-blocking dispatch sizes the fused-permute output by
// the current capacity; DeepEP: the current capacity is the per-rank layout
// stride).
//
// HBM-bound: reads T rows and writes up to T*K rows. Kernels:
//   dispatch_tile<ONEPASS, SMALL> : one CTA (8 warps) per layout tile, about
//                    one per SM. Thread 0 starts bulk async loads of the
//                    tile's rows into a shared-memory ring before the layout
//                    is known (the rows do not depend on it). The one-pass
//                    form (the default, a cooperative launch; it first waits
//                    for the previous kernel in the stream) counts its tile,
//                    meets every other CTA at a grid barrier and derives its
//                    prefixes from all tiles' counts; with SMALL (calls of
//                    few pairs) every CTA counts all of the call's ids instead
//                    and there is no barrier; the fused form waits for the
//                    separate count and scan kernels. Then all warps compute
//                    the tile's positions into shared memory, and warp 0
//                    streams the rows out: lane k issues the bulk store of
//                    destination k; warps 1-7 write scores and sources. CTAs
//                    that finish their own tokens take the last ones of the
//                    others from a shared pool. Completion of loads is tracked
//                    by mbarriers (bounded waits); a slot is reused only after
//                    its stores have read it (cp.async.bulk.wait_group.read).
//   permute_bulk   : the same ring for a standalone permute (positions from
//                    global memory, prefetched two tokens ahead), one warp per
//                    CTA, one CTA per SM, tokens strided by the grid.
//   permute_vec    : a CTA per token (grid-stride); each thread loads its
//                    16-byte vectors of the row once and stores them to every
//                    destination row.
// No multicast and no clusters: plain 1-D bulk copies within one CTA.
#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kVecThreads = 128;
constexpr int kBulkLag = 2;            // store groups in flight before a slot is reused
constexpr int kPoolAhead = 2;          // pool tokens taken ahead of the one being copied
constexpr int kBulkMaxStages = 32;
constexpr int kBulkSmemBudget = 200 * 1024;
constexpr int kFusedSmemCap = 227 * 1024 - 1024;   // dynamic shared memory of the fused kernel
constexpr int kOnepassStaticReserve = 2048;         // the one-pass kernel's extra static arrays

int slot_bytes_of(int64_t row_bytes) { return (int)((row_bytes + 127) / 128 * 128); }

template <int U>
__global__ void __launch_bounds__(kVecThreads)
permute_vec_kernel(PermuteArgs a)
{
    __shared__ int s_pos[kMaxTopk];
    griddep_wait();
    const int64_t V = a.row_bytes / 16;
    const int4* __restrict__ x = static_cast<const int4*>(a.x);
    int4* __restrict__ rx = static_cast<int4*>(a.recv_x);

    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        if (threadIdx.x < a.K) {
            const int64_t q = t * a.K + threadIdx.x;
            const int p = __ldcg(a.pos + q);
            s_pos[threadIdx.x] = p;
            if (p >= 0) {
                a.recv_scores[p] = __ldcg(a.scores + q);
                a.recv_src[p] = (int32_t)q;
            }
        }
        __syncthreads();
        const int4* src = x + t * V;
        for (int64_t v0 = threadIdx.x; v0 < V; v0 += (int64_t)U * kVecThreads) {
            int4 r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + (int64_t)u * kVecThreads;
                if (v < V) r[u] = ld_cg_v4(src + v);
            }
            for (int k = 0; k < a.K; ++k) {
                const int p = s_pos[k];
                if (p < 0) continue;
                int4* dst = rx + (int64_t)p * V;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t v = v0 + (int64_t)u * kVecThreads;
                    if (v < V) dst[v] = r[u];
                }
            }
        }
        __syncthreads();
    }
    griddep_launch_dependents();
}

// After a timed-out wait: lets every load this CTA issued (tokens [from, to)
// except `skipped`, which was never issued) land before the CTA's shared memory
// is released, under one shared deadline.
__device__ void drain_loads(uint32_t bar0, int stages, int64_t from, int64_t to, int64_t skipped)
{
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    for (int64_t m = from; m < to; ++m)
        if (m != skipped)
            mbar_wait_until(bar0 + 8u * (uint32_t)(m % stages), (uint32_t)((m / stages) & 1),
                            deadline);
}

// One warp per CTA. Lane 0 issues the row loads; lane k < K issues the store
// of destination k and writes its score and source index. Tokens of CTA b:
// b, b + G, b + 2G, ... (G = gridDim.x). Slot of the i-th token: i % stages.
__global__ void __launch_bounds__(32, 1)
permute_bulk_kernel(PermuteArgs a, int stages, int slot_bytes)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kBulkMaxStages];
    const int lane = threadIdx.x;
    const int64_t G = gridDim.x;
    const int64_t b = blockIdx.x;
    griddep_wait();
    if (b >= a.T) return;
    const int64_t n_my = (a.T - 1 - b) / G + 1;
    const uint32_t bytes = static_cast<uint32_t>(a.row_bytes);
    const uint32_t slot0 = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    const uint8_t* __restrict__ x = static_cast<const uint8_t*>(a.x);
    uint8_t* __restrict__ rx = static_cast<uint8_t*>(a.recv_x);
    const int K = a.K;

    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8u * s, 1u);
        fence_mbar_init();
    }
    __syncwarp();

    const int64_t skipped = (b == 0) ? a.skip_load : -1;
    auto issue_load = [&](int64_t i) {
        if (i == skipped) return;
        const int s = (int)(i % stages);
        const uint32_t bar = bar0 + 8u * s;
        mbar_expect_tx(bar, bytes);
        bulk_g2s(slot0 + (uint32_t)s * (uint32_t)slot_bytes, x + (b + i * G) * a.row_bytes, bytes,
                 bar);
    };
    const int64_t n_pro = n_my < stages ? n_my : stages;
    if (lane == 0)
        for (int64_t i = 0; i < n_pro; ++i) issue_load(i);

    // Positions and scores of tokens i and i+1 live in registers; token i+2's
    // are fetched at the top of iteration i so their latency hides behind the wait.
    auto fetch = [&](int64_t i, int& p, float& w) {
        p = -1;
        w = 0.f;
        if (i < n_my && lane < K) {
            const int64_t q = (b + i * G) * K + lane;
            p = __ldcg(a.pos + q);
            w = __ldcg(a.scores + q);
        }
    };
    int p_cur, p_nxt;
    float w_cur, w_nxt;
    fetch(0, p_cur, w_cur);
    fetch(1, p_nxt, w_nxt);

    bool ok = true;
    int64_t i = 0;
    for (; i < n_my; ++i) {
        int p_nn;
        float w_nn;
        fetch(i + 2, p_nn, w_nn);
        const int s = (int)(i % stages);
        if (!mbar_wait(bar0 + 8u * s, (uint32_t)((i / stages) & 1))) {
            ok = false;
            break;
        }
        if (p_cur >= 0) {
            bulk_s2g(rx + (int64_t)p_cur * a.row_bytes, slot0 + (uint32_t)s * (uint32_t)slot_bytes,
                     bytes);
            a.recv_scores[p_cur] = w_cur;
            a.recv_src[p_cur] = (int32_t)((b + i * G) * K + lane);
        }
        bulk_commit();
        const int64_t j = i - kBulkLag;
        if (j >= 0 && j + stages < n_my) {
            bulk_wait_read<kBulkLag>();   // this lane's stores of token j have read their slot
            __syncwarp();
            if (lane == 0) issue_load(j + stages);
        }
        p_cur = p_nxt;
        w_cur = w_nxt;
        p_nxt = p_nn;
        w_nxt = w_nn;
    }
    bulk_wait_all();
    if (!ok && lane == 0) {
        atomicOr(a.err, kErrTimeout);
        int64_t issued_hi = (i - kBulkLag) + stages;   // loads issued for tokens < issued_hi
        if (issued_hi < n_pro) issued_hi = n_pro;
        drain_loads(bar0, stages, i, issued_hi < n_my ? issued_hi : n_my, skipped);
    }
    griddep_launch_dependents();
}

// Layout of a small call without a grid barrier: every CTA counts all of the
// call's pairs itself (its ids stay in L2 after the first CTA reads them), so
// the CTAs never wait for one another. s_tot[e] = pairs of expert e in the
// call; s_seed[e] = those before this tile's first pair; tile 0 also counts
// each rank's distinct tokens into s_rank[2] and reports invalid ids.
// Ends with __syncthreads.
__device__ void redundant_counts(const LayoutArgs& L, int tile, int* s_seed, int* s_tot,
                                 int (*s_rank)[kMaxRanks])
{
    const int64_t np = L.T * L.K;
    const int64_t p0 = (int64_t)tile * L.tpt * L.K;   // this tile's first pair
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e = threadIdx.x; e < L.Ep; e += blockDim.x) {
        s_seed[e] = 0;
        s_tot[e] = 0;
    }
    if (threadIdx.x < L.R) s_rank[2][threadIdx.x] = 0;
    __syncthreads();
    const int64_t np32 = (np + 31) & ~(int64_t)31;
    bool bad = false;
    // Warp w takes the 32-pair chunks w, w + 8, ...; each lane loads the ids of
    // kRedBatch chunks before matching them, so the loads are in flight together.
    constexpr int kRedBatch = 16;
    for (int64_t cb = (int64_t)warp * 32; cb < np32; cb += (int64_t)kRedBatch * kLayoutThreads) {
        int raw[kRedBatch];
#pragma unroll
        for (int u = 0; u < kRedBatch; ++u) {
            const int64_t i = cb + (int64_t)u * kLayoutThreads + lane;
            raw[u] = (i < np) ? __ldcg(L.ids + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < kRedBatch; ++u) {
            const int64_t c = cb + (int64_t)u * kLayoutThreads;
            if (c >= np32) break;   // the same for every lane of the warp
            const int e = valid_id(raw[u], L.E);
            bad |= (e != raw[u]);
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && lane == __ffs(peers) - 1) {
                atomicAdd(&s_tot[e], __popc(peers));
                // lanes of this chunk whose pair comes before the tile
                const unsigned before = (c + 32 <= p0) ? 0xffffffffu
                                        : (c >= p0)    ? 0u
                                                       : (1u << (unsigned)(p0 - c)) - 1u;
                const int nb = __popc(peers & before);
                if (nb) atomicAdd(&s_seed[e], nb);
            }
        }
    }
    if (tile == 0) {
        if (bad) atomicOr(L.err, kErrBadId);
        // Distinct tokens per rank over the call: the rank set of every token,
        // kTokBatch tokens per thread with their first 8 ids loaded together.
        constexpr int kTokBatch = 4;
        const int eloc = L.E / L.R;
        for (int64_t tb = threadIdx.x; tb < L.T; tb += (int64_t)kTokBatch * kLayoutThreads) {
            unsigned long long mask[kTokBatch];
#pragma unroll
            for (int u = 0; u < kTokBatch; ++u) {
                mask[u] = 0ull;
                const int64_t t = tb + (int64_t)u * kLayoutThreads;
                if (t >= L.T) continue;
                int e8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    e8[k] = (k < L.K) ? valid_id(__ldcg(L.ids + t * L.K + k), L.E) : -1;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (e8[k] >= 0) mask[u] |= 1ull << (e8[k] / eloc);
                for (int k = 8; k < L.K; ++k) {
                    const int e = valid_id(__ldcg(L.ids + t * L.K + k), L.E);
                    if (e >= 0) mask[u] |= 1ull << (e / eloc);
                }
            }
#pragma unroll
            for (int u = 0; u < kTokBatch; ++u)
                while (mask[u]) {
                    atomicAdd(&s_rank[2][__ffsll((long long)mask[u]) - 1], 1);
                    mask[u] &= mask[u] - 1ull;
                }
        }
    }
    __syncthreads();
}

// Receive rows of pool token t for lane k < K: read from the positions its
// owner tile published (L.pos), once that tile's ready word holds this call's
// generation. -1 if the word does not come within the wait limit (then
// kErrTimeout is set and the row is skipped).
__device__ __forceinline__ int pool_pos(const LayoutArgs& L, int64_t t, int k, uint32_t epoch,
                                        uint32_t* err)
{
    const uint32_t* flag = L.tile_ready + t / L.tpt;
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    while (true) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v == epoch) break;
        if (globaltimer_ns() > deadline) {
            atomicOr(err, kErrTimeout);
            return -1;
        }
        __nanosleep(32);
    }
    return __ldcg(L.pos + t * L.K + k);
}

// Positions + permute of one layout tile per CTA (see the file comment).
// ONEPASS: the layout is computed here too (onepass_layout; launched
// cooperatively, so every tile's CTA is resident for the grid barrier).
// Shared memory: [stages slots of slot_bytes][kLayoutWarps * Ep ints][tile pairs
// ints] (+ ONEPASS: [3 * Ep ints]).
//
// Rows are copied in a sequence of tokens through the ring: the tile's own
// tokens first, then (ONEPASS with pool_d > 0) tokens taken from a pool shared
// by all CTAs, so that CTAs which finish early take over the others' last
// rows. The pool holds the last d = min(pool_d, n - stages) tokens of every
// tile of n tokens; pool entry c is token c / ntiles of tile c % ntiles's
// share. Whoever copies a row, the owner tile writes its scores and sources
// and publishes its positions (L.pos) for the others.
template <bool ONEPASS, bool SMALL>
__global__ void __launch_bounds__(kLayoutThreads, 1)
dispatch_tile_kernel(LayoutArgs L, PermuteArgs a, int stages, int slot_bytes, int pool_d)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kBulkMaxStages];
    __shared__ int s_seq[kBulkMaxStages];   // pool token in each ring slot, -1: none
    int* s_base = reinterpret_cast<int*>(smem + (size_t)stages * slot_bytes);
    int* s_pos = s_base + kLayoutWarps * L.Ep;
    const int tile = blockIdx.x;
    const int64_t t0 = (int64_t)tile * L.tpt;
    const int64_t t1 = min(L.T, t0 + L.tpt);
    const int n_my = (int)(t1 - t0);
    const int64_t p0 = t0 * L.K;
    const int K = L.K;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bytes = static_cast<uint32_t>(a.row_bytes);
    const uint32_t slot0 = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    const uint8_t* __restrict__ x = static_cast<const uint8_t*>(a.x);
    uint8_t* __restrict__ rx = static_cast<uint8_t*>(a.recv_x);
    const bool pooled = ONEPASS && !SMALL && pool_d > 0;
    // This tile's pool share and the tokens it keeps.
    auto share = [&](int n) { return pooled ? min(pool_d, max(0, n - stages)) : 0; };
    const int n_static = n_my - share(n_my);
    const int n_pro = n_static < stages ? n_static : stages;
    const uint32_t pool_total = pooled ? (uint32_t)L.ntiles * (uint32_t)pool_d : 0u;
    bool pool_empty = !pooled;   // thread 0 only
    // Sequence indices issued before the copy loop starts.
    const int pool_first_issue = pooled ? max(n_pro, min(stages, kPoolAhead + 1)) : n_pro;

    const int64_t skipped = (tile == 0) ? a.skip_load : -1;
    // Whether receive row p is to be written: p >= 0 and inside the call's
    // R * S rows. Positions always are when the layout is sound; one outside
    // (possible only if the grid barrier's words were corrupted and it opened
    // early) is skipped and reported, so that no store leaves the buffer.
    const int64_t rows_cap = (int64_t)L.R * L.S;
    auto in_rows = [&](int p) {
        if (p < 0) return false;
        if ((int64_t)p < rows_cap) return true;
        atomicOr(a.err, kErrRowOob);
        return false;
    };
    // Starts the load of sequence index q into its slot: an own token, or the
    // next pool token (recorded in s_seq; -1 once the pool is empty).
    auto issue = [&](int q) {
        const int s = q % stages;
        int64_t t = -1;
        if (q < n_static) {
            if (q == skipped) return;
            t = t0 + q;
        } else {
            while (!pool_empty) {
                const uint32_t c = atomicAdd(L.gbar + 2, 1u);
                if (c >= pool_total) {
                    pool_empty = true;
                    break;
                }
                const int ot = (int)(c % (uint32_t)L.ntiles), j = (int)(c / (uint32_t)L.ntiles);
                const int64_t o0 = (int64_t)ot * L.tpt;
                const int on = (int)(min(L.T, o0 + L.tpt) - o0);
                const int od = share(on);
                if (j < od) {
                    t = o0 + (on - od) + j;
                    break;
                }
            }
            s_seq[s] = (int)t;
            if (t < 0) return;
        }
        const uint32_t bar = bar0 + 8u * s;
        mbar_expect_tx(bar, bytes);
        bulk_g2s(slot0 + (uint32_t)s * (uint32_t)slot_bytes, x + t * a.row_bytes, bytes, bar);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(bar0 + 8u * s, 1u);
            s_seq[s] = -1;
        }
        fence_mbar_init();
        // The rows do not depend on the layout: the fused form starts them
        // before waiting for it. Its predecessors are this call's count and
        // scan kernels, which allow it to start only after their own waits,
        // so every kernel before them has completed by then. (The one-pass
        // form waits on entry and starts them right after its histogram.)
        if constexpr (!ONEPASS)
            for (int i = 0; i < n_pro; ++i) issue(i);
    }

    uint32_t epoch = 0;
    if constexpr (ONEPASS) {
        // Inputs (ids, x, scores) may come from the previous kernel in the
        // stream: wait for it before the first read (this costs nothing
        // measurable, as the previous kernel is at its end by then).
        griddep_wait();
        __shared__ int s_rank[3][kMaxRanks];
        __shared__ int s_tok[kMaxRanks];
        __shared__ int s_wsum[kLayoutWarps];
        __shared__ int s_flag;
        __shared__ uint32_t s_epoch;
        const int tile_pairs = (int)(L.tpt * L.K);
        int* s_seed = s_pos + tile_pairs;
        int* s_tot = s_seed + L.Ep;
        int* s_off = s_tot + L.Ep;
        bool ok = true;
        if constexpr (SMALL) {
            // A small call: no grid barrier (see redundant_counts), no pool.
            redundant_counts(L, tile, s_seed, s_tot, s_rank);
            if (threadIdx.x == 0)
                for (int i = 0; i < n_pro; ++i) issue(i);
            layout_offsets(L, s_base, s_seed, s_tot, s_off, s_rank, s_wsum);
            s_epoch = 0u;
        } else {
            ok = onepass_layout(L, tile, s_base, s_seed, s_tot, s_off, s_rank, s_tok, s_wsum,
                                &s_flag, &s_epoch, s_pos, nullptr, [&] {
                                    for (int i = 0; i < n_pro; ++i) issue(i);
                                });
        }
        if (!ok) {   // barrier timed out: report, let this CTA's loads land, leave
            if (threadIdx.x == 0) {
                atomicOr(a.err, kErrTimeout);
                drain_loads(bar0, stages, 0, n_pro, skipped);
            }
            griddep_launch_dependents();
            return;
        }
        epoch = s_epoch;
        if (tile == 0) {
            for (int e = threadIdx.x; e < L.E; e += blockDim.x) {
                L.cnt[e] = s_tot[e];
                L.expert_offset[e] = s_off[e];
            }
            if (threadIdx.x < L.R) {
                L.rows_per_rank[threadIdx.x] = s_rank[0][threadIdx.x];
                L.rank_prefix[threadIdx.x] = s_rank[1][threadIdx.x];
                L.tokens_in_rank[threadIdx.x] = s_rank[2][threadIdx.x];
            }
        }
        // The barrier form kept the tile's ids in s_pos (onepass_layout).
        tile_positions(L, tile, s_base, L.pos, s_pos, s_seed,
                       SMALL ? nullptr : s_pos);   // ends with __syncthreads
        if (pooled) {
            // Publish this tile's positions for the CTAs that copy its pool rows:
            // the block barrier that ends tile_positions orders every thread's
            // position writes before thread 32's fence and release (cumulativity),
            // so warp 0 starts copying without waiting for the fence.
            if (threadIdx.x == 32) {
                __threadfence();
                asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(L.tile_ready + tile),
                             "r"(epoch)
                             : "memory");
            }
            // A tile shorter than the ring takes its first pool tokens now (the
            // pool's rows do not depend on any position).
            if (threadIdx.x == 0)
                for (int q = n_pro; q < pool_first_issue; ++q) issue(q);
            if (warp == 0) __syncwarp();   // s_seq, written by lane 0, is read by the warp
        }
    } else {
        griddep_wait();                                   // counts and offsets are ready
        tile_positions(L, tile, s_base, L.pos, s_pos);    // ends with __syncthreads
    }

    if (warp == 0) {
        bool ok = true;
        int i = 0;
        int next = pool_first_issue;   // next sequence index to issue (the same in every lane)
        for (;; ++i) {
            const int s = i % stages;
            int64_t t = -1;
            if (i < n_static) {
                t = t0 + i;
            } else if (pooled) {
                t = s_seq[s];
            }
            if (t < 0) break;
            if (!mbar_wait(bar0 + 8u * s, (uint32_t)((i / stages) & 1))) {
                ok = false;
                break;
            }
            if (lane < K) {
                const int p = (i < n_static) ? s_pos[i * K + lane]
                                             : pool_pos(L, t, lane, epoch, a.err);
                if (in_rows(p))
                    bulk_s2g(rx + (int64_t)p * a.row_bytes,
                             slot0 + (uint32_t)s * (uint32_t)slot_bytes, bytes);
            }
            bulk_commit();
            // Loads up to the last index whose slot is free: own tokens as far
            // ahead as the ring allows (a slot is reused once the stores of
            // kBulkLag groups back have read it), pool tokens only kPoolAhead
            // ahead, so that no CTA holds many pool tokens when the pool runs
            // dry (a token's stores take longer than a row load).
            int target = (i >= kBulkLag) ? i - kBulkLag + stages : stages - 1;
            target = pooled ? min(target, max(n_static - 1, i + kPoolAhead))
                            : min(target, n_my - 1);
            if (next <= target) {
                if (target >= stages) bulk_wait_read<kBulkLag>();
                __syncwarp();
                if (lane == 0)
                    for (int q = next; q <= target; ++q) issue(q);
                next = target + 1;
            }
            __syncwarp();
        }
        bulk_wait_all();
        if (!ok && lane == 0) {
            atomicOr(a.err, kErrTimeout);
            // Loads were issued for sequence indices below `next`; pool indices
            // whose slot holds no token had none.
            const int hi = next;
            const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
            for (int m = i; m < hi; ++m) {
                if (m >= n_static && (!pooled || s_seq[m % stages] < 0)) continue;
                if (m == skipped) continue;
                mbar_wait_until(bar0 + 8u * (uint32_t)(m % stages), (uint32_t)((m / stages) & 1),
                                deadline);
            }
        }
    } else {
        const int np = n_my * K;
        for (int j = threadIdx.x - 32; j < np; j += kLayoutThreads - 32) {
            const int p = s_pos[j];
            if (in_rows(p)) {
                a.recv_scores[p] = __ldcg(a.scores + p0 + j);
                a.recv_src[p] = (int32_t)(p0 + j);
            }
        }
    }
    griddep_launch_dependents();
}

int vec_unroll(int64_t row_bytes)
{
    const int64_t V = row_bytes / 16;
    int64_t u = (V + kVecThreads - 1) / kVecThreads;
    if (u < 1) u = 1;
    if (u > 8) u = 8;
    return (int)u;
}

}  // namespace

cudaError_t plan_permute(int impl, int64_t row_bytes, int K, int E, int num_sms, int tiles_per_sm,
                         PermutePlan* plan)
{
    (void)E;
    plan->impl = impl;
    plan->stages = 0;
    plan->smem_bytes = 0;
    plan->fused_smem_cap = 0;
    const int slot = slot_bytes_of(row_bytes);
    if (impl == 2) {
        int stages = kBulkSmemBudget / slot;
        if (stages > kBulkMaxStages) stages = kBulkMaxStages;
        if (stages < kBulkLag + 2 || row_bytes > (1 << 20) || K > 32) {
            plan->impl = impl = 1;   // rows too large for a useful ring, or K > a warp
        } else {
            plan->stages = stages;
            plan->smem_bytes = stages * slot;
            cudaError_t e = cudaFuncSetAttribute(permute_bulk_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 plan->smem_bytes);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(dispatch_tile_kernel<false, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemCap);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(dispatch_tile_kernel<true, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kFusedSmemCap - kOnepassStaticReserve);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(dispatch_tile_kernel<true, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kFusedSmemCap - kOnepassStaticReserve);
            if (e != cudaSuccess) return e;
            // Each fused CTA on an SM gets its share (minus the per-CTA reserve).
            plan->fused_smem_cap =
                tiles_per_sm <= 1 ? kFusedSmemCap : (kFusedSmemCap + 1024) / tiles_per_sm - 1536;
            plan->grid = num_sms;
            return cudaSuccess;
        }
    }
    int per_sm = 0;
    cudaError_t e;
    switch (vec_unroll(row_bytes)) {
#define EP_OCC(U)                                                                              \
    case U:                                                                                    \
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, permute_vec_kernel<U>,       \
                                                          kVecThreads, 0);                     \
        break;
        EP_OCC(1) EP_OCC(2) EP_OCC(3) EP_OCC(4) EP_OCC(5) EP_OCC(6) EP_OCC(7) EP_OCC(8)
#undef EP_OCC
        default:
            return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    plan->grid = num_sms * (per_sm > 0 ? per_sm : 1);
    return cudaSuccess;
}

cudaError_t launch_permute(const PermuteArgs& a, const PermutePlan& plan, const LaunchOpts& o)
{
    if (a.T <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)(a.T < plan.grid ? a.T : plan.grid);
    if (plan.impl == 2)
        return launch_kernel(permute_bulk_kernel, dim3(grid), dim3(32), (size_t)plan.smem_bytes, o,
                             a, plan.stages, slot_bytes_of(a.row_bytes));
    switch (vec_unroll(a.row_bytes)) {
#define EP_LAUNCH(U) \
    case U:          \
        return launch_kernel(permute_vec_kernel<U>, dim3(grid), dim3(kVecThreads), 0, o, a);
        EP_LAUNCH(1) EP_LAUNCH(2) EP_LAUNCH(3) EP_LAUNCH(4)
        EP_LAUNCH(5) EP_LAUNCH(6) EP_LAUNCH(7) EP_LAUNCH(8)
#undef EP_LAUNCH
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dispatch_fused(const LayoutArgs& l, const PermuteArgs& p,
                                  const PermutePlan& plan, const LaunchOpts& o)
{
    if (plan.impl != 2 || plan.fused_smem_cap <= 0 || l.K > 32) return cudaErrorNotSupported;
    if (l.ntiles <= 0) return cudaSuccess;
    const int64_t tile_pairs = l.tpt * l.K;
    if (tile_pairs > kMaxTilePairs) return cudaErrorNotSupported;
    const int slot = slot_bytes_of(p.row_bytes);
    const int64_t fixed = ((int64_t)kLayoutWarps * l.Ep + tile_pairs) * 4;
    int64_t stages = (plan.fused_smem_cap - fixed) / slot;
    if (stages > kBulkMaxStages) stages = kBulkMaxStages;
    if (stages < kBulkLag + 2) return cudaErrorNotSupported;
    const size_t smem = (size_t)(stages * slot + fixed);
    return launch_kernel(dispatch_tile_kernel<false, false>, dim3(l.ntiles), dim3(kLayoutThreads),
                         smem, o, l, p, (int)stages, slot, 0);
}

cudaError_t launch_dispatch_onepass(const LayoutArgs& l, const PermuteArgs& p,
                                    const PermutePlan& plan, const LaunchOpts& o, bool pdl_ok,
                                    int pool_pct, int64_t small_pairs)
{
    if (plan.impl != 2 || plan.fused_smem_cap <= 0 || l.K > 32 || !l.gbar || l.ntiles <= 0)
        return cudaErrorNotSupported;
    const int64_t tile_pairs = l.tpt * l.K;
    if (tile_pairs > kMaxTilePairs) return cudaErrorNotSupported;
    const int slot = slot_bytes_of(p.row_bytes);
    const int64_t fixed = ((int64_t)kLayoutWarps * l.Ep + tile_pairs + 3 * (int64_t)l.Ep) * 4;
    int64_t stages = (plan.fused_smem_cap - kOnepassStaticReserve - fixed) / slot;
    if (stages > kBulkMaxStages) stages = kBulkMaxStages;
    if (stages < kBulkLag + 2) return cudaErrorNotSupported;
    const size_t smem = (size_t)(stages * slot + fixed);
    // A call of at most small_pairs pairs counts all its ids in every CTA
    // instead of meeting at the grid barrier (and then has no pool): a kernel
    // of its own, so that the barrier form carries none of its code.
    const bool small = l.T * l.K <= small_pairs;
    void (*kernel)(LayoutArgs, PermuteArgs, int, int, int) =
        small ? dispatch_tile_kernel<true, true> : dispatch_tile_kernel<true, false>;
    // Every CTA must be resident at once for the grid barrier.
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kLayoutThreads, smem) !=
            cudaSuccess)
        return cudaErrorNotSupported;
    if ((int64_t)per_sm * sms < l.ntiles) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(l.ntiles);
    cfg.blockDim = dim3(kLayoutThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = o.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (o.pdl && pdl_ok) ? 2 : 1;
    // Tokens of each full tile given to the shared pool. A tile keeps at least
    // a ring's worth of its own tokens (those are loaded before the layout is
    // known), so tiles that fit the ring give none and there is no pool.
    int64_t pool_d = 0;
    if (!small && l.tile_ready && pool_pct > 0) {
        pool_d = l.tpt * (pool_pct < 100 ? pool_pct : 100) / 100;
        if (pool_d > l.tpt - stages) pool_d = l.tpt - stages;
        if (pool_d < 0) pool_d = 0;
    }
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, l, p, (int)stages, slot, (int)pool_d);
    if (e == cudaErrorCooperativeLaunchTooLarge) {   // fewer SMs than the device reports (MPS)
        cudaGetLastError();
        return cudaErrorNotSupported;
    }
    if (e == cudaSuccess && o.launches) ++*o.launches;
    return e;
}

namespace {
__global__ void coop_probe_kernel(int* out)
{
    if (threadIdx.x == 0 && blockIdx.x == 0 && out) *out = 1;
}
}  // namespace

bool probe_cooperative_pdl()
{
    int* d = nullptr;
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return false;
    bool ok = false;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(32);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, coop_probe_kernel, d) == cudaSuccess &&
        cudaLaunchKernelEx(&cfg, coop_probe_kernel, d) == cudaSuccess &&
        cudaStreamSynchronize(s) == cudaSuccess)
        ok = true;
    cudaGetLastError();
    cudaStreamDestroy(s);
    return ok;
}

}  // namespace ep
