// dedup.cu - per-rank dedupe: one receive row per distinct (token, rank), and
// the receiver's expansion of those rows into the per-expert layout.
//
// A dispatcher that sends each token to a destination rank once, however
// many of that rank's experts it selected, moves fewer rows ("Unify expert
// parallel token dispatcher API", "Backend behavior": DeepEP's per-rank
// layout; "ep: graph-safe worst-token HT dispatch+combine", "Internode":
// per-rank counts on the device). Rank r owns rows [r*P, r*P +
// tokens_in_rank[r]) in ascending token order; each row carries its source
// token and, per k, the local expert index (or -1) and the score (or 0).
//
// Kernels (after the layout's count and scan, which also leave each tile's
// exclusive prefix of distinct tokens per rank):
//   dedup_fused  : the default. One CTA (8 warps) per layout tile. Thread 0
//                  starts bulk async loads of the tile's rows into a shared-
//                  memory ring before waiting for the scan; then all warps
//                  compute the tile's per-expert positions (kept for the
//                  expansion) and each token's dedupe row per rank (warp
//                  ballots rank the tile's tokens that hit rank r, in token
//                  order) into shared memory; then warp 0 streams the rows out
//                  (lane r issues the bulk store for rank r, r + 32) while
//                  warps 1-7 write sources, local expert indices and scores.
//   dedup_pos + dedup_copy : the same in two kernels (after the layout's
//                  positions), for tiles whose tables do not fit in shared
//                  memory: a CTA per token copies the row in 16-byte vectors.
//   dedup_expand : a CTA per token; copies each pair's dedupe row to its
//                  per-expert receive row (the receiver's expansion).
#include "ep_device.cuh"
#include "ep_next.cuh"

namespace ep {
namespace {

constexpr int kCopyThreads = 128;
constexpr int kLag = 4;                            // store groups in flight before a slot is reused
constexpr int kMaxStages = 32;
constexpr int kFusedSmemCap = 227 * 1024 - 1024;   // dynamic shared memory of the fused kernel
constexpr int kOnepassStatic = 2048;               // the one-pass kernel's extra static arrays

int slot_bytes_of(int64_t row_bytes) { return (int)((row_bytes + 127) / 128 * 128); }

__device__ __forceinline__ unsigned long long rank_mask(const int32_t* ids, int64_t t, int K,
                                                        int E, int eloc)
{
    unsigned long long m = 0ull;
#pragma unroll 8
    for (int k = 0; k < K; ++k) {
        const int e = valid_id(__ldcg(ids + t * K + k), E);
        if (e >= 0) m |= 1ull << (e / eloc);
    }
    return m;
}

// Dedupe row of each (token, rank) of layout tile `tile`: written to
// a.tok_pos[t][r] and, if s_tok is given, to s_tok[i * R + r] (i = token in the
// tile); -1 where the token selects none of rank r's experts. s_rbase holds
// kLayoutWarps * kMaxRanks ints. The distinct tokens per rank of the tiles
// before this one come from s_tokpre[r] if given, else from the scan's
// l.tile_tok_pre. Ends with __syncthreads.
__device__ __forceinline__ void tile_dedup_rows(const LayoutArgs& l, const DedupArgs& a, int tile,
                                                int (*s_rbase)[kMaxRanks], int* s_tok,
                                                const int* s_tokpre = nullptr)
{
    const int64_t t0 = (int64_t)tile * l.tpt;
    const int64_t t1 = min(l.T, t0 + l.tpt);
    const int n = (int)(t1 - t0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int R = a.R, eloc = a.E / a.R;
    const int seg = (((n + kLayoutWarps - 1) / kLayoutWarps) + 31) & ~31;
    const int w_begin = warp * seg;
    const int w_end = min(n, w_begin + seg);

    for (int i = threadIdx.x; i < kLayoutWarps * kMaxRanks; i += blockDim.x)
        s_rbase[i / kMaxRanks][i % kMaxRanks] = 0;
    __syncthreads();

    // Pass 1: tokens of this warp's segment that hit each rank.
    for (int c = w_begin; c < w_begin + seg; c += 32) {
        const int i = c + lane;
        const unsigned long long m = (i < w_end) ? rank_mask(a.ids, t0 + i, a.K, a.E, eloc) : 0ull;
        for (int r = 0; r < R; ++r) {
            const unsigned b = __ballot_sync(0xffffffffu, (m >> r) & 1ull);
            if (lane == 0) s_rbase[warp][r] += __popc(b);
        }
        __syncwarp();
    }
    __syncthreads();

    // Exclusive prefix over warps, seeded with the rank's base row and the
    // distinct tokens of all earlier tiles.
    if (threadIdx.x < R) {
        const int r = threadIdx.x;
        int base = (int)((int64_t)r * a.P) +
                   (s_tokpre ? s_tokpre[r] : __ldcg(l.tile_tok_pre + (int64_t)tile * R + r));
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int c = s_rbase[w][r];
            s_rbase[w][r] = base;
            base += c;
        }
    }
    __syncthreads();

    // Pass 2: row = running base + tokens hitting the rank in lower lanes.
    for (int c = w_begin; c < w_begin + seg; c += 32) {
        const int i = c + lane;
        const bool in = i < w_end;
        const unsigned long long m = in ? rank_mask(a.ids, t0 + i, a.K, a.E, eloc) : 0ull;
        for (int r = 0; r < R; ++r) {
            const bool bit = (m >> r) & 1ull;
            const unsigned b = __ballot_sync(0xffffffffu, bit);
            const int base = s_rbase[warp][r];
            if (in) {
                const int q = bit ? base + __popc(b & lanemask_lt(lane)) : -1;
                a.tok_pos[(t0 + i) * R + r] = q;
                if (s_tok) s_tok[i * R + r] = q;
            }
            __syncwarp();
            if (lane == 0) s_rbase[warp][r] = base + __popc(b);
            __syncwarp();
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kLayoutThreads)
dedup_pos_kernel(LayoutArgs l, DedupArgs a)
{
    __shared__ int s_rbase[kLayoutWarps][kMaxRanks];
    griddep_wait();
    griddep_launch_dependents();
    tile_dedup_rows(l, a, blockIdx.x, s_rbase, nullptr);
}

template <int U>
__global__ void __launch_bounds__(kCopyThreads)
dedup_copy_kernel(DedupArgs a)
{
    __shared__ int s_row[kMaxRanks];
    __shared__ int s_rank[kMaxRanks];
    __shared__ int s_n;
    griddep_wait();
    const int64_t V = a.row_bytes / 16;
    const int eloc = a.E / a.R;
    const int4* __restrict__ x = static_cast<const int4*>(a.x);
    int4* __restrict__ rx = static_cast<int4*>(a.recv_x);

    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        if (threadIdx.x == 0) {
            int n = 0;
            for (int r = 0; r < a.R; ++r) {
                const int q = __ldcg(a.tok_pos + t * a.R + r);
                if (q >= 0) {
                    s_row[n] = q;
                    s_rank[n] = r;
                    ++n;
                }
            }
            s_n = n;
        }
        __syncthreads();
        const int n = s_n;
        // Per destination row: source token, local expert index and score per k.
        for (int j = threadIdx.x; j < n * a.K; j += kCopyThreads) {
            const int d = j / a.K, k = j % a.K;
            const int q = s_row[d], r = s_rank[d];
            const int e = valid_id(__ldcg(a.ids + t * a.K + k), a.E);
            const bool mine = e >= 0 && e / eloc == r;
            a.recv_topk_idx[(int64_t)q * a.K + k] = mine ? e - r * eloc : -1;
            a.recv_topk_w[(int64_t)q * a.K + k] = mine ? __ldcg(a.scores + t * a.K + k) : 0.0f;
            if (k == 0) a.recv_tok_src[q] = (int32_t)t;
        }
        const int4* src = x + t * V;
        for (int64_t v0 = threadIdx.x; v0 < V; v0 += (int64_t)U * kCopyThreads) {
            int4 r4[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + (int64_t)u * kCopyThreads;
                if (v < V) r4[u] = ld_cg_v4(src + v);
            }
            for (int d = 0; d < n; ++d) {
                int4* dst = rx + (int64_t)s_row[d] * V;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t v = v0 + (int64_t)u * kCopyThreads;
                    if (v < V) dst[v] = r4[u];
                }
            }
        }
        __syncthreads();
    }
    griddep_launch_dependents();
}

// Loads this CTA issued for tokens [from, to) land before its shared memory is
// released (after a timed-out wait), under one deadline.
__device__ void drain_ring(uint32_t bar0, int stages, int from, int to)
{
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    for (int m = from; m < to; ++m)
        mbar_wait_until(bar0 + 8u * (uint32_t)(m % stages), (uint32_t)((m / stages) & 1), deadline);
}

// Streams the tile's rows out of the shared-memory ring (warp 0: lane r issues
// the bulk store of the token's row for rank r) while warps 1-7 write each
// dedupe row's source token, local expert indices and scores. keep(q): whether
// dedupe row q is written. The ring's first n_pro loads were issued already;
// issue_load(i) starts the load of the tile's token i. On a timed-out wait it
// reports EP_DEVERR_TIMEOUT and lets the loads in flight land.
template <typename Keep, typename IssueLoad>
__device__ __forceinline__ void dedup_stream_tile(const DedupArgs& a, int64_t t0, int n_my,
                                                  int n_pro, int stages, int slot_bytes,
                                                  uint32_t slot0, uint32_t bar0,
                                                  const int* s_tok, Keep keep,
                                                  IssueLoad issue_load)
{
    const int R = a.R, K = a.K, eloc = a.E / a.R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bytes = static_cast<uint32_t>(a.row_bytes);
    uint8_t* __restrict__ rx = static_cast<uint8_t*>(a.recv_x);
    if (warp == 0) {
        bool ok = true;
        int i = 0;
        for (; i < n_my; ++i) {
            const int s = i % stages;
            if (!mbar_wait(bar0 + 8u * s, (uint32_t)((i / stages) & 1))) {
                ok = false;
                break;
            }
            for (int r = lane; r < R; r += 32) {
                const int q = s_tok[i * R + r];
                if (keep(q))
                    bulk_s2g(rx + (int64_t)q * a.row_bytes, slot0 + (uint32_t)s * (uint32_t)slot_bytes,
                             bytes);
            }
            bulk_commit();
            const int j = i - kLag;
            if (j >= 0 && j + stages < n_my) {
                bulk_wait_read<kLag>();
                __syncwarp();
                if (lane == 0) issue_load(j + stages);
            }
        }
        bulk_wait_all();
        if (!ok && lane == 0) {
            atomicOr(a.err, kErrTimeout);
            int issued_hi = (i - kLag) + stages;   // loads issued for tokens < issued_hi
            if (issued_hi < n_pro) issued_hi = n_pro;
            drain_ring(bar0, stages, i, issued_hi < n_my ? issued_hi : n_my);
        }
    } else {
        // Per dedupe row: source token, and per k the local expert index and score.
        const int per_tok = R * K;
        for (int j = threadIdx.x - 32; j < n_my * per_tok; j += kLayoutThreads - 32) {
            const int i = j / per_tok, r = (j / K) % R, k = j % K;
            const int q = s_tok[i * R + r];
            if (!keep(q)) continue;
            const int64_t t = t0 + i;
            const int e = valid_id(__ldcg(a.ids + t * K + k), a.E);
            const bool mine = e >= 0 && e / eloc == r;
            a.recv_topk_idx[(int64_t)q * K + k] = mine ? e - r * eloc : -1;
            a.recv_topk_w[(int64_t)q * K + k] = mine ? __ldcg(a.scores + t * K + k) : 0.0f;
            if (k == 0) a.recv_tok_src[q] = (int32_t)t;
        }
    }
}

// Positions + dedupe rows + copies of one layout tile per CTA (file comment).
// Shared memory: [stages slots][kLayoutWarps * Ep ints][kLayoutWarps * kMaxRanks
// ints][tile tokens * R ints].
__global__ void __launch_bounds__(kLayoutThreads, 1)
dedup_fused_kernel(LayoutArgs L, DedupArgs a, int stages, int slot_bytes)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kMaxStages];
    int* s_base = reinterpret_cast<int*>(smem + (size_t)stages * slot_bytes);
    int (*s_rbase)[kMaxRanks] = reinterpret_cast<int (*)[kMaxRanks]>(s_base + kLayoutWarps * L.Ep);
    int* s_tok = s_base + kLayoutWarps * L.Ep + kLayoutWarps * kMaxRanks;
    const int tile = blockIdx.x;
    const int64_t t0 = (int64_t)tile * L.tpt;
    const int64_t t1 = min(L.T, t0 + L.tpt);
    const int n_my = (int)(t1 - t0);
    const uint32_t bytes = static_cast<uint32_t>(a.row_bytes);
    const uint32_t slot0 = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    const uint8_t* __restrict__ x = static_cast<const uint8_t*>(a.x);
    const int n_pro = n_my < stages ? n_my : stages;

    auto issue_load = [&](int i) {
        const int s = i % stages;
        const uint32_t bar = bar0 + 8u * s;
        mbar_expect_tx(bar, bytes);
        bulk_g2s(slot0 + (uint32_t)s * (uint32_t)slot_bytes, x + (t0 + i) * a.row_bytes, bytes, bar);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8u * s, 1u);
        fence_mbar_init();
        // The rows do not depend on the layout: start them before waiting for it.
        for (int i = 0; i < n_pro; ++i) issue_load(i);
    }

    griddep_wait();                                   // counts and offsets are ready
    tile_positions(L, tile, s_base, L.pos, nullptr);  // per-expert rows, for the expansion
    tile_dedup_rows(L, a, tile, s_rbase, s_tok);      // ends with __syncthreads

    dedup_stream_tile(a, t0, n_my, n_pro, stages, slot_bytes, slot0, bar0, s_tok,
                      [](int q) { return q >= 0; }, issue_load);
    griddep_launch_dependents();
}

// The dedupe dispatch in one cooperative kernel: the one-pass layout (this
// tile's counts, a grid barrier, every tile's counts summed from L2) replaces
// the count and scan kernels, then the same positions, dedupe rows and copies
// as dedup_fused. Thread 0 starts the tile's first row loads right after the
// histogram. Shared memory: dedup_fused's, then [3 * Ep ints].
__global__ void __launch_bounds__(kLayoutThreads, 1)
dedup_onepass_kernel(LayoutArgs L, DedupArgs a, int stages, int slot_bytes)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kMaxStages];
    __shared__ int s_rank[3][kMaxRanks];
    __shared__ int s_tk[kMaxRanks];
    __shared__ int s_tokpre[kMaxRanks];
    __shared__ int s_wsum[kLayoutWarps];
    __shared__ int s_flag;
    __shared__ uint32_t s_epoch;
    int* s_base = reinterpret_cast<int*>(smem + (size_t)stages * slot_bytes);
    int (*s_rbase)[kMaxRanks] = reinterpret_cast<int (*)[kMaxRanks]>(s_base + kLayoutWarps * L.Ep);
    int* s_tok = s_base + kLayoutWarps * L.Ep + kLayoutWarps * kMaxRanks;
    int* s_seed = s_tok + L.tpt * a.R;
    int* s_tot = s_seed + L.Ep;
    int* s_off = s_tot + L.Ep;
    const int tile = blockIdx.x;
    const int64_t t0 = (int64_t)tile * L.tpt;
    const int64_t t1 = min(L.T, t0 + L.tpt);
    const int n_my = (int)(t1 - t0);
    const int R = a.R;
    const uint32_t bytes = static_cast<uint32_t>(a.row_bytes);
    const uint32_t slot0 = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    const uint8_t* __restrict__ x = static_cast<const uint8_t*>(a.x);
    const int n_pro = n_my < stages ? n_my : stages;
    // Whether dedupe row q is to be written: q >= 0 and inside the call's R * P
    // rows. Rows always are when the layout is sound; one outside (possible
    // only if the grid barrier's words were corrupted and it opened early) is
    // skipped and reported, so that no store leaves the buffer.
    const int64_t rows_cap = (int64_t)R * a.P;
    auto in_rows = [&](int q) {
        if (q < 0) return false;
        if ((int64_t)q < rows_cap) return true;
        atomicOr(a.err, kErrRowOob);
        return false;
    };

    auto issue_load = [&](int i) {
        const int s = i % stages;
        const uint32_t bar = bar0 + 8u * s;
        mbar_expect_tx(bar, bytes);
        bulk_g2s(slot0 + (uint32_t)s * (uint32_t)slot_bytes, x + (t0 + i) * a.row_bytes, bytes, bar);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8u * s, 1u);
        fence_mbar_init();
    }
    // Inputs may come from the previous kernel in the stream.
    griddep_wait();
    const bool ok_layout =
        onepass_layout(L, tile, s_base, s_seed, s_tot, s_off, s_rank, s_tk, s_wsum, &s_flag,
                       &s_epoch, nullptr, s_tokpre, [&] {
                           for (int i = 0; i < n_pro; ++i) issue_load(i);
                       });
    if (!ok_layout) {   // barrier timed out: report, let this CTA's loads land, leave
        if (threadIdx.x == 0) {
            atomicOr(a.err, kErrTimeout);
            drain_ring(bar0, stages, 0, n_pro);
        }
        griddep_launch_dependents();
        return;
    }
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
    tile_positions(L, tile, s_base, L.pos, nullptr, s_seed);   // per-expert rows, for the expansion
    tile_dedup_rows(L, a, tile, s_rbase, s_tok, s_tokpre);     // ends with __syncthreads

    dedup_stream_tile(a, t0, n_my, n_pro, stages, slot_bytes, slot0, bar0, s_tok, in_rows,
                      issue_load);
    griddep_launch_dependents();
}

__global__ void __launch_bounds__(kCopyThreads)
dedup_expand_kernel(DedupArgs a, const int32_t* pos, void* y)
{
    __shared__ int s_dst[kMaxTopk];
    __shared__ int s_src[kMaxTopk];
    griddep_wait();
    const int64_t V = a.row_bytes / 16;
    const int eloc = a.E / a.R;
    const int4* __restrict__ rx = static_cast<const int4*>(a.recv_x);
    int4* __restrict__ out = static_cast<int4*>(y);

    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        if (threadIdx.x < a.K) {
            const int64_t q = t * a.K + threadIdx.x;
            const int p = __ldcg(pos + q);
            const int e = valid_id(__ldcg(a.ids + q), a.E);
            int src = -1;
            if (p >= 0 && e >= 0) {
                src = __ldcg(a.tok_pos + t * a.R + e / eloc);
                if (src < 0) atomicOr(a.err, kErrRowOob);   // ids differ from the dispatch's
            }
            s_dst[threadIdx.x] = (src >= 0) ? p : -1;
            s_src[threadIdx.x] = src;
        }
        __syncthreads();
        for (int k = 0; k < a.K; ++k) {
            const int p = s_dst[k];
            if (p < 0) continue;
            const int4* s = rx + (int64_t)s_src[k] * V;
            int4* d = out + (int64_t)p * V;
            for (int64_t v = threadIdx.x; v < V; v += kCopyThreads) d[v] = ld_cg_v4(s + v);
        }
        __syncthreads();
    }
    griddep_launch_dependents();
}

int copy_unroll(int64_t row_bytes)
{
    int64_t u = (row_bytes / 16 + kCopyThreads - 1) / kCopyThreads;
    return (int)(u < 1 ? 1 : (u > 8 ? 8 : u));
}

int copy_grid(int64_t T)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t g = (int64_t)(sms > 0 ? sms : 1) * 8;
    return (int)(T < g ? T : g);
}

}  // namespace

cudaError_t launch_dedup(const LayoutArgs& l, const DedupArgs& a, const LaunchOpts& o)
{
    if (a.T <= 0) return cudaSuccess;
    cudaError_t e = launch_kernel(dedup_pos_kernel, dim3(l.ntiles), dim3(kLayoutThreads), 0, o, l, a);
    if (e != cudaSuccess) return e;
    const dim3 g(copy_grid(a.T)), b(kCopyThreads);
    switch (copy_unroll(a.row_bytes)) {
#define EP_COPY(U) \
    case U:        \
        return launch_kernel(dedup_copy_kernel<U>, g, b, 0, o, a);
        EP_COPY(1) EP_COPY(2) EP_COPY(3) EP_COPY(4) EP_COPY(5) EP_COPY(6) EP_COPY(7) EP_COPY(8)
#undef EP_COPY
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dedup_fused(const LayoutArgs& l, const DedupArgs& a, const LaunchOpts& o)
{
    if (l.ntiles <= 0 || a.T <= 0) return cudaSuccess;
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e = cudaFuncSetAttribute(
            dedup_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemCap);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int slot = slot_bytes_of(a.row_bytes);
    const int64_t fixed =
        ((int64_t)kLayoutWarps * l.Ep + (int64_t)kLayoutWarps * kMaxRanks + l.tpt * a.R) * 4;
    int64_t stages = (kFusedSmemCap - fixed) / slot;
    if (stages > kMaxStages) stages = kMaxStages;
    if (a.row_bytes > (1 << 20) || stages < kLag + 2) return cudaErrorNotSupported;
    const size_t smem = (size_t)(stages * slot + fixed);
    return launch_kernel(dedup_fused_kernel, dim3(l.ntiles), dim3(kLayoutThreads), smem, o, l, a,
                         (int)stages, slot);
}

cudaError_t launch_dedup_onepass(const LayoutArgs& l, const DedupArgs& a, const LaunchOpts& o,
                                 bool pdl_ok)
{
    // An empty call still writes its (zero) layout: the separate kernels do that.
    if (l.ntiles <= 0 || a.T <= 0 || !l.gbar) return cudaErrorNotSupported;
    static bool attr_set = false;
    if (!attr_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(dedup_onepass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kFusedSmemCap - kOnepassStatic);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int slot = slot_bytes_of(a.row_bytes);
    const int64_t fixed = ((int64_t)kLayoutWarps * l.Ep + (int64_t)kLayoutWarps * kMaxRanks +
                           l.tpt * a.R + 3 * (int64_t)l.Ep) * 4;
    int64_t stages = (kFusedSmemCap - kOnepassStatic - fixed) / slot;
    if (stages > kMaxStages) stages = kMaxStages;
    if (a.row_bytes > (1 << 20) || stages < kLag + 2) return cudaErrorNotSupported;
    const size_t smem = (size_t)(stages * slot + fixed);
    // Every CTA must be resident at once for the grid barrier.
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dedup_onepass_kernel,
                                                      kLayoutThreads, smem) != cudaSuccess)
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
    const cudaError_t e =
        cudaLaunchKernelEx(&cfg, dedup_onepass_kernel, l, a, (int)stages, slot);
    if (e == cudaErrorCooperativeLaunchTooLarge) {   // fewer SMs than the device reports (MPS)
        cudaGetLastError();
        return cudaErrorNotSupported;
    }
    if (e == cudaSuccess && o.launches) ++*o.launches;
    return e;
}

cudaError_t launch_dedup_expand(const DedupArgs& a, const int32_t* pos, void* y,
                                const LaunchOpts& o)
{
    if (a.T <= 0) return cudaSuccess;
    return launch_kernel(dedup_expand_kernel, dim3(copy_grid(a.T)), dim3(kCopyThreads), 0, o, a,
                         pos, y);
}

}  // namespace ep
