// permute.cu - dispatch permute: copy each token row into the receive rows
// of its experts, with the row's score and source pair index.
//
// Follows "Unify expert parallel token dispatcher API", section "Backend
// behavior" (HybridEP: non-blocking dispatch sizes the fused-permute output by
// the current capacity; DeepEP: the current capacity is the per-rank layout
// stride).
//
// HBM-bound: reads T rows and writes up to T*K rows. Three kernels:
//   dispatch_fused : the default. One CTA (8 warps) per layout tile, about one
//                    per SM. Thread 0 starts bulk async loads of the tile's
//                    rows into a shared-memory ring *before* waiting for the
//                    layout scan (the rows do not depend on it), then all
//                    warps compute the tile's positions into shared memory,
//                    then warp 0 streams the rows out: lane k issues the bulk
//                    store of destination k; warps 1-7 write scores and
//                    sources. Completion of loads is tracked by mbarriers
//                    (bounded waits); a slot is reused only after its stores
//                    have read it (cp.async.bulk.wait_group.read).
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
constexpr int kBulkLag = 4;            // store groups in flight before a slot is reused
constexpr int kBulkMaxStages = 32;
constexpr int kBulkSmemBudget = 200 * 1024;
constexpr int kFusedSmemCap = 227 * 1024 - 1024;   // dynamic shared memory of the fused kernel

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

// Positions + permute of one layout tile per CTA (see the file comment).
// Shared memory: [stages slots of slot_bytes][kLayoutWarps * Ep ints][tile pairs ints].
__global__ void __launch_bounds__(kLayoutThreads, 1)
dispatch_fused_kernel(LayoutArgs L, PermuteArgs a, int stages, int slot_bytes)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kBulkMaxStages];
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
    const int n_pro = n_my < stages ? n_my : stages;

    const int64_t skipped = (tile == 0) ? a.skip_load : -1;
    auto issue_load = [&](int i) {
        if (i == skipped) return;
        const int s = i % stages;
        const uint32_t bar = bar0 + 8u * s;
        mbar_expect_tx(bar, bytes);
        bulk_g2s(slot0 + (uint32_t)s * (uint32_t)slot_bytes, x + (t0 + i) * a.row_bytes, bytes,
                 bar);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8u * s, 1u);
        fence_mbar_init();
        // The rows do not depend on the layout: start them before waiting for it.
        for (int i = 0; i < n_pro; ++i) issue_load(i);
    }

    griddep_wait();                                   // counts and offsets are ready
    tile_positions(L, tile, s_base, L.pos, s_pos);    // ends with __syncthreads

    if (warp == 0) {
        bool ok = true;
        int i = 0;
        for (; i < n_my; ++i) {
            const int s = i % stages;
            if (!mbar_wait(bar0 + 8u * s, (uint32_t)((i / stages) & 1))) {
                ok = false;
                break;
            }
            if (lane < K) {
                const int p = s_pos[i * K + lane];
                if (p >= 0)
                    bulk_s2g(rx + (int64_t)p * a.row_bytes,
                             slot0 + (uint32_t)s * (uint32_t)slot_bytes, bytes);
            }
            bulk_commit();
            const int j = i - kBulkLag;
            if (j >= 0 && j + stages < n_my) {
                bulk_wait_read<kBulkLag>();
                __syncwarp();
                if (lane == 0) issue_load(j + stages);
            }
        }
        bulk_wait_all();
        if (!ok && lane == 0) {
            atomicOr(a.err, kErrTimeout);
            int issued_hi = (i - kBulkLag) + stages;
            if (issued_hi < n_pro) issued_hi = n_pro;
            drain_loads(bar0, stages, i, issued_hi < n_my ? issued_hi : n_my, skipped);
        }
    } else {
        const int np = n_my * K;
        for (int j = threadIdx.x - 32; j < np; j += kLayoutThreads - 32) {
            const int p = s_pos[j];
            if (p >= 0) {
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
            e = cudaFuncSetAttribute(dispatch_fused_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmemCap);
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
    return launch_kernel(dispatch_fused_kernel, dim3(l.ntiles), dim3(kLayoutThreads), smem, o, l,
                         p, (int)stages, slot);
}

}  // namespace ep
