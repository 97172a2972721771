// permute.cu - dispatch permute: copy each token row into the receive rows
// of its experts, with the row's score and source pair index.
//
// Follows "Unify expert parallel token dispatcher API", section "Backend
// behavior" (HybridEP: non-blocking dispatch sizes the fused-permute output by
// the current capacity; DeepEP: the current capacity is the per-rank layout
// stride). Positions come from the layout kernels; this file only moves data.
//
// The kernel is HBM-bound: it reads T rows and writes up to T*K rows. Two
// implementations:
//   vec  : a CTA per token (grid-stride); each thread loads its 16-byte
//          vectors of the row once (non-coherent, no L1 allocation) and stores
//          them to every destination row.
//   bulk : one warp per CTA drives bulk async copies: a row goes global ->
//          shared memory once (completion tracked by an mbarrier), then each
//          lane k copies it shared -> global to its destination row; a ring of
//          row slots keeps several loads and stores in flight per SM. No
//          multicast, no cluster: plain 1-D bulk copies within one CTA.
#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr int kVecThreads = 128;
constexpr int kBulkLag = 4;            // store groups in flight before a slot is reused
constexpr int kBulkMaxStages = 32;
constexpr int kBulkSmemBudget = 200 * 1024;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // bounded mbarrier wait (then EP_DEVERR_TIMEOUT)

__device__ __forceinline__ int4 ld_stream_v4(const int4* p)
{
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int U>
__global__ void __launch_bounds__(kVecThreads)
permute_vec_kernel(PermuteArgs a)
{
    __shared__ int s_pos[kMaxTopk];
    const int64_t V = a.row_bytes / 16;
    const int4* __restrict__ x = static_cast<const int4*>(a.x);
    int4* __restrict__ rx = static_cast<int4*>(a.recv_x);

    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        if (threadIdx.x < a.K) {
            const int64_t q = t * a.K + threadIdx.x;
            const int p = a.pos[q];
            s_pos[threadIdx.x] = p;
            if (p >= 0) {
                a.recv_scores[p] = a.scores[q];
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
                if (v < V) r[u] = ld_stream_v4(src + v);
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
}

// ---- bulk async copy helpers (inline PTX) ---------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: false if the phase has not completed by the deadline
// (nanoseconds of %globaltimer).
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

    auto issue_load = [&](int64_t i) {
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
            p = __ldg(a.pos + q);
            w = __ldg(a.scores + q);
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
        const uint32_t parity = (uint32_t)((i / stages) & 1);
        if (!mbar_wait(bar0 + 8u * s, parity)) {
            ok = false;
            break;
        }
        if (p_cur >= 0) {
            bulk_s2g(rx + (int64_t)p_cur * a.row_bytes, slot0 + (uint32_t)s * (uint32_t)slot_bytes,
                     bytes);
            const int64_t q = (b + i * G) * K + lane;
            a.recv_scores[p_cur] = w_cur;
            a.recv_src[p_cur] = (int32_t)q;
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
    if (!ok) {
        if (lane == 0) {
            atomicOr(a.err, kErrTimeout);
            // Let loads already issued land before the CTA's shared memory is
            // released, under one shared deadline.
            int64_t issued_hi = (i - kBulkLag) + stages;   // loads issued for tokens < issued_hi
            if (issued_hi < n_pro) issued_hi = n_pro;
            const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
            for (int64_t m = i; m < n_my && m < issued_hi; ++m)
                if (!mbar_wait_until(bar0 + 8u * (uint32_t)(m % stages),
                                     (uint32_t)((m / stages) & 1), deadline))
                    break;
        }
    }
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

cudaError_t plan_permute(int impl, int64_t row_bytes, int K, int num_sms, PermutePlan* plan)
{
    plan->impl = impl;
    plan->stages = 0;
    plan->smem_bytes = 0;
    const int slot = (int)((row_bytes + 127) / 128 * 128);
    if (impl == 2) {
        int stages = kBulkSmemBudget / slot;
        if (stages > kBulkMaxStages) stages = kBulkMaxStages;
        if (stages < kBulkLag + 2 || row_bytes > (1 << 20) || K > 32) {
            plan->impl = impl = 1;   // rows too large for a useful ring: vector path
        } else {
            plan->stages = stages;
            plan->smem_bytes = stages * slot;
            cudaError_t e = cudaFuncSetAttribute(permute_bulk_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 plan->smem_bytes);
            if (e != cudaSuccess) return e;
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

cudaError_t launch_permute(const PermuteArgs& a, const PermutePlan& plan, cudaStream_t s,
                           int64_t* launches)
{
    if (a.T <= 0) return cudaSuccess;
    const unsigned grid = (unsigned)(a.T < plan.grid ? a.T : plan.grid);
    if (plan.impl == 2) {
        permute_bulk_kernel<<<grid, 32, plan.smem_bytes, s>>>(a, plan.stages,
                                                              (int)((a.row_bytes + 127) / 128 * 128));
    } else {
        switch (vec_unroll(a.row_bytes)) {
#define EP_LAUNCH(U)                                                        \
    case U:                                                                 \
        permute_vec_kernel<U><<<grid, kVecThreads, 0, s>>>(a);              \
        break;
            EP_LAUNCH(1) EP_LAUNCH(2) EP_LAUNCH(3) EP_LAUNCH(4)
            EP_LAUNCH(5) EP_LAUNCH(6) EP_LAUNCH(7) EP_LAUNCH(8)
#undef EP_LAUNCH
            default:
                return cudaErrorInvalidValue;
        }
    }
    ++*launches;
    return cudaGetLastError();
}

}  // namespace ep
