// combine.cu - weighted un-permute of expert outputs back to token order.
//
// Follows "fix(moe): equalize and align per-rank token counts for HybridEP
// dispatch", section "Fix" (combine() slices the padded rows back off: only
// rows t < T are produced) and "ep: graph-safe worst-token HT
// dispatch+combine", section "Internode", item 3 (the true received total is
// read from the device prefix sum, never the padded row count: a row past
// its rank's total is never read).
//
// For each token t and element d:
//   acc = +0.0f; for k = 0..K-1 with a valid row p: acc = fmaf(s[t][k], y[p][d], acc)
//   out[t][d] = acc rounded to the output type (bf16: round to nearest even).
// A gather: each output element is produced by exactly one thread, in a fixed
// k order, with no atomics, so results are bitwise reproducible. HBM-bound:
// reads up to T*K rows, writes T rows.
//
// NaN results: IEEE 754-2008 section 6.2 fixes only that an operation with a
// NaN result returns a quiet NaN, not which one (the hardware's own is
// 7fffffff). Every NaN this file's arithmetic produces is stored as the
// canonical quiet NaN: 7fc00000 in fp32, 7fc0 in bf16 (positive, quiet bit,
// empty payload), so results are the same bits on every machine.
#include <cuda_bf16.h>

#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kLoadBatch = 8;   // rows of one token loaded before their FMAs

// Elements per 16-byte vector of the input type (0 = bf16, 1 = fp32).
template <int IN>
struct InVec {
    static constexpr int kElems = IN == 0 ? 8 : 4;
};

template <int IN>
__device__ __forceinline__ void fma_vec(float* acc, const int4& r, float w);

template <>
__device__ __forceinline__ void fma_vec<0>(float* acc, const int4& r, float w)
{
    const uint32_t u[4] = {(uint32_t)r.x, (uint32_t)r.y, (uint32_t)r.z, (uint32_t)r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 word.
        const float lo = __uint_as_float(u[i] << 16);
        const float hi = __uint_as_float(u[i] & 0xffff0000u);
        acc[2 * i] = __fmaf_rn(w, lo, acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(w, hi, acc[2 * i + 1]);
    }
}

template <>
__device__ __forceinline__ void fma_vec<1>(float* acc, const int4& r, float w)
{
    acc[0] = __fmaf_rn(w, __int_as_float(r.x), acc[0]);
    acc[1] = __fmaf_rn(w, __int_as_float(r.y), acc[1]);
    acc[2] = __fmaf_rn(w, __int_as_float(r.z), acc[2]);
    acc[3] = __fmaf_rn(w, __int_as_float(r.w), acc[3]);
}

constexpr uint32_t kNanF32 = 0x7fc00000u;   // the canonical quiet NaN
constexpr uint32_t kNanBf16 = 0x7fc0u;

// v, or the canonical quiet NaN where v is a NaN.
__device__ __forceinline__ float canonical_nan(float v)
{
    return v != v ? __uint_as_float(kNanF32) : v;
}

// Two fp32 values to bf16 (round to nearest even; a NaN to the canonical quiet
// NaN), lo in the low half (the lower address).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x (low address) = lo
    uint32_t r = *reinterpret_cast<uint32_t*>(&h);
    if (lo != lo) r = (r & 0xffff0000u) | kNanBf16;
    if (hi != hi) r = (r & 0x0000ffffu) | (kNanBf16 << 16);
    return r;
}

// Stores the N = InVec<IN>::kElems accumulators of vector v of token t.
template <int IN, int OUT>
__device__ __forceinline__ void store_out(void* out, int64_t t, int64_t D, int64_t v,
                                          const float* acc)
{
    constexpr int N = InVec<IN>::kElems;
    const int64_t e0 = t * D + v * N;
    if constexpr (OUT == 0) {
        uint16_t* o = static_cast<uint16_t*>(out) + e0;
        if constexpr (N == 8) {
            int4 w;
            w.x = (int)pack_bf16x2(acc[0], acc[1]);
            w.y = (int)pack_bf16x2(acc[2], acc[3]);
            w.z = (int)pack_bf16x2(acc[4], acc[5]);
            w.w = (int)pack_bf16x2(acc[6], acc[7]);
            *reinterpret_cast<int4*>(o) = w;
        } else {
            uint2 w;
            w.x = pack_bf16x2(acc[0], acc[1]);
            w.y = pack_bf16x2(acc[2], acc[3]);
            *reinterpret_cast<uint2*>(o) = w;
        }
    } else {
        float* o = static_cast<float*>(out) + e0;
#pragma unroll
        for (int i = 0; i < N; i += 4)
            *reinterpret_cast<float4*>(o + i) =
                make_float4(canonical_nan(acc[i]), canonical_nan(acc[i + 1]),
                            canonical_nan(acc[i + 2]), canonical_nan(acc[i + 3]));
    }
}

template <int IN, int OUT, bool SPLIT>
__global__ void __launch_bounds__(kCombineThreads)
combine_vec_kernel(CombineArgs a)
{
    constexpr int N = InVec<IN>::kElems;
    __shared__ int s_pos[kMaxTopk];
    __shared__ float s_w[kMaxTopk];
    griddep_wait();
    const int64_t V = a.D / N;
    const int4* __restrict__ y = static_cast<const int4*>(a.y);
    // Work item w = (token w / vsplit, vector chunk w % vsplit): a call with
    // fewer tokens than CTAs (SPLIT) spreads each token's row over vsplit CTAs,
    // so that each thread has fewer dependent load rounds. Without SPLIT the
    // chunk is the whole row, resolved at compile time.
    const int64_t nch = SPLIT ? a.vsplit : 1;
    const int64_t per = (V + nch - 1) / nch;   // vectors per chunk

    for (int64_t w = blockIdx.x; w < a.T * nch; w += gridDim.x) {
        const int64_t t = w / nch, ch = w % nch;
        if (threadIdx.x < a.K) {
            const int64_t q = t * a.K + threadIdx.x;
            int p = __ldcg(a.pos + q);
            // Keep the row only if it lies inside its rank's true total.
            if (p >= 0 && !row_valid(p, a.S, a.R, a.rank_prefix, a.packed)) {
                if (ch == 0) atomicOr(a.err, kErrRowOob);
                p = -1;
            }
            s_pos[threadIdx.x] = p;
            s_w[threadIdx.x] = a.unit_weights ? 1.0f : __ldcg(a.scores + q);
            if (a.gather_out && ch == 0)
                a.gather_out[q] = (p >= 0 && a.gather_in) ? __ldcg(a.gather_in + p) : 0.0f;
        }
        __syncthreads();
        const int64_t v_end = min(V, (ch + 1) * per);
        for (int64_t v = ch * per + threadIdx.x; v < v_end; v += kCombineThreads) {
            float acc[N];
#pragma unroll
            for (int i = 0; i < N; ++i) acc[i] = 0.0f;
            for (int k0 = 0; k0 < a.K; k0 += kLoadBatch) {
                int4 r[kLoadBatch];
#pragma unroll
                for (int j = 0; j < kLoadBatch; ++j) {
                    const int k = k0 + j;
                    const int p = (k < a.K) ? s_pos[k] : -1;
                    if (p >= 0) r[j] = ld_cg_v4(y + (int64_t)p * V + v);
                }
#pragma unroll
                for (int j = 0; j < kLoadBatch; ++j) {
                    const int k = k0 + j;
                    const int p = (k < a.K) ? s_pos[k] : -1;
                    if (p >= 0) fma_vec<IN>(acc, r[j], s_w[k]);
                }
            }
            store_out<IN, OUT>(a.out, t, a.D, v, acc);
        }
        __syncthreads();
    }
    griddep_launch_dependents();
}

// Unpacks the N elements of a 16-byte vector of the input type to fp32.
template <int IN>
__device__ __forceinline__ void unpack(const int4& r, float* f)
{
    if constexpr (IN == 0) {
        const uint32_t u[4] = {(uint32_t)r.x, (uint32_t)r.y, (uint32_t)r.z, (uint32_t)r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(u[i] << 16);
            f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
    } else {
        f[0] = __int_as_float(r.x);
        f[1] = __int_as_float(r.y);
        f[2] = __int_as_float(r.z);
        f[3] = __int_as_float(r.w);
    }
}

// Packs N fp32 values to a 16-byte vector of the type (bf16: round to nearest
// even); NaNs become the canonical quiet NaN.
template <int IN>
__device__ __forceinline__ int4 pack(const float* f)
{
    if constexpr (IN == 0) {
        return make_int4((int)pack_bf16x2(f[0], f[1]), (int)pack_bf16x2(f[2], f[3]),
                         (int)pack_bf16x2(f[4], f[5]), (int)pack_bf16x2(f[6], f[7]));
    } else {
        return make_int4(__float_as_int(canonical_nan(f[0])), __float_as_int(canonical_nan(f[1])),
                         __float_as_int(canonical_nan(f[2])), __float_as_int(canonical_nan(f[3])));
    }
}

// Backward of combine, one CTA per token (grid-stride): for each valid pair,
// grad_y[pos][d] = s * grad_out[t][d] (one fp32 product, rounded to the row
// type) and, if requested, grad_scores[t][k] = <grad_out[t], y[pos]>: per-thread
// fp32 FMA chains over the thread's vectors, then a fixed butterfly across the
// warp and a fixed sum over warps (deterministic, order documented).
template <int IN>
__global__ void __launch_bounds__(kCombineThreads)
combine_backward_kernel(CombineBwdArgs a)
{
    constexpr int N = InVec<IN>::kElems;
    constexpr int kWarps = kCombineThreads / 32;
    __shared__ int s_pos[kMaxTopk];
    __shared__ float s_w[kMaxTopk];
    __shared__ float s_red[kWarps][kLoadBatch];
    griddep_wait();
    const int64_t V = a.D / N;
    const int4* __restrict__ gout = static_cast<const int4*>(a.grad_out);
    const int4* __restrict__ y = static_cast<const int4*>(a.y);
    int4* __restrict__ gy = static_cast<int4*>(a.grad_y);
    const bool want_scores = a.grad_scores != nullptr;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        if (threadIdx.x < a.K) {
            const int64_t q = t * a.K + threadIdx.x;
            int p = __ldcg(a.pos + q);
            // Keep the row only if it lies inside its rank's true total.
            if (p >= 0 && !row_valid(p, a.S, a.R, a.rank_prefix, a.packed)) {
                atomicOr(a.err, kErrRowOob);
                p = -1;
            }
            s_pos[threadIdx.x] = p;
            s_w[threadIdx.x] = __ldcg(a.scores + q);
        }
        __syncthreads();
        for (int k0 = 0; k0 < a.K; k0 += kLoadBatch) {
            float part[kLoadBatch];
#pragma unroll
            for (int j = 0; j < kLoadBatch; ++j) part[j] = 0.0f;
            for (int64_t v = threadIdx.x; v < V; v += kCombineThreads) {
                float gf[N];
                unpack<IN>(ld_cg_v4(gout + t * V + v), gf);
                int4 yv[kLoadBatch];
                if (want_scores) {
#pragma unroll
                    for (int j = 0; j < kLoadBatch; ++j) {
                        const int k = k0 + j;
                        const int p = (k < a.K) ? s_pos[k] : -1;
                        if (p >= 0) yv[j] = ld_cg_v4(y + (int64_t)p * V + v);
                    }
                }
#pragma unroll
                for (int j = 0; j < kLoadBatch; ++j) {
                    const int k = k0 + j;
                    const int p = (k < a.K) ? s_pos[k] : -1;
                    if (p < 0) continue;
                    float o[N];
#pragma unroll
                    for (int e = 0; e < N; ++e) o[e] = __fmul_rn(s_w[k], gf[e]);
                    gy[(int64_t)p * V + v] = pack<IN>(o);
                    if (want_scores) {
                        float yf[N];
                        unpack<IN>(yv[j], yf);
#pragma unroll
                        for (int e = 0; e < N; ++e) part[j] = __fmaf_rn(gf[e], yf[e], part[j]);
                    }
                }
            }
            if (want_scores) {
#pragma unroll
                for (int j = 0; j < kLoadBatch; ++j)
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        part[j] += __shfl_xor_sync(0xffffffffu, part[j], off);
                if (lane == 0)
#pragma unroll
                    for (int j = 0; j < kLoadBatch; ++j) s_red[warp][j] = part[j];
                __syncthreads();
                if (threadIdx.x < kLoadBatch && k0 + (int)threadIdx.x < a.K) {
                    const int k = k0 + threadIdx.x;
                    float sum = 0.0f;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) sum += s_red[w][threadIdx.x];
                    a.grad_scores[t * a.K + k] = (s_pos[k] >= 0) ? canonical_nan(sum) : 0.0f;
                }
                __syncthreads();
            }
        }
        __syncthreads();
    }
    griddep_launch_dependents();
}

template <int IN, int OUT>
cudaError_t occupancy(int* per_sm)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, combine_vec_kernel<IN, OUT, false>,
                                                         kCombineThreads, 0);
}

}  // namespace

cudaError_t plan_combine(int in_dtype, int num_sms, int per_sm_cap, int* grid)
{
    int per_sm = 0;
    cudaError_t e = in_dtype == 0 ? occupancy<0, 0>(&per_sm) : occupancy<1, 1>(&per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm_cap > 0 && per_sm > per_sm_cap) per_sm = per_sm_cap;
    *grid = num_sms * (per_sm > 0 ? per_sm : 1);
    return cudaSuccess;
}

cudaError_t launch_combine(const CombineArgs& args, int grid, const LaunchOpts& opts)
{
    if (args.T <= 0) return cudaSuccess;
    // The combine follows the expert (or, with an identity expert, the permute)
    // and would only start early to wait: launch it in plain stream order. In a
    // captured graph an early-launched combine behind the bulk permute measured
    // slower than a plain dependency.
    LaunchOpts o = opts;
    o.pdl = false;
    // Fewer tokens than CTAs: split each token's row into chunks of at least one
    // vector per thread, as many as the grid has room for.
    CombineArgs a = args;
    const int64_t V = a.D / (a.in_dtype == 0 ? 8 : 4);
    int64_t nch = 1;
    if (a.T < grid) {
        const int64_t by_grid = grid / a.T;
        const int64_t by_row = (V + kCombineThreads - 1) / kCombineThreads;
        nch = by_grid < by_row ? by_grid : by_row;
        if (nch < 1) nch = 1;
    }
    a.vsplit = (int)nch;
    const int64_t items = a.T * nch;
    const dim3 g((unsigned)(items < grid ? items : grid)), b(kCombineThreads);
    if (nch > 1) {
        if (a.in_dtype == 0 && a.out_dtype == 0)
            return launch_kernel(combine_vec_kernel<0, 0, true>, g, b, 0, o, a);
        if (a.in_dtype == 0 && a.out_dtype == 1)
            return launch_kernel(combine_vec_kernel<0, 1, true>, g, b, 0, o, a);
        if (a.in_dtype == 1 && a.out_dtype == 0)
            return launch_kernel(combine_vec_kernel<1, 0, true>, g, b, 0, o, a);
        return launch_kernel(combine_vec_kernel<1, 1, true>, g, b, 0, o, a);
    }
    if (a.in_dtype == 0 && a.out_dtype == 0)
        return launch_kernel(combine_vec_kernel<0, 0, false>, g, b, 0, o, a);
    if (a.in_dtype == 0 && a.out_dtype == 1)
        return launch_kernel(combine_vec_kernel<0, 1, false>, g, b, 0, o, a);
    if (a.in_dtype == 1 && a.out_dtype == 0)
        return launch_kernel(combine_vec_kernel<1, 0, false>, g, b, 0, o, a);
    return launch_kernel(combine_vec_kernel<1, 1, false>, g, b, 0, o, a);
}

cudaError_t launch_combine_backward(const CombineBwdArgs& a, int grid, const LaunchOpts& opts)
{
    if (a.T <= 0) return cudaSuccess;
    LaunchOpts o = opts;
    o.pdl = false;
    const dim3 g((unsigned)(a.T < grid ? a.T : grid)), b(kCombineThreads);
    if (a.dtype == 0) return launch_kernel(combine_backward_kernel<0>, g, b, 0, o, a);
    return launch_kernel(combine_backward_kernel<1>, g, b, 0, o, a);
}

}  // namespace ep
