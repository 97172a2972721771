// patterns.cu - the HBM access patterns of the hot path, with nothing else in
// the kernel, so a benchmark can time each pattern's ceiling on this GPU and
// set the dispatch and the combine against it.
//
// The dispatch reads each token row once and writes it to K places (a 1:K
// fan-out into K rank regions); the combine reads K rows and writes one (a K:1
// gather). ep_pattern_probe moves whole rows in those shapes, and in the plain
// read, write and copy shapes, with the same kernel structure as the combine:
// one 128-thread CTA per row (grid-stride over rows), 16-byte vectors,
// L2-coherent loads, as many CTAs per SM as fit. What is computed on the way
// (an XOR of the words) only keeps the loads live.
#include <cuda_runtime.h>

#include "ep.h"
#include "ep_device.cuh"

namespace {

constexpr int kThreads = 128;
constexpr int kMaxFan = 64;

struct PatternArgs {
    const int4* src;
    int4* dst;
    int64_t rows;
    int64_t V;      // 16-byte vectors per row
    int fan;
};

__device__ __forceinline__ int4 xor4(int4 a, int4 b)
{
    return make_int4(a.x ^ b.x, a.y ^ b.y, a.z ^ b.z, a.w ^ b.w);
}

// READ: row r of src XOR-reduced into one 16-byte word, dst[r].
__global__ void __launch_bounds__(kThreads) pattern_read(PatternArgs a)
{
    __shared__ int4 s_part[kThreads / 32];
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        int4 acc = make_int4(0, 0, 0, 0);
        for (int64_t v = threadIdx.x; v < a.V; v += kThreads)
            acc = xor4(acc, ep::ld_cg_v4(a.src + r * a.V + v));
        for (int off = 16; off > 0; off >>= 1) {
            acc.x ^= __shfl_xor_sync(0xffffffffu, acc.x, off);
            acc.y ^= __shfl_xor_sync(0xffffffffu, acc.y, off);
            acc.z ^= __shfl_xor_sync(0xffffffffu, acc.z, off);
            acc.w ^= __shfl_xor_sync(0xffffffffu, acc.w, off);
        }
        if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            int4 t = s_part[0];
            for (int w = 1; w < kThreads / 32; ++w) t = xor4(t, s_part[w]);
            a.dst[r] = t;
        }
        __syncthreads();
    }
}

// WRITE: every vector of row r of dst set to (r, v, r, v).
__global__ void __launch_bounds__(kThreads) pattern_write(PatternArgs a)
{
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x)
        for (int64_t v = threadIdx.x; v < a.V; v += kThreads)
            a.dst[r * a.V + v] = make_int4((int)r, (int)v, (int)r, (int)v);
}

// COPY: dst[r] = src[r].
__global__ void __launch_bounds__(kThreads) pattern_copy(PatternArgs a)
{
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x)
        for (int64_t v = threadIdx.x; v < a.V; v += kThreads)
            a.dst[r * a.V + v] = ep::ld_cg_v4(a.src + r * a.V + v);
}

// FANOUT: dst[j*rows + r] = src[r] for j < fan (each vector loaded once).
__global__ void __launch_bounds__(kThreads) pattern_fanout(PatternArgs a)
{
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x)
        for (int64_t v = threadIdx.x; v < a.V; v += kThreads) {
            const int4 x = ep::ld_cg_v4(a.src + r * a.V + v);
            for (int j = 0; j < a.fan; ++j) a.dst[((int64_t)j * a.rows + r) * a.V + v] = x;
        }
}

// GATHER: dst[r] = XOR over j < fan of src[j*rows + r] (loads in batches of 8
// before their use, as the combine issues its K loads).
__global__ void __launch_bounds__(kThreads) pattern_gather(PatternArgs a)
{
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x)
        for (int64_t v = threadIdx.x; v < a.V; v += kThreads) {
            int4 acc = make_int4(0, 0, 0, 0);
            for (int j0 = 0; j0 < a.fan; j0 += 8) {
                int4 x[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j0 + j < a.fan)
                        x[j] = ep::ld_cg_v4(a.src + ((int64_t)(j0 + j) * a.rows + r) * a.V + v);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j0 + j < a.fan) acc = xor4(acc, x[j]);
            }
            a.dst[r * a.V + v] = acc;
        }
}

}  // namespace

extern "C" ep_status ep_pattern_probe(int32_t pattern, const void* src, void* dst, int64_t rows,
                                      int64_t row_bytes, int32_t fan, ep_stream_t stream)
{
    if (rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return EP_ERR_INVALID_ARG;
    if (pattern < EP_PATTERN_READ || pattern > EP_PATTERN_GATHER) return EP_ERR_INVALID_ARG;
    const bool fans = pattern == EP_PATTERN_FANOUT || pattern == EP_PATTERN_GATHER;
    if (fans && (fan < 1 || fan > kMaxFan)) return EP_ERR_INVALID_ARG;
    if (!dst || (pattern != EP_PATTERN_WRITE && !src)) return EP_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u)
        return EP_ERR_ALIGNMENT;
    if (rows == 0) return EP_OK;
    PatternArgs a{static_cast<const int4*>(src), static_cast<int4*>(dst), rows, row_bytes / 16,
                  fans ? fan : 1};
    void (*k)(PatternArgs) = pattern == EP_PATTERN_READ    ? pattern_read
                             : pattern == EP_PATTERN_WRITE ? pattern_write
                             : pattern == EP_PATTERN_COPY  ? pattern_copy
                             : pattern == EP_PATTERN_FANOUT ? pattern_fanout
                                                            : pattern_gather;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, 0) != cudaSuccess)
        return EP_ERR_CUDA;
    int64_t grid = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    if (grid > rows) grid = rows;
    const ep::LaunchOpts o{static_cast<cudaStream_t>(stream), false, nullptr};
    return ep::launch_kernel(k, dim3((unsigned)grid), dim3(kThreads), 0, o, a) == cudaSuccess
               ? EP_OK
               : EP_ERR_CUDA;
}
