// expert_gemm.cu - the expert consumer between dispatch and combine: a
// grouped GEMM  y[p] = x[p] * W_e^T  over the receive rows of every expert,
// driven by the per-expert counts and offsets the layout left on the device
// ("ep: graph-safe worst-token HT dispatch+combine", "Internode" item 2: the
// counts stay on the device so graph-mode consumers never touch the host;
// "Tests": layout -> dispatch -> expert -> combine). No host round trip: the
// tile list is derived on the device from the counts.
//
// sm_103a tensor cores, written directly:
//   - one CTA per SM, persistent over tiles of 128 rows x BN output columns
//     of one expert (tile order: the BN-wide column blocks of one row block
//     first, so the row block is reused from L2);
//   - warp 0 (one thread) streams 64-wide K slices of the row block and of
//     the expert's weights into a 4-stage shared-memory ring with TMA tensor
//     copies (128-byte swizzle), completion on mbarriers;
//   - warp 1 owns two BN-column fp32 accumulators in tensor memory (TMEM)
//     and one thread issues tcgen05.mma (M=128, N=BN, K=16, bf16 inputs, fp32
//     accumulate) from shared-memory descriptors, committing each stage back
//     to the ring and each finished tile to the epilogue; tiles alternate
//     between the accumulators so the epilogue overlaps the next tile;
//   - warps 2-5 read the accumulator with tcgen05.ld (each warp its 32-lane
//     quarter), round to bf16 and store the rows that belong to the expert.
// Every wait is bounded; on a timeout the CTA reports EP_DEVERR_TIMEOUT,
// waits for its copies and MMAs in flight, frees its TMEM and returns.
#include <cuda.h>

#include <mutex>

#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kBM = 128;            // rows per tile = TMEM lanes = UMMA M
constexpr int kBK = 64;             // K per stage: one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;          // K per tcgen05.mma for 16-bit inputs
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;   // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr int kEpilogueThreads = 128;

template <int BN>
struct Tile {
    static constexpr uint32_t kBytesA = kBM * kBK * 2;
    static constexpr uint32_t kBytesB = BN * kBK * 2;
    static constexpr uint32_t kStageBytes = kBytesA + kBytesB;
    // Instruction descriptor, kind::f16: fp32 accumulate (bits 4-5 = 1), A and
    // B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
    // N >> 3 at bits 17-22, M >> 4 at bits 24-28.
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                       ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
    // Two accumulators, so the epilogue of one tile overlaps the MMAs of the next.
    static constexpr uint32_t kTmemCols = 2 * BN;
};

// Shared-memory matrix descriptor for a K-major tile written by TMA with the
// 128-byte swizzle: start address >> 4 (bits 0-13), leading offset 16 B
// (unused for this layout), stride 1024 B between 8-row groups (bits 32-45),
// descriptor version 1 (bits 46-47), swizzle mode 128B = 2 (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() > deadline) {
            *abort = 1;
            return false;
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Expert of m-tile number mt: the e with s_mtile[e] <= mt < s_mtile[e+1].
__device__ __forceinline__ int expert_of(const int* s_mtile, int E, int mt)
{
    int lo = 0, hi = E;   // invariant: s_mtile[lo] <= mt < s_mtile[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_mtile[mid] <= mt) lo = mid;
        else hi = mid;
    }
    return lo;
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                   GemmArgs a)
{
    using C = Tile<BN>;
    extern __shared__ uint8_t smem_raw[];
    // Swizzled tiles want 1024-byte alignment.
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    const uint32_t tiles_u32 = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * C::kStageBytes);
    const uint32_t full0 = smem_u32(bars);                 // kStages
    const uint32_t empty0 = full0 + 8u * kStages;          // kStages
    const uint32_t accum_full0 = empty0 + 8u * kStages;    // 2: one per accumulator
    const uint32_t accum_empty0 = accum_full0 + 16u;       // 2
    const uint32_t drain = accum_empty0 + 16u;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    int* s_mtile = const_cast<int*>(reinterpret_cast<volatile int*>(s_abort + 1));   // [E + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;
    const int k_iters = (int)(a.din / kBK);
    const int n_blocks = (int)(a.dout / BN);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full0 + 8u * s, 1u);
            mbar_init(empty0 + 8u * s, 1u);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accum_full0 + 8u * b, 1u);
            mbar_init(accum_empty0 + 8u * b, (uint32_t)kEpilogueThreads);
        }
        mbar_init(drain, 1u);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(s_tmem), C::kTmemCols);
        tmem_relinquish();
    }

    griddep_wait();   // counts, offsets and the receive rows come from earlier kernels

    // Prefix over experts of their 128-row tiles (warp 0, 32 experts at a time).
    if (warp == 0) {
        int carry = 0;
        if (lane == 0) s_mtile[0] = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            int m = (e < E) ? (__ldcg(a.cnt + e) + kBM - 1) / kBM : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, m, d);
                if (lane >= d) m += n;
            }
            if (e < E) s_mtile[e + 1] = carry + m;
            carry += __shfl_sync(0xffffffffu, m, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int total_tiles = s_mtile[E] * n_blocks;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer --------------------------------------------------
        int g = 0;   // k-slices issued
        for (int t = blockIdx.x; t < total_tiles && !*s_abort; t += gridDim.x) {
            const int mt = t / n_blocks, nb = t % n_blocks;
            const int e = expert_of(s_mtile, E, mt);
            const int row0 = __ldcg(a.expert_offset + e) + (mt - s_mtile[e]) * kBM;
            const int wrow0 = e * (int)a.dout + nb * BN;
            for (int k = 0; k < k_iters; ++k, ++g) {
                const int s = g % kStages;
                const uint32_t ph = (uint32_t)((g / kStages) & 1);
                if (!wait_or_abort(empty0 + 8u * s, ph ^ 1u, s_abort)) break;
                mbar_expect_tx(full0 + 8u * s, C::kStageBytes);
                const uint32_t sa = tiles_u32 + (uint32_t)s * C::kStageBytes;
                tma_load_2d(sa, &tm_x, k * kBK, row0, full0 + 8u * s);
                tma_load_2d(sa + C::kBytesA, &tm_w, k * kBK, wrow0, full0 + 8u * s);
            }
        }
        // Let the copies this thread issued land before shared memory goes away.
        const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
        for (int i = (g > kStages ? g - kStages : 0); i < g; ++i)
            mbar_wait_until(full0 + 8u * (uint32_t)(i % kStages), (uint32_t)((i / kStages) & 1),
                            deadline);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----------------------------------------------------
        int g = 0, tl = 0;
        bool issued = false;
        for (int t = blockIdx.x; t < total_tiles && !*s_abort; t += gridDim.x, ++tl) {
            const int acc = tl & 1, use = tl >> 1;      // accumulator and its use count
            if (!wait_or_abort(accum_empty0 + 8u * acc, (uint32_t)((use & 1) ^ 1), s_abort)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
            bool ok = true;
            for (int k = 0; k < k_iters; ++k, ++g) {
                const int s = g % kStages;
                if (!wait_or_abort(full0 + 8u * s, (uint32_t)((g / kStages) & 1), s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = tiles_u32 + (uint32_t)s * C::kStageBytes;
#pragma unroll
                for (int j = 0; j < kBK / kUmmaK; ++j)
                    umma_bf16(d_tmem, sw128_desc(sa + j * kUmmaK * 2),
                              sw128_desc(sa + C::kBytesA + j * kUmmaK * 2), C::kIdesc,
                              (k | j) != 0 ? 1u : 0u);
                issued = true;
                umma_commit(empty0 + 8u * s);   // frees the stage once these MMAs finish
            }
            if (!ok) break;
            umma_commit(accum_full0 + 8u * acc);   // the tile's accumulator is complete
        }
        if (issued) {   // every MMA this thread issued has finished before TMEM is freed
            umma_commit(drain);
            mbar_wait(drain, 0u);
        }
    } else if (warp >= 2) {
        // ---- epilogue: TMEM -> bf16 -> global ------------------------------
        const int quarter = warp & 3;                  // TMEM lanes this warp may read
        const int r_in = quarter * 32 + lane;          // accumulator row = tile row
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        uint16_t* y = static_cast<uint16_t*>(a.y);
        int tl = 0;
        for (int t = blockIdx.x; t < total_tiles && !*s_abort; t += gridDim.x, ++tl) {
            const int acc = tl & 1, use = tl >> 1;
            if (!wait_or_abort(accum_full0 + 8u * acc, (uint32_t)(use & 1), s_abort)) break;
            tc_fence_after();
            const uint32_t t_acc = t_lane + (uint32_t)(acc * BN);
            const int mt = t / n_blocks, nb = t % n_blocks;
            const int e = expert_of(s_mtile, E, mt);
            const int m_in = (mt - s_mtile[e]) * kBM;
            const int rows = min(kBM, __ldcg(a.cnt + e) - m_in);
            const int64_t row = (int64_t)__ldcg(a.expert_offset + e) + m_in + r_in;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t v[32];
                tmem_ld32(t_acc + (uint32_t)c, v);
                tmem_wait_ld();
                if (r_in < rows) {
                    int4* dst = reinterpret_cast<int4*>(y + row * a.dout + nb * BN + c);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        int4 w;
                        w.x = (int)pack_bf16x2_rn(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
                        w.y = (int)pack_bf16x2_rn(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
                        w.z = (int)pack_bf16x2_rn(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
                        w.w = (int)pack_bf16x2_rn(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
                        dst[q] = w;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(accum_empty0 + 8u * acc);
        }
    }

    if (threadIdx.x == 0 && *s_abort) atomicOr(a.err, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    griddep_launch_dependents();
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 tensor map over [rows][inner] with a box of [box_rows][64] and the
// 128-byte swizzle the UMMA descriptors expect.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int BN>
size_t gemm_smem_bytes(int E)
{
    return 1024 + (size_t)kStages * Tile<BN>::kStageBytes + 8 * (2 * kStages + 5) + 8 +
           4 * (size_t)(E + 1);
}

template <int BN>
cudaError_t launch_bn(const GemmArgs& a, const void* x, int64_t rows, const void* w, int grid,
                      const LaunchOpts& o)
{
    CUtensorMap tx, tw;
    if (!make_map(&tx, x, (uint64_t)a.din, (uint64_t)rows, kBM) ||
        !make_map(&tw, w, (uint64_t)a.din, (uint64_t)a.E * (uint64_t)a.dout, BN))
        return cudaErrorInvalidValue;
    const size_t smem = gemm_smem_bytes<BN>(a.E);
    cudaError_t e = cudaFuncSetAttribute(expert_gemm_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(expert_gemm_kernel<BN>, dim3(grid), dim3(kGemmThreads), smem, o, tx, tw, a);
}

}  // namespace

cudaError_t launch_expert_gemm(const GemmArgs& a, const void* x, int64_t rows, const void* w,
                               int grid, const LaunchOpts& o)
{
    if (a.din % kBK != 0 || a.dout % 128 != 0) return cudaErrorInvalidValue;
    if (a.dout % 256 == 0) return launch_bn<256>(a, x, rows, w, grid, o);
    return launch_bn<128>(a, x, rows, w, grid, o);
}

}  // namespace ep
