// expert_gemm.cu - the expert consumer between dispatch and combine: a
// grouped GEMM  y[p] = x[p] * W_e^T  over the receive rows of every expert,
// driven by the per-expert counts and offsets the layout left on the device
// ("ep: graph-safe worst-token HT dispatch+combine", "Internode" item 2: the
// counts stay on the device so graph-mode consumers never touch the host;
// "Tests": layout -> dispatch -> expert -> combine). No host round trip: the
// tile list is derived on the device from the counts.
//
// sm_103a tensor cores, written directly:
//   - one CTA per SM, persistent over output tiles of 128 rows x BN columns
//     of one expert (tile order: the column blocks of one row block first,
//     so the row block is reused from L2);
//   - light experts (at most light_rows rows: their weights are read from
//     HBM for one or two row tiles, so their tiles wait on memory) and heavy
//     ones (weights reused from L2 by many row tiles, so their tiles wait on
//     the tensor cores) form two tile sequences, each in expert order, that
//     are interleaved in proportion to their lengths: at every point of the
//     schedule both kinds run side by side, instead of a tensor-bound phase
//     followed by a memory-bound one when the routing is skewed;
//   - warp 0 (one thread) streams BK-wide K slices of the row block and of
//     the expert's weights into a shared-memory ring with TMA tensor copies
//     (128-byte swizzle for BK = 64, 64-byte for BK = 32), completion on
//     mbarriers;
//   - warp 1 owns two BN-column fp32 accumulators in tensor memory (TMEM)
//     and one thread issues tcgen05.mma (M=128, N=BN, K=16, bf16 inputs, fp32
//     accumulate) from shared-memory descriptors, committing each stage back
//     to the ring and each finished tile to the epilogue; tiles alternate
//     between the accumulators so the epilogue overlaps the next tile;
//   - warps 2-5 read the accumulator with tcgen05.ld (each warp its 32-lane
//     quarter), round to bf16 and store the rows that belong to the expert.
//
// A single-CTA 128 x 256 MMA reads 12 KB of operands from shared memory per
// K=16 step; with the ring's copies writing as much again, this kernel's MMAs
// ran at 1.46 PFLOP/s even with the copies switched off, against 2.42 PFLOP/s
// for a bare stream of the same MMAs from fixed operands.
//
// Two-SM variant (PAIR, the default where dout % 256 == 0): a cluster of two
// CTAs computes 256 x 256 tiles with tcgen05.mma.cta_group::2 (M = 256):
//   - CTA r holds rows [128r, 128r + 128) of the tile and the W rows
//     [128r, 128r + 128) of the column block, so each SM reads 8 KB per K=16
//     step and takes 32 KB per 64-wide slice into shared memory instead of 48;
//   - both CTAs' TMA copies complete on the leader's (rank 0) full barrier;
//     the leader's one MMA thread issues for both SMs, and its commits arrive
//     on both CTAs' barriers (stage release, accumulator ready);
//   - each CTA's epilogue drains its own TMEM (its 128 rows x 256 columns) and
//     tells the leader, which reuses an accumulator only after both have;
//   - an expert's last rows, when at most 128 remain, run as one M = 128 tile
//     across the pair (64 rows per CTA, loaded with a 64-row box). Its
//     accumulator holds the CTA's 64 rows twice in 128 columns: lanes 0-63
//     with output columns [0, 128), lanes 64-127 with [128, 256), so every
//     epilogue warp drains 32 rows x 128 columns.
// Tiles cover 256 rows of one expert, so an expert's last tile is padded to
// 256 rows when more than 128 remain (to 128 otherwise).
//
// Every wait is bounded; on a timeout the CTA reports EP_DEVERR_TIMEOUT,
// waits (bounded) for its copies and MMAs in flight, frees its TMEM and
// returns.
#include <cuda.h>

#include <mutex>

#include "ep_device.cuh"
#include "ep_next.cuh"

namespace ep {
namespace {

constexpr int kBM = 128;            // rows per tile = TMEM lanes = UMMA M
constexpr int kUmmaK = 16;          // K per tcgen05.mma for 16-bit inputs
constexpr int kGemmThreads = 192;   // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 epilogue
constexpr int kPairBN = 256;
constexpr uint16_t kBothCtas = 0x3;
constexpr int kSmemLimit = 232448;  // dynamic shared memory per CTA on sm_103

// Bytes after the ring: barriers, TMEM address, abort flag, the two
// per-expert tile prefixes (heavy, light) and the per-expert row counts (all
// sized for the largest expert count).
template <int STAGES>
constexpr int tail_bytes()
{
    return 8 * (2 * STAGES + 5) + 8 + 8 * (kMaxExperts + 1) + 4 * kMaxExperts;
}

template <int BN_, int BK_, int STAGES_, bool PAIR_>
struct Cfg {
    static constexpr int BN = BN_, BK = BK_, STAGES = STAGES_;
    static constexpr bool PAIR = PAIR_;
    static constexpr int kTileRows = PAIR ? 2 * kBM : kBM;          // rows of one work unit
    static constexpr int kRowsB = PAIR ? BN / 2 : BN;               // W rows this CTA holds
    static constexpr uint32_t kBytesA = kBM * BK * 2;
    static constexpr uint32_t kBytesB = kRowsB * BK * 2;
    static constexpr uint32_t kStageBytes = kBytesA + kBytesB;      // per CTA
    // Instruction descriptor, kind::f16: fp32 accumulate (bits 4-5 = 1), A and
    // B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
    // N >> 3 at bits 17-22, M >> 4 at bits 24-28 (M = 256 across a pair).
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                       ((uint32_t)(BN >> 3) << 17) |
                                       ((uint32_t)(kTileRows >> 4) << 24);
    // Pairs: an expert's last rows, when at most 128 are left, run as M = 128
    // across the pair (64 rows per CTA; same N).
    static constexpr uint32_t kIdescHalf = (kIdesc & ~(0x1Fu << 24)) |
                                           ((uint32_t)((kTileRows / 2) >> 4) << 24);
    static constexpr uint32_t kBytesAHalf = kBytesA / 2;
    static constexpr uint32_t kTmemCols = 2 * BN;                   // two accumulators per CTA
    // Epilogue warps that release an accumulator (both CTAs for a pair).
    static constexpr uint32_t kReleaseCount = PAIR ? 8u : 4u;
    // One K slice of a row is one swizzle span: 128 bytes (BK = 64) or 64 (BK = 32).
    static constexpr uint32_t kSpan = BK * 2;
    static constexpr uint64_t kSwizzleMode = (BK == 64) ? 2 : 4;   // descriptor: 128B = 2, 64B = 4
    static constexpr uint32_t kSbo = 8 * kSpan;                     // bytes between 8-row groups
    static constexpr size_t kSmem = 1024 + (size_t)STAGES * kStageBytes + tail_bytes<STAGES>();
    static_assert(BK == 64 || BK == 32, "K slice is one 128- or 64-byte swizzle span");
    static_assert(!PAIR || BN == kPairBN, "pairs use 256-column tiles");
    static_assert(kSmem <= (size_t)kSmemLimit, "ring does not fit in shared memory");
};

// Shared-memory matrix descriptor for a K-major tile written by TMA with the
// 128- or 64-byte swizzle: start address >> 4 (bits 0-13), leading offset 16 B
// (unused for these layouts), stride between 8-row groups >> 4 (bits 32-45),
// descriptor version 1 (bits 46-47), swizzle mode (bits 61-63).
template <class C>
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
           ((uint64_t)(C::kSbo >> 4) << 32) | ((uint64_t)1 << 46) | (C::kSwizzleMode << 61);
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

// Pair form: the data lands in this CTA's shared memory, the completion on an
// mbarrier that may be the peer's (bar: a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, int c0,
                                                 int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// shared::cluster address of the same offset in CTA rank of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, int rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its shared::cluster address (any CTA of the cluster).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
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

// tcgen05 allocation, MMA and commit; a kernel uses one CTA group throughout
// (PAIR: cta_group::2, issued for both CTAs of the pair).
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    if (PAIR)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         dst_smem),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         dst_smem),
                     "r"(ncols)
                     : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_relinquish()
{
    if (PAIR) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    else asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    if (PAIR)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
}

template <bool PAIR>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    if (PAIR)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrives on bar once the MMAs issued so far finish; PAIR: on bar in both CTAs.
template <bool PAIR>
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    if (PAIR)
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
            "[%0], %1;" ::"r"(bar),
            "h"(kBothCtas)
            : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
}

// Arrives on this CTA's bar only.
template <bool PAIR>
__device__ __forceinline__ void umma_commit_local(uint32_t bar)
{
    if (PAIR)
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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

__device__ __forceinline__ void cluster_sync()
{
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ int cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return (int)r;
}

__device__ __forceinline__ int cluster_index()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return (int)r;
}

__device__ __forceinline__ int cluster_count()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return (int)r;
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

// Index e with pre[e] <= i < pre[e+1] of a non-decreasing prefix (i < pre[E]).
__device__ __forceinline__ int expert_of(const int* pre, int E, int i)
{
    int lo = 0, hi = E;   // invariant: pre[lo] <= i < pre[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= i) lo = mid;
        else hi = mid;
    }
    return lo;
}

struct TileRef {
    int e;       // expert
    int mt;      // row tile (of kTileRows rows) within the expert
    int nb;      // column block
    bool half;   // pairs: the expert's last rows, at most kTileRows / 2 of them (M = 128)
};

// The schedule: uh heavy units then, interleaved with them in proportion,
// total - uh light ones. Within a class, unit v = (row tile of the class's
// prefix, column block), column blocks fastest.
struct Schedule {
    const int* heavy;   // [E + 1] prefix of the heavy experts' row tiles (light: 0)
    const int* light;   // [E + 1] prefix of the light experts' row tiles (heavy: 0)
    const int* cnt;     // [E] rows of each expert
    int uh, total;      // heavy units, all units
    int tile_rows;      // rows of a full row tile
    bool halves;        // pairs: last row tiles of at most tile_rows / 2 rows run as M = 128
};

// Unit u is the h-th heavy unit when floor((u + 1) uh / total) steps past
// h = floor(u uh / total), else the (u - h)-th light one: the heavy units
// before u are exactly floor(u uh / total), so every unit of both classes
// appears once.
__device__ __forceinline__ TileRef tile_of(const Schedule& q, int E, int nbk, int u)
{
    const int h = (int)(((int64_t)u * q.uh) / q.total);
    const bool heavy = (int)(((int64_t)(u + 1) * q.uh) / q.total) > h;
    const int* pre = heavy ? q.heavy : q.light;
    const int v = heavy ? h : u - h;
    TileRef p;
    const int mt = v / nbk;
    p.nb = v % nbk;
    p.e = expert_of(pre, E, mt);
    p.mt = mt - pre[p.e];
    p.half = q.halves && q.cnt[p.e] - p.mt * q.tile_rows <= q.tile_rows / 2;
    return p;
}

// tm_a: box of [128 rows][BK] over the receive rows; tm_a_half: [64 rows][BK]
// (pairs' M = 128 tiles); tm_b: box of [kRowsB rows][BK] over the weights
// (half a column block per CTA for pairs).
template <class C>
__global__ void __launch_bounds__(kGemmThreads, 1)
expert_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_a_half,
                   const __grid_constant__ CUtensorMap tm_b, GemmArgs a)
{
    constexpr int STAGES = C::STAGES, BN = C::BN, BK = C::BK;
    constexpr bool PAIR = C::PAIR;
    extern __shared__ uint8_t smem_raw[];
    // Swizzled tiles want 1024-byte alignment; the offset is the same in both
    // CTAs of a pair (the MMA reads the peer's tiles, and copies and arrivals
    // reach the peer, at the same CTA-relative offsets).
    const uint32_t raw_u32 = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
    const uint32_t tiles_u32 = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
    const uint32_t full0 = smem_u32(bars);                 // STAGES (pairs: the leader's count)
    const uint32_t empty0 = full0 + 8u * STAGES;           // STAGES
    const uint32_t accum_full0 = empty0 + 8u * STAGES;     // 2: one per accumulator
    const uint32_t accum_empty0 = accum_full0 + 16u;       // 2 (pairs: the leader's count)
    const uint32_t drain = accum_empty0 + 16u;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    int* s_heavy = const_cast<int*>(reinterpret_cast<volatile int*>(s_abort + 1));   // [E + 1]
    int* s_light = s_heavy + (kMaxExperts + 1);                                        // [E + 1]
    int* s_cnt = s_light + (kMaxExperts + 1);                                          // [E]
    const int E = a.E;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = PAIR ? cluster_rank() : 0;
    const bool leader = r == 0;
    const int first = PAIR ? cluster_index() : (int)blockIdx.x;
    const int step = PAIR ? cluster_count() : (int)gridDim.x;
    const int k_iters = (int)(a.din / BK);
    const int nbk = (int)(a.dout / BN);
    // The barriers the MMA thread waits on live in the leader (rank 0).
    const uint32_t lead_full0 = PAIR ? map_to_rank(full0, 0) : full0;
    const uint32_t lead_accum_empty0 = PAIR ? map_to_rank(accum_empty0, 0) : accum_empty0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8u * s, 1u);
            mbar_init(empty0 + 8u * s, 1u);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accum_full0 + 8u * b, 1u);
            mbar_init(accum_empty0 + 8u * b, C::kReleaseCount);
        }
        mbar_init(drain, 1u);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc<PAIR>(smem_u32(s_tmem), C::kTmemCols);
        tmem_relinquish<PAIR>();
    }

    griddep_wait();   // counts, offsets and the receive rows come from earlier kernels

    // Prefixes over experts of their row tiles (kTileRows rows each), one per
    // class: experts with at most light_rows rows are light.
    if (warp == 0) {
        int carry_h = 0, carry_l = 0;
        if (lane == 0) s_heavy[0] = s_light[0] = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = (e < E) ? __ldcg(a.cnt + e) : 0;
            if (e < E) s_cnt[e] = c;
            const int m = (c + C::kTileRows - 1) / C::kTileRows;
            const bool is_light = c <= a.light_rows;
            int mh = is_light ? 0 : m, ml = is_light ? m : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int nh = __shfl_up_sync(0xffffffffu, mh, d);
                const int nl = __shfl_up_sync(0xffffffffu, ml, d);
                if (lane >= d) {
                    mh += nh;
                    ml += nl;
                }
            }
            if (e < E) {
                s_heavy[e + 1] = carry_h + mh;
                s_light[e + 1] = carry_l + ml;
            }
            carry_h += __shfl_sync(0xffffffffu, mh, 31);
            carry_l += __shfl_sync(0xffffffffu, ml, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // the peer's barriers exist before any copy or arrival reaches them
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    Schedule q;
    q.heavy = s_heavy;
    q.light = s_light;
    q.cnt = s_cnt;
    q.tile_rows = C::kTileRows;
    q.halves = PAIR;
    q.uh = s_heavy[E] * nbk;
    q.total = q.uh + s_light[E] * nbk;
    const int total = q.total;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer (each CTA fills its own ring) --------------------
        int g = 0;   // k-slices issued
        for (int u = first; u < total && !*s_abort; u += step) {
            const TileRef p = tile_of(q, E, nbk, u);
            const int row0 = __ldcg(a.expert_offset + p.e) + p.mt * C::kTileRows +
                             r * (p.half ? kBM / 2 : kBM);
            const int wrow0 = p.e * (int)a.dout + p.nb * BN + r * C::kRowsB;
            for (int k = 0; k < k_iters; ++k, ++g) {
                const int s = g % STAGES;
                const uint32_t ph = (uint32_t)((g / STAGES) & 1);
                if (!wait_or_abort(empty0 + 8u * s, ph ^ 1u, s_abort)) break;
                const uint32_t sa = tiles_u32 + (uint32_t)s * C::kStageBytes;
                const uint32_t sb = sa + C::kBytesA;
                const int kc = k * BK;
                if (!PAIR) {
                    const uint32_t fb = full0 + 8u * s;
                    mbar_expect_tx(fb, C::kStageBytes);
                    tma_load_2d(sa, &tm_a, kc, row0, fb);
                    tma_load_2d(sb, &tm_b, kc, wrow0, fb);
                } else {
                    // Both CTAs' copies complete on the leader's barrier, which
                    // expects the bytes of both (an M = 128 tile: 64 rows of x per CTA).
                    if (leader)
                        mbar_expect_tx(full0 + 8u * s,
                                       2u * (p.half ? C::kBytesAHalf + C::kBytesB : C::kStageBytes));
                    const uint32_t fb = lead_full0 + 8u * s;
                    tma_load_2d_pair(sa, p.half ? &tm_a_half : &tm_a, kc, row0, fb);
                    tma_load_2d_pair(sb, &tm_b, kc, wrow0, fb);
                }
            }
        }
        // The copies this thread issued land before shared memory goes away
        // (a pair's copies are tracked by the leader's barrier: wait for the
        // MMAs to release the stages instead).
        const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
        for (int i = (g > STAGES ? g - STAGES : 0); i < g; ++i) {
            const uint32_t s = (uint32_t)(i % STAGES), par = (uint32_t)((i / STAGES) & 1);
            if (PAIR) mbar_wait_until(empty0 + 8u * s, par, deadline);
            else mbar_wait_until(full0 + 8u * s, par, deadline);
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ---- MMA issuer (pairs: the leader's, for both SMs) ----------------
        int g = 0, tl = 0;
        bool issued = false;
        for (int u = first; u < total && !*s_abort; u += step, ++tl) {
            const int acc = tl & 1, use = tl >> 1;      // accumulator and its use count
            if (!wait_or_abort(accum_empty0 + 8u * acc, (uint32_t)((use & 1) ^ 1), s_abort)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
            const uint32_t idesc = tile_of(q, E, nbk, u).half ? C::kIdescHalf : C::kIdesc;
            bool ok = true;
            for (int k = 0; k < k_iters; ++k, ++g) {
                const int s = g % STAGES;
                if (!wait_or_abort(full0 + 8u * s, (uint32_t)((g / STAGES) & 1), s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = tiles_u32 + (uint32_t)s * C::kStageBytes;
#pragma unroll
                for (int j = 0; j < BK / kUmmaK; ++j)
                    umma_bf16<PAIR>(d_tmem, smem_desc<C>(sa + j * kUmmaK * 2),
                                    smem_desc<C>(sa + C::kBytesA + j * kUmmaK * 2), idesc,
                                    (k | j) != 0 ? 1u : 0u);
                issued = true;
                umma_commit<PAIR>(empty0 + 8u * s);   // frees the stage (in both CTAs of a pair)
            }
            if (!ok) break;
            umma_commit<PAIR>(accum_full0 + 8u * acc);   // the tile's accumulator is complete
        }
        if (issued) {   // every MMA this thread issued has finished before TMEM is freed
            umma_commit_local<PAIR>(drain);
            mbar_wait(drain, 0u);
        }
    } else if (warp >= 2) {
        // ---- epilogue: TMEM -> bf16 -> global ------------------------------
        const int quarter = warp & 3;                  // TMEM lanes this warp may read
        const int r_in = quarter * 32 + lane;          // accumulator row = tile row (of this CTA)
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        uint16_t* y = static_cast<uint16_t*>(a.y);
        int tl = 0;
        for (int u = first; u < total && !*s_abort; u += step, ++tl) {
            const int acc = tl & 1, use = tl >> 1;
            if (!wait_or_abort(accum_full0 + 8u * acc, (uint32_t)(use & 1), s_abort)) break;
            tc_fence_after();
            const uint32_t t_acc = t_lane + (uint32_t)(acc * BN);
            const TileRef p = tile_of(q, E, nbk, u);
            // The rows this warp drains and the output columns they cover. A full
            // tile: lane quarter w holds this CTA's tile rows 32w..32w+31, every
            // column. A pair's M = 128 tile: the CTA's 64 rows appear twice, lanes
            // 0-63 with output columns [0, BN/2) and lanes 64-127 with
            // [BN/2, BN), both in accumulator columns [0, BN/2).
            const int sub = p.half ? 32 * (quarter & 1) + lane : r_in;
            const int col0 = p.half ? (BN / 2) * (quarter >> 1) : 0;
            const int ncols = p.half ? BN / 2 : BN;
            const int part = p.half ? kBM / 2 : kBM;       // rows of this CTA's part
            const int m_in = p.mt * C::kTileRows + r * part;
            const int rows = min(part, q.cnt[p.e] - m_in);
            const int64_t row = (int64_t)__ldcg(a.expert_offset + p.e) + m_in + sub;
#pragma unroll 1
            for (int c = 0; c < ncols; c += 32) {
                uint32_t v[32];
                tmem_ld32(t_acc + (uint32_t)c, v);
                tmem_wait_ld();
                if (sub < rows) {
                    int4* dst = reinterpret_cast<int4*>(y + row * a.dout + p.nb * BN + col0 + c);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        int4 w;
                        w.x = (int)pack_bf16x2_rn(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1]));
                        w.y = (int)pack_bf16x2_rn(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
                        w.z = (int)pack_bf16x2_rn(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]));
                        w.w = (int)pack_bf16x2_rn(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
                        dst[g] = w;
                    }
                }
            }
            // This warp's reads of the accumulator are done: one arrival per
            // warp on the leader's barrier.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR) mbar_arrive_cluster(lead_accum_empty0 + 8u * acc);
                else mbar_arrive(accum_empty0 + 8u * acc);
            }
        }
    }

    if (threadIdx.x == 0 && *s_abort) atomicOr(a.err, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    // Pairs: the leader's MMAs (which read the peer's shared memory and write
    // its TMEM) and its arrivals on the peer are done before either CTA frees
    // TMEM or exits.
    if (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<PAIR>(tmem, C::kTmemCols);
    }
    griddep_launch_dependents();
}

// Ring depths: as many stages as fit next to the tail (at most 12); a stage
// holds 128 rows and the CTA's rows_b rows of W.
template <int ROWS_B, int BK>
constexpr int stages_for()
{
    const int fit = (kSmemLimit - 1024 - tail_bytes<12>()) / (int)((kBM + ROWS_B) * BK * 2);
    return fit > 12 ? 12 : fit;
}

template <int BN, int BK, bool PAIR>
using CfgOf = Cfg<BN, BK, stages_for<(PAIR ? BN / 2 : BN), BK>(), PAIR>;

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

// 2-D bf16 tensor map over [rows][inner] with a box of [box_rows][bk] and the
// swizzle the UMMA descriptors expect (one swizzle span per box row).
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
              int bk)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)bk, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void set_attrs(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, bool pair, bool pdl)
{
    int n = 0;
    if (pair) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg->attrs = attr;
    cfg->numAttrs = n;
}

// CTAs of the persistent cluster grid of `kernel` (its dynamic shared memory
// attribute already set): twice the clusters that fit at once (one CTA per SM),
// within the SM budget; 0 if no cluster fits. Cached per kernel and device.
template <typename Kernel>
int cluster_grid(Kernel kernel, size_t smem, int num_sms)
{
    static std::mutex mu;
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    int fit = (dev >= 0 && dev < 64) ? cached[dev] : 0;
    if (fit == 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        cfg.gridDim = dim3((unsigned)(sms & ~1));
        cfg.blockDim = dim3(kGemmThreads);
        cfg.dynamicSmemBytes = smem;
        set_attrs(&cfg, attr, true, false);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            return 0;
        }
        fit = 2 * n;
        if (dev >= 0 && dev < 64) cached[dev] = fit;
    }
    const int budget = num_sms & ~1;
    return fit < budget ? fit : budget;
}

template <class C>
cudaError_t launch_cfg(const GemmArgs& a, const void* x, int64_t rows, const void* w, int num_sms,
                       const LaunchOpts& o, int* grid_used)
{
    cudaError_t e = cudaFuncSetAttribute(expert_gemm_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    int grid = num_sms;
    if (C::PAIR) {
        grid = cluster_grid(expert_gemm_kernel<C>, C::kSmem, num_sms);
        if (grid < 2) return cudaErrorNotSupported;
    }
    CUtensorMap ta, ta_half, tb;
    const uint64_t wrows = (uint64_t)a.E * (uint64_t)a.dout;
    if (!make_map(&ta, x, (uint64_t)a.din, (uint64_t)rows, kBM, C::BK) ||
        !make_map(&ta_half, x, (uint64_t)a.din, (uint64_t)rows, kBM / 2, C::BK) ||
        !make_map(&tb, w, (uint64_t)a.din, wrows, C::kRowsB, C::BK))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = o.stream;
    set_attrs(&cfg, attr, C::PAIR, o.pdl);
    e = cudaLaunchKernelEx(&cfg, expert_gemm_kernel<C>, ta, ta_half, tb, a);
    if (e == cudaSuccess && o.launches) ++*o.launches;
    *grid_used = grid;
    return e;
}

template <int BK>
cudaError_t launch_bk(const GemmArgs& a, const void* x, int64_t rows, const void* w, int grid,
                      const LaunchOpts& o, int* kernel_used, int* grid_used)
{
    if (a.kind >= 2 && a.dout % kPairBN == 0) {
        *kernel_used = 2;
        const cudaError_t e = launch_cfg<CfgOf<kPairBN, BK, true>>(a, x, rows, w, grid, o, grid_used);
        if (e != cudaErrorNotSupported) return e;
    }
    *kernel_used = 1;
    if (a.dout % 256 == 0)
        return launch_cfg<CfgOf<256, BK, false>>(a, x, rows, w, grid, o, grid_used);
    return launch_cfg<CfgOf<128, BK, false>>(a, x, rows, w, grid, o, grid_used);
}

}  // namespace

cudaError_t launch_expert_gemm(const GemmArgs& a, const void* x, int64_t rows, const void* w,
                               int grid, const LaunchOpts& o, int* kernel_used, int* grid_used)
{
    if (a.din % 64 != 0 || a.dout % 128 != 0) return cudaErrorInvalidValue;
    if (a.bk == 32) return launch_bk<32>(a, x, rows, w, grid, o, kernel_used, grid_used);
    return launch_bk<64>(a, x, rows, w, grid, o, kernel_used, grid_used);
}

}  // namespace ep
