// ep_api.cu - the C ABI declared in include/ep.h: buffer set-up over a
// caller-owned workspace, argument checks, and the stream-ordered calls that
// enqueue the layout, permute and combine kernels.
//
// The buffer follows "Unify expert parallel token dispatcher API": the
// lifetime maximum num_max_tokens_per_rank sizes persistent storage once
// ("API design"; "Backend behavior": DeepEP and HybridEP preallocate), and
// each call lays out its current capacity inside it without growing it. The
// graph-safety rules follow "ep: graph-safe worst-token HT dispatch+combine":
// no host handshake, no host-mapped counters, counts stay on the device.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "ep.h"
#include "ep_kernels.cuh"
#include "ep_next.cuh"

struct ep_buffer {
    ep_config cfg;
    int device;
    int num_sms;
    int64_t row_bytes;
    int64_t s_max;          // roundup4(N_max) * K
    int64_t max_tiles;      // layout tiles the tables hold
    int ep_stride;          // row stride of the tile tables: roundup4(E)
    bool pdl;               // launch with programmatic dependent launch
    int tiles_per_sm;       // layout tiles (fused-dispatch CTAs) per SM
    int gemm_kind;          // expert GEMM kernel (GemmArgs::kind), 0: chosen per call
    int gemm_bk;            // expert GEMM K slice per ring stage (64 or 32)
    int gemm_light_rows;    // expert GEMM: experts with at most this many rows are light
    bool dedup_fused;       // dedupe dispatch in one kernel after the counts
    bool onepass;           // dispatch as one cooperative kernel where it fits
    bool debug;             // EP_DEBUG: sentinel fill and checks of the receive rows
    bool nvtx;              // EP_NVTX: an NVTX range around every call
    bool coop_pdl;          // cooperative launches take programmatic serialization
    uint32_t* gbar;         // [4] the one-pass dispatch's grid barrier and token-pool counter
    uint32_t* tile_ready;   // [max_tiles] the one-pass dispatch's per-tile ready words
    int dispatch_pool_pct;  // share of each tile's tokens in the one-pass dispatch's pool
    int64_t dispatch_small_pairs;   // calls this small count every id in every CTA, no barrier
    int combine_per_sm;     // combine CTAs per SM at most (0: as many as fit)
    int gemm_kernel;        // last expert GEMM: 0 none, 1 single-CTA, 2 two-SM
    int gemm_grid;
    int64_t test_skip_load; // test hook (EP_TEST_SKIP_LOAD), -1 = off
    size_t ws_bytes;
    // carved device pointers
    uint8_t* recv_x;
    float* recv_scores;
    int32_t* recv_src;
    int32_t* pos;
    int32_t* cnt;
    int32_t* expert_offset;
    int32_t* rows_per_rank;
    int32_t* rank_prefix;
    int32_t* tokens_in_rank;
    int32_t* tile_cnt;
    int32_t* tile_pre;
    int32_t* tile_tok;
    int32_t* tile_tok_pre;
    int32_t* tok_pos;
    int32_t* tok_src;
    uint32_t* err;
    // plans
    ep::PermutePlan permute;
    int combine_grid;
    // state of the last layout on this buffer (host-side scalars only)
    bool has_layout;
    bool last_dedup;        // the last dispatch wrote dedupe rows
    int64_t last_T, last_N, last_S;
    int64_t launches;
};

namespace {

constexpr size_t kAlign = 256;
// Expert GEMM schedule: experts with at most this many rows are light (their
// weights feed one or two 128-row tiles, so those tiles wait on HBM).
constexpr int kGemmLightRows = 256;
// One-pass dispatch: percent of each tile's tokens in the shared token pool
// (CTAs that finish their own share early copy the rest of the others').
constexpr int kDispatchPoolPct = 25;
// One-pass dispatch: calls of at most this many (token, k) pairs count all of
// their ids in every CTA instead of meeting at the grid barrier.
constexpr int64_t kDispatchSmallPairs = 2048;
// Combine CTAs per SM at most (0: as many as fit).
constexpr int kCombinePerSm = 0;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int64_t pad4(int64_t n) { return (n + 3) / 4 * 4; }

int64_t elem_bytes(int32_t dtype) { return dtype == EP_BF16 ? 2 : 4; }

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Validates a configuration; fills the derived sizes. Host-only.
bool check_config(const ep_config* c, int64_t* row_bytes, int64_t* s_max, int64_t* max_tiles)
{
    if (!c) return false;
    if (c->num_max_tokens_per_rank < 1 || c->hidden < 1) return false;
    if (c->dtype != EP_BF16 && c->dtype != EP_F32) return false;
    if (c->num_experts < 1 || c->num_experts > ep::kMaxExperts) return false;
    if (c->num_ranks < 1 || c->num_ranks > ep::kMaxRanks) return false;
    if (c->num_experts % c->num_ranks != 0) return false;
    if (c->topk < 1 || c->topk > c->num_experts || c->topk > ep::kMaxTopk) return false;
    if (c->num_sms < 0) return false;
    if (c->permute_impl < EP_PERMUTE_DEFAULT || c->permute_impl > EP_PERMUTE_BULK) return false;
    if (c->layout_mode != EP_LAYOUT_STRIDED && c->layout_mode != EP_LAYOUT_PACKED) return false;
    const int64_t rb = c->hidden * elem_bytes(c->dtype);
    if (rb % 16 != 0) return false;
    const int64_t s = pad4(c->num_max_tokens_per_rank) * c->topk;
    // Receive rows and pair indices are int32 on the device.
    if (s > INT32_MAX / c->num_ranks) return false;
    if (c->num_max_tokens_per_rank * c->topk > INT32_MAX) return false;
    *row_bytes = rb;
    *s_max = s;
    *max_tiles = ep::max_tiles(c->num_max_tokens_per_rank, c->topk);
    return true;
}

struct Carve {
    size_t off = 0;
    size_t take(size_t bytes)
    {
        const size_t at = off;
        off = align_up(off + (bytes ? bytes : 1));
        return at;
    }
};

struct Offsets {
    size_t recv_x, recv_scores, recv_src, pos, cnt, expert_offset, rows_per_rank, rank_prefix,
        tokens_in_rank, tile_cnt, tile_pre, tile_tok, tile_tok_pre, tok_pos, tok_src, tile_ready,
        gbar, err, total;
};

Offsets layout_workspace(const ep_config* c, int64_t row_bytes, int64_t s_max, int64_t max_tiles)
{
    const size_t rows = (size_t)c->num_ranks * (size_t)s_max;
    const size_t E = (size_t)c->num_experts, R = (size_t)c->num_ranks;
    const size_t Ep = (size_t)ep::round_up4(c->num_experts);
    Carve cv;
    Offsets o;
    o.recv_x = cv.take(rows * (size_t)row_bytes);
    o.recv_scores = cv.take(rows * 4);
    o.recv_src = cv.take(rows * 4);
    o.pos = cv.take((size_t)c->num_max_tokens_per_rank * (size_t)c->topk * 4);
    o.cnt = cv.take(E * 4);
    o.expert_offset = cv.take(E * 4);
    o.rows_per_rank = cv.take(R * 4);
    o.rank_prefix = cv.take(R * 4);
    o.tokens_in_rank = cv.take(R * 4);
    o.tile_cnt = cv.take((size_t)max_tiles * Ep * 4);
    o.tile_pre = cv.take((size_t)max_tiles * Ep * 4);
    o.tile_tok = cv.take((size_t)max_tiles * R * 4);
    o.tile_tok_pre = cv.take((size_t)max_tiles * R * 4);
    o.tok_pos = cv.take((size_t)c->num_max_tokens_per_rank * R * 4);
    o.tok_src = cv.take(R * (size_t)pad4(c->num_max_tokens_per_rank) * 4);
    o.tile_ready = cv.take((size_t)max_tiles * 4);
    o.gbar = cv.take(16);
    o.err = cv.take(4);   // last: the workspace ends after the error word
    o.total = cv.off;
    return o;
}

cudaStream_t as_stream(ep_stream_t s) { return static_cast<cudaStream_t>(s); }

// True if the stream is capturing (or the query failed: treat as capturing,
// so no host synchronisation is attempted).
bool capturing(cudaStream_t s)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return true;
    return st != cudaStreamCaptureStatusNone;
}

ep_status check_call(const ep_buffer* b, const void* ids, int64_t T, int64_t N)
{
    if (!b) return EP_ERR_INVALID_ARG;
    if (T < 0 || N < T) return EP_ERR_INVALID_ARG;
    if (N > b->cfg.num_max_tokens_per_rank) return EP_ERR_CAPACITY;
    if (T > 0 && !ids) return EP_ERR_INVALID_ARG;
    if (!is_aligned(ids, 4)) return EP_ERR_ALIGNMENT;
    return EP_OK;
}

void fill_layout(const ep_buffer* b, ep_layout* out)
{
    if (!out) return;
    out->tokens_per_expert = b->cnt;
    out->expert_offset = b->expert_offset;
    out->rows_per_rank = b->rows_per_rank;
    out->rank_prefix = b->rank_prefix;
    out->tokens_in_rank = b->tokens_in_rank;
    out->pos = b->pos;
    out->num_tokens = b->last_T;
    out->padded_tokens = pad4(b->last_N);
    out->rank_stride = b->last_S;
    out->packed = b->cfg.layout_mode == EP_LAYOUT_PACKED ? 1 : 0;
}

void fill_dispatch(const ep_buffer* b, ep_dispatch_out* out)
{
    if (!out) return;
    out->recv_x = b->recv_x;
    out->recv_scores = b->recv_scores;
    out->recv_src = b->recv_src;
    fill_layout(b, &out->layout);
}

ep::LaunchOpts opts(ep_buffer* b, cudaStream_t s) { return ep::LaunchOpts{s, b->pdl, &b->launches}; }

// An NVTX range for the lifetime of a call when EP_NVTX=1.
struct Range {
    bool on;
    Range(const ep_buffer* b, const char* name) : on(b && b->nvtx)
    {
        if (on) nvtxRangePushA(name);
    }
    ~Range()
    {
        if (on) nvtxRangePop();
    }
};

// EP_DEBUG: the call's receive rows (R * S) get the 0xFF sentinel before a permute.
bool debug_fill(ep_buffer* b, int64_t S, cudaStream_t s)
{
    return !b->debug || cudaMemsetAsync(b->recv_x, 0xFF,
                                        (size_t)b->cfg.num_ranks * (size_t)S * (size_t)b->row_bytes,
                                        s) == cudaSuccess;
}

// EP_DEBUG: rows inside each rank's true total written, the rest untouched.
bool debug_check(ep_buffer* b, const void* rows, cudaStream_t s)
{
    if (!b->debug) return true;
    ep::SentinelArgs a;
    a.recv_x = static_cast<const uint8_t*>(rows);
    a.S = b->last_S;
    a.row_bytes = b->row_bytes;
    a.R = b->cfg.num_ranks;
    a.packed = b->cfg.layout_mode == EP_LAYOUT_PACKED;
    a.rows_per_rank = b->rows_per_rank;
    a.rank_prefix = b->rank_prefix;
    a.err = b->err;
    return ep::launch_sentinel_check(a, b->num_sms, opts(b, s)) == cudaSuccess;
}

ep::LayoutArgs layout_args(ep_buffer* b, const int32_t* ids, int64_t T, int64_t N)
{
    ep::LayoutArgs a;
    a.ids = ids;
    a.T = T;
    a.S = pad4(N) * b->cfg.topk;
    a.tpt = ep::tokens_per_tile(T, b->cfg.topk, b->num_sms * b->tiles_per_sm);
    a.ntiles = (int)ep::tile_count(T, a.tpt);
    a.K = b->cfg.topk;
    a.E = b->cfg.num_experts;
    a.R = b->cfg.num_ranks;
    a.Ep = b->ep_stride;
    a.tile_cnt = b->tile_cnt;
    a.tile_pre = b->tile_pre;
    a.tile_tok = b->tile_tok;
    a.tile_tok_pre = nullptr;
    a.cnt = b->cnt;
    a.expert_offset = b->expert_offset;
    a.rows_per_rank = b->rows_per_rank;
    a.rank_prefix = b->rank_prefix;
    a.tokens_in_rank = b->tokens_in_rank;
    a.pos = b->pos;
    a.err = b->err;
    a.gbar = b->gbar;
    a.tile_ready = b->tile_ready;
    a.packed = b->cfg.layout_mode == EP_LAYOUT_PACKED;
    return a;
}

ep::PermuteArgs permute_args(ep_buffer* b, const void* x, const float* scores)
{
    ep::PermuteArgs a;
    a.x = x;
    a.scores = scores;
    a.pos = b->pos;
    a.recv_x = b->recv_x;
    a.recv_scores = b->recv_scores;
    a.recv_src = b->recv_src;
    a.T = b->last_T;
    a.K = b->cfg.topk;
    a.row_bytes = b->row_bytes;
    a.err = b->err;
    a.skip_load = b->test_skip_load;
    return a;
}

void remember_layout(ep_buffer* b, int64_t T, int64_t N)
{
    b->has_layout = true;
    b->last_dedup = false;
    b->last_T = T;
    b->last_N = N;
    b->last_S = pad4(N) * b->cfg.topk;
}

ep_status enqueue_layout(ep_buffer* b, const int32_t* ids, int64_t T, int64_t N, cudaStream_t s)
{
    if (ep::launch_layout(layout_args(b, ids, T, N), opts(b, s)) != cudaSuccess) return EP_ERR_CUDA;
    remember_layout(b, T, N);
    return EP_OK;
}

ep_status enqueue_permute(ep_buffer* b, const void* x, const float* scores, cudaStream_t s)
{
    return ep::launch_permute(permute_args(b, x, scores), b->permute, opts(b, s)) == cudaSuccess
               ? EP_OK
               : EP_ERR_CUDA;
}

// Layout counts, then positions + permute fused into one kernel when the call
// fits it, else the positions and permute kernels one after the other.
ep_status enqueue_dispatch(ep_buffer* b, const void* x, const float* scores, const int32_t* ids,
                           int64_t T, int64_t N, cudaStream_t s)
{
    const ep::LayoutArgs la = layout_args(b, ids, T, N);
    const ep::LaunchOpts o = opts(b, s);
    if (b->permute.impl == EP_PERMUTE_BULK) {
        if (b->onepass) {
            const cudaError_t e1 = ep::launch_dispatch_onepass(
                la, permute_args(b, x, scores), b->permute, o, b->coop_pdl, b->dispatch_pool_pct,
                b->dispatch_small_pairs);
            if (e1 == cudaSuccess) {
                remember_layout(b, T, N);
                return EP_OK;
            }
            if (e1 != cudaErrorNotSupported) return EP_ERR_CUDA;
        }
        if (ep::launch_layout_counts(la, o) != cudaSuccess) return EP_ERR_CUDA;
        remember_layout(b, T, N);
        const cudaError_t e = ep::launch_dispatch_fused(la, permute_args(b, x, scores), b->permute, o);
        if (e == cudaSuccess) return EP_OK;
        if (e != cudaErrorNotSupported) return EP_ERR_CUDA;
        if (ep::launch_layout_positions(la, o) != cudaSuccess) return EP_ERR_CUDA;
        return enqueue_permute(b, x, scores, s);
    }
    if (ep::launch_layout(la, o) != cudaSuccess) return EP_ERR_CUDA;
    remember_layout(b, T, N);
    return enqueue_permute(b, x, scores, s);
}

ep_status check_rows(const ep_buffer* b, const void* x, const float* scores)
{
    if (b->last_T > 0 && (!x || !scores)) return EP_ERR_INVALID_ARG;
    if (!is_aligned(x, 16) || !is_aligned(scores, 4)) return EP_ERR_ALIGNMENT;
    return EP_OK;
}

// ---- environment knobs, read once at ep_buffer_init ------------------------

bool env_is(const char* name, const char* value)
{
    const char* v = std::getenv(name);
    return v && std::strcmp(v, value) == 0;
}

int64_t env_int(const char* name, int64_t fallback)
{
    const char* v = std::getenv(name);
    return (v && *v) ? std::strtoll(v, nullptr, 10) : fallback;
}

void read_knobs(ep_buffer* b)
{
    b->pdl = !env_is("EP_PDL", "0");
    // Fused-dispatch CTAs per SM (1 or 2).
    b->tiles_per_sm = env_is("EP_TILES_PER_SM", "2") ? 2 : 1;
    // EP_GEMM_KERNEL=1 / 2 forces the expert GEMM's kernel (single-CTA
    // 128-row tiles, 2-SM 256-row tiles); 0 chooses per call.
    b->gemm_kind = env_is("EP_GEMM_KERNEL", "1") ? 1 : env_is("EP_GEMM_KERNEL", "2") ? 2 : 0;
    // EP_GEMM_BK=32 or 64: the expert GEMM's K slice per ring stage.
    b->gemm_bk = env_is("EP_GEMM_BK", "32") ? 32 : 64;
    // EP_GEMM_LIGHT_ROWS=n: experts with at most n rows are scheduled as light
    // (0: one sequence in expert order).
    const int64_t lr = env_int("EP_GEMM_LIGHT_ROWS", kGemmLightRows);
    b->gemm_light_rows = lr > 0 ? (int)std::min<int64_t>(lr, INT32_MAX) : 0;
    // EP_DEDUP_FUSED=0 runs the dedupe dispatch as positions + copy kernels.
    b->dedup_fused = !env_is("EP_DEDUP_FUSED", "0");
    // EP_DISPATCH_ONEPASS=0 keeps the dispatch as count + scan + fused.
    b->onepass = !env_is("EP_DISPATCH_ONEPASS", "0");
    // EP_DISPATCH_POOL=p: percent of each tile's tokens the one-pass dispatch
    // puts in its shared pool (0: every CTA copies only its own tile).
    const int64_t pool = env_int("EP_DISPATCH_POOL", kDispatchPoolPct);
    b->dispatch_pool_pct = (int)std::min<int64_t>(std::max<int64_t>(pool, 0), 100);
    // EP_COMBINE_PER_SM=n: at most n combine CTAs per SM (0: as many as fit).
    b->combine_per_sm = (int)std::min<int64_t>(std::max<int64_t>(env_int("EP_COMBINE_PER_SM",
                                                                         kCombinePerSm), 0), 64);
    // EP_DISPATCH_SMALL_PAIRS=n: one-pass dispatches of at most n (token, k)
    // pairs count every id in every CTA instead of meeting at the grid barrier.
    b->dispatch_small_pairs = std::max<int64_t>(env_int("EP_DISPATCH_SMALL_PAIRS",
                                                        kDispatchSmallPairs), 0);
    // Debugging: EP_DEBUG=1 (sentinel checks), EP_NVTX=1 (NVTX ranges).
    b->debug = env_is("EP_DEBUG", "1");
    b->nvtx = env_is("EP_NVTX", "1");
    // Test hook: make one bounded wait of the bulk permute run out.
    b->test_skip_load = env_int("EP_TEST_SKIP_LOAD", -1);
}

}  // namespace

extern "C" {

size_t ep_buffer_required_bytes(const ep_config* cfg)
{
    int64_t rb, s_max, tiles;
    if (!check_config(cfg, &rb, &s_max, &tiles)) return 0;
    return layout_workspace(cfg, rb, s_max, tiles).total;
}

ep_status ep_buffer_init(const ep_config* cfg, void* workspace, size_t workspace_bytes,
                         ep_buffer** out)
{
    if (!out) return EP_ERR_INVALID_ARG;
    *out = nullptr;
    int64_t rb, s_max, tiles;
    if (!check_config(cfg, &rb, &s_max, &tiles)) return EP_ERR_INVALID_ARG;
    const Offsets o = layout_workspace(cfg, rb, s_max, tiles);
    if (!workspace || !is_aligned(workspace, kAlign) || workspace_bytes < o.total)
        return EP_ERR_WORKSPACE;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, workspace) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_WORKSPACE;
    }
    if ((attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) ||
        attr.device != dev)
        return EP_ERR_WORKSPACE;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return EP_ERR_CUDA;

    ep_buffer* b = new (std::nothrow) ep_buffer();
    if (!b) return EP_ERR_HOST_ALLOC;
    b->cfg = *cfg;
    b->device = dev;
    // SM budget: the config's, else EP_NUM_SMS, else every SM.
    const int budget = cfg->num_sms > 0 ? cfg->num_sms : (int)env_int("EP_NUM_SMS", 0);
    b->num_sms = (budget > 0 && budget < sms) ? budget : sms;
    b->row_bytes = rb;
    b->s_max = s_max;
    b->max_tiles = tiles;
    b->ep_stride = ep::round_up4(cfg->num_experts);
    read_knobs(b);
    b->ws_bytes = o.total;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    b->recv_x = w + o.recv_x;
    b->recv_scores = reinterpret_cast<float*>(w + o.recv_scores);
    b->recv_src = reinterpret_cast<int32_t*>(w + o.recv_src);
    b->pos = reinterpret_cast<int32_t*>(w + o.pos);
    b->cnt = reinterpret_cast<int32_t*>(w + o.cnt);
    b->expert_offset = reinterpret_cast<int32_t*>(w + o.expert_offset);
    b->rows_per_rank = reinterpret_cast<int32_t*>(w + o.rows_per_rank);
    b->rank_prefix = reinterpret_cast<int32_t*>(w + o.rank_prefix);
    b->tokens_in_rank = reinterpret_cast<int32_t*>(w + o.tokens_in_rank);
    b->tile_cnt = reinterpret_cast<int32_t*>(w + o.tile_cnt);
    b->tile_pre = reinterpret_cast<int32_t*>(w + o.tile_pre);
    b->tile_tok = reinterpret_cast<int32_t*>(w + o.tile_tok);
    b->tile_tok_pre = reinterpret_cast<int32_t*>(w + o.tile_tok_pre);
    b->tok_pos = reinterpret_cast<int32_t*>(w + o.tok_pos);
    b->tok_src = reinterpret_cast<int32_t*>(w + o.tok_src);
    b->err = reinterpret_cast<uint32_t*>(w + o.err);
    b->gbar = reinterpret_cast<uint32_t*>(w + o.gbar);
    b->tile_ready = reinterpret_cast<uint32_t*>(w + o.tile_ready);
    b->coop_pdl = ep::probe_cooperative_pdl();

    const int impl = cfg->permute_impl == EP_PERMUTE_DEFAULT ? EP_PERMUTE_BULK : cfg->permute_impl;
    if (ep::plan_permute(impl, rb, cfg->topk, cfg->num_experts, b->num_sms, b->tiles_per_sm,
                         &b->permute) != cudaSuccess ||
        ep::plan_combine(cfg->dtype == EP_BF16 ? 0 : 1, b->num_sms, b->combine_per_sm,
                         &b->combine_grid) !=
            cudaSuccess ||
        cudaMemset(b->err, 0, sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(b->gbar, 0, 4 * sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(b->tile_ready, 0, (size_t)b->max_tiles * 4) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        delete b;
        return EP_ERR_CUDA;
    }
    *out = b;
    return EP_OK;
}

ep_status ep_buffer_destroy(ep_buffer* buf)
{
    delete buf;
    return EP_OK;
}

ep_status ep_dispatch_layout(ep_buffer* buf, const int32_t* ids, int64_t T, int64_t N,
                             ep_stream_t stream, ep_layout* out, int32_t* host_counts)
{
    const Range range(buf, "ep_dispatch_layout");
    ep_status st = check_call(buf, ids, T, N);
    if (st != EP_OK) return st;
    cudaStream_t s = as_stream(stream);
    if (host_counts && capturing(s)) return EP_ERR_CAPTURE_HOST_SYNC;
    st = enqueue_layout(buf, ids, T, N, s);
    if (st != EP_OK) return st;
    fill_layout(buf, out);
    if (host_counts) {
        if (cudaMemcpyAsync(host_counts, buf->cnt, sizeof(int32_t) * buf->cfg.num_experts,
                            cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return EP_ERR_CUDA;
    }
    return EP_OK;
}

ep_status ep_dispatch(ep_buffer* buf, const void* x, const float* scores, const int32_t* ids,
                      int64_t T, int64_t N, ep_stream_t stream, ep_dispatch_out* out)
{
    const Range range(buf, "ep_dispatch");
    ep_status st = check_call(buf, ids, T, N);
    if (st != EP_OK) return st;
    if (T > 0 && (!x || !scores)) return EP_ERR_INVALID_ARG;
    if (!is_aligned(x, 16) || !is_aligned(scores, 4)) return EP_ERR_ALIGNMENT;
    if (!debug_fill(buf, pad4(N) * buf->cfg.topk, as_stream(stream))) return EP_ERR_CUDA;
    st = enqueue_dispatch(buf, x, scores, ids, T, N, as_stream(stream));
    if (st != EP_OK) return st;
    if (!debug_check(buf, buf->recv_x, as_stream(stream))) return EP_ERR_CUDA;
    fill_dispatch(buf, out);
    return EP_OK;
}

ep_status ep_dispatch_permute(ep_buffer* buf, const void* x, const float* scores,
                              ep_stream_t stream, ep_dispatch_out* out)
{
    const Range range(buf, "ep_dispatch_permute");
    if (!buf) return EP_ERR_INVALID_ARG;
    if (!buf->has_layout) return EP_ERR_NO_LAYOUT;
    ep_status st = check_rows(buf, x, scores);
    if (st != EP_OK) return st;
    if (!debug_fill(buf, buf->last_S, as_stream(stream))) return EP_ERR_CUDA;
    st = enqueue_permute(buf, x, scores, as_stream(stream));
    if (st != EP_OK) return st;
    if (!debug_check(buf, buf->recv_x, as_stream(stream))) return EP_ERR_CUDA;
    fill_dispatch(buf, out);
    return EP_OK;
}

ep_status ep_combine(ep_buffer* buf, const void* y, const float* scores, int64_t T, void* out,
                     int32_t out_dtype, ep_stream_t stream)
{
    const Range range(buf, "ep_combine");
    if (!buf) return EP_ERR_INVALID_ARG;
    if (!buf->has_layout || T != buf->last_T) return EP_ERR_NO_LAYOUT;
    if (out_dtype != EP_BF16 && out_dtype != EP_F32) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!y || !scores || !out)) return EP_ERR_INVALID_ARG;
    if (!is_aligned(y, 16) || !is_aligned(out, 16) || !is_aligned(scores, 4))
        return EP_ERR_ALIGNMENT;
    ep::CombineArgs a;
    a.y = y;
    a.scores = scores;
    a.pos = buf->pos;
    a.rank_prefix = buf->rank_prefix;
    a.out = out;
    a.T = T;
    a.K = buf->cfg.topk;
    a.R = buf->cfg.num_ranks;
    a.S = buf->last_S;
    a.D = buf->cfg.hidden;
    a.in_dtype = buf->cfg.dtype == EP_BF16 ? 0 : 1;
    a.out_dtype = out_dtype == EP_BF16 ? 0 : 1;
    a.err = buf->err;
    a.packed = buf->cfg.layout_mode == EP_LAYOUT_PACKED;
    a.unit_weights = false;
    a.gather_in = nullptr;
    a.gather_out = nullptr;
    if (y == buf->recv_x && !debug_check(buf, y, as_stream(stream))) return EP_ERR_CUDA;
    if (ep::launch_combine(a, buf->combine_grid, opts(buf, as_stream(stream))) != cudaSuccess)
        return EP_ERR_CUDA;
    return EP_OK;
}

ep_status ep_combine_backward(ep_buffer* buf, const void* grad_out, const void* y,
                              const float* scores, int64_t T, void* grad_y, float* grad_scores,
                              ep_stream_t stream)
{
    const Range range(buf, "ep_combine_backward");
    if (!buf) return EP_ERR_INVALID_ARG;
    if (!buf->has_layout || T != buf->last_T) return EP_ERR_NO_LAYOUT;
    if (T > 0 && (!grad_out || !scores || !grad_y || (grad_scores && !y)))
        return EP_ERR_INVALID_ARG;
    if (!is_aligned(grad_out, 16) || !is_aligned(y, 16) || !is_aligned(grad_y, 16) ||
        !is_aligned(scores, 4) || !is_aligned(grad_scores, 4))
        return EP_ERR_ALIGNMENT;
    ep::CombineBwdArgs a;
    a.grad_out = grad_out;
    a.y = y;
    a.scores = scores;
    a.pos = buf->pos;
    a.rank_prefix = buf->rank_prefix;
    a.grad_y = grad_y;
    a.grad_scores = grad_scores;
    a.T = T;
    a.K = buf->cfg.topk;
    a.R = buf->cfg.num_ranks;
    a.S = buf->last_S;
    a.D = buf->cfg.hidden;
    a.dtype = buf->cfg.dtype == EP_BF16 ? 0 : 1;
    a.err = buf->err;
    a.packed = buf->cfg.layout_mode == EP_LAYOUT_PACKED;
    if (ep::launch_combine_backward(a, buf->combine_grid, opts(buf, as_stream(stream))) !=
        cudaSuccess)
        return EP_ERR_CUDA;
    return EP_OK;
}

ep_status ep_dispatch_backward(ep_buffer* buf, const void* grad_recv_x,
                               const float* grad_recv_scores, int64_t T, void* grad_x,
                               int32_t grad_x_dtype, float* grad_scores, ep_stream_t stream)
{
    const Range range(buf, "ep_dispatch_backward");
    if (!buf) return EP_ERR_INVALID_ARG;
    if (!buf->has_layout || T != buf->last_T) return EP_ERR_NO_LAYOUT;
    if (grad_x_dtype != EP_BF16 && grad_x_dtype != EP_F32) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!grad_recv_x || !grad_x)) return EP_ERR_INVALID_ARG;
    if (!is_aligned(grad_recv_x, 16) || !is_aligned(grad_x, 16) ||
        !is_aligned(grad_recv_scores, 4) || !is_aligned(grad_scores, 4))
        return EP_ERR_ALIGNMENT;
    ep::CombineArgs a;
    a.y = grad_recv_x;
    a.scores = nullptr;
    a.pos = buf->pos;
    a.rank_prefix = buf->rank_prefix;
    a.out = grad_x;
    a.T = T;
    a.K = buf->cfg.topk;
    a.R = buf->cfg.num_ranks;
    a.S = buf->last_S;
    a.D = buf->cfg.hidden;
    a.in_dtype = buf->cfg.dtype == EP_BF16 ? 0 : 1;
    a.out_dtype = grad_x_dtype == EP_BF16 ? 0 : 1;
    a.err = buf->err;
    a.packed = buf->cfg.layout_mode == EP_LAYOUT_PACKED;
    a.unit_weights = true;
    a.gather_in = grad_recv_scores;
    a.gather_out = grad_scores;
    if (ep::launch_combine(a, buf->combine_grid, opts(buf, as_stream(stream))) != cudaSuccess)
        return EP_ERR_CUDA;
    return EP_OK;
}

ep::DedupArgs dedup_args(ep_buffer* b, const void* x, const float* scores, const int32_t* ids,
                         int64_t T, int64_t N)
{
    ep::DedupArgs a;
    a.x = x;
    a.scores = scores;
    a.ids = ids;
    a.T = T;
    a.K = b->cfg.topk;
    a.E = b->cfg.num_experts;
    a.R = b->cfg.num_ranks;
    a.P = pad4(N);
    a.row_bytes = b->row_bytes;
    a.recv_x = b->recv_x;
    a.recv_tok_src = b->tok_src;
    a.recv_topk_idx = b->recv_src;     // the per-expert sources' region holds R*P*K ints
    a.recv_topk_w = b->recv_scores;    // and the scores' region R*P*K floats
    a.tok_pos = b->tok_pos;
    a.err = b->err;
    return a;
}

ep_status ep_dispatch_dedup(ep_buffer* buf, const void* x, const float* scores, const int32_t* ids,
                            int64_t T, int64_t N, ep_stream_t stream, ep_dedup_out* out)
{
    const Range range(buf, "ep_dispatch_dedup");
    ep_status st = check_call(buf, ids, T, N);
    if (st != EP_OK) return st;
    if (T > 0 && (!x || !scores)) return EP_ERR_INVALID_ARG;
    if (!is_aligned(x, 16) || !is_aligned(scores, 4)) return EP_ERR_ALIGNMENT;
    cudaStream_t s = as_stream(stream);
    ep::LayoutArgs la = layout_args(buf, ids, T, N);
    la.tile_tok_pre = buf->tile_tok_pre;
    const ep::LaunchOpts o = opts(buf, s);
    const ep::DedupArgs da = dedup_args(buf, x, scores, ids, T, N);
    // One cooperative kernel where it fits; else count + scan, then the fused
    // kernel (or positions + copies).
    const cudaError_t e0 = (buf->onepass && buf->dedup_fused)
                               ? ep::launch_dedup_onepass(la, da, o, buf->coop_pdl)
                               : cudaErrorNotSupported;
    if (e0 != cudaSuccess && e0 != cudaErrorNotSupported) return EP_ERR_CUDA;
    if (e0 == cudaErrorNotSupported) {
        if (ep::launch_layout_counts(la, o) != cudaSuccess) return EP_ERR_CUDA;
        const cudaError_t e =
            buf->dedup_fused ? ep::launch_dedup_fused(la, da, o) : cudaErrorNotSupported;
        if (e == cudaErrorNotSupported) {
            if (ep::launch_layout_positions(la, o) != cudaSuccess ||
                ep::launch_dedup(la, da, o) != cudaSuccess)
                return EP_ERR_CUDA;
        } else if (e != cudaSuccess) {
            return EP_ERR_CUDA;
        }
    }
    remember_layout(buf, T, N);
    buf->last_dedup = true;
    if (out) {
        out->recv_x = buf->recv_x;
        out->recv_tok_src = buf->tok_src;
        out->recv_topk_idx = buf->recv_src;
        out->recv_topk_w = buf->recv_scores;
        out->tok_pos = buf->tok_pos;
        out->rows_per_rank_stride = pad4(N);
        fill_layout(buf, &out->layout);
    }
    return EP_OK;
}

ep_status ep_dedup_expand(ep_buffer* buf, const int32_t* ids, void* y_recv, ep_stream_t stream)
{
    const Range range(buf, "ep_dedup_expand");
    if (!buf) return EP_ERR_INVALID_ARG;
    if (!buf->has_layout || !buf->last_dedup) return EP_ERR_NO_LAYOUT;
    if (buf->last_T > 0 && (!ids || !y_recv)) return EP_ERR_INVALID_ARG;
    if (!is_aligned(ids, 4) || !is_aligned(y_recv, 16)) return EP_ERR_ALIGNMENT;
    // y_recv must not overlap the workspace that holds the dedupe rows.
    const uint8_t* y0 = static_cast<const uint8_t*>(y_recv);
    const uint8_t* w0 = buf->recv_x;
    const uint8_t* w1 = reinterpret_cast<const uint8_t*>(buf->err) + 4;
    const size_t ybytes = (size_t)buf->cfg.num_ranks * (size_t)buf->last_S * (size_t)buf->row_bytes;
    if (y0 && y0 < w1 && w0 < y0 + ybytes) return EP_ERR_INVALID_ARG;
    const ep::DedupArgs a = dedup_args(buf, nullptr, nullptr, ids, buf->last_T, buf->last_N);
    return ep::launch_dedup_expand(a, buf->pos, y_recv, opts(buf, as_stream(stream))) ==
                   cudaSuccess
               ? EP_OK
               : EP_ERR_CUDA;
}

ep_status ep_expert_gemm(ep_buffer* buf, const void* x_recv, const void* weights, int64_t din,
                         int64_t dout, void* y_recv, ep_stream_t stream)
{
    const Range range(buf, "ep_expert_gemm");
    if (!buf) return EP_ERR_INVALID_ARG;
    if (!buf->has_layout) return EP_ERR_NO_LAYOUT;
    if (buf->cfg.dtype != EP_BF16) return EP_ERR_INVALID_ARG;
    if (din < 64 || din % 64 != 0 || dout < 128 || dout % 128 != 0) return EP_ERR_INVALID_ARG;
    if (!x_recv || !weights || !y_recv) return EP_ERR_INVALID_ARG;
    if (!is_aligned(x_recv, 16) || !is_aligned(weights, 16) || !is_aligned(y_recv, 16))
        return EP_ERR_ALIGNMENT;
    const int64_t rows = (int64_t)buf->cfg.num_ranks * buf->last_S;
    if (rows <= 0) return EP_OK;
    if ((int64_t)buf->cfg.num_experts * dout > INT32_MAX) return EP_ERR_CAPACITY;
    // Row tiles times column blocks (and work units) are counted in int32.
    if ((rows / 128 + buf->cfg.num_experts) * (dout / 128) > INT32_MAX) return EP_ERR_CAPACITY;
    ep::GemmArgs a;
    a.cnt = buf->cnt;
    a.expert_offset = buf->expert_offset;
    a.y = y_recv;
    a.din = din;
    a.dout = dout;
    a.E = buf->cfg.num_experts;
    // 2-SM row tiles cover 256 rows of one expert: worth it when experts hold
    // at least 512 routed rows on average (the last call's T * K / E), else
    // the padding of each expert's last tile costs more than the pair saves.
    a.kind = buf->gemm_kind > 0
                 ? buf->gemm_kind
                 : (buf->last_T * buf->cfg.topk >= (int64_t)512 * buf->cfg.num_experts ? 2 : 1);
    a.bk = buf->gemm_bk;
    a.light_rows = buf->gemm_light_rows;
    a.err = buf->err;
    int kernel = 0, grid = 0;
    const cudaError_t e = ep::launch_expert_gemm(a, x_recv, rows, weights, buf->num_sms,
                                                 opts(buf, as_stream(stream)), &kernel, &grid);
    if (e == cudaSuccess) {
        buf->gemm_kernel = kernel;
        buf->gemm_grid = grid;
    }
    if (e == cudaErrorInvalidValue) return EP_ERR_INVALID_ARG;
    return e == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

ep_status ep_get_device_error(ep_buffer* buf, ep_stream_t stream, uint32_t* flags)
{
    if (!buf || !flags) return EP_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    if (capturing(s)) return EP_ERR_CAPTURE_HOST_SYNC;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, buf->err, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(buf->err, 0, sizeof v, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return EP_ERR_CUDA;
    // A timed-out grid barrier leaves its arrival counts behind: start them over
    // (generation, pool counter and the tiles' ready words with them, so that no
    // ready word of an earlier call can match a generation counted anew).
    if ((v & EP_DEVERR_TIMEOUT) &&
        (cudaMemsetAsync(buf->gbar, 0, 4 * sizeof(uint32_t), s) != cudaSuccess ||
         cudaMemsetAsync(buf->tile_ready, 0, (size_t)buf->max_tiles * 4, s) != cudaSuccess ||
         cudaStreamSynchronize(s) != cudaSuccess))
        return EP_ERR_CUDA;
    *flags = v;
    return EP_OK;
}

ep_status ep_buffer_query(const ep_buffer* buf, ep_buffer_info* info)
{
    if (!buf || !info) return EP_ERR_INVALID_ARG;
    info->workspace_bytes = (int64_t)buf->ws_bytes;
    info->max_rank_stride = buf->s_max;
    info->kernel_launches = buf->launches;
    info->device = buf->device;
    info->num_sms = buf->num_sms;
    info->permute_impl = buf->permute.impl;
    info->permute_grid = buf->permute.grid;
    info->combine_grid = buf->combine_grid;
    info->bulk_stages = buf->permute.stages;
    info->gemm_kernel = buf->gemm_kernel;
    info->gemm_grid = buf->gemm_grid;
    return EP_OK;
}

int64_t ep_pad_tokens(int64_t n) { return n < 0 ? -1 : pad4(n); }

int64_t ep_derive_max_tokens_pretrain(int64_t local_batch_size, int64_t seq_len, int64_t cp,
                                      int64_t tp)
{
    if (local_batch_size <= 0 || seq_len <= 0 || cp <= 0 || tp <= 0) return -1;
    const int64_t shards = cp * tp;
    return local_batch_size * ((seq_len + shards - 1) / shards);
}

int64_t ep_derive_max_tokens_inference(int64_t max_num_batched_tokens, int64_t cp, int64_t tp)
{
    if (max_num_batched_tokens <= 0 || cp <= 0 || tp <= 0) return -1;
    const int64_t shards = cp * tp;
    return (max_num_batched_tokens + shards - 1) / shards;
}

ep_status ep_validate_max_tokens(int64_t configured, int64_t derived)
{
    if (configured <= 0) return EP_ERR_INVALID_ARG;
    if (configured < derived) return EP_ERR_CAPACITY;
    return EP_OK;
}

const char* ep_status_string(ep_status s)
{
    switch (s) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID_ARG: return "invalid argument";
        case EP_ERR_CAPACITY: return "num_tokens_per_rank exceeds num_max_tokens_per_rank";
        case EP_ERR_ALIGNMENT: return "pointer or row size misaligned";
        case EP_ERR_WORKSPACE: return "workspace too small, misaligned or not device memory";
        case EP_ERR_CAPTURE_HOST_SYNC: return "synchronous call on a capturing stream";
        case EP_ERR_CUDA: return "CUDA runtime error";
        case EP_ERR_NO_LAYOUT: return "no layout for this call on the buffer";
        case EP_ERR_HOST_ALLOC: return "host-side buffer handle could not be allocated";
    }
    return "unknown status";
}

}  // extern "C"
