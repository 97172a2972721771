/*
 * ep.h - C ABI of the GB300 MoE token dispatch / combine library (libep_gb300.so).
 *
 * One process drives one GPU. "Ranks" are R logical partitions of this GPU's
 * receive buffer: experts are split into R contiguous blocks of E/R experts,
 * and rank r owns receive rows [r*S, (r+1)*S) (the default strided layout;
 * EP_LAYOUT_PACKED puts the ranks' rows back to back). Everything here follows the
 * token-dispatcher pages:
 *   [titan] "Unify expert parallel token dispatcher API" (pytorch/torchtitan
 *           pull 3970): sections "API design", "Backend behavior",
 *           "Capacity derivation".
 *   [align] "fix(moe): equalize and align per-rank token counts for HybridEP
 *           dispatch" (NVIDIA-NeMo/Automodel pull 3641): "Problem", "Fix".
 *   [graph] "ep: graph-safe worst-token HT dispatch+combine (internode +
 *           intranode)" (uccl pull 18): "Internode" items 1-3, "Intranode".
 *   [flex]  "Inference: enable flex dispatcher (DeepEP/HybridEP) for prefill"
 *           (Megatron-LM pull 4321): the SM budget knob.
 *
 * Notation: T = materialised tokens (rows of x_TD), N = num_tokens_per_rank
 * (T <= N <= N_max), P = N rounded up to a multiple of 4, K = top-k,
 * E = experts, R = logical ranks, D = hidden size, S = P*K receive rows per
 * rank for the current call.
 *
 * Conventions for every call:
 *  - Pointers named *_TD, *_TK, y_recv, out_TD are DEVICE pointers owned by
 *    the caller; they must stay valid until the stream work completes.
 *    Hidden-row pointers (x_TD, y_recv, out_TD) must be 16-byte aligned;
 *    ids and scores 4-byte aligned. Row-major, densely packed.
 *  - topk_expert_ids_TK is int32 [T][K]; -1 means "no expert". Any other id
 *    outside [0, E) is treated as -1 and raises EP_DEVERR_BAD_ID.
 *    topk_scores_TK is fp32 [T][K]. x_TD is [T][D] of the configured dtype.
 *  - Calls are stream-ordered and asynchronous; none allocates memory, none
 *    reads device memory on the host (except the calls documented as
 *    synchronous, which refuse to run while the stream is capturing), and
 *    none writes host-mapped memory from a kernel. Every dispatch/combine
 *    sequence can therefore be captured in a CUDA graph and replayed with new
 *    routing written into the same input buffers ([graph] "Internode" item 1,
 *    "Intranode").
 *  - A host-side argument error returns a status and enqueues nothing.
 *    Data errors found on the device (bad ids, rows outside a rank's true
 *    total) set sticky bits in the buffer's device error word; kernels never
 *    trap and never write out of bounds. Read them with ep_get_device_error.
 *  - Outputs that live in the workspace (layout arrays, receive buffers) are
 *    overwritten by the next call on the same buffer. A buffer is not
 *    thread-safe; use one buffer per concurrent stream of calls.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EP_API __attribute__((visibility("default")))
#else
#define EP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t passed as an opaque pointer (NULL = the legacy default stream). */
typedef void* ep_stream_t;

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,       /* bad shape, null pointer, bad enum */
    EP_ERR_CAPACITY = 2,          /* num_tokens_per_rank > num_max_tokens_per_rank, or sizes overflow */
    EP_ERR_ALIGNMENT = 3,         /* pointer or row size not aligned as documented */
    EP_ERR_WORKSPACE = 4,         /* workspace too small, misaligned or not device memory */
    EP_ERR_CAPTURE_HOST_SYNC = 5, /* a synchronous call was made on a capturing stream */
    EP_ERR_CUDA = 6,              /* a CUDA runtime call or launch failed */
    EP_ERR_NO_LAYOUT = 7,         /* combine/permute before any layout on this buffer, or T differs */
    EP_ERR_HOST_ALLOC = 8         /* the host-side buffer handle could not be allocated */
} ep_status;

typedef enum { EP_BF16 = 0, EP_F32 = 1 } ep_dtype;

typedef enum {
    EP_PERMUTE_DEFAULT = 0,       /* the library's choice */
    EP_PERMUTE_VEC = 1,           /* 16-byte vector loads/stores through registers */
    EP_PERMUTE_BULK = 2           /* bulk async copies staged through shared memory */
} ep_permute_impl;

typedef enum {
    EP_LAYOUT_STRIDED = 0,        /* worst-token mode: rank r's rows start at r*S */
    EP_LAYOUT_PACKED = 1          /* exact mode: ranks back to back, rows [0, true total) */
} ep_layout_mode;

/* Device error word bits (sticky until ep_get_device_error clears them). */
#define EP_DEVERR_BAD_ID 0x1u     /* an id outside [-1, E) was seen; treated as -1 */
#define EP_DEVERR_ROW_OOB 0x2u    /* combine met a row outside its rank's true total, or the
                                     one-pass dispatch computed a row outside the call's R*S
                                     rows (only after its barrier words were corrupted);
                                     skipped */
#define EP_DEVERR_TIMEOUT 0x4u    /* a bounded device-side wait gave up; outputs invalid */
/* Only with EP_DEBUG=1 (read at ep_buffer_init): the dispatch fills its receive
 * rows with 0xFF before the permute and checks them after it; the combine
 * repeats the check when it reads the receive buffer itself. */
#define EP_DEVERR_DEBUG_UNWRITTEN 0x8u  /* a row inside a rank's true total kept the 0xFF fill */
#define EP_DEVERR_DEBUG_STRAY 0x10u     /* a row past a rank's true total was written */

/* Lifetime configuration ([titan] "API design": the dispatcher configuration
 * carries the lifetime maximum num_max_tokens_per_rank; persistent storage is
 * sized from it once and never grows inside dispatch). */
typedef struct {
    int64_t num_max_tokens_per_rank; /* N_max >= 1 */
    int64_t hidden;                  /* D >= 1; D * element size must be a multiple of 16 */
    int32_t num_experts;             /* E, 1 <= E <= 1024, E % R == 0 */
    int32_t num_ranks;               /* R, 1 <= R <= 64 logical ranks */
    int32_t topk;                    /* K, 1 <= K <= min(E, 64) */
    int32_t dtype;                   /* ep_dtype of x_TD and the receive buffer */
    int32_t num_sms;                 /* SMs the copy kernels may use; 0 = the environment
                                        variable EP_NUM_SMS if set, else all ([flex]) */
    int32_t permute_impl;            /* ep_permute_impl */
    int32_t layout_mode;             /* ep_layout_mode: where each rank's rows start.
                                        STRIDED ([titan] "Backend behavior": the current
                                        capacity is the per-rank stride; [graph] worst-token
                                        mode): rank r owns rows [r*S, r*S + rows_per_rank[r]).
                                        PACKED ([graph] num_worst_tokens == 0, receive sized
                                        by the true counts): rank r owns rows
                                        [rank_prefix[r-1], rank_prefix[r]), expert e starts
                                        after all lower experts, the valid rows are exactly
                                        [0, rank_prefix[R-1]); read the counts with exact
                                        mode (host_tokens_per_expert) to size consumers. */
} ep_config;

/* Opaque handle; the library owns this host-side object, the caller owns the workspace. */
typedef struct ep_buffer ep_buffer;

/* Layout of one call. All pointers are device pointers into the workspace. */
typedef struct {
    int32_t* tokens_per_expert; /* [E] pairs routed to each expert: [titan] "API design"
                                   num_local_tokens_per_expert_E; [graph] "Internode" item 2 */
    int32_t* expert_offset;     /* [E] first receive row of expert e: r(e)*S + counts of the
                                   lower experts of the same rank */
    int32_t* rows_per_rank;     /* [R] receive rows used by rank r (its true total) */
    int32_t* rank_prefix;       /* [R] inclusive prefix of rows_per_rank; the last entry is the
                                   true received total ([graph] "Internode" item 3) */
    int32_t* tokens_in_rank;    /* [R] distinct tokens with at least one expert on rank r */
    int32_t* pos;               /* [T][K] receive row of pair (t,k), or -1; rows of one expert
                                   follow ascending t*K+k */
    int64_t num_tokens;         /* T */
    int64_t padded_tokens;      /* P = roundup4(N) ([align] "Problem" item 2, "Fix") */
    int64_t rank_stride;        /* S = P*K rows reserved per rank ([titan] "Backend behavior");
                                   the strided layout's per-rank stride */
    int32_t packed;             /* 1 if rows are placed by EP_LAYOUT_PACKED */
} ep_layout;

/* Result of a dispatch: views into the workspace. recv_x is [R*S][D] of the
 * configured dtype (rank r's rows start at r*S), recv_scores fp32 [R*S] and
 * recv_src int32 [R*S] (source pair index t*K+k). Only rows
 * [r*S, r*S + rows_per_rank[r]) of each rank are defined; the tail of each
 * rank's block holds stale data from earlier calls and must not be read. */
typedef struct {
    void* recv_x;
    float* recv_scores;
    int32_t* recv_src;
    ep_layout layout;
} ep_dispatch_out;

/* Result of a per-rank dedupe dispatch: views into the workspace. Rank r owns
 * rows [r*rows_per_rank_stride, r*rows_per_rank_stride + tokens_in_rank[r]) of
 * recv_x ([R*P][D], configured dtype), in ascending token order, one row per
 * distinct (token, rank). recv_tok_src [R*P] is the row's token, recv_topk_idx
 * [R*P][K] its local expert index on that rank per k (or -1), recv_topk_w
 * [R*P][K] the score of those pairs (or 0). tok_pos [T][R] is the row of
 * (t, r) or -1. layout is the same call's per-expert layout. The dedupe rows
 * share the per-expert receive rows' storage: a later dispatch overwrites them. */
typedef struct {
    void* recv_x;
    int32_t* recv_tok_src;
    int32_t* recv_topk_idx;
    float* recv_topk_w;
    int32_t* tok_pos;
    int64_t rows_per_rank_stride;   /* P = roundup4(N) */
    ep_layout layout;
} ep_dedup_out;

/* Read-only facts about a buffer (for tuning and for counting launches). */
typedef struct {
    int64_t workspace_bytes;    /* bytes the buffer uses from the workspace */
    int64_t max_rank_stride;    /* S_max = roundup4(N_max) * K */
    int64_t kernel_launches;    /* kernels this buffer has launched so far */
    int32_t device;             /* CUDA device the buffer was created on */
    int32_t num_sms;            /* SMs the copy kernels use */
    int32_t permute_impl;       /* resolved ep_permute_impl */
    int32_t permute_grid;       /* CTAs of the permute kernel */
    int32_t combine_grid;       /* CTAs of the combine kernel */
    int32_t bulk_stages;        /* shared-memory row slots per CTA of the bulk permute */
    int32_t gemm_kernel;        /* last ep_expert_gemm launch: 0 none, 1 single-CTA
                                   128-row tiles, 2 two-SM 256-row tiles (CTA pairs) */
    int32_t gemm_grid;          /* CTAs of that launch */
} ep_buffer_info;

/* Bytes of device workspace ep_buffer_init needs for this configuration, or 0
 * if the configuration is invalid. Host-only; never touches the GPU.
 * Sized once from N_max ([titan] "API design"; "Backend behavior": persistent
 * buffers are preallocated): receive rows R * roundup4(N_max) * K of D
 * elements, their scores and sources, the [N_max][K] positions and the
 * layout arrays. */
EP_API size_t ep_buffer_required_bytes(const ep_config* cfg);

/* Create a buffer over caller-owned device workspace ([titan] "API design": the
 * lifetime maximum num_max_tokens_per_rank sizes persistent storage once;
 * "Backend behavior": DeepEP and HybridEP preallocate). workspace must be
 * device memory on the current device, 256-byte aligned, at least
 * ep_buffer_required_bytes(cfg) bytes, and must outlive the buffer. The
 * current device at this call is the buffer's device. Synchronous (clears
 * the device error word). Returns EP_ERR_INVALID_ARG for a bad cfg,
 * EP_ERR_WORKSPACE for an unusable workspace, EP_ERR_CUDA if no device,
 * EP_ERR_HOST_ALLOC if the host-side handle cannot be allocated. */
EP_API ep_status ep_buffer_init(const ep_config* cfg, void* workspace, size_t workspace_bytes,
                         ep_buffer** out);

/* Release the host-side handle. Does not free the workspace. NULL is a no-op.
 * (Plumbing: no page passage defines it.) */
EP_API ep_status ep_buffer_destroy(ep_buffer* buf);

/* Dispatch layout ([titan] "API design"; [graph] "Internode" items 2-3):
 * per-expert counts, per-rank totals, their inclusive prefix, distinct
 * tokens per rank, expert offsets and the receive row of every (t, k) pair,
 * computed on the device from topk_expert_ids_TK [T][K]. num_tokens = T,
 * num_tokens_per_rank = N (0 <= T <= N <= N_max); rows T..P-1 are padding
 * that routes to no expert ([align] "Fix"). Fills *out (may be NULL).
 * host_tokens_per_expert: NULL for worst-token mode (counts stay on the
 * device, fully asynchronous); non-NULL for exact mode ([graph] "Internode"
 * item 1, num_worst_tokens == 0): the E counts are copied to this host array
 * and the call synchronizes the stream; refused with EP_ERR_CAPTURE_HOST_SYNC
 * while the stream is capturing. */
EP_API ep_status ep_dispatch_layout(ep_buffer* buf, const int32_t* topk_expert_ids_TK, int64_t num_tokens,
                             int64_t num_tokens_per_rank, ep_stream_t stream, ep_layout* out,
                             int32_t* host_tokens_per_expert);

/* Dispatch = layout + permute ([titan] "API design" dispatch(x_TD,
 * topk_scores_TK, topk_expert_ids_TK, ..., num_tokens_per_rank);
 * "Backend behavior": the current capacity sets the per-rank stride of the
 * preallocated buffer and sizes the permute output). For every pair with a
 * row p: recv_x[p] = x_TD[t], recv_scores[p] = topk_scores_TK[t][k],
 * recv_src[p] = t*K + k. Fills *out (may be NULL). */
EP_API ep_status ep_dispatch(ep_buffer* buf, const void* x_TD, const float* topk_scores_TK,
                      const int32_t* topk_expert_ids_TK, int64_t num_tokens,
                      int64_t num_tokens_per_rank, ep_stream_t stream, ep_dispatch_out* out);

/* The permute half of ep_dispatch alone ([titan] "Backend behavior": rows go to
 * the receive buffer with the current capacity as the per-rank stride), using
 * the layout of the last
 * ep_dispatch_layout / ep_dispatch on this buffer (same T; x_TD and
 * topk_scores_TK have that T). EP_ERR_NO_LAYOUT if there is none. */
EP_API ep_status ep_dispatch_permute(ep_buffer* buf, const void* x_TD, const float* topk_scores_TK,
                              ep_stream_t stream, ep_dispatch_out* out);

/* Combine ([align] "Fix": combine() slices the padded rows back off;
 * [graph] "Internode" item 3: the true total comes from the device prefix
 * sum). Uses the layout of the last dispatch on this buffer; num_tokens must
 * equal its T. y_recv is the expert output in the receive layout
 * ([R*S][D], configured dtype; may alias recv_x). For t < T:
 *   out_TD[t][d] = round( fma-chain over k = 0..K-1 with pos >= 0 of
 *                         topk_scores_TK[t][k] * y_recv[pos[t][k]][d] )
 * accumulated in fp32 from +0 in ascending k with one fused multiply-add
 * per term, no atomics, then rounded to out_dtype (bf16: round to nearest
 * even; fp32: unchanged). A token with no expert gets a +0 row. Rows of
 * y_recv beyond a rank's true total are never read (EP_DEVERR_ROW_OOB).
 * out_TD is [T][D] of out_dtype. */
EP_API ep_status ep_combine(ep_buffer* buf, const void* y_recv, const float* topk_scores_TK,
                     int64_t num_tokens, void* out_TD, int32_t out_dtype, ep_stream_t stream);

/* Backward of ep_combine, for training ([align] "Testing": the unequal-count
 * run must reproduce the equal-count run bit for bit in the forward AND the
 * backward pass; the page does not spell the backward out, it is the
 * derivative of the combine). Uses the layout of the last dispatch on this
 * buffer; num_tokens must equal its T. grad_out_TD is [T][D] and y_recv,
 * grad_y_recv are [R*S][D], all of the configured dtype. For every valid pair:
 *   grad_y_recv[pos[t][k]][d] = topk_scores_TK[t][k] * grad_out_TD[t][d]
 *   (one fp32 product, rounded to the dtype; rows no pair references are not
 *   written), and, when grad_scores_TK (fp32 [T][K]) is non-NULL,
 *   grad_scores_TK[t][k] = sum_d grad_out_TD[t][d] * y_recv[pos[t][k]][d]
 *   (fp32 per-thread FMA chains reduced in a fixed order: deterministic; 0 for
 *   a pair without a valid row). y_recv is read only for grad_scores_TK. */
EP_API ep_status ep_combine_backward(ep_buffer* buf, const void* grad_out_TD, const void* y_recv,
                                     const float* topk_scores_TK, int64_t num_tokens,
                                     void* grad_y_recv, float* grad_scores_TK, ep_stream_t stream);

/* Backward of ep_dispatch, its adjoint ([align] "Testing": forward and backward
 * of unequal-count runs reproduce the equal-count run bitwise). grad_recv_x is
 * [R*S][D] of the configured dtype; grad_x_TD [T][D] of grad_x_dtype:
 *   grad_x_TD[t][d] = sum over valid k (ascending, fp32 from +0) of
 *                     grad_recv_x[pos[t][k]][d], rounded to grad_x_dtype;
 * and, when grad_scores_TK is non-NULL, grad_scores_TK[t][k] =
 * grad_recv_scores[pos[t][k]] (0 without a valid row or without
 * grad_recv_scores): the scores' gradient through recv_scores. */
EP_API ep_status ep_dispatch_backward(ep_buffer* buf, const void* grad_recv_x,
                                      const float* grad_recv_scores, int64_t num_tokens,
                                      void* grad_x_TD, int32_t grad_x_dtype,
                                      float* grad_scores_TK, ep_stream_t stream);

/* Per-rank dedupe dispatch: each token is sent to each destination rank
 * once, however many of that rank's experts it selected ([titan] "Backend
 * behavior": DeepEP's per-rank layout stride; [graph] "Internode": per-rank
 * token counts on the device), then expanded to experts at the receiver
 * (ep_dedup_expand). Arguments as ep_dispatch; results in *out (see
 * ep_dedup_out). Also computes the per-expert layout (counts, offsets,
 * positions) of the call. On DeepSeek-style routing it writes about 40% of
 * the rows ep_dispatch writes. */
EP_API ep_status ep_dispatch_dedup(ep_buffer* buf, const void* x_TD, const float* topk_scores_TK,
                                   const int32_t* topk_expert_ids_TK, int64_t num_tokens,
                                   int64_t num_tokens_per_rank, ep_stream_t stream,
                                   ep_dedup_out* out);

/* The receiver's expansion of the last ep_dispatch_dedup on this buffer into
 * the per-expert layout ([titan] "Backend behavior": DeepEP's per-rank layout,
 * each token sent once per rank and spread over that rank's experts there): y_recv[pos[t][k]] = dedupe row of (t, rank of
 * topk_expert_ids_TK[t][k]) for every routed pair; y_recv is [R*S][D] of the
 * configured dtype, caller-owned, outside the workspace, and then feeds
 * ep_combine like recv_x. topk_expert_ids_TK must be the dedupe call's ids
 * (a pair whose rank row is missing raises EP_DEVERR_ROW_OOB and is skipped).
 * EP_ERR_NO_LAYOUT unless the buffer's last dispatch was ep_dispatch_dedup. */
EP_API ep_status ep_dedup_expand(ep_buffer* buf, const int32_t* topk_expert_ids_TK, void* y_recv,
                                 ep_stream_t stream);

/* The expert consumer between dispatch and combine: a grouped GEMM driven by
 * the per-expert counts and offsets that the last layout on this buffer left
 * on the device ([graph] "Internode" item 2: counts stay on the device so
 * consumers never touch the host; "Tests": layout -> dispatch -> expert ->
 * combine). For every expert e and each of its rows p = expert_offset[e] + j,
 * j < tokens_per_expert[e]:
 *     y_recv[p][o] = sum_i x_recv[p][i] * weights[e][o][i]
 * with bf16 inputs, fp32 accumulation on the tensor cores (tcgen05) and one
 * round to bf16. x_recv is [R*S][din] and y_recv [R*S][dout] in the receive
 * layout (strided or packed; x_recv may be recv_x with din = D), weights is
 * [E][dout][din]; all bf16 device memory, 16-byte aligned. din % 64 == 0,
 * dout % 128 == 0; bf16 buffers only (EP_ERR_INVALID_ARG otherwise). Rows of
 * y_recv that belong to no expert are not written. Summation order inside the
 * tensor cores is the hardware's: results are within the fp32 summation bound
 * of the exact product, not bitwise fixed across GPU models. Tiles: 256 rows
 * on an SM pair (tcgen05 cta_group::2; an expert's last 128 rows or fewer as
 * one 128-row pair tile) when dout % 256 == 0 and the last call routed at
 * least 512 rows per expert on average (T * K >= 512 * E), else 128 rows per
 * SM; all issue the same K order, so they agree bit for bit.
 * The environment variable EP_GEMM_KERNEL=1 (128-row) or 2 (256-row), read at
 * ep_buffer_init, forces one of them. Schedule: the tiles of experts with at
 * most 256 rows (memory-bound: their weights serve one or two tiles) are
 * interleaved in proportion with the others' (tensor-bound: weights reused
 * from L2), so skewed routing keeps both HBM and the tensor cores busy;
 * EP_GEMM_LIGHT_ROWS=n sets the threshold (0: all tiles in expert order).
 * The schedule changes which SM computes a tile, never its K order. */
EP_API ep_status ep_expert_gemm(ep_buffer* buf, const void* x_recv, const void* weights,
                                int64_t din, int64_t dout, void* y_recv, ep_stream_t stream);

/* Synchronously read and clear the device error word (EP_DEVERR_* bits).
 * Refused with EP_ERR_CAPTURE_HOST_SYNC while the stream is capturing. Status
 * stays on the device and is read only here ([graph] "Internode" item 1: no
 * host handshake on the dispatch path). */
EP_API ep_status ep_get_device_error(ep_buffer* buf, ep_stream_t stream, uint32_t* flags);

/* Read-only facts about buf. (Plumbing: no page passage defines it.) */
EP_API ep_status ep_buffer_query(const ep_buffer* buf, ep_buffer_info* info);

/* The dispatch layout of ep_dispatch_layout, for callers that cannot allocate
 * device memory or keep a workspace (for example an op inside a host framework
 * that owns every device allocation and only hands it input and output
 * tensors). The layout is ep_dispatch_layout's ([titan] "API design";
 * [graph] "Internode" item 2: counts stay on the device); the pages have no
 * variant without a workspace: it exists for such callers.
 * No buffer is involved and nothing is allocated: the caller passes
 * topk_expert_ids_TK [T][K] and the outputs (device pointers, 4-byte aligned):
 * tokens_per_expert [E], expert_offset [E], rows_per_rank [R], rank_prefix [R],
 * tokens_in_rank [R] and pos [T][K], with the same meaning and values as the
 * ep_layout fields; error_flags (nullable) is a device word the kernels OR
 * EP_DEVERR_BAD_ID into (the caller zeroes it). The kernels' other global
 * memory is a library-owned 4 MiB device array per GPU, held until the
 * process exits; a call whose tile tables need more,
 *   ceil(T / max(1, 2048/K)) * (2*roundup4(E) + R) * 4 bytes (plus alignment),
 * is rejected with EP_ERR_CAPACITY (about 516k tokens at E=256, R=8, K=8;
 * about 126k at E=1024, R=64, K=8; ep_dispatch_layout_noalloc_scratch_bytes
 * gives the exact figure). The first call on each device (with that device
 * current) looks up the array's device address; make it before any stream
 * capture. The address is kept per device and context: after a
 * cudaDeviceReset, or in another context of the device, the next call looks
 * it up again (so that call, too, must come before any capture). All calls
 * share the array, so calls whose GPU work overlaps (other streams or
 * threads) race: serialize them. Asynchronous on stream. */
EP_API ep_status ep_dispatch_layout_noalloc(const int32_t* topk_expert_ids_TK, int64_t num_tokens,
                                            int64_t num_tokens_per_rank, int32_t topk,
                                            int32_t num_experts, int32_t num_ranks,
                                            int32_t* tokens_per_expert, int32_t* expert_offset,
                                            int32_t* rows_per_rank, int32_t* rank_prefix,
                                            int32_t* tokens_in_rank, int32_t* pos,
                                            uint32_t* error_flags, ep_stream_t stream);

/* Size of the fixed device array behind ep_dispatch_layout_noalloc (per GPU). */
#define EP_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/* Bytes of that array a call of ep_dispatch_layout_noalloc with these sizes
 * needs; the call is accepted when this is at most EP_NOALLOC_SCRATCH_BYTES.
 * Host-only arithmetic: no device is touched. 0 for a non-positive topk,
 * num_experts or num_ranks, or a negative num_tokens. (Plumbing: no page
 * passage defines it.) */
EP_API size_t ep_dispatch_layout_noalloc_scratch_bytes(int64_t num_tokens, int32_t topk,
                                                       int32_t num_experts, int32_t num_ranks);

/* roundup4(n): the padded per-rank token count ([align] "Problem" item 2, "Fix"). */
EP_API int64_t ep_pad_tokens(int64_t n);

/* [titan] "Capacity derivation", Pretraining: local_batch_size *
 * ceil_div(seq_len, cp * tp). Returns -1 if any argument is not positive. */
EP_API int64_t ep_derive_max_tokens_pretrain(int64_t local_batch_size, int64_t seq_len, int64_t cp,
                                      int64_t tp);

/* [titan] "Capacity derivation", vLLM inference: ceil_div(max_num_batched_tokens,
 * cp * tp). Returns -1 if any argument is not positive. */
EP_API int64_t ep_derive_max_tokens_inference(int64_t max_num_batched_tokens, int64_t cp, int64_t tp);

/* [titan] "Capacity derivation": an explicitly configured num_max_tokens_per_rank
 * must be positive and at least the derived requirement. Returns EP_OK,
 * EP_ERR_INVALID_ARG (not positive) or EP_ERR_CAPACITY (too small). */
EP_API ep_status ep_validate_max_tokens(int64_t configured, int64_t derived);

/* Access patterns of the hot path, for ep_pattern_probe. */
typedef enum {
    EP_PATTERN_READ = 0,     /* dst[r] (16 bytes) = XOR of the words of src row r */
    EP_PATTERN_WRITE = 1,    /* dst row r filled (src unused) */
    EP_PATTERN_COPY = 2,     /* dst row r = src row r */
    EP_PATTERN_FANOUT = 3,   /* dst row j*rows + r = src row r, j < fan (the dispatch's shape) */
    EP_PATTERN_GATHER = 4    /* dst row r = XOR of src rows j*rows + r, j < fan (the combine's) */
} ep_pattern;

/* Measurement aid (plumbing: no page passage defines it). Moves `rows` rows of
 * row_bytes (a multiple of 16) in one of the shapes above, with the combine's
 * kernel structure (a 128-thread CTA per row, 16-byte vectors, as many CTAs
 * per SM as fit) and nothing else in the kernel, so that a benchmark can time
 * the HBM ceiling of the dispatch's 1:fan fan-out and the combine's fan:1
 * gather on this GPU. src and dst are device pointers, 16-byte aligned, sized
 * for the pattern (FANOUT: dst holds fan*rows rows; GATHER: src holds
 * fan*rows rows; READ: dst holds rows 16-byte words); 1 <= fan <= 64.
 * Asynchronous on stream; EP_ERR_INVALID_ARG / EP_ERR_ALIGNMENT on bad
 * arguments, with nothing enqueued. */
EP_API ep_status ep_pattern_probe(int32_t pattern, const void* src, void* dst, int64_t rows,
                                  int64_t row_bytes, int32_t fan, ep_stream_t stream);

/* Static description of a status code. (Plumbing: no page passage defines it.) */
EP_API const char* ep_status_string(ep_status s);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
