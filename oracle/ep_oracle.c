/*
 * ep_oracle.c - CPU oracle for MoE expert-parallel token dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY. This is the correctness reference the CUDA library
 * is checked against. Only the tests, the smoke check and the benchmark's CPU
 * baseline load it. The product path never calls it, and it shares no code,
 * header, table or constant with the CUDA library.
 *
 * Plain, single-threaded, unoptimised C (compiled with -ffp-contract=off).
 * Each function names the passage it follows. Pages, by title:
 *   [titan] "Unify expert parallel token dispatcher API" (pytorch/torchtitan
 *           pull 3970): "API design", "Backend behavior", "Capacity derivation".
 *   [align] "fix(moe): equalize and align per-rank token counts for HybridEP
 *           dispatch" (NVIDIA-NeMo/Automodel pull 3641): "Problem", "Fix",
 *           "Testing".
 *   [graph] "ep: graph-safe worst-token HT dispatch+combine (internode +
 *           intranode)" (uccl pull 18): "Internode" items 2 and 3, "Tests".
 *
 * Where the pages leave a step open, the reading taken is stated at the step.
 * Every function here is pinned by the CPU tests (worked values printed on the
 * pages, closed forms, library-routine cross-checks, brute force on tiny
 * inputs, hand-worked IEEE-754 encodings, NaN results included).
 *
 * NaN results. The pages say nothing about NaNs. IEEE 754-2008 section 6.2
 * asks an arithmetic operation with a NaN result for a quiet NaN but leaves
 * its payload to a recommendation (6.2.3), says nothing about which of
 * several NaN operands propagates, and gives a NaN's sign no meaning (6.3);
 * hosts differ (the default NaN is ffc00000 on x86, 7fc00000 on Arm). So a
 * NaN produced by the arithmetic here (combine's fma chain, the backward's
 * products and sums) is delivered as THE canonical quiet NaN, 7fc00000 (bf16
 * 7fc0), and only a format conversion of a given NaN keeps its sign and
 * leading payload bits (6.2.3). Copies (dispatch, dedupe) keep every bit.
 *
 * Conventions: ids are int32, -1 means "no expert"; scores are fp32; hidden
 * rows are either fp32 or bf16 stored as uint16 bit patterns. Return value 0 =
 * success, 1 = invalid argument, 2 = out of memory (host scratch), 3 = a
 * computed receive row outside the receive buffer (refused, never written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ENOMEM 2
#define ORC_EBOUNDS 3   /* a computed receive row outside the receive buffer */

/* Element kinds of hidden rows, as the Python wrapper passes them. */
#define ORC_BF16 0
#define ORC_F32 1

/* Sticky data-error bits reported by layout and combine. */
#define ORC_ERR_BAD_ID 1u   /* an id outside [-1, E): treated as -1 */
#define ORC_ERR_ROW_OOB 2u  /* a combine row outside its rank's received range */

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0     /* tests build deliberately broken copies (1..N) */
#endif

/* ------------------------------------------------------------------------ */
/* Padding and capacity                                                       */
/* ------------------------------------------------------------------------ */

/* ceil(a / b) for a >= 0, b > 0. [titan] "Capacity derivation" uses
 * ceil_div so that a sequence length not divisible by the sharding degree
 * is never under-allocated. */
int64_t oracle_ceil_div(int64_t a, int64_t b)
{
#if ORACLE_MUTANT == 10
    return a / b;                                   /* mutant: floor division */
#else
    return (a + b - 1) / b;
#endif
}

/* Padded per-rank token count: the per-call count rounded up to a multiple
 * of 4. [align] "Problem" item 2 (the count must be a multiple of 4 because
 * the metadata allgather wants bytes_per_rank % 16 == 0 on a 4-byte-per-token
 * array) and "Fix" (round the group max up to the 4-token alignment). */
int64_t oracle_pad_tokens(int64_t n)
{
#if ORACLE_MUTANT == 9
    return oracle_ceil_div(n, 8) * 8;               /* mutant: wrong alignment */
#else
    return oracle_ceil_div(n, 4) * 4;
#endif
}

/* [titan] "Capacity derivation" / "Pretraining":
 *   num_token_shards = context_parallel_degree * tensor_parallel_degree
 *   num_max_tokens_per_rank = local_batch_size * ceil_div(seq_len, num_token_shards)
 * Returns -1 on a non-positive argument. */
int64_t oracle_num_max_tokens_pretrain(int64_t local_batch_size, int64_t seq_len,
                                       int64_t cp, int64_t tp)
{
    if (local_batch_size <= 0 || seq_len <= 0 || cp <= 0 || tp <= 0) return -1;
    int64_t num_token_shards = cp * tp;
    return local_batch_size * oracle_ceil_div(seq_len, num_token_shards);
}

/* [titan] "Capacity derivation" / "vLLM inference":
 *   num_max_tokens_per_rank = ceil_div(max_num_batched_tokens, cp * tp)
 * Returns -1 on a non-positive argument. */
int64_t oracle_num_max_tokens_inference(int64_t max_num_batched_tokens, int64_t cp, int64_t tp)
{
    if (max_num_batched_tokens <= 0 || cp <= 0 || tp <= 0) return -1;
    return oracle_ceil_div(max_num_batched_tokens, cp * tp);
}

/* Rows reserved per logical rank for the current call: every (token, k)
 * pair of every padded token could land on one rank, so S = P * K with
 * P = oracle_pad_tokens(N). [titan] "Backend behavior" (DeepEP: the current
 * capacity, not the lifetime maximum, is the per-rank layout stride). */
int64_t oracle_rank_stride(int64_t num_tokens_per_rank, int64_t K)
{
#if ORACLE_MUTANT == 5
    return num_tokens_per_rank * K;                 /* mutant: stride ignores padding */
#else
    return oracle_pad_tokens(num_tokens_per_rank) * K;
#endif
}

/* ------------------------------------------------------------------------ */
/* Argument checks ([titan] "API design": x_TD.shape[0] <= num_tokens_per_rank;
 * experts are split into R equal contiguous blocks, one per logical rank).     */
/* ------------------------------------------------------------------------ */

static int check_shape(int64_t T, int64_t N, int32_t K, int32_t E, int32_t R)
{
    if (T < 0 || N < T) return ORC_EINVAL;
    if (E <= 0 || R <= 0 || E % R != 0) return ORC_EINVAL;
    if (K <= 0 || K > E) return ORC_EINVAL;
    return ORC_OK;
}

/* Logical rank owning expert e: contiguous blocks of E/R experts (the pages
 * are silent on the map; contiguous blocks is the plainest reading). */
static int32_t rank_of(int32_t e, int32_t E, int32_t R)
{
#if ORACLE_MUTANT == 4
    (void)E;
    return e % R;                                   /* mutant: strided map */
#else
    return e / (E / R);
#endif
}

/* Padded view of the router output: rows t < T keep their ids (an id
 * outside [-1, E) becomes -1 and raises ORC_ERR_BAD_ID); rows T <= t < P get
 * -1 everywhere. [align] "Fix": padded rows route to no expert. */
static int32_t* padded_ids(const int32_t* ids, int64_t T, int64_t P, int32_t K, int32_t E,
                           uint32_t* err)
{
    int32_t* p = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1) * (size_t)K);
    if (!p) return NULL;
    for (int64_t t = 0; t < P; ++t) {
        for (int32_t k = 0; k < K; ++k) {
            int32_t v = -1;
#if ORACLE_MUTANT == 11
            if (t < P) {                            /* mutant: padded rows read garbage ids */
                v = (t < T) ? ids[t * K + k] : (int32_t)((t * K + k) % E);
#else
            if (t < T) {
                v = ids[t * K + k];
#endif
                if (v < -1 || v >= E) {
                    *err |= ORC_ERR_BAD_ID;
                    v = -1;
                }
            }
            p[t * K + k] = v;
        }
    }
    return p;
}

/* Dense routing map and probabilities of the padded token block, as the
 * aligned dispatcher builds them. [align] "Fix": hidden states, routing map
 * and probabilities are padded to P rows; padded rows are all-False with zero
 * probability. map_PE is P x E bytes (1 = routed), probs_PE is P x E fp32
 * (the top-k score at the chosen experts, 0 elsewhere). A duplicated id in a
 * token sets its map entry once and keeps the last score written. */
int oracle_routing_map(const int32_t* ids, const float* scores, int64_t T, int64_t N,
                       int32_t K, int32_t E, uint8_t* map_PE, float* probs_PE, uint32_t* err)
{
    if (T < 0 || N < T || K <= 0 || E <= 0) return ORC_EINVAL;
    int64_t P = oracle_pad_tokens(N);
    if (P < N) return ORC_EINVAL;                   /* the padded block covers every token */
    int32_t* ip = padded_ids(ids, T, P, K, E, err);
    if (!ip) return ORC_ENOMEM;
    memset(map_PE, 0, (size_t)P * (size_t)E);
    for (int64_t i = 0; i < P * E; ++i) probs_PE[i] = 0.0f;
    for (int64_t t = 0; t < P; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = ip[t * K + k];
            if (e < 0) continue;
            map_PE[t * E + e] = 1;
            probs_PE[t * E + e] = (t < T) ? scores[t * K + k] : 0.0f;
        }
    free(ip);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Layout: per-expert counts, per-rank totals and prefix sums, positions.     */
/* ------------------------------------------------------------------------ */

/* Dispatch layout for one call.
 *
 * Inputs: ids [T][K]; T materialised tokens; N = num_tokens_per_rank
 * (T <= N); K, E, R.
 * Outputs (all int32):
 *   cnt_E[e]            pairs (t, k) routed to expert e: the per-expert
 *                       token counts ([titan] "API design",
 *                       num_local_tokens_per_expert_E; [graph] "Internode"
 *                       item 2, device-side per-expert counts).
 *   rows_per_rank_R[r]  sum of cnt_E over the experts of rank r.
 *   rank_prefix_R[r]    inclusive prefix of rows_per_rank_R; its last entry
 *                       is the true received total ([graph] "Internode"
 *                       item 3, gbl_rank_prefix_sum).
 *   tokens_in_rank_R[r] tokens with at least one expert on rank r.
 *   expert_offset_E[e]  first receive row of expert e: r(e) * S + the counts
 *                       of the lower experts of the same rank.
 *   pos_TK[t][k]        receive row of pair (t, k), or -1 when it has no
 *                       expert. Rows of one expert follow ascending flat
 *                       pair index t*K + k (reading: a stable order; the
 *                       pages do not fix one, and combine does not depend on
 *                       it).
 *   *S_out              rows per rank for this call, P * K.
 * packed = 0 (worst-token mode, [graph] "Internode" items 2-3): rank r's rows
 * start at r * S. packed = 1 (exact mode, [graph] num_worst_tokens == 0, where
 * the receive side is sized by the true counts): ranks follow each other with
 * no gap, so expert e starts at the counts of all lower experts and the valid
 * rows are exactly [0, rank_prefix[R-1]).
 * The steps follow the plain definition: pad (rows T..P-1 get -1), count,
 * scan, then hand out rows with a running cursor per expert in flat order.
 */
int oracle_layout(const int32_t* ids, int64_t T, int64_t N, int32_t K, int32_t E, int32_t R,
                  int32_t packed, int32_t* cnt_E, int32_t* expert_offset_E,
                  int32_t* rows_per_rank_R, int32_t* rank_prefix_R, int32_t* tokens_in_rank_R,
                  int32_t* pos_TK, int64_t* S_out, uint32_t* err)
{
    if (check_shape(T, N, K, E, R) != ORC_OK) return ORC_EINVAL;
#if ORACLE_MUTANT == 26
    int64_t P = oracle_pad_tokens(T);               /* mutant: capacity from T, not N */
    int64_t S = oracle_rank_stride(T, K);
    if (P < T || S < P * K) return ORC_EINVAL;
#else
    int64_t P = oracle_pad_tokens(N);
    int64_t S = oracle_rank_stride(N, K);
    if (P < N || S < P * K) return ORC_EINVAL;      /* the padded block covers every token */
#endif
    int32_t* ip = padded_ids(ids, T, P, K, E, err);
    if (!ip) return ORC_ENOMEM;

    /* Step 1: per-expert counts over the whole padded block. */
    for (int32_t e = 0; e < E; ++e) cnt_E[e] = 0;
    for (int64_t t = 0; t < P; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = ip[t * K + k];
            if (e >= 0) cnt_E[e] += 1;
        }

    /* Step 2: per-rank row totals, distinct tokens, inclusive prefix. */
    for (int32_t r = 0; r < R; ++r) {
        rows_per_rank_R[r] = 0;
        tokens_in_rank_R[r] = 0;
    }
    for (int32_t e = 0; e < E; ++e) rows_per_rank_R[rank_of(e, E, R)] += cnt_E[e];
    for (int64_t t = 0; t < P; ++t)
        for (int32_t r = 0; r < R; ++r) {
            int hit = 0;
            for (int32_t k = 0; k < K; ++k) {
                int32_t e = ip[t * K + k];
#if ORACLE_MUTANT == 8
                if (e >= 0 && rank_of(e, E, R) == r) hit += 1;  /* mutant: counts pairs */
#else
                if (e >= 0 && rank_of(e, E, R) == r) hit = 1;
#endif
            }
            tokens_in_rank_R[r] += hit;
        }
    int32_t run = 0;
    for (int32_t r = 0; r < R; ++r) {
#if ORACLE_MUTANT == 18
        rank_prefix_R[r] = run;                     /* mutant: exclusive prefix */
        run += rows_per_rank_R[r];
#else
        run += rows_per_rank_R[r];
        rank_prefix_R[r] = run;
#endif
    }

    /* Step 3: first row of each expert: inside its rank's block of S rows
     * (strided), or after every lower expert (packed). */
    for (int32_t e = 0; e < E; ++e) {
        int32_t r = rank_of(e, E, R);
#if ORACLE_MUTANT == 14
        int64_t off = (int64_t)r * S;                   /* mutant: packed mode ignored */
        for (int32_t f = 0; f < e; ++f)
            if (rank_of(f, E, R) == r) off += cnt_E[f];
#else
        int64_t off = packed ? 0 : (int64_t)r * S;
        for (int32_t f = 0; f < e; ++f)
            if (packed || rank_of(f, E, R) == r) off += cnt_E[f];
#endif
#if ORACLE_MUTANT == 3
        off += cnt_E[e];                            /* mutant: inclusive offset */
#endif
        expert_offset_E[e] = (int32_t)off;
    }

    /* Step 4: hand out rows in ascending flat pair order. */
    int64_t* cursor = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
    if (!cursor) {
        free(ip);
        return ORC_ENOMEM;
    }
    for (int32_t e = 0; e < E; ++e) cursor[e] = expert_offset_E[e];
#if ORACLE_MUTANT == 6
    for (int64_t t = T - 1; t >= 0; --t)            /* mutant: reverse token order */
#else
    for (int64_t t = 0; t < T; ++t)
#endif
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = ip[t * K + k];
            if (e < 0) {
                pos_TK[t * K + k] = -1;
            } else {
                pos_TK[t * K + k] = (int32_t)cursor[e];
                cursor[e] += 1;
            }
        }
    free(cursor);
    free(ip);
    *S_out = S;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Dispatch: copy each routed token row into its expert's receive rows.       */
/* ------------------------------------------------------------------------ */

/* Dispatch (permute) for one call. [titan] "Backend behavior" (HybridEP: the
 * current capacity sizes the fused-permute output; DeepEP: the current
 * capacity is the per-rank stride) and [align] "Fix".
 *
 * x is [T][row_bytes] (any element type; rows are copied byte for byte).
 * recv_x must hold R * S rows of row_bytes, recv_scores and recv_src R * S
 * entries, where S = oracle_rank_stride(N, K). For each pair with a row p:
 *   recv_x[p] = x[t], recv_scores[p] = scores[t][k], recv_src[p] = t*K + k.
 * Receive rows past a rank's true total are left as the caller filled them.
 * The layout outputs are written as oracle_layout writes them. A position
 * outside the R * S receive rows returns ORC_EBOUNDS before anything is
 * written there.
 */
int oracle_dispatch(const void* x, int64_t row_bytes, const float* scores, const int32_t* ids,
                    int64_t T, int64_t N, int32_t K, int32_t E, int32_t R, int32_t packed,
                    void* recv_x,
                    float* recv_scores, int32_t* recv_src, int32_t* cnt_E,
                    int32_t* expert_offset_E, int32_t* rows_per_rank_R, int32_t* rank_prefix_R,
                    int32_t* tokens_in_rank_R, int32_t* pos_TK, int64_t* S_out, uint32_t* err)
{
    if (row_bytes <= 0) return ORC_EINVAL;
    int rc = oracle_layout(ids, T, N, K, E, R, packed, cnt_E, expert_offset_E, rows_per_rank_R,
                           rank_prefix_R, tokens_in_rank_R, pos_TK, S_out, err);
    if (rc != ORC_OK) return rc;
    const uint8_t* xb = (const uint8_t*)x;
    uint8_t* rb = (uint8_t*)recv_x;
    /* The receive buffer holds R * S rows; a position outside it cannot come
     * from a correct layout, and is refused instead of written. */
    const int64_t rows = (int64_t)R * *S_out;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int64_t p = pos_TK[t * K + k];
            if (p < 0) continue;
            if (p >= rows) return ORC_EBOUNDS;
            memcpy(rb + p * row_bytes, xb + t * row_bytes, (size_t)row_bytes);
            recv_scores[p] = scores[t * K + k];
#if ORACLE_MUTANT == 19
            recv_src[p] = (int32_t)t;                   /* mutant: token, not pair index */
#else
            recv_src[p] = (int32_t)(t * K + k);
#endif
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                              */
/* ------------------------------------------------------------------------ */

/* fp32 -> bf16, round to nearest, ties to even, from the IEEE-754 definition:
 * bf16 keeps the top 16 bits of the fp32 encoding; the dropped low 16 bits
 * round up when above half an ulp, or exactly half with an odd kept bit.
 * A carry out of the mantissa correctly bumps the exponent (and overflows the
 * largest finite values to infinity). A NaN converts as IEEE 754-2008 6.2.3
 * recommends for a narrowing conversion: a quiet NaN of the same sign that
 * keeps the leading payload bits which fit (fp32 significand bits 21..16
 * become bf16 bits 5..0; the quiet bit 6 is set). */
uint16_t oracle_bf16_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
#if ORACLE_MUTANT == 30
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)0x7fc0u;                   /* mutant: drops sign and payload */
#elif ORACLE_MUTANT != 25
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
#endif
#if ORACLE_MUTANT == 7
    return (uint16_t)(u >> 16);                     /* mutant: truncation */
#else
    uint32_t low = u & 0xffffu;
    uint32_t kept = u >> 16;
#if ORACLE_MUTANT == 28
    if (low >= 0x8000u) kept += 1u;                 /* mutant: ties away from zero */
#else
    if (low > 0x8000u || (low == 0x8000u && (kept & 1u))) kept += 1u;
#endif
    return (uint16_t)kept;
#endif
}

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 word. */
float oracle_f32_from_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* The canonical quiet NaN (positive, quiet bit set, zero payload) in place of
 * whatever NaN the host's arithmetic produced; other values pass unchanged.
 * Every NaN result of the arithmetic below goes through this (see the NaN
 * reading at the top of the file). */
static float canonical_nan(float v)
{
#if ORACLE_MUTANT == 29
    return v;                                       /* mutant: the host's own NaN */
#else
    if (isnan(v)) {
        const uint32_t q = 0x7fc00000u;
        memcpy(&v, &q, sizeof v);
    }
    return v;
#endif
}

static float load_elem(const void* base, int kind, int64_t i)
{
    if (kind == ORC_BF16) return oracle_f32_from_bf16(((const uint16_t*)base)[i]);
    return ((const float*)base)[i];
}

/* ------------------------------------------------------------------------ */
/* Combine: weighted un-permute back to token order.                          */
/* ------------------------------------------------------------------------ */

/* Whether receive row p holds data: inside its rank's true total ([graph]
 * "Internode" item 3), i.e. p - r*S < rank_prefix[r] - rank_prefix[r-1] for
 * r = p / S (strided), or p < rank_prefix[R-1] (packed). */
static int row_ok(int64_t p, const int32_t* rank_prefix_R, int64_t S, int32_t R, int32_t packed)
{
    if (p < 0) return 0;
    if (packed) return p < (int64_t)rank_prefix_R[R - 1];
    int64_t r = (S > 0) ? p / S : R;
    if (r >= R) return 0;
    int64_t lo = (r > 0) ? rank_prefix_R[r - 1] : 0;
    return p - r * S < (int64_t)rank_prefix_R[r] - lo;
}

/* Combine for one call. [align] "Fix" (combine() slices the padded rows
 * back off) and [graph] "Internode" item 3 (the true received total comes
 * from the device prefix sum, not the padded row count).
 *
 * y is the expert output in the receive layout: R * S rows of D elements of
 * kind y_kind. For every token t < T and element d:
 *     acc = +0.0f
 *     for k = 0 .. K-1 with pos[t][k] >= 0:  acc = fmaf(scores[t][k], y[pos][d], acc)
 *     out[t][d] = acc (fp32) or its bf16 rounding (round to nearest even),
 *                 the canonical quiet NaN where acc is a NaN.
 * The accumulation is fp32 in ascending k, one fused multiply-add per term
 * (reading: the pages fix no order; this is the fixed top-k order). A NaN
 * stays a NaN through the rest of the chain, so replacing the final value is
 * the same as replacing every NaN along the way. A row p
 * of rank r = p / S is used only when p - r*S < rank_prefix[r] -
 * rank_prefix[r-1] (the rank's true total); any other row raises
 * ORC_ERR_ROW_OOB and contributes nothing. Only rows t < T are written: the
 * padded tail does not exist in the output.
 */
int oracle_combine(const void* y, int y_kind, int64_t D, const float* scores,
                   const int32_t* pos_TK, const int32_t* rank_prefix_R, int64_t S, int64_t T,
                   int32_t K, int32_t R, int32_t packed, void* out, int out_kind, uint32_t* err)
{
    if (T < 0 || D <= 0 || K <= 0 || R <= 0 || S < 0) return ORC_EINVAL;
    if ((y_kind != ORC_BF16 && y_kind != ORC_F32) || (out_kind != ORC_BF16 && out_kind != ORC_F32))
        return ORC_EINVAL;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t d = 0; d < D; ++d) {
            float acc = 0.0f;
#if ORACLE_MUTANT == 1
            for (int32_t k = 0; k < K - 1; ++k) {   /* mutant: drops the last term */
#elif ORACLE_MUTANT == 17
            for (int32_t k = K - 1; k >= 0; --k) {  /* mutant: descending k */
#else
            for (int32_t k = 0; k < K; ++k) {
#endif
                int64_t p = pos_TK[t * K + k];
                if (p < 0) continue;
                if (!row_ok(p, rank_prefix_R, S, R, packed)) {
                    *err |= ORC_ERR_ROW_OOB;
                    continue;
                }
                float v = load_elem(y, y_kind, p * D + d);
#if ORACLE_MUTANT == 2
                acc = fmaf(-scores[t * K + k], v, acc); /* mutant: wrong sign */
#else
                acc = fmaf(scores[t * K + k], v, acc);
#endif
            }
#if ORACLE_MUTANT == 24
            if (fabsf(acc) < 1.17549435e-38f) acc = 0.0f;   /* mutant: flushes subnormals */
#endif
            acc = canonical_nan(acc);
            if (out_kind == ORC_F32)
                ((float*)out)[t * D + d] = acc;
            else
                ((uint16_t*)out)[t * D + d] = oracle_bf16_from_f32(acc);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Backward of combine and dispatch.                                          */
/* ------------------------------------------------------------------------ */

static void store_elem(void* base, int kind, int64_t i, float v)
{
    if (kind == ORC_BF16)
        ((uint16_t*)base)[i] = oracle_bf16_from_f32(v);
    else
        ((float*)base)[i] = v;
}

/* Backward of combine. The pages require the backward pass to be reproduced
 * bit for bit like the forward ([align] "Testing": unequal-count forward AND
 * backward bitwise-match the equal-count run) but do not spell it out; it is
 * the derivative of out[t] = sum_k s[t][k] * y[pos[t][k]]:
 *   grad_y[pos[t][k]][d] = s[t][k] * grad_out[t][d]   (one fp32 product,
 *                          rounded to y's kind), for every valid pair;
 *   grad_scores[t][k]    = sum_d grad_out[t][d] * y[pos[t][k]][d], summed in
 *                          fp64 in ascending d and rounded once to fp32
 *                          (0 for a pair without a valid row).
 * A NaN product or sum is the canonical quiet NaN.
 * Rows of grad_y that no valid pair references are left as the caller filled
 * them. A pair whose row lies outside its rank's true total raises
 * ORC_ERR_ROW_OOB and contributes nothing. grad_scores may be NULL. */
int oracle_combine_backward(const void* grad_out, int g_kind, const void* y, int y_kind,
                            int64_t D, const float* scores, const int32_t* pos_TK,
                            const int32_t* rank_prefix_R, int64_t S, int64_t T, int32_t K,
                            int32_t R, int32_t packed, void* grad_y, float* grad_scores,
                            uint32_t* err)
{
    if (T < 0 || D <= 0 || K <= 0 || R <= 0 || S < 0) return ORC_EINVAL;
    if ((g_kind != ORC_BF16 && g_kind != ORC_F32) || (y_kind != ORC_BF16 && y_kind != ORC_F32))
        return ORC_EINVAL;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int64_t p = pos_TK[t * K + k];
#if ORACLE_MUTANT == 23
            float dot = 0.0f;                           /* mutant: fp32 dot */
#else
            double dot = 0.0;
#endif
            if (p >= 0 && !row_ok(p, rank_prefix_R, S, R, packed)) {
                *err |= ORC_ERR_ROW_OOB;
                p = -1;
            }
            if (p >= 0) {
#if ORACLE_MUTANT == 12
                float s = scores[t * K];                /* mutant: always the first score */
#else
                float s = scores[t * K + k];
#endif
                for (int64_t d = 0; d < D; ++d) {
                    float g = load_elem(grad_out, g_kind, t * D + d);
                    store_elem(grad_y, y_kind, p * D + d, canonical_nan(s * g));
                    dot += (double)g * (double)load_elem(y, y_kind, p * D + d);
                }
            }
            if (grad_scores) grad_scores[t * K + k] = canonical_nan((float)dot);
        }
    return ORC_OK;
}

/* Backward of dispatch: the derivative of recv_x[pos[t][k]] = x[t] and
 * recv_scores[pos[t][k]] = s[t][k]:
 *   grad_x[t][d]      = sum over valid k (ascending) of grad_recv[pos[t][k]][d],
 *                       accumulated in fp32 from +0 (the same chain as
 *                       combine with unit weights, a NaN sum canonical) and
 *                       rounded to grad_x's kind;
 *   grad_scores[t][k] = grad_recv_scores[pos[t][k]] (0 without a valid row).
 * grad_recv_scores and grad_scores may be NULL (then that part is skipped). */
int oracle_dispatch_backward(const void* grad_recv, int g_kind, int64_t D,
                             const float* grad_recv_scores, const int32_t* pos_TK,
                             const int32_t* rank_prefix_R, int64_t S, int64_t T, int32_t K,
                             int32_t R, int32_t packed, void* grad_x, int x_kind,
                             float* grad_scores, uint32_t* err)
{
    if (T < 0 || D <= 0 || K <= 0 || R <= 0 || S < 0) return ORC_EINVAL;
    if ((g_kind != ORC_BF16 && g_kind != ORC_F32) || (x_kind != ORC_BF16 && x_kind != ORC_F32))
        return ORC_EINVAL;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t d = 0; d < D; ++d) {
            float acc = 0.0f;
#if ORACLE_MUTANT == 13
            for (int32_t k = 1; k < K; ++k) {           /* mutant: drops the first term */
#else
            for (int32_t k = 0; k < K; ++k) {
#endif
                int64_t p = pos_TK[t * K + k];
                if (!row_ok(p, rank_prefix_R, S, R, packed)) continue;
                acc = fmaf(1.0f, load_elem(grad_recv, g_kind, p * D + d), acc);
            }
            store_elem(grad_x, x_kind, t * D + d, canonical_nan(acc));
        }
        for (int32_t k = 0; k < K; ++k) {
            int64_t p = pos_TK[t * K + k];
            int ok = row_ok(p, rank_prefix_R, S, R, packed);
            if (p >= 0 && !ok) *err |= ORC_ERR_ROW_OOB;
            if (grad_scores)
                grad_scores[t * K + k] = (ok && grad_recv_scores) ? grad_recv_scores[p] : 0.0f;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Per-rank dedupe: one row per (token, destination rank).                     */
/* ------------------------------------------------------------------------ */

/* Dispatch with one receive row per distinct (token, rank), the transport
 * format of a dispatcher that sends a token to a rank once however many of
 * that rank's experts it selected ([titan] "Backend behavior": DeepEP's
 * per-rank layout; [graph] "Internode": per-rank token counts). Rank r owns
 * rows [r*P, r*P + tokens_in_rank[r]); its rows are the tokens with at least
 * one expert on r, in ascending token order (reading: the stable order, as
 * for expert rows). For row q of token t on rank r:
 *   recv_tok_x[q] = x[t], recv_tok_src[q] = t,
 *   recv_topk_idx[q][k] = e - r*E_loc if pair (t,k) routes to expert e of
 *                         rank r, else -1 (a local expert index),
 *   recv_topk_w[q][k]   = scores[t][k] for those pairs, else 0;
 * and tok_pos[t][r] = q, or -1 when t has no expert on r. Receive buffers hold
 * R * P rows (P = oracle_pad_tokens(N)). */
int oracle_dispatch_dedup(const void* x, int64_t row_bytes, const float* scores,
                          const int32_t* ids, int64_t T, int64_t N, int32_t K, int32_t E,
                          int32_t R, void* recv_tok_x, int32_t* recv_tok_src,
                          int32_t* recv_topk_idx, float* recv_topk_w, int32_t* tok_pos_TR,
                          int32_t* tokens_in_rank_R, uint32_t* err)
{
    if (check_shape(T, N, K, E, R) != ORC_OK || row_bytes <= 0) return ORC_EINVAL;
    const int64_t P = oracle_pad_tokens(N);
    const int32_t eloc = E / R;
    for (int32_t r = 0; r < R; ++r) {
        int64_t q = (int64_t)r * P;
        for (int64_t t = 0; t < T; ++t) {
            int hit = 0;
            for (int32_t k = 0; k < K; ++k) {
                int32_t e = ids[t * K + k];
                if (e < -1 || e >= E) {
                    *err |= ORC_ERR_BAD_ID;
                    e = -1;
                }
                if (e >= 0 && rank_of(e, E, R) == r) hit = 1;
            }
            if (!hit) {
                tok_pos_TR[t * R + r] = -1;
                continue;
            }
#if ORACLE_MUTANT == 16
            for (int32_t dup = 0; dup < K; ++dup) {     /* mutant: one row per pair */
                if (dup > 0) {
                    int32_t e = ids[t * K + dup];
                    if (e < 0 || e >= E || rank_of(e, E, R) != r) continue;
                }
#endif
            if (q >= (int64_t)(r + 1) * P) return ORC_EINVAL;   /* a rank never exceeds P rows */
            tok_pos_TR[t * R + r] = (int32_t)q;
            memcpy((uint8_t*)recv_tok_x + q * row_bytes, (const uint8_t*)x + t * row_bytes,
                   (size_t)row_bytes);
            recv_tok_src[q] = (int32_t)t;
            for (int32_t k = 0; k < K; ++k) {
                int32_t e = ids[t * K + k];
                int mine = e >= 0 && e < E && rank_of(e, E, R) == r;
#if ORACLE_MUTANT == 21
                recv_topk_idx[q * K + k] = mine ? e : -1;  /* mutant: global expert id */
#else
                recv_topk_idx[q * K + k] = mine ? e - r * eloc : -1;
#endif
                recv_topk_w[q * K + k] = mine ? scores[t * K + k] : 0.0f;
            }
            ++q;
#if ORACLE_MUTANT == 16
            }
#endif
        }
        tokens_in_rank_R[r] = (int32_t)(q - (int64_t)r * P);
    }
    return ORC_OK;
}

/* The receiver's expansion of the dedupe rows into the expert layout of
 * oracle_dispatch: for every pair (t,k) with a receive row p = pos[t][k],
 *   y[p] = recv_tok_x[tok_pos[t][r(e)]]
 * where e = ids[t][k]. y holds the expert layout's rows (R * S of row_bytes). */
int oracle_dedup_expand(const void* recv_tok_x, int64_t row_bytes, const int32_t* tok_pos_TR,
                        const int32_t* pos_TK, const int32_t* ids, int64_t T, int32_t K,
                        int32_t E, int32_t R, void* y)
{
    if (T < 0 || K <= 0 || E <= 0 || R <= 0 || E % R != 0 || row_bytes <= 0) return ORC_EINVAL;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k) {
            const int64_t p = pos_TK[t * K + k];
            const int32_t e = ids[t * K + k];
            if (p < 0 || e < 0 || e >= E) continue;
#if ORACLE_MUTANT == 22
            const int64_t q = tok_pos_TR[t * R + (rank_of(e, E, R) + 1) % R];   /* mutant */
            if (q < 0) continue;
#else
            const int64_t q = tok_pos_TR[t * R + rank_of(e, E, R)];
            if (q < 0) return ORC_EINVAL;
#endif
            memcpy((uint8_t*)y + p * row_bytes, (const uint8_t*)recv_tok_x + q * row_bytes,
                   (size_t)row_bytes);
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Expert consumer: grouped GEMM over each expert's receive rows.             */
/* ------------------------------------------------------------------------ */

/* The expert computation between dispatch and combine, as a grouped linear
 * layer driven by the device-side counts ([graph] "Internode" item 2: per-
 * expert counts stay on the device for the consumers; "Tests": layout ->
 * dispatch -> expert -> combine). For every expert e and each of its rows
 * p = expert_offset[e] + j, j < cnt[e]:
 *     y[p][o] = sum_i x[p][i] * w[e][o][i]      (o < dout, i < din)
 * summed in fp64 in ascending i (each product of two bf16 values is exact in
 * fp64) and rounded once, from fp64 straight to bf16 (oracle_bf16_from_f64: no
 * intermediate fp32 rounding). x and y are in the receive layout (rows of
 * din / dout bf16 values), w is [E][dout][din] bf16. Rows of y that belong to
 * no expert are left as the caller filled them. */
/* fp64 -> bf16 in one rounding, to nearest with ties to even. bf16 has 8
 * significant bits, fp32's exponent range and subnormals spaced 2^-133 apart.
 * With v = m * 2^e, 0.5 <= |m| < 1 (frexp), the bf16 values near v are spaced
 * 2^(e-8), but never closer than 2^-133; v over that spacing, rounded to an
 * integer with ties to even (nearbyint in the default rounding mode), times
 * the spacing is the result: it has at most 8 significant bits and fits fp32
 * exactly, except at 2^128 and beyond, which is infinity. A NaN gives the
 * canonical quiet NaN (the sum is arithmetic, see the NaN reading above). */
uint16_t oracle_bf16_from_f64(double v)
{
    if (isnan(v)) return (uint16_t)0x7fc0u;
#if ORACLE_MUTANT == 31
    return oracle_bf16_from_f32((float)v);          /* mutant: rounds twice, via fp32 */
#endif
    if (v != 0.0 && !isinf(v)) {
        int e;
        (void)frexp(v, &e);
        int q = e - 8;
        if (q < -133) q = -133;
        v = ldexp(nearbyint(ldexp(v, -q)), q);
        if (fabs(v) >= 0x1p128) v = v > 0 ? INFINITY : -INFINITY;
    }
    float f = (float)v;                 /* exact: v is a bf16 value (or 0, inf) */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

int oracle_expert_gemm(const uint16_t* x, const uint16_t* w, const int32_t* cnt_E,
                       const int32_t* expert_offset_E, int32_t E, int64_t din, int64_t dout,
                       uint16_t* y)
{
    if (E <= 0 || din <= 0 || dout <= 0) return ORC_EINVAL;
    for (int32_t e = 0; e < E; ++e) {
#if ORACLE_MUTANT == 15
        const uint16_t* we = w + (int64_t)((e + 1) % E) * dout * din;   /* mutant: next expert */
#else
        const uint16_t* we = w + (int64_t)e * dout * din;
#endif
        for (int64_t j = 0; j < cnt_E[e]; ++j) {
            int64_t p = (int64_t)expert_offset_E[e] + j;
            for (int64_t o = 0; o < dout; ++o) {
#if ORACLE_MUTANT == 20
                float acc = 0.0f;                       /* mutant: fp32 sum */
#else
                double acc = 0.0;
#endif
                for (int64_t i = 0; i < din; ++i)
                    acc += (double)oracle_f32_from_bf16(x[p * din + i]) *
#if ORACLE_MUTANT == 27
                           (double)oracle_f32_from_bf16(we[i * dout + o]);   /* mutant: W^T */
#else
                           (double)oracle_f32_from_bf16(we[o * din + i]);
#endif
                y[p * dout + o] = oracle_bf16_from_f64((double)acc);
            }
        }
    }
    return ORC_OK;
}

/* Number of deliberately broken builds the tests can request (ORACLE_MUTANT). */
int oracle_mutant_id(void) { return ORACLE_MUTANT; }
