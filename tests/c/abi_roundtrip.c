/*
 * abi_roundtrip.c - the C ABI used from plain C (no Python, no torch): create a
 * buffer over cudaMalloc'ed workspace, dispatch and combine one call, read the
 * device error word, and compare every layout array, every defined receive row
 * and the combined output bit for bit with the CPU oracle, a separate library
 * (test infrastructure; it shares no code with libep_gb300).
 *
 * Built and run by tests/test_c_abi_gpu.py. Exit status 0 and "c-abi ok" on
 * success; the first mismatch is printed otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ep.h"

/* The oracle's entry points (oracle/ep_oracle.c), declared here. */
int oracle_dispatch(const void* x, int64_t row_bytes, const float* scores, const int32_t* ids,
                    int64_t T, int64_t N, int32_t K, int32_t E, int32_t R, int32_t packed,
                    void* recv_x, float* recv_scores, int32_t* recv_src, int32_t* cnt_E,
                    int32_t* expert_offset_E, int32_t* rows_per_rank_R, int32_t* rank_prefix_R,
                    int32_t* tokens_in_rank_R, int32_t* pos_TK, int64_t* S_out, uint32_t* err);
int oracle_combine(const void* y, int y_kind, int64_t D, const float* scores,
                   const int32_t* pos_TK, const int32_t* rank_prefix_R, int64_t S, int64_t T,
                   int32_t K, int32_t R, int32_t packed, void* out, int out_kind, uint32_t* err);
enum { ORACLE_BF16 = 0 };

enum { T = 777, N = 780, N_MAX = 800, D = 256, E = 64, K = 4, R = 8 };

static uint64_t rng_state = 0x243F6A8885A308D3ull;
static uint32_t next_u32(void)
{
    rng_state = rng_state * 6364136223846793005ull + 1442695040888963407ull;
    return (uint32_t)(rng_state >> 32);
}

#define CK(call)                                                                   \
    do {                                                                           \
        cudaError_t e_ = (call);                                                   \
        if (e_ != cudaSuccess) {                                                   \
            printf("CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
            return 1;                                                              \
        }                                                                          \
    } while (0)
#define EPK(call)                                                                  \
    do {                                                                           \
        ep_status s_ = (call);                                                     \
        if (s_ != EP_OK) {                                                         \
            printf("ep error %s at %s:%d\n", ep_status_string(s_), __FILE__, __LINE__); \
            return 1;                                                              \
        }                                                                          \
    } while (0)

static int same(const char* what, const void* a, const void* b, size_t n)
{
    if (memcmp(a, b, n) == 0) return 1;
    printf("mismatch: %s\n", what);
    return 0;
}

int main(void)
{
    /* Inputs: bf16 rows, K distinct experts per token, positive scores. */
    uint16_t* x = (uint16_t*)malloc((size_t)T * D * 2);
    int32_t* ids = (int32_t*)malloc((size_t)T * K * 4);
    float* sc = (float*)malloc((size_t)T * K * 4);
    for (size_t i = 0; i < (size_t)T * D; ++i) x[i] = (uint16_t)(0x3C00u + (next_u32() & 0x07FFu));
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int e, dup;
            do {
                e = (int)(next_u32() % E);
                dup = 0;
                for (int j = 0; j < k; ++j) dup |= ids[t * K + j] == e;
            } while (dup);
            ids[t * K + k] = e;
            sc[t * K + k] = (float)(1 + next_u32() % 1000) / 1000.0f;
        }

    ep_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.num_max_tokens_per_rank = N_MAX;
    cfg.hidden = D;
    cfg.num_experts = E;
    cfg.num_ranks = R;
    cfg.topk = K;
    cfg.dtype = EP_BF16;
    const size_t need = ep_buffer_required_bytes(&cfg);
    if (need == 0) {
        printf("configuration rejected\n");
        return 1;
    }
    void *ws, *dx, *dids, *dsc, *dout;
    CK(cudaMalloc(&ws, need));
    CK(cudaMalloc(&dx, (size_t)T * D * 2));
    CK(cudaMalloc(&dids, (size_t)T * K * 4));
    CK(cudaMalloc(&dsc, (size_t)T * K * 4));
    CK(cudaMalloc(&dout, (size_t)T * D * 2));
    CK(cudaMemcpy(dx, x, (size_t)T * D * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dids, ids, (size_t)T * K * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dsc, sc, (size_t)T * K * 4, cudaMemcpyHostToDevice));

    ep_buffer* buf = NULL;
    EPK(ep_buffer_init(&cfg, ws, need, &buf));
    ep_dispatch_out d;
    EPK(ep_dispatch(buf, dx, (const float*)dsc, (const int32_t*)dids, T, N, NULL, &d));
    EPK(ep_combine(buf, d.recv_x, (const float*)dsc, T, dout, EP_BF16, NULL));
    CK(cudaDeviceSynchronize());
    uint32_t flags = 0;
    EPK(ep_get_device_error(buf, NULL, &flags));
    if (flags != 0) {
        printf("device error word 0x%x\n", flags);
        return 1;
    }

    const int64_t S = d.layout.rank_stride;
    const size_t rows = (size_t)R * (size_t)S;
    int32_t g_cnt[E], g_off[E], g_rpr[R], g_rp[R], g_tir[R];
    int32_t* g_pos = (int32_t*)malloc((size_t)T * K * 4);
    uint16_t* g_rx = (uint16_t*)malloc(rows * D * 2);
    uint16_t* g_out = (uint16_t*)malloc((size_t)T * D * 2);
    CK(cudaMemcpy(g_cnt, d.layout.tokens_per_expert, sizeof g_cnt, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(g_off, d.layout.expert_offset, sizeof g_off, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(g_rpr, d.layout.rows_per_rank, sizeof g_rpr, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(g_rp, d.layout.rank_prefix, sizeof g_rp, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(g_tir, d.layout.tokens_in_rank, sizeof g_tir, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(g_pos, d.layout.pos, (size_t)T * K * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(g_rx, d.recv_x, rows * D * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(g_out, dout, (size_t)T * D * 2, cudaMemcpyDeviceToHost));

    /* The oracle on the same inputs. */
    int32_t o_cnt[E], o_off[E], o_rpr[R], o_rp[R], o_tir[R];
    int32_t* o_pos = (int32_t*)malloc((size_t)T * K * 4);
    uint16_t* o_rx = (uint16_t*)calloc(rows * D, 2);
    float* o_rs = (float*)calloc(rows, 4);
    int32_t* o_src = (int32_t*)calloc(rows, 4);
    uint16_t* o_out = (uint16_t*)malloc((size_t)T * D * 2);
    int64_t oS = 0;
    uint32_t oerr = 0;
    if (oracle_dispatch(x, D * 2, sc, ids, T, N, K, E, R, 0, o_rx, o_rs, o_src, o_cnt, o_off,
                        o_rpr, o_rp, o_tir, o_pos, &oS, &oerr) != 0 ||
        oracle_combine(o_rx, ORACLE_BF16, D, sc, o_pos, o_rp, oS, T, K, R, 0, o_out,
                       ORACLE_BF16, &oerr) != 0 ||
        oerr != 0) {
        printf("oracle failed\n");
        return 1;
    }
    if (oS != S) {
        printf("rank stride %lld vs oracle %lld\n", (long long)S, (long long)oS);
        return 1;
    }
    int ok = same("tokens_per_expert", g_cnt, o_cnt, sizeof g_cnt) &&
             same("expert_offset", g_off, o_off, sizeof g_off) &&
             same("rows_per_rank", g_rpr, o_rpr, sizeof g_rpr) &&
             same("rank_prefix", g_rp, o_rp, sizeof g_rp) &&
             same("tokens_in_rank", g_tir, o_tir, sizeof g_tir) &&
             same("pos", g_pos, o_pos, (size_t)T * K * 4);
    for (int r = 0; ok && r < R; ++r)
        ok = same("receive rows", g_rx + (size_t)r * S * D, o_rx + (size_t)r * S * D,
                  (size_t)o_rpr[r] * D * 2);
    ok = ok && same("combine output", g_out, o_out, (size_t)T * D * 2);
    EPK(ep_buffer_destroy(buf));
    cudaFree(ws);
    if (!ok) return 1;
    printf("c-abi ok: T=%d D=%d E=%d K=%d R=%d, %d rows\n", T, D, E, K, R, o_rp[R - 1]);
    return 0;
}
