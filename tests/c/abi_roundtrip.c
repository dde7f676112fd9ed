/*
 * A C99 program that uses libmoeep through include/moe_ep.h and the CUDA
 * runtime's C API only (no C++, no Python): one HT forward of 300 tokens --
 * route with a node limit ("NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式"),
 * the receive-count query, a bf16 dispatch and the combine ("NCCL EP 论文解读",
 * item "核心功能函数") -- with identity experts, so the combined tokens must equal
 * the input tokens within one bf16 ulp (the score-normalised weights of a token
 * sum to 1 up to fp32 rounding).  Also checks that every token's experts are
 * distinct, in range and on at most topk_groups nodes, and that the row map is
 * a bijection onto the receive rows.  Prints "c abi ok" and exits 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "moe_ep.h"

#define T 300
#define E 64
#define R 16
#define H 1024
#define K 4
#define G 8
#define KG 4

static int fail(const char* what, int code)
{
    fprintf(stderr, "FAIL: %s (%d)\n", what, code);
    return 1;
}

#define CHECK_EP(call)                                  \
    do {                                                \
        int st_ = (call);                               \
        if (st_ != MOE_EP_OK) return fail(#call, st_);  \
    } while (0)
#define CHECK_CUDA(call)                                        \
    do {                                                        \
        cudaError_t e_ = (call);                                \
        if (e_ != cudaSuccess) return fail(#call, (int)e_);     \
    } while (0)

static uint32_t lcg(uint64_t* s)
{
    *s = *s * 6364136223846793005ull + 1442695040888963407ull;
    return (uint32_t)(*s >> 33);
}

/* fp32 -> bf16 bits, nearest even (finite inputs) */
static uint16_t bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* bf16 bits as an ordered integer: adjacent values differ by 1 */
static int32_t ordered(uint16_t b)
{
    return (b & 0x8000u) ? -(int32_t)(b & 0x7fffu) : (int32_t)b;
}

int main(void)
{
    static float scores[T * E];
    static uint16_t x[T * H], out[T * H];
    static int32_t idx[T * K], row[T * K], seen[T * K];
    uint64_t s = 12345;
    for (int i = 0; i < T * E; ++i) scores[i] = (float)(lcg(&s) >> 8) * (1.0f / 16777216.0f);
    for (int i = 0; i < T * H; ++i) {
        const float u = (float)(lcg(&s) >> 8) * (1.0f / 16777216.0f);
        x[i] = bf16(4.0f * u - 2.0f);
    }

    float *d_scores = NULL, *d_w = NULL;
    void *d_x = NULL, *d_recv = NULL, *d_out = NULL;
    int32_t *d_idx = NULL, *d_src = NULL, *d_cnt = NULL;
    CHECK_CUDA(cudaMalloc((void**)&d_scores, sizeof scores));
    CHECK_CUDA(cudaMalloc((void**)&d_w, sizeof(float) * T * K));
    CHECK_CUDA(cudaMalloc(&d_x, sizeof x));
    CHECK_CUDA(cudaMalloc(&d_recv, sizeof(uint16_t) * (size_t)T * K * H));
    CHECK_CUDA(cudaMalloc(&d_out, sizeof out));
    CHECK_CUDA(cudaMalloc((void**)&d_idx, sizeof idx));
    CHECK_CUDA(cudaMalloc((void**)&d_src, sizeof(int32_t) * T * K));
    CHECK_CUDA(cudaMalloc((void**)&d_cnt, sizeof(int32_t) * E));
    CHECK_CUDA(cudaMemcpy(d_scores, scores, sizeof scores, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_x, x, sizeof x, cudaMemcpyHostToDevice));

    moe_ep_group_t g = NULL;
    moe_ep_handle_t h = NULL;
    CHECK_EP(moe_ep_create_group(&g, MOE_EP_HT, E, R, T, H));
    CHECK_EP(moe_ep_create_handle(g, K, &h));
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));

    const moe_ep_route_opts_t opts = {K, G, KG, 0, MOE_EP_W_SCORE_NORM};
    CHECK_EP(moe_ep_route(h, d_scores, T, &opts, d_idx, d_w, stream));
    int64_t total = 0;
    static int32_t per_rank[R], per_expert[E];
    CHECK_EP(moe_ep_get_num_recv_tokens(h, &total, per_rank, per_expert, stream));
    if (total != (int64_t)T * K) return fail("receive rows", (int)total);
    CHECK_EP(moe_ep_dispatch(h, d_x, 0, d_recv, NULL, d_src, d_cnt, total, stream));
    CHECK_EP(moe_ep_combine(h, d_recv, d_w, d_out, total, stream));
    CHECK_EP(moe_ep_copy_layout(h, NULL, NULL, NULL, NULL, d_src, stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));
    CHECK_CUDA(cudaMemcpy(out, d_out, sizeof out, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(idx, d_idx, sizeof idx, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(row, d_src, sizeof row, cudaMemcpyDeviceToHost));

    for (int t = 0; t < T; ++t) {
        unsigned nodes = 0;
        for (int j = 0; j < K; ++j) {
            const int e = idx[t * K + j];
            if (e < 0 || e >= E) return fail("expert id", e);
            for (int jj = 0; jj < j; ++jj)
                if (idx[t * K + jj] == e) return fail("repeated expert", e);
            nodes |= 1u << (e / (E / G));
        }
        if (__builtin_popcount(nodes) > KG) return fail("nodes per token", (int)nodes);
    }
    int64_t sum = 0;
    for (int e = 0; e < E; ++e) sum += per_expert[e];
    if (sum != total) return fail("per-expert counts", (int)sum);
    for (int i = 0; i < T * K; ++i) {
        const int r = row[i];
        if (r < 0 || r >= T * K || seen[r]) return fail("row map", r);
        seen[r] = 1;
    }
    for (int i = 0; i < T * H; ++i) {
        const int32_t d = ordered(out[i]) - ordered(x[i]);
        if (d > 1 || d < -1) return fail("round trip (bf16 ulp)", d);
    }

    CHECK_EP(moe_ep_destroy_handle(h));
    CHECK_EP(moe_ep_destroy_group(g));
    cudaStreamDestroy(stream);
    cudaFree(d_scores);
    cudaFree(d_w);
    cudaFree(d_x);
    cudaFree(d_recv);
    cudaFree(d_out);
    cudaFree(d_idx);
    cudaFree(d_src);
    cudaFree(d_cnt);
    printf("c abi ok\n");
    return 0;
}
