// Dispatch pack: every (token, j) pair with a receive row gets a copy of its
// token, as bf16 or as FP8 e4m3 with one fp32 scale per 128 elements.
//
// "NCCL EP 论文解读", item "通信模式": the send phase reads the token, writes it to
// the buffer and quantises in-kernel when FP8 is on.  "NVSHMEM 与 DeepEP：GPU 发起
// 的通信", section "高吞吐模式": dispatch payload FP8 with fine-grained scaling,
// one scale per 128 elements.  Here the "send" to logical rank r is a store
// into rank r's rows of the receive buffer in this GPU's memory.
//
// HBM-bound (read 2H bytes per token, write k rows).  One warp per token: the
// k lanes compute the pair rows from the layout (and store the row map), then
// the warp reads the token once in 16-byte vectors, converts it once (FP8) and
// streams it to the k rows.  No block-level barrier anywhere.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "layout_dev.cuh"

namespace moeep {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;  // 8 warps, 8 tokens in flight per CTA

// Rows of token t: lane j < k gets row(t, j); also stores the row map and the
// source id of every written row.
__device__ __forceinline__ int place_token(const RowArgs& ra, int t, int lane, int32_t* row,
                                           int32_t* recv_src)
{
    const int r = token_pair_row(ra, t, lane);
    if (lane < ra.k) {
        row[(size_t)t * ra.k + lane] = r;
        if (r >= 0 && recv_src) recv_src[r] = t;
    }
    return r;
}

template <int U>
__global__ void __launch_bounds__(kThreads) dispatch_bf16_kernel(
    RowArgs ra, const uint4* __restrict__ x, int nvec, int32_t* __restrict__ row,
    uint4* __restrict__ recv_x, int32_t* __restrict__ recv_src, const int32_t* __restrict__ cnt,
    int32_t* __restrict__ recv_cnt)
{
    if (blockIdx.x == 0 && recv_cnt)
        for (int e = threadIdx.x; e < ra.E; e += blockDim.x) recv_cnt[e] = cnt[e];
    const int lane = threadIdx.x & 31, wpc = blockDim.x >> 5;
    for (int t = blockIdx.x * wpc + (threadIdx.x >> 5); t < ra.T; t += gridDim.x * wpc) {
        const int r = place_token(ra, t, lane, row, recv_src);
        const uint4* xt = x + (size_t)t * nvec;
        for (int c0 = 0; c0 < nvec; c0 += 32 * U) {
            uint4 buf[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = c0 + u * 32 + lane;
                if (v < nvec) buf[u] = __ldg(xt + v);
            }
            for (int j = 0; j < ra.k; ++j) {
                const int rj = __shfl_sync(kFull, r, j);
                if (rj < 0) continue;
                uint4* dst = recv_x + (size_t)rj * nvec;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = c0 + u * 32 + lane;
                    if (v < nvec) dst[v] = buf[u];
                }
            }
        }
    }
}

// A half-warp (16 lanes x 8 elements) covers exactly one 128-element block.
template <int U>
__global__ void __launch_bounds__(kThreads) dispatch_fp8_kernel(
    RowArgs ra, const uint4* __restrict__ x, int nvec, int32_t* __restrict__ row,
    uint2* __restrict__ recv_q, float* __restrict__ recv_scale, int32_t* __restrict__ recv_src,
    const int32_t* __restrict__ cnt, int32_t* __restrict__ recv_cnt)
{
    if (blockIdx.x == 0 && recv_cnt)
        for (int e = threadIdx.x; e < ra.E; e += blockDim.x) recv_cnt[e] = cnt[e];
    const int lane = threadIdx.x & 31, wpc = blockDim.x >> 5;
    const int nblk = nvec / 16;
    for (int t = blockIdx.x * wpc + (threadIdx.x >> 5); t < ra.T; t += gridDim.x * wpc) {
        const int r = place_token(ra, t, lane, row, recv_src);
        const uint4* xt = x + (size_t)t * nvec;
        for (int c0 = 0; c0 < nvec; c0 += 32 * U) {
            uint2 q[U];
            float sc[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = c0 + u * 32 + lane;
                const uint4 raw = (v < nvec) ? __ldg(xt + v) : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                float f[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    f[2 * i] = __uint_as_float(w[i] << 16);
                    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
                }
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
                const float scale = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
                uint32_t packed[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                        make_float2(__fdiv_rn(f[4 * h + 0], scale), __fdiv_rn(f[4 * h + 1], scale)),
                        __NV_SATFINITE, __NV_E4M3);
                    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                        make_float2(__fdiv_rn(f[4 * h + 2], scale), __fdiv_rn(f[4 * h + 3], scale)),
                        __NV_SATFINITE, __NV_E4M3);
                    packed[h] = (uint32_t)lo | ((uint32_t)hi << 16);
                }
                q[u] = make_uint2(packed[0], packed[1]);
                sc[u] = scale;
            }
            for (int j = 0; j < ra.k; ++j) {
                const int rj = __shfl_sync(kFull, r, j);
                if (rj < 0) continue;
                uint2* dst = recv_q + (size_t)rj * nvec;
                float* sdst = recv_scale + (size_t)rj * nblk;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = c0 + u * 32 + lane;
                    if (v < nvec) {
                        dst[v] = q[u];
                        if ((lane & 15) == 0) sdst[v >> 4] = sc[u];
                    }
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_dispatch(const RowArgs& ra, const void* x, int H, int fp8, int32_t* row,
                            void* recv_x, float* recv_scale, int32_t* recv_src,
                            const int32_t* cnt, int32_t* recv_cnt, int sm_count, cudaStream_t s)
{
    const int nvec = H / 8;
    const int wpc = kThreads / 32;
    int blocks = (ra.T + wpc - 1) / wpc;
    if (blocks < 1) blocks = 1;
    if (blocks > sm_count * 8) blocks = sm_count * 8;
    if (fp8)
        dispatch_fp8_kernel<4><<<blocks, kThreads, 0, s>>>(ra, (const uint4*)x, nvec, row,
                                                           (uint2*)recv_x, recv_scale, recv_src,
                                                           cnt, recv_cnt);
    else
        dispatch_bf16_kernel<7><<<blocks, kThreads, 0, s>>>(ra, (const uint4*)x, nvec, row,
                                                            (uint4*)recv_x, recv_src, cnt, recv_cnt);
    return cudaGetLastError();
}

}  // namespace moeep
