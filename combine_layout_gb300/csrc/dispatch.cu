// Dispatch pack: every (token, j) pair with a receive row gets a copy of its
// token, as bf16 or as FP8 e4m3 with one fp32 scale per 128 elements.
//
// "NCCL EP 论文解读", item "通信模式": the send phase reads the token, writes it to
// the buffer and quantises in-kernel when FP8 is on.  "NVSHMEM 与 DeepEP：GPU 发起
// 的通信", section "高吞吐模式": dispatch payload FP8 with fine-grained scaling,
// one scale per 128 elements.  Here the "send" to logical rank r is a store
// into rank r's rows of the receive buffer in this GPU's memory.
//
// The work is HBM-bound (read H*2 bytes per token, write k rows): each CTA
// takes one token at a time, reads it once in 16-byte vectors, converts it
// once (FP8) and streams it to the k destination rows.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moeep {
namespace {

constexpr int kThreads = 128;
constexpr int kUnroll = 8;  // 16-byte vectors held per thread per pass

__device__ __forceinline__ void load_rows(const int32_t* __restrict__ row, int t, int k,
                                          int32_t* __restrict__ recv_src, int* s_row)
{
    if (threadIdx.x < k) {
        const int r = row[(size_t)t * k + threadIdx.x];
        s_row[threadIdx.x] = r;
        if (r >= 0 && recv_src) recv_src[r] = t;
    }
}

__global__ void __launch_bounds__(kThreads) dispatch_bf16_kernel(
    const uint4* __restrict__ x, int T, int k, int nvec, const int32_t* __restrict__ row,
    uint4* __restrict__ recv_x, int32_t* __restrict__ recv_src, const int32_t* __restrict__ cnt,
    int32_t* __restrict__ recv_cnt, int E)
{
    __shared__ int s_row[kMaxTopk];
    if (blockIdx.x == 0 && recv_cnt)
        for (int e = threadIdx.x; e < E; e += blockDim.x) recv_cnt[e] = cnt[e];

    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        load_rows(row, t, k, recv_src, s_row);
        __syncthreads();
        const uint4* xt = x + (size_t)t * nvec;
        for (int v0 = threadIdx.x; v0 < nvec; v0 += kUnroll * kThreads) {
            uint4 buf[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * kThreads;
                if (v < nvec) buf[u] = __ldg(xt + v);
            }
            for (int j = 0; j < k; ++j) {
                const int r = s_row[j];
                if (r < 0) continue;
                uint4* dst = recv_x + (size_t)r * nvec;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int v = v0 + u * kThreads;
                    if (v < nvec) dst[v] = buf[u];
                }
            }
        }
        __syncthreads();
    }
}

// Half-warp (16 lanes x 8 elements) covers exactly one 128-element block.
__global__ void __launch_bounds__(kThreads) dispatch_fp8_kernel(
    const uint4* __restrict__ x, int T, int k, int nvec, const int32_t* __restrict__ row,
    uint2* __restrict__ recv_q, float* __restrict__ recv_scale, int32_t* __restrict__ recv_src,
    const int32_t* __restrict__ cnt, int32_t* __restrict__ recv_cnt, int E)
{
    __shared__ int s_row[kMaxTopk];
    if (blockIdx.x == 0 && recv_cnt)
        for (int e = threadIdx.x; e < E; e += blockDim.x) recv_cnt[e] = cnt[e];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nblk = nvec / 16;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        load_rows(row, t, k, recv_src, s_row);
        __syncthreads();
        const uint4* xt = x + (size_t)t * nvec;
        // the loop bound is uniform per warp so that every shuffle has all 32 lanes
        for (int v0 = warp * 32; v0 < nvec; v0 += kThreads) {
            const int v = v0 + lane;
            const bool act = v < nvec;
            uint4 raw = act ? __ldg(xt + v) : make_uint4(0u, 0u, 0u, 0u);
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
            for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
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
            if (act) {
                const uint2 q = make_uint2(packed[0], packed[1]);
                for (int j = 0; j < k; ++j) {
                    const int r = s_row[j];
                    if (r < 0) continue;
                    recv_q[(size_t)r * nvec + v] = q;
                    if ((lane & 15) == 0) recv_scale[(size_t)r * nblk + v / 16] = scale;
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_dispatch(const void* x, int T, int H, int k, int fp8, const int32_t* row,
                            void* recv_x, float* recv_scale, int32_t* recv_src,
                            const int32_t* cnt, int32_t* recv_cnt, int E, int sm_count,
                            cudaStream_t s)
{
    const int nvec = H / 8;
    int blocks = T < 1 ? 1 : T;
    const int cap = sm_count * 16;
    if (blocks > cap) blocks = cap;
    if (fp8)
        dispatch_fp8_kernel<<<blocks, kThreads, 0, s>>>(
            (const uint4*)x, T, k, nvec, row, (uint2*)recv_x, recv_scale, recv_src, cnt, recv_cnt, E);
    else
        dispatch_bf16_kernel<<<blocks, kThreads, 0, s>>>((const uint4*)x, T, k, nvec, row,
                                                         (uint4*)recv_x, recv_src, cnt, recv_cnt, E);
    return cudaGetLastError();
}

}  // namespace moeep
