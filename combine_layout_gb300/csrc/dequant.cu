// Receive-side dequantisation: the FP8 e4m3 rows of the receive layout, with
// their fp32 scale per 128 elements, into bf16 rows of the same layout --
// the expert-major input of a bf16 expert GEMM ("NCCL EP 论文解读", "Tensor
// Layouts": the expert-major layout is fed to the GEMM directly; "NVSHMEM 与
// DeepEP：GPU 发起的通信", section "高吞吐模式": FP8 dispatch with fine-grained
// scaling).  y = bf16_rn(float(q) * scale), the product taken in fp32.
//
// Only the rows the layout defines are written: HT expert e's rows
// off[e] .. off[e] + cnt[e] (padding rows of an aligned layout are left
// alone), LL slots e * S .. e * S + cnt[e].  The rows are enumerated on the
// device from the counts, so no host synchronisation is needed: every CTA
// rebuilds the prefix of the counts in shared memory and its warps take rows
// in grid-stride order, one row per warp, 16 FP8 values per lane and vector.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moeep {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t dequant_pair(uint16_t two_fp8, float s)
{
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two_fp8, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));  // exact
    const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, s), __fmul_rn(f.y, s));
    return *reinterpret_cast<const uint32_t*>(&b);
}

__global__ void __launch_bounds__(kThreads) dequant_kernel(const int32_t* __restrict__ cnt,
                                                           const int32_t* __restrict__ off, int E,
                                                           int S, int mode, int H,
                                                           const uint4* __restrict__ q,
                                                           const float* __restrict__ scale,
                                                           uint4* __restrict__ y)
{
    griddep_wait();
    __shared__ int s_pre[kMaxExperts + 1];
    __shared__ int s_part[kThreads];
    // exclusive prefix of the actual counts
    const int tid = threadIdx.x;
    const int per = (E + kThreads - 1) / kThreads;
    const int lo = min(tid * per, E), hi = min(lo + per, E);
    int sum = 0;
    for (int e = lo; e < hi; ++e) sum += __ldg(cnt + e);
    s_part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int i = 0; i < kThreads; ++i) {
            const int v = s_part[i];
            s_part[i] = run;
            run += v;
        }
        s_pre[E] = run;
    }
    __syncthreads();
    int run = s_part[tid];
    for (int e = lo; e < hi; ++e) {
        s_pre[e] = run;
        run += __ldg(cnt + e);
    }
    __syncthreads();

    const int total = s_pre[E];
    const int lane = tid & 31, wpc = kThreads / 32;
    const int nvq = H / 16;   // 16-byte vectors of FP8 per row
    const int nbk = H / 128;  // scales per row
    for (int i = blockIdx.x * wpc + (tid >> 5); i < total; i += gridDim.x * wpc) {
        // expert of defined row i: the last e with s_pre[e] <= i
        int a = 0, b = E;
        while (b - a > 1) {
            const int m = (a + b) >> 1;
            if (s_pre[m] <= i) a = m; else b = m;
        }
        const int e = a;
        const int row = (mode == MOE_EP_HT ? __ldg(off + e) : e * S) + (i - s_pre[e]);
        const uint4* qr = q + (size_t)row * nvq;
        const float* sr = scale + (size_t)row * nbk;
        uint4* yr = y + (size_t)row * (H / 8);
        constexpr int U = 7;  // vectors in flight per lane
        for (int v0 = lane; v0 < nvq; v0 += 32 * U) {
            uint4 w[U];
            float s[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + 32 * u;
                if (v < nvq) {
                    w[u] = __ldg(qr + v);
                    s[u] = __ldg(sr + (v >> 3));  // 16 values lie in one 128-block
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + 32 * u;
                if (v >= nvq) break;
                const uint32_t x[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
                uint32_t o[8];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    o[2 * c] = dequant_pair((uint16_t)(x[c] & 0xffffu), s[u]);
                    o[2 * c + 1] = dequant_pair((uint16_t)(x[c] >> 16), s[u]);
                }
                yr[2 * v] = make_uint4(o[0], o[1], o[2], o[3]);
                yr[2 * v + 1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_dequant(const int32_t* cnt, const int32_t* off, int E, int S, int mode, int H,
                           const uint8_t* q, const float* scale, void* y, int sm_count,
                           cudaStream_t s)
{
    return launch_pdl(dequant_kernel, dim3(sm_count * 8), dim3(kThreads), s, cnt, off, E, S, mode, H,
                      (const uint4*)q, scale, (uint4*)y);
}

}  // namespace moeep
