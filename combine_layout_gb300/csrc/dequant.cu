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

#include <atomic>

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

// Exclusive prefix of the actual counts into s_pre[0..E] (s_pre[E] = the
// number of defined rows); all threads of the CTA.
__device__ __forceinline__ void count_prefix(const int32_t* __restrict__ cnt, int E, int* s_pre,
                                             int* s_part)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (E + nt - 1) / nt;
    const int lo = min(tid * per, E), hi = min(lo + per, E);
    int sum = 0;
    for (int e = lo; e < hi; ++e) sum += __ldg(cnt + e);
    // block-wide exclusive scan of the per-thread sums: warp scans, then the
    // warp totals (s_part holds the nt / 32 totals)
    const int lane = tid & 31, warp = tid >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += s_part[w];
    if (tid == nt - 1) s_pre[E] = run + sum;
    for (int e = lo; e < hi; ++e) {
        s_pre[e] = run;
        run += __ldg(cnt + e);
    }
    __syncthreads();
}

// Row of the i-th defined row: expert e = the last e with s_pre[e] <= i.
__device__ __forceinline__ int defined_row(const int* s_pre, int E, int i,
                                           const int32_t* __restrict__ off, int S, int mode)
{
    int a = 0, b = E;
    while (b - a > 1) {
        const int m = (a + b) >> 1;
        if (s_pre[m] <= i) a = m; else b = m;
    }
    return (mode == MOE_EP_HT ? __ldg(off + a) : a * S) + (i - s_pre[a]);
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
    __shared__ int s_part[32];
    const int tid = threadIdx.x;
    count_prefix(cnt, E, s_pre, s_part);
    const int total = s_pre[E];
    const int lane = tid & 31, wpc = kThreads / 32;
    const int nvq = H / 16;   // 16-byte vectors of FP8 per row
    const int nbk = H / 128;  // scales per row
    for (int i = blockIdx.x * wpc + (tid >> 5); i < total; i += gridDim.x * wpc) {
        const int row = defined_row(s_pre, E, i, off, S, mode);
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

// ---------------------------------------------------------------------------
// TMA-staged variant (H % 512 == 0: a row's scales are a whole number of
// 16-byte units).  Every CTA keeps kStages rows in flight in shared memory:
// one thread issues a bulk copy (cp.async.bulk, completion counted on the
// stage's mbarrier) of each defined row's FP8 values and scales; all threads
// convert the staged row and store bf16 with 16-byte stores.  The copies hold
// no registers, so far more bytes are in flight per SM than with loads into
// registers.  Every mbarrier wait is bounded: a wait that gives up latches
// kErrTimeout, the CTA stops converting, waits (bounded) for the copies it
// still has in flight and returns.

constexpr int kStages = 8;
constexpr int kTmaMaxThreads = 512;
// CTAs per SM (shared memory permitting).  Measured on the 4096-token,
// 7168-wide FP8 layout: 3 CTAs x 8 stages 120 us; 2 x 8 139 us, 2 x 12
// 137 us, 4 x 6 133 us, 6 x 4 130 us.
constexpr int kTmaPerSm = 3;
constexpr uint32_t kWaitPolls = 1u << 22;  // try_wait polls before a wait gives up

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    for (uint32_t it = 0; it < kWaitPolls; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

__global__ void __launch_bounds__(kTmaMaxThreads) dequant_tma_kernel(const int32_t* __restrict__ cnt,
                                                               const int32_t* __restrict__ off,
                                                               int E, int S, int mode, int H,
                                                               const uint8_t* __restrict__ q,
                                                               const float* __restrict__ scale,
                                                               uint4* __restrict__ y,
                                                               unsigned* err)
{
    griddep_wait();
    extern __shared__ __align__(128) unsigned char s_buf[];  // kStages x (H + H/32) bytes
    __shared__ __align__(8) unsigned long long s_bar[kStages];
    __shared__ int s_row[kStages];
    __shared__ int s_pre[kMaxExperts + 1];
    __shared__ int s_part[32];
    __shared__ int s_fail;
    const int tid = threadIdx.x;
    count_prefix(cnt, E, s_pre, s_part);
    const int total = s_pre[E];
    const int first = blockIdx.x;
    const int mine = first < total ? (total - 1 - first) / (int)gridDim.x + 1 : 0;
    const uint32_t qbytes = (uint32_t)H, sbytes = (uint32_t)(H / 32), stage = qbytes + sbytes;
    const int nvq = H / 16, nbk = H / 128;
    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(smem_u32(&s_bar[st]));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_fail = 0;
    }
    __syncthreads();
    // thread 0: stage n's row into buffer n % kStages
    auto issue = [&](int n) {
        const int st = n % kStages;
        const int row = defined_row(s_pre, E, first + n * (int)gridDim.x, off, S, mode);
        s_row[st] = row;
        const uint32_t bar = smem_u32(&s_bar[st]);
        unsigned char* dst = s_buf + (size_t)st * stage;
        mbar_expect_tx(bar, stage);
        bulk_load(smem_u32(dst), q + (size_t)row * H, qbytes, bar);
        bulk_load(smem_u32(dst + qbytes), scale + (size_t)row * nbk, sbytes, bar);
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < min(kStages, mine); ++issued) issue(issued);
    int n = 0;
    for (; n < mine; ++n) {
        const int st = n % kStages;
        const bool ok = mbar_wait(smem_u32(&s_bar[st]), (uint32_t)((n / kStages) & 1));
        if (ok) {
            const uint4* qs = reinterpret_cast<const uint4*>(s_buf + (size_t)st * stage);
            const float* ss = reinterpret_cast<const float*>(s_buf + (size_t)st * stage + qbytes);
            uint4* yr = y + (size_t)s_row[st] * (H / 8);
            for (int v = tid; v < nvq; v += (int)blockDim.x) {
                const uint4 w = qs[v];
                const float sc = ss[v >> 3];
                const uint32_t x[4] = {w.x, w.y, w.z, w.w};
                uint32_t o[8];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    o[2 * c] = dequant_pair((uint16_t)(x[c] & 0xffffu), sc);
                    o[2 * c + 1] = dequant_pair((uint16_t)(x[c] >> 16), sc);
                }
                yr[2 * v] = make_uint4(o[0], o[1], o[2], o[3]);
                yr[2 * v + 1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
        } else {
            s_fail = 1;
        }
        __syncthreads();  // the stage is free again (and s_fail is seen by all)
        if (s_fail) break;
        if (tid == 0 && issued < mine) issue(issued++);
    }
    if (s_fail && tid == 0) {
        err[kErrTimeout] = 1u;
        // the copies still in flight into this CTA's shared memory: wait for
        // them (bounded) before the CTA exits
        for (int m = n; m < issued; ++m)
            mbar_wait(smem_u32(&s_bar[m % kStages]), (uint32_t)((m / kStages) & 1));
    }
}

// The TMA kernel's dynamic shared memory limit, raised once per device (the
// attribute belongs to the device's copy of the kernel) and size.
constexpr int kMaxDevices = 64;
std::atomic<int> g_tma_smem[kMaxDevices];

cudaError_t allow_tma_smem(int smem)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && g_tma_smem[dev].load() >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(dequant_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        int cur = g_tma_smem[dev].load();
        while (cur < smem && !g_tma_smem[dev].compare_exchange_weak(cur, smem)) {
        }
    }
    return e;
}

}  // namespace

cudaError_t launch_dequant(const int32_t* cnt, const int32_t* off, int E, int S, int mode, int H,
                           const uint8_t* q, const float* scale, void* y, int64_t max_rows,
                           int sm_count, unsigned* err, cudaStream_t s)
{
    const size_t stage = (size_t)H + H / 32;
    const size_t smem = kStages * stage;
    int per_sm = (int)((200 * 1024) / smem);
    per_sm = per_sm < 1 ? 1 : (per_sm > kTmaPerSm ? kTmaPerSm : per_sm);
    // staging pays once every CTA has rings of rows to stream; a small batch
    // (LL decode) is latency-bound and does better with a warp per row on
    // every SM, leaving shared memory to kernels of other streams
    const bool tma = H % 512 == 0 && ((uintptr_t)q & 15u) == 0 && ((uintptr_t)scale & 15u) == 0 &&
                     smem <= 160 * 1024 && max_rows >= (int64_t)kStages * sm_count * per_sm;
    if (!tma) {
        // one warp per row: no more CTAs than the rows can keep busy
        const int64_t want = (max_rows + kThreads / 32 - 1) / (kThreads / 32);
        const int blocks = (int)(want < 1 ? 1 : (want < sm_count * 8 ? want : sm_count * 8));
        return launch_pdl(dequant_kernel, dim3(blocks), dim3(kThreads), s, cnt, off, E, S, mode,
                          H, (const uint4*)q, scale, (uint4*)y);
    }
    const cudaError_t e = allow_tma_smem((int)smem);
    if (e != cudaSuccess) return e;
    // two vectors of a staged row per thread (the thread count matters little)
    int thr = (H / 16 / 2 + 31) / 32 * 32;
    thr = thr > kTmaMaxThreads ? kTmaMaxThreads : thr;
    return launch_pdl_smem(dequant_tma_kernel, dim3(sm_count * per_sm), dim3(thr), smem, s,
                           cnt, off, E, S, mode, H, q, scale, (uint4*)y, err);
}

}  // namespace moeep
