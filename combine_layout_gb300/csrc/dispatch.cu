// Dispatch pack: every (token, j) pair with a receive row gets a copy of its
// token, as bf16 or as FP8 e4m3 with one fp32 scale per 128 elements.
//
// "NCCL EP 论文解读", item "通信模式": the send phase reads the token, writes it to
// the buffer and quantises in-kernel when FP8 is on.  "NVSHMEM 与 DeepEP：GPU 发起
// 的通信", section "高吞吐模式": dispatch payload FP8 with fine-grained scaling,
// one scale per 128 elements.  Here the "send" to logical rank r is a store
// into rank r's rows of the receive buffer in this GPU's memory.
//
// HBM-bound (read 2H bytes per token, write k rows).  One CTA per token (or
// per column slice of a token: every token of a small batch, the last few
// hundred tokens of a large bf16 batch): its
// threads start reading the token (16-byte vectors, all in flight at once)
// and warp 0 computes the k pair rows from the layout and stores the row map
// (bf16: while the token's loads are in flight; FP8: after its own share of
// the conversion, when the raw vectors no longer hold registers -- 55.7 us
// against 64.8 us on the 4096-token, 7168-wide shape); then the token is
// streamed to the k rows, each row written by the whole CTA in one burst.
// (Measured on the same shape: this beats one warp per token and TMA bulk
// copies through shared memory.)
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "layout_dev.cuh"

namespace moeep {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 128;
constexpr int kUnroll = 8;  // 16-byte vectors per thread per pass (H <= 8192 in one pass)

// CTA 0: the caller's copies of the column counts and offsets; with a
// deferred layout, first the layout's counts and offsets from the tile words
// (the router left that to the first consumer).
template <int NT = kThreads>
__device__ __forceinline__ void copy_counts(const RowArgs& ra, const int32_t* cnt,
                                            int32_t* recv_cnt, const LayoutArgs& fin)
{
    if (fin.deferred) {
        finish_layout_from_words<NT>(fin, recv_cnt);
        return;
    }
    for (int c = threadIdx.x; c <= ra.ncols; c += blockDim.x) {
        if (recv_cnt && c < ra.ncols) recv_cnt[c] = cnt[c];
        if (ra.off_out) ra.off_out[c] = ra.off[c];
    }
}

// Warp 0: rows of token t into s_row; with `write` (the token's first slice)
// also the row map, recv_src and the rank masks.
__device__ __forceinline__ void place_token(const RowArgs& ra, int t, int32_t* row,
                                            int32_t* recv_src, int* s_row, bool write)
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        uint32_t m = 0u;
        const int r = token_pair_row(ra, t, lane, &m);
        if (lane < ra.k) {
            s_row[lane] = r;
            if (write) {
                row[(size_t)t * ra.k + lane] = r;
                if (r >= 0 && recv_src) recv_src[r] = t;
                if (r >= 0 && ra.mask) ra.mask[r] = m;
            }
        }
    }
}

// One CTA per work item: a token's row or one of its equal column slices
// (split: small batches slice every token, so several CTAs share a token's
// rows; large batches slice only the last few hundred tokens, which shortens
// the launch's tail; the grid is exactly one CTA per item).  U vectors per
// thread per pass: the slice's own count where it fits in one pass, so no registers are
// held for vectors a row does not have (fewer registers, more CTAs per SM and
// more of the token rows in flight).  NT threads: 128, or 64 for rows of at
// most 512 vectors (H <= 4096), so that a CTA still holds U = 8 vectors per
// thread and an SM holds as many bytes of token rows in flight as with wider
// rows.  early: x was complete before the layout's producer started, so the
// first pass is read before waiting for that producer (while the router
// finishes the layout).  The token is read with the evict-first policy: it
// is read once, and the L2 it does not take keeps more of the rows just
// written for a consumer that reads them back (4096 x 7168, k = 8: step
// 157.2 -> 156.7 us; 8192 x 4096, k = 2: 65.2 -> 64.1 us).
template <int U, int NT>
__global__ void __launch_bounds__(NT) dispatch_bf16_kernel(
    RowArgs ra, const uint4* __restrict__ x, int nvec, TokenSplit split, int32_t* __restrict__ row,
    uint4* __restrict__ recv_x, int32_t* __restrict__ recv_src, const int32_t* __restrict__ cnt,
    int32_t* __restrict__ recv_cnt, LayoutArgs fin, int early)
{
    __shared__ int s_row[kMaxTopk];
    const bool item = (int)blockIdx.x < split_items(split, ra.T);
    int t = 0, vb = 0, ve = 0;
    if (item) split_item(split, blockIdx.x, nvec, t, vb, ve);
    const uint4* xt = x + (size_t)t * nvec;
    uint4 buf[U];
    auto load = [&](int pass) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = pass + threadIdx.x + u * NT;
            if (v < ve) buf[u] = __ldcs(xt + v);  // read once: evict first
        }
    };
    auto store = [&](int pass) {
        for (int j = 0; j < ra.k; ++j) {
            const int r = s_row[j];
            if (r < 0) continue;
            uint4* dst = recv_x + (size_t)r * nvec;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = pass + threadIdx.x + u * NT;
                if (v < ve) dst[v] = buf[u];
            }
        }
    };
    if (early && item) load(vb);
    griddep_wait();
    if (blockIdx.x == 0) copy_counts<NT>(ra, cnt, recv_cnt, fin);
    if (!item) {
        send_arrive(ra.sig);
        return;
    }
    if (!early) load(vb);
    place_token(ra, t, row, recv_src, s_row, vb == 0);
    __syncthreads();
    store(vb);
    for (int pass = vb + U * NT; pass < ve; pass += U * NT) {  // rows wider than one pass
        load(pass);
        store(pass);
    }
    send_arrive(ra.sig);
}

// FP8 e4m3 of one 16-byte vector of eight bf16 values; a half-warp (16 lanes
// x 8 elements) holds one 128-element block.  All 32 lanes must call it
// (the block maximum is reduced with shuffles).  *scale receives the block's
// scale amax / 448 (1 when the block is all zeros).
__device__ __forceinline__ uint2 quant8(const uint4& raw, float* scale_out)
{
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
    // Quotients rounded to nearest (IEEE) by Markstein's method: with r =
    // RN(1/d), q0 = RN(a*r) is within 1 ulp of a/d and RN(q0 + (a - q0*d)*r)
    // is exactly RN(a/d), the remainder being exact in one fma -- provided
    // nothing overflows or underflows, which 2^-80 <= amax <= 2^100
    // guarantees both for the scale amax / 448 and for every element quotient
    // whose e4m3 code depends on its low bits (smaller quotients all give the
    // code 0).  Other blocks divide directly.
    const bool fast = amax >= 0x1p-80f && amax <= 0x1p+100f;  // uniform per block
    float scale, rs;
    if (fast) {
        constexpr float kR448 = 0x1.24924ap-9f;  // RN(1/448)
        const float s0 = __fmul_rn(amax, kR448);
        scale = __fmaf_rn(__fmaf_rn(-s0, 448.f, amax), kR448, s0);
        rs = __frcp_rn(scale);
    } else {
        scale = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
        rs = 0.f;
    }
    float qt[8];
    if (fast) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float q0 = __fmul_rn(f[i], rs);
            const float rem = __fmaf_rn(-q0, scale, f[i]);
            qt[i] = (f[i] == 0.f) ? f[i] : __fmaf_rn(rem, rs, q0);  // keep the sign of 0
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) qt[i] = __fdiv_rn(f[i], scale);
    }
    uint32_t packed[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(qt[4 * h + 0], qt[4 * h + 1]), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(qt[4 * h + 2], qt[4 * h + 3]), __NV_SATFINITE, __NV_E4M3);
        packed[h] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *scale_out = scale;
    return make_uint2(packed[0], packed[1]);
}

// General FP8 dispatch (any H, multiple of 128): thread i handles vectors
// i + u*128 of each pass of kUnroll*128 vectors.
__global__ void __launch_bounds__(kThreads) dispatch_fp8_kernel(
    RowArgs ra, const uint4* __restrict__ x, int nvec, int nsplit, int32_t* __restrict__ row,
    uint2* __restrict__ recv_q, float* __restrict__ recv_scale, int32_t* __restrict__ recv_src,
    const int32_t* __restrict__ cnt, int32_t* __restrict__ recv_cnt, LayoutArgs fin)
{
    griddep_wait();
    __shared__ int s_row[kMaxTopk];
    if (blockIdx.x == 0) copy_counts(ra, cnt, recv_cnt, fin);
    const int lane = threadIdx.x & 31;
    const int nblk = nvec / 16;
    const int chunk = nvec / nsplit;  // a multiple of 16 vectors: whole 128-blocks
    for (int it = blockIdx.x; it < ra.T * nsplit; it += gridDim.x) {
        const int t = it / nsplit, sl = it - t * nsplit;
        const int vb = sl * chunk, ve = vb + chunk;
        const uint4* xt = x + (size_t)t * nvec;
        // the pass loop is uniform across the CTA (it holds a barrier and
        // half-warp shuffles; lanes past the slice end carry zeros)
        for (int pass = vb; pass < ve; pass += kUnroll * kThreads) {
            const int v0 = pass + threadIdx.x;
            uint4 raw[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * kThreads;
                raw[u] = (v < ve) ? __ldg(xt + v) : make_uint4(0u, 0u, 0u, 0u);
            }
            uint2 q[kUnroll];
            float sc[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) q[u] = quant8(raw[u], &sc[u]);
            if (pass == vb) place_token(ra, t, row, recv_src, s_row, sl == 0);
            __syncthreads();
            for (int j = 0; j < ra.k; ++j) {
                const int r = s_row[j];
                if (r < 0) continue;
                uint2* dst = recv_q + (size_t)r * nvec;
                float* sdst = recv_scale + (size_t)r * nblk;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int v = v0 + u * kThreads;
                    if (v < ve) {
                        dst[v] = q[u];
                        if ((lane & 15) == 0) sdst[v >> 4] = sc[u];
                    }
                }
            }
        }
        __syncthreads();
    }
    send_arrive(ra.sig);
}

// FP8 dispatch for slices of exactly NV * 128 vectors (a row of
// NV * 128 * nsplit vectors, H = 1024 * NV * nsplit): no bounds checks, and
// the slice's NV * 8 scales go through shared memory so every row's scales
// are one coalesced store.
template <int NV>
__global__ void __launch_bounds__(kThreads) dispatch_fp8_fit_kernel(
    RowArgs ra, const uint4* __restrict__ x, int nsplit, int32_t* __restrict__ row,
    uint2* __restrict__ recv_q, float* __restrict__ recv_scale, int32_t* __restrict__ recv_src,
    const int32_t* __restrict__ cnt, int32_t* __restrict__ recv_cnt, LayoutArgs fin)
{
    constexpr int chunk = NV * kThreads, cblk = chunk / 16;
    griddep_wait();
    __shared__ int s_row[kMaxTopk];
    __shared__ float s_sc[cblk];
    if (blockIdx.x == 0) copy_counts(ra, cnt, recv_cnt, fin);
    const int tid = threadIdx.x;
    const int nvec = chunk * nsplit, nblk = cblk * nsplit;
    for (int it = blockIdx.x; it < ra.T * nsplit; it += gridDim.x) {
        const int t = it / nsplit, sl = it - t * nsplit;
        const uint4* xt = x + (size_t)t * nvec + sl * chunk;
        uint4 raw[NV];
#pragma unroll
        for (int u = 0; u < NV; ++u) raw[u] = __ldg(xt + tid + u * kThreads);
        uint2 q[NV];
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            float sc;
            q[u] = quant8(raw[u], &sc);
            if ((tid & 15) == 0) s_sc[(tid + u * kThreads) >> 4] = sc;
        }
        place_token(ra, t, row, recv_src, s_row, sl == 0);
        __syncthreads();
        for (int j = 0; j < ra.k; ++j) {
            const int r = s_row[j];
            if (r < 0) continue;
            uint2* dst = recv_q + (size_t)r * nvec + sl * chunk;
#pragma unroll
            for (int u = 0; u < NV; ++u) dst[tid + u * kThreads] = q[u];
            if (tid < cblk) recv_scale[(size_t)r * nblk + sl * cblk + tid] = s_sc[tid];
        }
        __syncthreads();
    }
    send_arrive(ra.sig);
}

}  // namespace

int slices_for(int T, int units, int sm_count)
{
    if (T <= 0 || units <= 1) return 1;
    const int want = (2 * sm_count + T - 1) / T;  // about two CTAs per SM
    if (want <= 1) return 1;
    for (int d = want; d <= units; ++d)
        if (units % d == 0) return d;
    return units;
}

TokenSplit token_split(int T, int units, int sm_count, int max_slice_units, int min_tokens)
{
    TokenSplit s{T, slices_for(T, units, sm_count), 1};
    if (s.nsa != 1 || units <= max_slice_units || T < min_tokens) return s;
    int d = 2;
    while (d < units && (units % d != 0 || units / d > max_slice_units)) ++d;
    // the tail: an eighth of the tokens, at most three per SM (measured on
    // 4096 x 7168, k = 8: dispatch 82.2 -> 80.1 us with its last 512 tokens
    // in 4 slices, combine 77.0 -> 74.6 us with them in 7)
    int tail = T / 8;
    if (tail > 3 * sm_count) tail = 3 * sm_count;
    s.th = T - tail;
    s.nsb = d;
    return s;
}

cudaError_t launch_dispatch(const RowArgs& ra, const void* x, int H, int fp8, int32_t* row,
                            void* recv_x, float* recv_scale, int32_t* recv_src,
                            const int32_t* cnt, int32_t* recv_cnt, int sm_count, cudaStream_t s,
                            const LayoutArgs* fin_in, int early)
{
    LayoutArgs fin{};
    if (fin_in) fin = *fin_in;
    fin.deferred = fin_in ? 1 : 0;
    const int nvec = H / 8;
    const int T = ra.T < 1 ? 1 : ra.T;
    if (fp8 && nvec % kThreads == 0 && nvec / kThreads <= 8 * 8) {
        const int units = nvec / kThreads;  // 128-vector units of a row
        const int nsplit = slices_for(T, units, sm_count);
        if (units / nsplit <= 8) {
            const int blocks = T * nsplit;
#define MOEEP_FP8_FIT(N)                                                                         \
    case N:                                                                                      \
        return launch_pdl(dispatch_fp8_fit_kernel<N>, dim3(blocks), dim3(kThreads), s, ra,      \
                          (const uint4*)x, nsplit, row, (uint2*)recv_x, recv_scale, recv_src,   \
                          cnt, recv_cnt, fin);
            switch (units / nsplit) {
            MOEEP_FP8_FIT(1)
            MOEEP_FP8_FIT(2)
            MOEEP_FP8_FIT(3)
            MOEEP_FP8_FIT(4)
            MOEEP_FP8_FIT(5)
            MOEEP_FP8_FIT(6)
            MOEEP_FP8_FIT(7)
            MOEEP_FP8_FIT(8)
            }
#undef MOEEP_FP8_FIT
        }
    }
    // 128-element blocks (16 vectors) are the slicing unit of the other kernels
    if (fp8) {
        const int nsplit = (nvec % 16 == 0) ? slices_for(T, nvec / 16, sm_count) : 1;
        return launch_pdl(dispatch_fp8_kernel, dim3(T * nsplit), dim3(kThreads), s, ra,
                          (const uint4*)x, nvec, nsplit, row, (uint2*)recv_x, recv_scale,
                          recv_src, cnt, recv_cnt, fin);
    }
    // bf16: tail slices of at most 256 vectors, from 16 tokens per SM (2048
    // tokens of 7168: 42.7 -> 43.1 us with a sliced tail, 1024: no change).
    // No tokens: one CTA, no item (it still copies the counts and raises a
    // send's signal).
    const TokenSplit split = (ra.T > 0 && nvec % 16 == 0)
                                 ? token_split(ra.T, nvec / 16, sm_count, 16, 16 * sm_count)
                                 : TokenSplit{ra.T > 0 ? ra.T : 0, 1, 1};
    int blocks = split_items(split, ra.T > 0 ? ra.T : 0);
    if (blocks < 1) blocks = 1;
    const int chunk = nvec / split.nsa;
    const bool narrow = chunk <= kUnroll * 64;  // 64 threads of up to 8 vectors
    const int nt = narrow ? 64 : kThreads;
    int per = (chunk + nt - 1) / nt;  // vectors per thread
    per = per < kUnroll ? per : kUnroll;
#define MOEEP_BF16(N, T_)                                                                         \
    return launch_pdl(dispatch_bf16_kernel<N, T_>, dim3(blocks), dim3(T_), s, ra, (const uint4*)x, \
                      nvec, split, row, (uint4*)recv_x, recv_src, cnt, recv_cnt, fin, early)
#define MOEEP_BF16_ALL(T_)           \
    switch (per) {                   \
    case 1: MOEEP_BF16(1, T_);       \
    case 2: MOEEP_BF16(2, T_);       \
    case 3: MOEEP_BF16(3, T_);       \
    case 4: MOEEP_BF16(4, T_);       \
    case 5: MOEEP_BF16(5, T_);       \
    case 6: MOEEP_BF16(6, T_);       \
    case 7: MOEEP_BF16(7, T_);       \
    default: MOEEP_BF16(kUnroll, T_); \
    }
    if (narrow) MOEEP_BF16_ALL(64);
    MOEEP_BF16_ALL(kThreads);
#undef MOEEP_BF16_ALL
#undef MOEEP_BF16
}

}  // namespace moeep
