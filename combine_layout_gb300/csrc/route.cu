// Node-limited (grouped) top-k router and the per-tile expert bitmaps.
//
// Routing follows "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": each node
// (a contiguous group of E/G experts) is scored by the sum of its m best expert
// scores, the best kg nodes are kept, and the k best experts among them are
// chosen.  Ties: the larger score wins; on equal scores the lower index wins
// (nodes and experts alike).  Group sums are formed in binary64 (the sum of
// two fp32 scores is exact there), so node decisions do not depend on fp32
// rounding of the sum.  NaN scores rank as -infinity.
//
// Work split: one warp per token, one CTA per 32-token tile.  Lane l holds up
// to `epl` consecutive experts of group l / lpg, so a group's experts live in
// lpg adjacent lanes and its top-m merges in log2(lpg) butterfly steps.
#include <limits.h>
#include <math.h>

#include "common.cuh"

namespace moeep {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int M>
__device__ __forceinline__ void insert_desc(float (&t)[M], float x)
{
#pragma unroll
    for (int q = 0; q < M; ++q) {
        if (x > t[q]) {
            float o = t[q];
            t[q] = x;
            x = o;
        }
    }
}

// (value, index) ordering: larger value first, lower index on ties.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

template <int EPL>
__device__ __forceinline__ void route_token(const float* __restrict__ s, const RouteParams& p,
                                            int lane, int& out_idx, float& out_w)
{
    const int grp = lane >> p.lpg_log2;
    const int sub = lane & (p.lpg - 1);
    const int first = sub * p.epl;           // offset of my first expert inside the group
    const int base = grp * p.gs + first;     // global id of my first expert

    float v[EPL];
    uint32_t inr = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const bool in = (grp < p.G) && (i < p.epl) && (first + i < p.gs);
        const float x = in ? __ldg(s + base + i) : -INFINITY;
        v[i] = isnan(x) ? -INFINITY : x;  // a NaN score ranks below every number
        if (in) inr |= 1u << i;
    }

    uint32_t ok = inr;
    if (p.limit) {
        float top[kMaxGroupTopk];
#pragma unroll
        for (int q = 0; q < kMaxGroupTopk; ++q) top[q] = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if ((inr >> i) & 1u) insert_desc(top, v[i]);
        for (int o = 1; o < p.lpg; o <<= 1) {
            float oth[kMaxGroupTopk];
#pragma unroll
            for (int q = 0; q < kMaxGroupTopk; ++q) oth[q] = __shfl_xor_sync(kFull, top[q], o);
#pragma unroll
            for (int q = 0; q < kMaxGroupTopk; ++q) insert_desc(top, oth[q]);
        }
        // the group's m best, summed in ascending order in binary64
        double gsum = 0.0;
#pragma unroll
        for (int q = kMaxGroupTopk - 1; q >= 0; --q)
            if (q < p.m) gsum += (double)top[q];
        int rank = 0;
        for (int n = 0; n < p.G; ++n) {
            const double o = __shfl_sync(kFull, gsum, n << p.lpg_log2);
            if (o > gsum || (o == gsum && n < grp)) ++rank;
        }
        if (rank >= p.kg) ok = 0;
    }

    // k rounds of warp arg-max; lane j keeps the j-th pick
    int my_i = 0;
    float my_v = 0.f;
    for (int j = 0; j < p.k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (((ok >> i) & 1u) && better(v[i], base + i, bv, bi)) {
                bv = v[i];
                bi = base + i;
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, o);
            const int oi = __shfl_xor_sync(kFull, bi, o);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        const int iw = bi - base;
        if (iw >= 0 && iw < EPL && ((ok >> iw) & 1u)) ok &= ~(1u << iw);
        if (lane == j) {
            my_i = (bi == INT_MAX) ? -1 : bi;  // unreachable while kg * gs >= k
            my_v = bv;
        }
    }

    const bool act = lane < p.k;
    float w;
    if (p.wmode == MOE_EP_W_SCORE_NORM) {
        float den = 0.f;
        for (int j = 0; j < p.k; ++j) den += __shfl_sync(kFull, my_v, j);
        w = __fdiv_rn(my_v, den);
    } else if (p.wmode == MOE_EP_W_SOFTMAX_TOPK) {
        const float mx = __shfl_sync(kFull, my_v, 0);
        const float ex = act ? expf(my_v - mx) : 0.f;
        float den = 0.f;
        for (int j = 0; j < p.k; ++j) den += __shfl_sync(kFull, ex, j);
        w = __fdiv_rn(ex, den);
    } else {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if ((inr >> i) & 1u) mx = fmaxf(mx, v[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if ((inr >> i) & 1u) z += expf(v[i] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(kFull, z, o);
        const float pj = act ? __fdiv_rn(expf(my_v - mx), z) : 0.f;
        float sel = 0.f;
        for (int j = 0; j < p.k; ++j) sel += __shfl_sync(kFull, pj, j);
        w = __fdiv_rn(pj, sel);
    }
    out_idx = my_i;
    out_w = w;
}

template <int EPL>
__global__ void __launch_bounds__(1024) route_kernel(const float* __restrict__ scores, int T,
                                                     RouteParams p, int32_t* __restrict__ topk_idx,
                                                     float* __restrict__ topk_w,
                                                     uint32_t* __restrict__ tile_word)
{
    extern __shared__ uint32_t s_word[];  // [E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < p.E; e += blockDim.x) s_word[e] = 0u;
    __syncthreads();

    const int tile = blockIdx.x;
    const int t = tile * kTileTokens + warp;
    if (t < T) {
        int e;
        float w;
        route_token<EPL>(scores + (size_t)t * p.E, p, lane, e, w);
        if (lane < p.k) {
            topk_idx[(size_t)t * p.k + lane] = e;
            if (topk_w) topk_w[(size_t)t * p.k + lane] = w;
            if (e >= 0) atomicOr(&s_word[e], 1u << warp);
        }
    }
    __syncthreads();
    for (int e = tid; e < p.E; e += blockDim.x) tile_word[(size_t)tile * p.E + e] = s_word[e];
}

__global__ void __launch_bounds__(256) layout_bits_kernel(const int32_t* __restrict__ topk_idx,
                                                          int T, int k, int E,
                                                          uint32_t* __restrict__ tile_word,
                                                          volatile unsigned* err)
{
    extern __shared__ uint32_t s_word[];  // [E]
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) s_word[e] = 0u;
    __syncthreads();
    const int tile = blockIdx.x;
    const int t0 = tile * kTileTokens;
    const int nt = min(kTileTokens, T - t0);
    for (int q = tid; q < nt * k; q += blockDim.x) {
        const int tl = q / k, j = q - tl * k;
        const int32_t* r = topk_idx + (size_t)(t0 + tl) * k;
        const int e = r[j];
        if (e == -1) continue;
        if (e < -1 || e >= E) {
            err[kErrRange] = 1u;
            continue;
        }
        bool dup = false;
        for (int jj = 0; jj < j; ++jj) dup |= (r[jj] == e);
        if (dup) {
            err[kErrDuplicate] = 1u;
            continue;
        }
        atomicOr(&s_word[e], 1u << tl);
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) tile_word[(size_t)tile * E + e] = s_word[e];
}

}  // namespace

cudaError_t launch_route(const float* scores, int T, const RouteParams& p, int32_t* topk_idx,
                         float* topk_w, uint32_t* tile_word, cudaStream_t s)
{
    if (T <= 0) return cudaSuccess;
    const int ntiles = (T + kTileTokens - 1) / kTileTokens;
    const size_t smem = sizeof(uint32_t) * (size_t)p.E;
    if (p.epl <= 1)
        route_kernel<1><<<ntiles, 1024, smem, s>>>(scores, T, p, topk_idx, topk_w, tile_word);
    else if (p.epl <= 2)
        route_kernel<2><<<ntiles, 1024, smem, s>>>(scores, T, p, topk_idx, topk_w, tile_word);
    else if (p.epl <= 4)
        route_kernel<4><<<ntiles, 1024, smem, s>>>(scores, T, p, topk_idx, topk_w, tile_word);
    else if (p.epl <= 8)
        route_kernel<8><<<ntiles, 1024, smem, s>>>(scores, T, p, topk_idx, topk_w, tile_word);
    else
        route_kernel<16><<<ntiles, 1024, smem, s>>>(scores, T, p, topk_idx, topk_w, tile_word);
    return cudaGetLastError();
}

cudaError_t launch_layout_bits(const int32_t* topk_idx, int T, int k, int E, uint32_t* tile_word,
                               volatile unsigned* err, cudaStream_t s)
{
    if (T <= 0) return cudaSuccess;
    const int ntiles = (T + kTileTokens - 1) / kTileTokens;
    layout_bits_kernel<<<ntiles, 256, sizeof(uint32_t) * (size_t)E, s>>>(topk_idx, T, k, E,
                                                                          tile_word, err);
    return cudaGetLastError();
}

}  // namespace moeep
