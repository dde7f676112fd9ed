// Device-side pieces of the per-expert counting and prefix layout, shared by
// the router / bitmap kernels (which finish the layout) and by the kernels
// that place pairs into receive rows (dispatch, row map).
//
// "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": count the tokens bound
// for every rank and every expert.  "NCCL EP 论文解读", item "算法模式": HT output
// in deterministic order with per-expert counts marking the boundaries;
// "低延迟模式" on the DeepEP page: fixed slots per (rank, local expert).
//
// Representation: tokens are grouped in tiles of 32; word tile_word[tile][e]
// has bit i set when token tile*32 + i chose expert e.  Then
//   cnt[e]            = sum over tiles of popc(word)
//   tile_base[tile][e] = pairs of expert e in earlier tiles
//   rank(t, e)         = tile_base[t/32][e] + popc(word & bits below t%32)
// is the number of earlier tokens that chose e, i.e. the stable in-expert rank.
#pragma once

#include "common.cuh"

namespace moeep {

// The last CTA of a layout-producing grid to finish computes, alone, the
// column prefix over tiles, the per-expert counts and the offsets.  Every CTA
// calls this after writing its tile words; only the last one returns true
// after doing the work.  No CTA waits on another: the counter only tells the
// CTA that arrives last that all words are written.
__device__ __forceinline__ void finish_layout_if_last(const LayoutArgs& a, int* s_scratch /*>= blockDim.x + 32 ints*/)
{
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(a.done, 1u) == gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    const int nthr = blockDim.x, tid = threadIdx.x;
    const int E = a.E, ntiles = a.ntiles;
    // tpc threads share one expert column, each scanning a contiguous run of
    // tiles; consecutive threads take consecutive columns (coalesced loads),
    // and each thread keeps kBatch independent loads in flight.
    constexpr int kBatch = 16;
    int tpc = 1;
    while (tpc * 2 * E <= nthr) tpc *= 2;
    const int cols_per_pass = nthr / tpc;
    const int col_in = tid % cols_per_pass, part = tid / cols_per_pass;
    const int rp = (ntiles + tpc - 1) / tpc;
    const int r0 = min(part * rp, ntiles), r1 = min(r0 + rp, ntiles);
    for (int c0 = 0; c0 < E; c0 += cols_per_pass) {
        const int col = c0 + col_in;
        const bool act = col < E && part < tpc;
        int sum = 0;
        if (act)
            for (int rb = r0; rb < r1; rb += kBatch) {
                uint32_t w[kBatch];
#pragma unroll
                for (int q = 0; q < kBatch; ++q)
                    w[q] = (rb + q < r1) ? __ldcg(a.tile_word + (size_t)(rb + q) * E + col) : 0u;
#pragma unroll
                for (int q = 0; q < kBatch; ++q) sum += __popc(w[q]);
            }
        s_scratch[tid] = sum;
        __syncthreads();
        if (act) {
            int base = 0, total = 0;
            for (int q = 0; q < tpc; ++q) {
                const int v = s_scratch[q * cols_per_pass + col_in];
                if (q < part) base += v;
                total += v;
            }
            int run = base;
            for (int rb = r0; rb < r1; rb += kBatch) {
                uint32_t w[kBatch];
#pragma unroll
                for (int q = 0; q < kBatch; ++q)
                    w[q] = (rb + q < r1) ? __ldcg(a.tile_word + (size_t)(rb + q) * E + col) : 0u;
#pragma unroll
                for (int q = 0; q < kBatch; ++q) {
                    if (rb + q < r1) a.tile_base[(size_t)(rb + q) * E + col] = run;
                    run += __popc(w[q]);
                }
            }
            if (part == 0) a.cnt[col] = total;
        }
        __syncthreads();
    }

    // exclusive prefix of cnt over experts -> off; per-rank sums
    const int per = (E + nthr - 1) / nthr;
    const int lo = min(tid * per, E), hi = min(lo + per, E);
    int sum = 0;
    for (int e = lo; e < hi; ++e) sum += a.cnt[e];
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    int* s_warp = s_scratch + nthr;
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane < nwarps) s_warp[lane] = v;
    }
    __syncthreads();
    int run = incl - sum + (warp > 0 ? s_warp[warp - 1] : 0);
    for (int e = lo; e < hi; ++e) {
        a.off[e] = run;
        run += a.cnt[e];
    }
    if (tid == nthr - 1) a.off[E] = s_warp[nwarps - 1];
    __syncthreads();
    const int L = E / a.R;
    for (int r = tid; r < a.R; r += nthr) {
        a.roff[r] = a.off[r * L];
        a.rcnt[r] = a.off[(r + 1) * L] - a.off[r * L];
    }
    if (tid == 0) {
        a.roff[a.R] = a.off[E];
        *a.done = 0u;  // ready for the next launch on this handle
    }
}

// Receive row of pair (t, lane) for lanes < k of a warp (-1 for lanes >= k and
// for pairs without a row).  All 32 lanes must call it (warp-collective).
// Invalid pairs -- id outside [0, E), or an expert repeated at an earlier j of
// the same token -- get -1.
__device__ __forceinline__ int token_pair_row(const RowArgs& a, int t, int lane)
{
    int e = -2 - lane;  // lanes >= k: distinct values that match nothing
    if (lane < a.k) e = __ldg(a.idx + (size_t)t * a.k + lane);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const bool dup = (peers & ((1u << lane) - 1u)) != 0u;
    if (lane >= a.k || e < 0 || e >= a.E || dup) return -1;
    const size_t q = (size_t)(t >> 5) * a.E + e;
    const int rank = __ldg(a.tile_base + q) + __popc(__ldg(a.tile_word + q) & ((1u << (t & 31)) - 1u));
    return (a.mode == MOE_EP_HT) ? __ldg(a.off + e) + rank : e * a.S + rank;
}

}  // namespace moeep
