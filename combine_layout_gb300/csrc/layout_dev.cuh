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

// Shared memory the layout tail needs (ints): partial sums, warp sums,
// per-expert counts and offsets.
constexpr int kTailSmemInts = 1024 + 32 + 2 * (kMaxExperts + 1);

// Sum of the four bytes of w.
__device__ __forceinline__ int byte_sum(uint32_t w) { return (int)__dp4a(w, 0x01010101u, 0u); }

// The last CTA of a layout-producing grid to finish computes, alone, the
// column prefix over tiles, the per-expert counts and the offsets.  Every CTA
// calls this after writing its tile words and per-tile counts; only the CTA
// that arrives last does the work.  No CTA waits on another: the counter only
// tells the CTA that arrives last that all tiles are written.
// The one-byte counts are stored expert-major, tile_cnt[e][tile], so a
// thread reads its run of tiles of one expert in 16-byte vectors, all in
// flight at once; global memory is read once and written once, and
// everything in between stays in shared memory.
__device__ __forceinline__ void finish_layout_if_last(const LayoutArgs& a, int* smem)
{
    // The barrier orders every thread's tile writes before thread 0's
    // GPU-scope fence, which orders them before the arrival count (one fence
    // per CTA: a fence in every thread costs microseconds).
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(a.done, 1u);
        __threadfence();
        s_last = (prev == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;

    const int nthr = blockDim.x, tid = threadIdx.x;
    const int E = a.E, ntiles = a.ntiles;
    int* s_part = smem;                 // [nthr]
    int* s_warp = smem + nthr;          // [32]
    int* s_cnt = s_warp + 32;           // [E]
    int* s_off = s_cnt + kMaxExperts;   // [E + 1]

    // tpc threads share one expert column, each taking a run of rp tiles
    // (a multiple of 16: whole vectors)
    constexpr int kVec = 8;  // 16-byte vectors held in registers (128 tiles)
    int tpc = 1;
    while (tpc * 2 * E <= nthr) tpc *= 2;
    const int cols_per_pass = nthr / tpc;
    const int col_in = tid % cols_per_pass, part = tid / cols_per_pass;
    const int rp = (((ntiles + tpc - 1) / tpc) + 15) & ~15;
    const int r0 = min(part * rp, ntiles), r1 = min(r0 + rp, ntiles);
    const int nv = (r1 - r0 + 15) / 16;
    for (int c0 = 0; c0 < E; c0 += cols_per_pass) {
        const int col = c0 + col_in;
        const bool act = col < E;
        const uint8_t* src = a.tile_cnt + (size_t)col * a.cnt_stride + r0;
        uint4 v[kVec];
        int sum = 0;
        if (act) {
            for (int b0 = 0; b0 < nv; b0 += kVec) {
#pragma unroll
                for (int i = 0; i < kVec; ++i)
                    v[i] = (b0 + i < nv) ? __ldcg(reinterpret_cast<const uint4*>(src) + b0 + i)
                                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int i = 0; i < kVec; ++i) {
                    const int t0 = r0 + 16 * (b0 + i);
                    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int lim = r1 - (t0 + 4 * q);  // bytes of this word that count
                        const uint32_t m = lim >= 4 ? 0xffffffffu : (lim <= 0 ? 0u : (1u << (8 * lim)) - 1u);
                        sum += byte_sum(w[q] & m);
                    }
                }
            }
        }
        s_part[tid] = sum;
        __syncthreads();
        if (act) {
            int run = 0, total = 0;
            for (int q = 0; q < tpc; ++q) {
                const int x = s_part[q * cols_per_pass + col_in];
                if (q < part) run += x;
                total += x;
            }
            for (int b0 = 0; b0 < nv; b0 += kVec) {
                if (nv > kVec) {  // runs longer than the registers hold: read again
#pragma unroll
                    for (int i = 0; i < kVec; ++i)
                        v[i] = (b0 + i < nv) ? __ldcg(reinterpret_cast<const uint4*>(src) + b0 + i)
                                             : make_uint4(0u, 0u, 0u, 0u);
                }
                const int nvb = min(kVec, nv - b0);
#pragma unroll
                for (int i = 0; i < kVec; ++i) {
                    if (i >= nvb) break;  // only the vectors that hold tiles
                    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                    const int t0 = r0 + 16 * (b0 + i);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        if (t0 + q < r1) {
                            a.tile_base[(size_t)(t0 + q) * E + col] = run;
                            run += (int)((w[q >> 2] >> (8 * (q & 3))) & 0xffu);
                        }
                    }
                }
            }
            if (part == 0) s_cnt[col] = total;
        }
        __syncthreads();
    }

    // exclusive prefix of the (padded) counts over experts (shared memory only)
    const int al = a.align;
    const int per = (E + nthr - 1) / nthr;
    const int lo = min(tid * per, E), hi = min(lo + per, E);
    int sum = 0;
    for (int e = lo; e < hi; ++e) sum += (s_cnt[e] + al - 1) / al * al;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        if (lane < nwarps) s_warp[lane] = x;
    }
    __syncthreads();
    int run = incl - sum + (warp > 0 ? s_warp[warp - 1] : 0);
    for (int e = lo; e < hi; ++e) {
        s_off[e] = run;
        run += (s_cnt[e] + al - 1) / al * al;
    }
    if (tid == nthr - 1) s_off[E] = s_warp[nwarps - 1];
    __syncthreads();
    for (int e = tid; e < E; e += nthr) {
        a.cnt[e] = s_cnt[e];
        a.off[e] = s_off[e];
    }
    if (tid == 0) a.off[E] = s_off[E];
    const int L = E / a.R;
    for (int r = tid; r < a.R; r += nthr) {
        int c = 0;
        for (int l = 0; l < L; ++l) c += s_cnt[r * L + l];
        a.roff[r] = s_off[r * L];
        a.rcnt[r] = c;
        if (a.host_out) a.host_out[E + 1 + r] = c;
    }
    if (tid == 0) {
        a.roff[a.R] = s_off[E];
        *a.done = 0u;  // ready for the next launch on this handle
    }
    if (a.host_out) {
        // the host's copy of the counts (one host synchronisation of HT mode
        // waits for these words, not for the rest of the stream)
        for (int e = tid; e <= E; e += nthr) a.host_out[e] = s_off[e];
        for (int e = tid; e < E; e += nthr) a.host_out[E + 1 + a.R + e] = s_cnt[e];
        __syncthreads();
        if (tid == 0) {
            __threadfence_system();
            reinterpret_cast<volatile unsigned*>(a.host_out)[E + 1 + a.R + E] = a.seq;
        }
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
