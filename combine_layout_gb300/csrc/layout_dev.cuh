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
// has bit i set when token tile*32 + i chose expert e.  Tiles are grouped 16
// at a time, and the byte counts popc(word) of one expert in one group form
// one 16-byte vector: tile_cnt[g][e][j] = popc(tile_word[16g + j][e]).  Then
//   cnt[e]           = sum of expert e's byte counts
//   grp_base[g][e]   = pairs of expert e in the groups before g
//   rank(t, e)       = grp_base[g][e] + sum of tile_cnt[g][e][0 .. j)
//                      + popc(word & bits below t%32),   tile = t/32 = 16g + j,
// is the number of earlier tokens that chose e, i.e. the stable in-expert rank.
// The last CTA of the producing grid writes E bases per 512 tokens (not per
// 32): one CTA's work is the serial part of the layout.
#pragma once

#include "common.cuh"

namespace moeep {

// Shared memory the layout tail needs (ints): per-part sums, warp sums,
// per-expert counts and offsets.
constexpr int kTailSmemInts = 1024 + 32 + 2 * kMaxExperts;

// Byte offset of tile `tile`'s count for column c (ncols columns).
__device__ __forceinline__ size_t tile_cnt_index(int tile, int c, int ncols)
{
    return ((size_t)(tile / kGroupTiles) * ncols + c) * kGroupTiles + (tile % kGroupTiles);
}

// Sum of the four bytes of w.
__device__ __forceinline__ int byte_sum(uint32_t w) { return (int)__dp4a(w, 0x01010101u, 0u); }

// Mask of the low n bytes of a word (n clamped to [0, 4]).
__device__ __forceinline__ uint32_t low_bytes(int n)
{
    return n >= 4 ? 0xffffffffu : (n <= 0 ? 0u : (1u << (8 * n)) - 1u);
}

// Sum of the first n of the 16 bytes in v.
__device__ __forceinline__ int vec_byte_sum(const uint4& v, int n)
{
    if (n >= 16) {
        const unsigned ones = 0x01010101u;
        return (int)__dp4a(v.w, ones, __dp4a(v.z, ones, __dp4a(v.y, ones, __dp4a(v.x, ones, 0u))));
    }
    return byte_sum(v.x & low_bytes(n)) + byte_sum(v.y & low_bytes(n - 4)) +
           byte_sum(v.z & low_bytes(n - 8)) + byte_sum(v.w & low_bytes(n - 12));
}

// Pairs of column c (an expert, or a node) in the tiles before `tile`.
__device__ __forceinline__ int pairs_before_tile(const uint8_t* tile_cnt, const int32_t* grp_base,
                                                 int ncols, int c, int tile)
{
    const int g = tile / kGroupTiles;
    const size_t q = (size_t)g * ncols + c;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(tile_cnt) + q);
    return __ldg(grp_base + q) + vec_byte_sum(v, tile - g * kGroupTiles);
}

// Vectors (groups) a thread of the last CTA keeps in flight.
constexpr int kTailVec = 8;

// The last CTA's work split for a launch of nthr threads per CTA (host side).
// A column (expert) is split into parts only when it has more than kTailVec
// groups; only as many warps as the work needs take part.
inline LayoutArgs tail_planned(LayoutArgs a, int nthr)
{
    const int ngroups = (a.ntiles + kGroupTiles - 1) / kGroupTiles;
    a.L = a.E / a.R;
    a.cols = a.E < nthr ? a.E : nthr;
    int parts = (ngroups + kTailVec - 1) / kTailVec;
    if (parts > nthr / a.cols) parts = nthr / a.cols;
    a.parts = parts < 1 ? 1 : parts;
    a.rg = (ngroups + a.parts - 1) / a.parts;
    a.per = (a.E + nthr - 1) / nthr;
    a.nact = ((a.E + a.per - 1) / a.per + 31) & ~31;
    const int ncol = (a.parts * a.cols + 31) & ~31;
    a.nwork = ncol > a.nact ? ncol : a.nact;
    return a;
}

// Byte counts of group g of column col from the tile words (tiles past
// ntiles count 0), stored to tile_cnt for the consumers.
__device__ __forceinline__ uint4 counts_from_words(const LayoutArgs& a, int g, int col)
{
    uint32_t c[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < kGroupTiles; ++j) {
        const int tile = g * kGroupTiles + j;
        const uint32_t w = tile < a.ntiles ? __ldcg(a.tile_word + (size_t)tile * a.E + col) : 0u;
        c[j >> 2] |= (uint32_t)__popc(w) << (8 * (j & 3));
    }
    const uint4 v = make_uint4(c[0], c[1], c[2], c[3]);
    reinterpret_cast<uint4*>(a.tile_cnt)[(size_t)g * a.E + col] = v;
    return v;
}

// Padded size of an expert block of c rows.
__device__ __forceinline__ int padded(int c, int align)
{
    return align == 1 ? c : (c + align - 1) / align * align;
}

// The last CTA of a layout-producing grid to finish computes, alone, the
// group bases (column prefix over groups of 16 tiles), the per-expert counts
// and the offsets.  Every CTA calls this after writing its tile words and
// per-tile counts; only the CTA that arrives last does the work.  No CTA waits
// on another: the counter only tells the CTA that arrives last that all tiles
// are written.
// The group vectors of consecutive experts are adjacent, so a warp's loads
// are contiguous; each thread keeps up to kTailVec groups in flight.  Only
// the first nwork threads (whole warps) go on: every warp of a 1024-thread
// CTA running the tail would cost 32 warps' issue slots per instruction of a
// serial chain.
__device__ __forceinline__ void finish_layout_if_last(const LayoutArgs& a, int* smem)
{
    // The barrier orders every thread's tile writes before thread 0's
    // arrival, an atomic add with release semantics at GPU scope; its acquire
    // side, with the barrier after it, orders the last CTA's reads after every
    // other CTA's writes.
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(a.done)
                     : "memory");
        s_last = (prev == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    const int tid = threadIdx.x, nwork = a.nwork;
    if (!s_last || tid >= nwork) return;

    const int E = a.E, ntiles = a.ntiles;
    const int ngroups = (ntiles + kGroupTiles - 1) / kGroupTiles;
    int* s_part = smem;                 // [nwork]
    int* s_warp = smem + 1024;          // [32]
    int* s_cnt = s_warp + 32;           // [E]
    int* s_off = s_cnt + kMaxExperts;   // [E]

    // Column pass: `parts` runs of rg consecutive groups per column; thread
    // (part, col) = (tid / cols, tid % cols).
    const int cols = a.cols, parts = a.parts, rg = a.rg;
    const int part = tid / cols, col_in = tid - part * cols;
    const int g0 = min(part * rg, ngroups), g1 = min(g0 + rg, ngroups);
    const uint4* vec = reinterpret_cast<const uint4*>(a.tile_cnt);
    for (int c0 = 0; c0 < E; c0 += cols) {
        const int col = c0 + col_in;
        const bool act = part < parts && col < E;
        int gs[kTailVec];
        int sum = 0;
        if (act && a.cnt_from_words) {  // at most two groups, one run
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                gs[i] = 0;
                if (g0 + i < g1)
                    gs[i] = vec_byte_sum(counts_from_words(a, g0 + i, col),
                                         ntiles - (g0 + i) * kGroupTiles);
                sum += gs[i];
            }
        } else if (act) {
            for (int b = g0; b < g1; b += kTailVec) {
                uint4 v[kTailVec];
#pragma unroll
                for (int i = 0; i < kTailVec; ++i)
                    v[i] = (b + i < g1) ? __ldcg(vec + (size_t)(b + i) * E + col)
                                        : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int i = 0; i < kTailVec; ++i) {
                    gs[i] = vec_byte_sum(v[i], ntiles - (b + i) * kGroupTiles);
                    sum += gs[i];
                }
            }
        }
        int run = 0, total = sum;
        if (parts > 1) {
            s_part[tid] = sum;
            asm volatile("bar.sync 1, %0;" ::"r"(nwork) : "memory");
            total = 0;
            for (int q = 0; q < parts; ++q) {
                const int x = s_part[q * cols + col_in];
                run += q < part ? x : 0;
                total += x;
            }
        }
        if (act) {
            for (int b = g0; b < g1; b += kTailVec) {
                if (g1 - g0 > kTailVec) {  // runs longer than the registers hold: read again
                    uint4 v[kTailVec];
#pragma unroll
                    for (int i = 0; i < kTailVec; ++i)
                        v[i] = (b + i < g1) ? __ldcg(vec + (size_t)(b + i) * E + col)
                                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int i = 0; i < kTailVec; ++i)
                        gs[i] = vec_byte_sum(v[i], ntiles - (b + i) * kGroupTiles);
                }
#pragma unroll
                for (int i = 0; i < kTailVec; ++i) {
                    if (b + i < g1) {
                        a.grp_base[(size_t)(b + i) * E + col] = run;
                        run += gs[i];
                    }
                }
            }
            if (part == 0) s_cnt[col] = total;
        }
        if (parts > 1) asm volatile("bar.sync 1, %0;" ::"r"(nwork) : "memory");
    }
    asm volatile("bar.sync 1, %0;" ::"r"(nwork) : "memory");

    // Prefix of the padded counts over experts: `per` consecutive experts per
    // thread, on the first nact threads (whole warps).
    const int per = a.per, nact = a.nact;
    const int al = a.align, L = a.L;
    const int lo = min(tid * per, E), hi = min(lo + per, E);
    const bool pre = tid < nact;
    int sum = 0, incl = 0;
    const int lane = tid & 31, warp = tid >> 5;
    if (pre) {
        for (int e = lo; e < hi; ++e) sum += padded(s_cnt[e], al);
        incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) s_warp[warp] = incl;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(nwork) : "memory");
    int32_t* const host = a.host_out;
    if (pre) {
        int run = incl - sum;
        for (int w = 0; w < warp; ++w) run += s_warp[w];
        for (int e = lo; e < hi; ++e) {
            const int c = s_cnt[e];
            a.cnt[e] = c;
            a.off[e] = run;
            s_off[e] = run;
            if (host) {
                host[e] = run;
                host[E + 1 + a.R + e] = c;
            }
            run += padded(c, al);
        }
        if (lo < E && hi == E) {  // the thread holding the last expert: the totals
            a.off[E] = run;
            a.roff[a.R] = run;
            if (host) host[E] = run;
        }
    }
    if (tid == 0) *a.done = 0u;  // ready for the next launch on this handle
    asm volatile("bar.sync 1, %0;" ::"r"(nwork) : "memory");
    for (int r = tid; r < a.R; r += nwork) {
        int c = 0;
        for (int l = 0; l < L; ++l) c += s_cnt[r * L + l];
        a.rcnt[r] = c;
        a.roff[r] = s_off[r * L];
        if (host) host[E + 1 + r] = c;
    }
    if (host) {
        // the host's copy of the counts (one host synchronisation of HT mode
        // waits for these words, not for the rest of the stream)
        asm volatile("bar.sync 1, %0;" ::"r"(nwork) : "memory");
        if (tid == 0) {
            __threadfence_system();
            reinterpret_cast<volatile unsigned*>(host)[E + 1 + a.R + E] = a.seq;
        }
    }
}

// Deferred LL layout (LayoutArgs.deferred: a few tiles, no padding),
// finished by one CTA of NT threads from the tile words alone:
// cnt[e] = sum over tiles of popc(word), off = exclusive prefix, rank counts
// and offsets from the expert offsets, recv_cnt (may be null) = cnt.  All
// NT threads of the CTA must call it (it holds barriers).  The words are
// spread over the threads, 8 loads in flight each, and summed per expert in
// shared memory: few registers, since the dispatch kernels inline this into
// their first CTA.
template <int NT>
__device__ __forceinline__ void finish_layout_from_words(const LayoutArgs& a, int32_t* recv_cnt)
{
    static_assert(NT % 32 == 0, "block size");
    constexpr int kU = 8;
    __shared__ int s_warp[NT / 32];
    __shared__ int s_cnt[kMaxExperts + 1];  // counts, then (in place) offsets
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = a.E;
    for (int e = tid; e < E; e += NT) s_cnt[e] = 0;
    __syncthreads();
    const int nw = a.ntiles * E;
    for (int q0 = tid; q0 < nw; q0 += NT * kU) {
        uint32_t w[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int q = q0 + u * NT;
            w[u] = q < nw ? __ldcg(a.tile_word + q) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int q = q0 + u * NT;
            if (q < nw && w[u]) atomicAdd(&s_cnt[q - (q / E) * E], __popc(w[u]));
        }
    }
    __syncthreads();
    const int per = (E + NT - 1) / NT;
    const int lo = min(tid * per, E), hi = min(lo + per, E);
    int sum = 0;
    for (int e = lo; e < hi; ++e) sum += s_cnt[e];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += s_warp[w];
    for (int e = lo; e < hi; ++e) {
        const int c = s_cnt[e];
        a.cnt[e] = c;
        a.off[e] = run;
        if (recv_cnt) recv_cnt[e] = c;
        s_cnt[e] = run;  // this thread's own experts: offsets in place of counts
        run += c;
    }
    if (lo < E && hi == E) {  // the thread holding the last expert: the total
        a.off[E] = run;
        s_cnt[E] = run;
    }
    __syncthreads();
    const int L = E / a.R;
    for (int r = tid; r <= a.R; r += NT) {
        a.roff[r] = s_cnt[r * L];
        if (r < a.R) a.rcnt[r] = s_cnt[(r + 1) * L] - s_cnt[r * L];
    }
}

// Receive row of pair (t, lane) for lanes < k of a warp (-1 for lanes >= k and
// for pairs without a row).  All 32 lanes must call it (warp-collective).
// Invalid pairs -- id outside [0, E), or an expert repeated at an earlier j of
// the same token -- get -1.  With G > 1 experts per column only the token's
// first valid pair in each column gets the row, and *mask receives the bits
// e % G of all the token's valid experts in that column.
__device__ __forceinline__ int token_pair_row(const RowArgs& a, int t, int lane, uint32_t* mask)
{
    const unsigned full = 0xffffffffu, lower = (1u << lane) - 1u;
    int e = -2 - lane;  // lanes >= k: distinct values that match nothing
    if (lane < a.k) e = __ldg(a.idx + (size_t)t * a.k + lane);
    const unsigned peers = __match_any_sync(full, e);
    const bool valid = lane < a.k && e >= 0 && e < a.E && (peers & lower) == 0u;
    int col = e;
    uint32_t m = 1u;
    if (a.G > 1) {  // warp-uniform
        col = valid ? e / a.G : -100 - lane;
        const unsigned cpeers = __match_any_sync(full, col);
        const uint32_t bit = valid ? 1u << (e - col * a.G) : 0u;
        m = 0u;
        for (int j = 0; j < a.k; ++j) {
            const uint32_t b = __shfl_sync(full, bit, j);
            if ((cpeers >> j) & 1u) m |= b;
        }
        if ((cpeers & lower) != 0u) return -1;  // a lower lane holds this column
    }
    *mask = m;
    if (!valid) return -1;
    const int tile = t / kTileTokens;
    int rank = __popc(__ldg(a.tile_word + (size_t)tile * a.ncols + col) & ((1u << (t & 31)) - 1u));
    if (a.from_words) {  // a few tiles: the earlier tiles' words, two loads in flight
#pragma unroll 2
        for (int tl = 0; tl < tile; ++tl)
            rank += __popc(__ldg(a.tile_word + (size_t)tl * a.ncols + col));
    } else {
        rank += pairs_before_tile(a.tile_cnt, a.grp_base, a.ncols, col, tile);
    }
    return (a.mode == MOE_EP_HT) ? __ldg(a.off + col) + rank : col * a.S + rank;
}

}  // namespace moeep
