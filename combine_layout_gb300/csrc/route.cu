// Node-limited (grouped) top-k router and the per-tile expert bitmaps.
//
// Routing follows "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": each node
// (a contiguous group of E/G experts) is scored by the sum of its m best expert
// scores, the best kg nodes are kept, and the k best experts among them are
// chosen, best first.  Ties: the larger score wins; on equal scores the lower
// index wins (nodes and experts alike).  Nodes are ranked by the exact sum of
// their m best scores: for m <= 2 an fp32 two-sum holds it exactly as a
// (hi, lo) pair, compared as one ordered 64-bit key (binary64 for larger m).
// NaN scores and NaN sums (inf + -inf) rank as -infinity; -0 equals +0.
// Scores are expected below 2^126 in magnitude, so a two-score sum cannot
// overflow fp32.
//
// Work split: one warp per token, one CTA per 32-token tile (batches up to
// 1024 tokens: four CTAs of 8 tokens per tile, so more SMs share the
// issue-bound selection; 16 experts or fewer without a node limit: 2 or 4
// tokens per warp, route_small_kernel).  The grid's last CTA finishes the layout, except
// for a deferred LL layout (at most 256 tokens), which the dispatch's first
// CTA finishes from the tile words.  Lane l holds up
// to `epl` consecutive experts of group l / lpg, so a group's experts live in
// lpg adjacent lanes and its top-m merges in log2(lpg) butterfly steps.  Each
// of the k picks is two warp reductions (redux.sync): the largest score key,
// then the lowest expert index holding it.  Scores are compared as
// order-preserving 32-bit keys (0 is below every score: "no candidate").
#include <limits.h>
#include <math.h>

#include "layout_dev.cuh"

namespace moeep {
namespace {

constexpr unsigned kFull = 0xffffffffu;
// Batches up to this many tokens (32 tiles, two groups of byte counts) are
// routed 8 tokens per CTA.
constexpr int kSplitMaxTokens = 1024;

__device__ __forceinline__ uint32_t score_key(float x)
{
    // fmaxf returns the other operand for a NaN (so NaN -> -inf); adding +0
    // turns -0 into +0 (round to nearest) and leaves every other value alone
    x = __fadd_rn(fmaxf(x, -INFINITY), 0.f);
    const uint32_t u = __float_as_uint(x);
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ uint64_t sum_key(double d)
{
    if (isnan(d)) d = -INFINITY;
    const uint64_t u = (uint64_t)__double_as_longlong(d);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

template <int M>
__device__ __forceinline__ void insert_desc(uint32_t (&t)[M], uint32_t x)
{
#pragma unroll
    for (int q = 0; q < M; ++q) {
        const uint32_t hi = max(t[q], x), lo = min(t[q], x);
        t[q] = hi;
        x = lo;
    }
}

// Compare-exchange on (key desc, index asc): afterwards slot a holds the better.
__device__ __forceinline__ void cx(uint32_t& ka, int& ia, uint32_t& kb, int& ib)
{
    const bool sw = kb > ka || (kb == ka && ib < ia);
    const uint32_t k0 = sw ? kb : ka, k1 = sw ? ka : kb;
    const int i0 = sw ? ib : ia, i1 = sw ? ia : ib;
    ka = k0;
    kb = k1;
    ia = i0;
    ib = i1;
}

// Sort a lane's candidates best first.  Eight and four: the optimal 19- and
// 5-comparator networks; other sizes: odd-even transposition (EPL rounds).
template <int EPL>
__device__ __forceinline__ void sort_desc(uint32_t (&k)[EPL], int (&ix)[EPL])
{
    if constexpr (EPL == 4) {
        constexpr int net[5][2] = {{0, 1}, {2, 3}, {0, 2}, {1, 3}, {1, 2}};
#pragma unroll
        for (int c = 0; c < 5; ++c) cx(k[net[c][0]], ix[net[c][0]], k[net[c][1]], ix[net[c][1]]);
    } else if constexpr (EPL == 8) {
        constexpr int net[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6},
                                    {3, 7}, {0, 1}, {2, 3}, {4, 5}, {6, 7}, {2, 4}, {3, 5},
                                    {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
        for (int c = 0; c < 19; ++c) cx(k[net[c][0]], ix[net[c][0]], k[net[c][1]], ix[net[c][1]]);
    } else {
#pragma unroll
        for (int r = 0; r < EPL; ++r)
#pragma unroll
            for (int i = r & 1; i + 1 < EPL; i += 2) cx(k[i], ix[i], k[i + 1], ix[i + 1]);
    }
}

// k picks from lane-sorted candidate lists: each pick is the largest head key
// of the warp, then the lowest expert index holding it; the winning lane pops
// its head.  Lane j keeps pick j; den sums the picked scores in pick order.
template <int N>
__device__ __forceinline__ void pick_k(uint32_t (&key)[N], int (&ix)[N], int k, int lane,
                                       int& my_i, uint32_t& my_k, uint32_t& first_k, float& den)
{
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
        const uint32_t hk = key[0];
        const uint32_t mk = __reduce_max_sync(kFull, hk);
        const uint32_t wi = __reduce_min_sync(kFull, (hk == mk) ? (uint32_t)ix[0] : 0xffffffffu);
        const bool found = mk != 0u;
        if (found && hk == mk && (uint32_t)ix[0] == wi) {
#pragma unroll
            for (int i = 0; i + 1 < N; ++i) {
                key[i] = key[i + 1];
                ix[i] = ix[i + 1];
            }
            key[N - 1] = 0u;
        }
        if (lane == j) {
            my_i = found ? (int)wi : -1;  // not found is unreachable while kg * gs >= k
            my_k = mk;
        }
        if (j == 0) first_k = mk;
        den += key_score(mk);
    }
}

// REDIST: the node-limited routing of 256 experts in 8 groups of 32 with 4
// groups kept and the top 8 taken by the sum of each group's best 2 (lanes
// of 8 experts, 4 lanes per group): the kept groups' experts are spread over
// the whole warp before the picks (4 per lane instead of 8 on half the
// lanes), which halves the sort and the pops.
template <int EPL, bool VEC, int MG, bool REDIST>
__device__ __forceinline__ void route_token(const float* __restrict__ s, const RouteParams& pin,
                                            int lane, int& out_idx, float& out_w)
{
    RouteParams p = pin;
    if constexpr (REDIST) {
        // the one shape this path serves (checked at launch), as constants:
        // loop bounds, shifts and lane predicates fold away
        p.E = 256;
        p.G = 8;
        p.gs = 32;
        p.lpg = 4;
        p.lpg_log2 = 2;
        p.epl = 8;
        p.kg = 4;
        p.m = 2;
        p.k = 8;
        p.limit = 1;
    }
    const int grp = lane >> p.lpg_log2;
    const int sub = lane & (p.lpg - 1);
    const int first = sub * p.epl;        // offset of my first expert inside the group
    const int base = grp * p.gs + first;  // global id of my first expert

    uint32_t key[EPL];
    uint32_t inr = 0;
    if (VEC) {
#pragma unroll
        for (int i4 = 0; i4 < EPL / 4; ++i4) {
            const bool in = (grp < p.G) && (4 * i4 < p.epl);
            float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
            if (in) f = __ldg(reinterpret_cast<const float4*>(s + base) + i4);
            key[4 * i4 + 0] = score_key(f.x);
            key[4 * i4 + 1] = score_key(f.y);
            key[4 * i4 + 2] = score_key(f.z);
            key[4 * i4 + 3] = score_key(f.w);
            if (in) inr |= 0xfu << (4 * i4);
        }
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const bool in = (grp < p.G) && (i < p.epl) && (first + i < p.gs);
            key[i] = in ? score_key(__ldg(s + base + i)) : 0u;
            if (in) inr |= 1u << i;
        }
    }

    uint32_t rem = inr;
    uint32_t key0[EPL];  // the scores before any pick (renormalised softmax needs all)
#pragma unroll
    for (int i = 0; i < EPL; ++i) key0[i] = key[i];
    if (p.limit) {
        uint32_t top[MG];  // the group's MG >= m best keys
#pragma unroll
        for (int q = 0; q < MG; ++q) top[q] = 0u;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if ((inr >> i) & 1u) insert_desc(top, key[i]);
        for (int o = 1; o < p.lpg; o <<= 1) {
            uint32_t oth[MG];
#pragma unroll
            for (int q = 0; q < MG; ++q) oth[q] = __shfl_xor_sync(kFull, top[q], o);
#pragma unroll
            for (int q = 0; q < MG; ++q) insert_desc(top, oth[q]);
        }
        // Group score: the exact sum of the group's m best scores.  For m <= 2
        // an fp32 two-sum gives it exactly as (hi, lo), and (hi, lo) pairs
        // order like the exact sums; larger m sums in binary64, ascending.
        unsigned long long gk;
        if (p.m <= 2) {
            const float a = key_score(top[0]);
            const float b = (p.m == 2) ? key_score(top[MG > 1 ? 1 : 0]) : 0.f;
            const float hi = __fadd_rn(b, a);
            float lo = 0.f;
            if (isfinite(hi)) {
                const float bb = __fsub_rn(hi, a);
                lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, bb)), __fsub_rn(b, bb));
            }
            gk = ((unsigned long long)score_key(hi) << 32) | score_key(lo);
        } else {
            double gsum = 0.0;
#pragma unroll
            for (int q = MG - 1; q >= 0; --q)
                if (q < p.m) gsum += (double)key_score(top[q]);
            gk = sum_key(gsum);
        }
        // ranked by the high word unless two groups share it (then exactly)
        const uint32_t gh = (uint32_t)(gk >> 32);
        int rank = 0;
        bool tie = false;
#pragma unroll 8
        for (int n = 0; n < p.G; ++n) {
            const uint32_t o = __shfl_sync(kFull, gh, n << p.lpg_log2);
            rank += (o > gh) ? 1 : 0;
            tie |= (o == gh && n != grp);
        }
        if (__any_sync(kFull, tie)) {
            rank = 0;
#pragma unroll 8
            for (int n = 0; n < p.G; ++n) {
                const unsigned long long o = __shfl_sync(kFull, gk, n << p.lpg_log2);
                rank += (o > gk || (o == gk && n < grp)) ? 1 : 0;
            }
        }
        if (grp >= p.G || rank >= p.kg) rem = 0u;
    }

    int my_i = -1;
    uint32_t my_k = 0u, first_k = 0u;
    float den = 0.f;
    if constexpr (REDIST) {
        // 8 groups of 32 experts (4 lanes of 8 each), 4 kept: gather the 128
        // kept experts onto all 32 lanes, 4 consecutive experts per lane, lanes
        // in ascending expert order (kept slot q = lane / 8 holds the q-th
        // kept group by index; lane pair (2l, 2l+1) of the slot takes source
        // lane l's two halves).  Exactly 4 group leaders are kept.
        uint32_t kept = __ballot_sync(kFull, sub == 0 && grp < p.G && (rem != 0u));
        const int q = lane >> 3;
#pragma unroll
        for (int i = 0; i < 3; ++i)
            if (i < q) kept &= kept - 1u;  // drop the q lowest kept leaders
        const int sgrp = (__ffs(kept) - 1) >> p.lpg_log2;
        const int src = (sgrp << p.lpg_log2) + ((lane >> 1) & 3);
        const bool upper = lane & 1;
        uint32_t ck[4];
        int ci[4];
        const int cbase = sgrp * p.gs + ((lane >> 1) & 3) * 8 + (upper ? 4 : 0);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t a = __shfl_sync(kFull, key[r], src);
            const uint32_t b = __shfl_sync(kFull, key[4 + r], src);
            ck[r] = upper ? b : a;
            ci[r] = cbase + r;
        }
        sort_desc<4>(ck, ci);
        pick_k<4>(ck, ci, p.k, lane, my_i, my_k, first_k, den);
    } else {
        // k picks from lane-sorted candidates (banned or absent: key 0, below
        // every score)
        int ix[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            if (!((rem >> i) & 1u)) key[i] = 0u;
            ix[i] = base + i;
        }
        sort_desc<EPL>(key, ix);
        pick_k<EPL>(key, ix, p.k, lane, my_i, my_k, first_k, den);
    }

    const bool act = lane < p.k;
    const float my_v = key_score(my_k);
    float w;
    if (p.wmode == MOE_EP_W_SCORE_NORM) {
        w = __fdiv_rn(my_v, den);
    } else if (p.wmode == MOE_EP_W_SOFTMAX_TOPK) {
        const float mx = key_score(first_k);
        const float ex = act ? expf(my_v - mx) : 0.f;
        float d = 0.f;
        for (int j = 0; j < p.k; ++j) d += __shfl_sync(kFull, ex, j);
        w = __fdiv_rn(ex, d);
    } else {
        uint32_t mloc = 0u;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if ((inr >> i) & 1u) mloc = max(mloc, key0[i]);
        const float mx = key_score(__reduce_max_sync(kFull, mloc));
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if ((inr >> i) & 1u) z += expf(key_score(key0[i]) - mx);
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

// One warp per token.  TPC = 32: a CTA routes a whole 32-token tile and
// writes its tile words and byte counts.  TPC = 8 (small batches): four CTAs
// share a tile, each writing its own byte of every tile word (the bits of its
// 8 tokens), so four times as many SMs do the selection work; the last CTA
// then derives the byte counts from the words.
template <int EPL, bool VEC, int MG, int TPC, bool REDIST = false>
__global__ void __launch_bounds__(TPC * 32, TPC == kTileTokens ? 1 : 2) route_kernel(
    const float* __restrict__ scores, int T, RouteParams p, int32_t* __restrict__ topk_idx,
    int32_t* __restrict__ idx_copy, float* __restrict__ topk_w, LayoutArgs la)
{
    constexpr int kParts = kTileTokens / TPC;
    griddep_wait();
    __shared__ uint32_t s_word[kMaxExperts];
    __shared__ int s_scratch[kTailSmemInts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < p.E; e += blockDim.x) s_word[e] = 0u;
    __syncthreads();

    const int tile = blockIdx.x / kParts, part = blockIdx.x % kParts;
    const int slot = part * TPC + warp;  // the token's bit in its tile word
    const int t = tile * kTileTokens + slot;
    if (t < T) {
        int e;
        float w;
        route_token<EPL, VEC, MG, REDIST>(scores + (size_t)t * p.E, p, lane, e, w);
        if (lane < p.k) {
            const size_t q = (size_t)t * p.k + lane;
            topk_idx[q] = e;
            idx_copy[q] = e;
            if (topk_w) topk_w[q] = w;
            if (e >= 0) atomicOr(&s_word[e], 1u << slot);
        }
    }
    __syncthreads();
    for (int e = tid; e < p.E; e += blockDim.x) {
        const uint32_t wd = s_word[e];
        if constexpr (kParts == 1) {
            la.tile_word[(size_t)tile * p.E + e] = wd;
            la.tile_cnt[tile_cnt_index(tile, e, p.E)] = (uint8_t)__popc(wd);
        } else {
            reinterpret_cast<uint8_t*>(la.tile_word)[((size_t)tile * p.E + e) * 4 + part] =
                (uint8_t)(wd >> (8 * part));
        }
    }
    griddep_launch_dependents();
    if (!la.deferred) finish_layout_if_last(la, s_scratch);
}

// Small expert counts without a node limit (E <= W, W = 8 or 16 lanes per
// token): 32 / W tokens per warp, one expert per lane of the token's W-lane
// segment, so no lane of the warp idles while E is far below 32.  A CTA of W
// warps routes one 32-token tile.  The selection and the weights are those of
// route_token: each pick is the largest key, then the lowest expert index
// holding it (here a butterfly over the segment); the weights' sums run in the
// same order (the j-ordered sums lane by lane; the full-softmax normaliser by
// the same butterfly levels, the lanes past E adding zeros), so for a single
// routing group both kernels give the same bits.
template <int W>
__global__ void __launch_bounds__(W * 32) route_small_kernel(
    const float* __restrict__ scores, int T, RouteParams p, int32_t* __restrict__ topk_idx,
    int32_t* __restrict__ idx_copy, float* __restrict__ topk_w, LayoutArgs la)
{
    constexpr int kTpw = 32 / W;  // tokens per warp
    griddep_wait();
    __shared__ uint32_t s_word[kMaxExperts];
    __shared__ int s_scratch[kTailSmemInts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sl = lane & (W - 1);  // the lane's expert (and output slot j)
    for (int e = tid; e < p.E; e += blockDim.x) s_word[e] = 0u;
    __syncthreads();

    const int tile = blockIdx.x;
    const int slot = warp * kTpw + lane / W;  // the token's bit in its tile word
    const int t = tile * kTileTokens + slot;
    const bool tok = t < T;
    const bool in = tok && sl < p.E;
    const uint32_t key0 = in ? score_key(__ldg(scores + (size_t)t * p.E + sl)) : 0u;
    uint32_t key = key0;
    int my_i = -1;
    uint32_t my_k = 0u, first_k = 0u;
    float den = 0.f;
    for (int j = 0; j < p.k; ++j) {
        uint32_t bk = key;
        int bi = key ? sl : W;  // no candidate: past every index
#pragma unroll
        for (int o = W / 2; o > 0; o >>= 1) {
            const uint32_t ok = __shfl_xor_sync(kFull, bk, o, W);
            const int oi = __shfl_xor_sync(kFull, bi, o, W);
            if (ok > bk || (ok == bk && oi < bi)) {
                bk = ok;
                bi = oi;
            }
        }
        const bool found = bk != 0u;
        if (found && sl == bi) key = 0u;  // the winner leaves the candidates
        if (sl == j) {
            my_i = found ? bi : -1;
            my_k = bk;
        }
        if (j == 0) first_k = bk;
        den += key_score(bk);
    }

    const bool act = sl < p.k;
    const float my_v = key_score(my_k);
    const int base = lane & ~(W - 1);  // the segment's first lane
    float w;
    if (p.wmode == MOE_EP_W_SCORE_NORM) {
        w = __fdiv_rn(my_v, den);
    } else if (p.wmode == MOE_EP_W_SOFTMAX_TOPK) {
        const float mx = key_score(first_k);
        const float ex = act ? expf(my_v - mx) : 0.f;
        float d = 0.f;
        for (int j = 0; j < p.k; ++j) d += __shfl_sync(kFull, ex, base + j);
        w = __fdiv_rn(ex, d);
    } else {
        uint32_t mloc = in ? key0 : 0u;
#pragma unroll
        for (int o = W / 2; o > 0; o >>= 1) mloc = max(mloc, __shfl_xor_sync(kFull, mloc, o, W));
        const float mx = key_score(mloc);
        float z = in ? expf(key_score(key0) - mx) : 0.f;
#pragma unroll
        for (int o = W / 2; o > 0; o >>= 1) z += __shfl_xor_sync(kFull, z, o, W);
        const float pj = act ? __fdiv_rn(expf(my_v - mx), z) : 0.f;
        float sel = 0.f;
        for (int j = 0; j < p.k; ++j) sel += __shfl_sync(kFull, pj, base + j);
        w = __fdiv_rn(pj, sel);
    }
    if (tok && act) {
        const size_t q = (size_t)t * p.k + sl;
        topk_idx[q] = my_i;
        idx_copy[q] = my_i;
        if (topk_w) topk_w[q] = w;
        if (my_i >= 0) atomicOr(&s_word[my_i], 1u << slot);
    }
    __syncthreads();
    for (int e = tid; e < p.E; e += blockDim.x) {
        const uint32_t wd = s_word[e];
        la.tile_word[(size_t)tile * p.E + e] = wd;
        la.tile_cnt[tile_cnt_index(tile, e, p.E)] = (uint8_t)__popc(wd);
    }
    griddep_launch_dependents();
    if (!la.deferred) finish_layout_if_last(la, s_scratch);
}

__global__ void __launch_bounds__(256) layout_bits_kernel(const int32_t* __restrict__ topk_idx,
                                                          int T, int k,
                                                          int32_t* __restrict__ idx_copy,
                                                          LayoutArgs la, volatile unsigned* err)
{
    griddep_wait();
    __shared__ uint32_t s_word[kMaxExperts];
    __shared__ int s_scratch[kTailSmemInts];
    const int tid = threadIdx.x, E = la.E;
    for (int e = tid; e < E; e += blockDim.x) s_word[e] = 0u;
    __syncthreads();
    const int tile = blockIdx.x;
    const int t0 = tile * kTileTokens;
    const int nt = min(kTileTokens, T - t0);
    for (int q = tid; q < nt * k; q += blockDim.x) {
        const int tl = q / k, j = q - tl * k;
        const int32_t* r = topk_idx + (size_t)(t0 + tl) * k;
        const int e = r[j];
        idx_copy[(size_t)(t0 + tl) * k + j] = e;
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
    for (int e = tid; e < E; e += blockDim.x) {
        const uint32_t wd = s_word[e];
        la.tile_word[(size_t)tile * E + e] = wd;
        la.tile_cnt[tile_cnt_index(tile, e, E)] = (uint8_t)__popc(wd);
    }
    griddep_launch_dependents();
    if (!la.deferred) finish_layout_if_last(la, s_scratch);
}

template <int EPL, bool VEC>
cudaError_t launch_route_mg(const float* scores, int T, const RouteParams& p, int32_t* topk_idx,
                     int32_t* idx_copy, float* topk_w, const LayoutArgs& la, cudaStream_t s)
{
    const int ntiles = (T + kTileTokens - 1) / kTileTokens;
    // the group list holds MG >= m keys (m = 1, 2: two; 3, 4: four)
    const bool mg2 = !p.limit || p.m <= 2;
    if constexpr (EPL == 8 && VEC) {
        // 8 groups of 32 experts, 4 kept (every lane holds a whole group's
        // quarter): the kept experts are spread over the warp before the picks
        if (p.limit && p.m == 2 && p.k == 8 && p.G == 8 && p.lpg == 4 && p.gs == 32 &&
            p.kg == 4) {
            if (T <= kSplitMaxTokens) {
                LayoutArgs lt = tail_planned(la, 256);
                lt.cnt_from_words = 1;
                return launch_pdl(route_kernel<8, true, 2, 8, true>,
                                  dim3(ntiles * (kTileTokens / 8)), dim3(256), s, scores, T, p,
                                  topk_idx, idx_copy, topk_w, lt);
            }
            return launch_pdl(route_kernel<8, true, 2, kTileTokens, true>, dim3(ntiles),
                              dim3(1024), s, scores, T, p, topk_idx, idx_copy, topk_w,
                              tail_planned(la, 1024));
        }
    }
    if (T <= kSplitMaxTokens) {  // small batch: 8 tokens per CTA
        LayoutArgs lt = tail_planned(la, 256);
        lt.cnt_from_words = 1;
        const dim3 grid(ntiles * (kTileTokens / 8)), block(256);
        if (mg2)
            return launch_pdl(route_kernel<EPL, VEC, 2, 8>, grid, block, s, scores, T, p,
                              topk_idx, idx_copy, topk_w, lt);
        return launch_pdl(route_kernel<EPL, VEC, 4, 8>, grid, block, s, scores, T, p, topk_idx,
                          idx_copy, topk_w, lt);
    }
    const LayoutArgs lt = tail_planned(la, 1024);
    if (mg2)
        return launch_pdl(route_kernel<EPL, VEC, 2, kTileTokens>, dim3(ntiles), dim3(1024), s,
                          scores, T, p, topk_idx, idx_copy, topk_w, lt);
    return launch_pdl(route_kernel<EPL, VEC, 4, kTileTokens>, dim3(ntiles), dim3(1024), s,
                      scores, T, p, topk_idx, idx_copy, topk_w, lt);
}

template <int EPL>
cudaError_t launch_route_epl(const float* scores, int T, const RouteParams& p, int32_t* topk_idx,
                             int32_t* idx_copy, float* topk_w, const LayoutArgs& la,
                             cudaStream_t s)
{
    if (EPL >= 4 && p.vec4)
        return launch_route_mg<EPL, (EPL >= 4)>(scores, T, p, topk_idx, idx_copy, topk_w, la, s);
    return launch_route_mg<EPL, false>(scores, T, p, topk_idx, idx_copy, topk_w, la, s);
}

}  // namespace

cudaError_t launch_route(const float* scores, int T, const RouteParams& p, int32_t* topk_idx,
                         int32_t* idx_copy, float* topk_w, const LayoutArgs& la, cudaStream_t s)
{
    if (T <= 0) return cudaSuccess;
    if (!p.limit && p.E <= 16) {  // small expert counts: several tokens per warp
        const int ntiles = (T + kTileTokens - 1) / kTileTokens;
        if (p.E <= 8)
            return launch_pdl(route_small_kernel<8>, dim3(ntiles), dim3(8 * 32), s, scores, T, p,
                              topk_idx, idx_copy, topk_w, tail_planned(la, 8 * 32));
        return launch_pdl(route_small_kernel<16>, dim3(ntiles), dim3(16 * 32), s, scores, T, p,
                          topk_idx, idx_copy, topk_w, tail_planned(la, 16 * 32));
    }
    if (p.epl <= 1) return launch_route_epl<1>(scores, T, p, topk_idx, idx_copy, topk_w, la, s);
    if (p.epl <= 2) return launch_route_epl<2>(scores, T, p, topk_idx, idx_copy, topk_w, la, s);
    if (p.epl <= 4) return launch_route_epl<4>(scores, T, p, topk_idx, idx_copy, topk_w, la, s);
    if (p.epl <= 8) return launch_route_epl<8>(scores, T, p, topk_idx, idx_copy, topk_w, la, s);
    return launch_route_epl<16>(scores, T, p, topk_idx, idx_copy, topk_w, la, s);
}

cudaError_t launch_layout_bits(const int32_t* topk_idx, int T, int k, int32_t* idx_copy,
                               const LayoutArgs& la, volatile unsigned* err, cudaStream_t s)
{
    if (T <= 0) return cudaSuccess;
    const int ntiles = (T + kTileTokens - 1) / kTileTokens;
    return launch_pdl(layout_bits_kernel, dim3(ntiles), dim3(256), s, topk_idx, T, k, idx_copy,
                      tail_planned(la, 256), err);
}

}  // namespace moeep
