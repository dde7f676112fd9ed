// Per-expert counting and prefix layout.
//
// "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": the high-throughput mode
// first counts the tokens bound for every rank and every expert (the "layout").
// "NCCL EP 论文解读", item "算法模式": the HT output is 2D with per-expert counts
// and a deterministic order.  Here the order is (expert, token), which is
// (rank, local expert, token) because expert e = r * L + l.
//
// Input: tile_word[tile][e], bit i set when token tile*32+i chose expert e.
//   scan kernel:   tile_base[tile][e] = pairs of expert e in earlier tiles,
//                  cnt[e] = all pairs of expert e.
//   rowmap kernel: off = exclusive prefix of cnt (each CTA recomputes it in
//                  shared memory; CTA 0 publishes off, rcnt, roff), then
//                  row[t][j] = base(e) + tile_base[tile][e]
//                              + popc(tile_word[tile][e] & bits below t),
//                  base(e) = off[e] (HT) or e * S (LL: slot within [r][l]).
#include "common.cuh"

namespace moeep {
namespace {

constexpr int kScanWarps = 8;

__global__ void __launch_bounds__(kScanWarps * 32) layout_scan_kernel(
    const uint32_t* __restrict__ tile_word, int ntiles, int E, int32_t* __restrict__ tile_base,
    int32_t* __restrict__ cnt)
{
    __shared__ int part[kScanWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + lane;
    const bool col = e < E;
    const int chunk = (ntiles + kScanWarps - 1) / kScanWarps;
    const int r0 = min(warp * chunk, ntiles);
    const int r1 = min(r0 + chunk, ntiles);

    int local = 0;
    if (col)
        for (int r = r0; r < r1; ++r) local += __popc(__ldg(tile_word + (size_t)r * E + e));
    part[warp][lane] = local;
    __syncthreads();
    int base = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kScanWarps; ++w) {
        const int v = part[w][lane];
        if (w < warp) base += v;
        total += v;
    }
    if (col) {
        int run = base;
        for (int r = r0; r < r1; ++r) {
            tile_base[(size_t)r * E + e] = run;
            run += __popc(__ldg(tile_word + (size_t)r * E + e));
        }
        if (warp == 0) cnt[e] = total;
    }
}

// Exclusive prefix of cnt[0..E) into s_off[0..E], by all threads of the CTA.
__device__ void block_exclusive_scan(const int32_t* __restrict__ cnt, int E, int* s_off,
                                     int* s_warp)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;
    const int per = (E + nthreads - 1) / nthreads;
    const int lo = min(tid * per, E), hi = min(lo + per, E);
    int sum = 0;
    for (int e = lo; e < hi; ++e) sum += cnt[e];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane < nwarps) s_warp[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    int run = incl - sum + (warp > 0 ? s_warp[warp - 1] : 0);
    for (int e = lo; e < hi; ++e) {
        s_off[e] = run;
        run += cnt[e];
    }
    if (tid == nthreads - 1) s_off[E] = s_warp[nwarps - 1];
    __syncthreads();
}

__global__ void __launch_bounds__(256) rowmap_kernel(
    const int32_t* __restrict__ topk_idx, int T, int k, int E, int R, int mode, int S,
    const uint32_t* __restrict__ tile_word, const int32_t* __restrict__ tile_base,
    const int32_t* __restrict__ cnt, int32_t* __restrict__ off, int32_t* __restrict__ rcnt,
    int32_t* __restrict__ roff, int32_t* __restrict__ row)
{
    extern __shared__ int s_off[];  // [E + 1]
    __shared__ int s_warp[32];
    block_exclusive_scan(cnt, E, s_off, s_warp);

    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) off[e] = s_off[e];
        const int L = E / R;
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            roff[r] = s_off[r * L];
            rcnt[r] = s_off[(r + 1) * L] - s_off[r * L];
        }
        if (threadIdx.x == 0) roff[R] = s_off[E];
    }

    const int64_t n = (int64_t)T * k;
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n;
         p += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(p / k), j = (int)(p - (int64_t)t * k);
        const int32_t* r = topk_idx + (size_t)t * k;
        const int e = r[j];
        bool valid = (e >= 0 && e < E);
        for (int jj = 0; jj < j; ++jj) valid &= (r[jj] != e);
        if (!valid) {
            row[p] = -1;
            continue;
        }
        const int tile = t / kTileTokens, bit = t % kTileTokens;
        const size_t q = (size_t)tile * E + e;
        const int rank = __ldg(tile_base + q) + __popc(__ldg(tile_word + q) & ((1u << bit) - 1u));
        row[p] = (mode == MOE_EP_HT) ? s_off[e] + rank : e * S + rank;
    }
}

}  // namespace

cudaError_t launch_layout_scan(const uint32_t* tile_word, int ntiles, int E, int32_t* tile_base,
                               int32_t* cnt, cudaStream_t s)
{
    if (ntiles <= 0) {
        return cudaMemsetAsync(cnt, 0, sizeof(int32_t) * (size_t)E, s);
    }
    layout_scan_kernel<<<(E + 31) / 32, kScanWarps * 32, 0, s>>>(tile_word, ntiles, E, tile_base,
                                                                 cnt);
    return cudaGetLastError();
}

cudaError_t launch_rowmap(const int32_t* topk_idx, int T, int k, int E, int R, int mode, int S,
                          const uint32_t* tile_word, const int32_t* tile_base, const int32_t* cnt,
                          int32_t* off, int32_t* rcnt, int32_t* roff, int32_t* row,
                          int sm_count, cudaStream_t s)
{
    const int64_t n = (int64_t)T * k;
    int64_t blocks = (n + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > (int64_t)sm_count * 8) blocks = (int64_t)sm_count * 8;
    rowmap_kernel<<<(int)blocks, 256, sizeof(int) * (size_t)(E + 1), s>>>(
        topk_idx, T, k, E, R, mode, S, tile_word, tile_base, cnt, off, rcnt, roff, row);
    return cudaGetLastError();
}

}  // namespace moeep
