// Per-rank dedup path (HT): the receiver-side kernels.
//
// "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": the routing simulation
// counts the copies of a token sent once per destination GPU ("按目标卡去重"),
// and combine sends back the weighted sum of the expert outputs in BF16.
// The dispatch of one copy per (token, rank) reuses the dispatch kernels with
// a layout whose columns are ranks (RowArgs.G = E/R).  Here:
//   - expand_kernel: each dedup row q (token t = dsrc[q], local experts
//     dmask[q], rank r found from rank_off) is copied, payload bytes as they
//     are, to the expert-major HT row of every expert r*L + l in the mask --
//     the rows the direct dispatch writes, found from the expert layout.
//   - combine_partial_kernel: each dedup row gets the BF16 weighted sum of its
//     rank's expert outputs for that token (fp32 fma chain in j order, one
//     rounding).  The source-side sum of the partials is combine_kernel with
//     unit weights over the dedup row map.
// HBM-bound copies and gathers with 16-byte vectors.
#include "bf16x8.cuh"
#include "layout_dev.cuh"

namespace moeep {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 128;
constexpr int kUnroll = 8;  // 16-byte vectors per thread per pass

// Rank of dedup row q (all 32 lanes of a warp): ranks whose block ends at or
// before q.
__device__ __forceinline__ int row_rank(const int32_t* rank_off, int R, int q, int lane)
{
    int r = 0;
    for (int b = 0; b < R; b += 32) {
        const int i = b + lane;
        r += __popc(__ballot_sync(kFull, i < R && __ldg(rank_off + i + 1) <= q));
    }
    return r;
}

// HT row of (token t, expert e) in the expert layout.
__device__ __forceinline__ int expert_row(const RowArgs& ex, int t, int e)
{
    const int tile = t / kTileTokens;
    return __ldg(ex.off + e) + pairs_before_tile(ex.tile_cnt, ex.grp_base, ex.E, e, tile) +
           __popc(__ldg(ex.tile_word + (size_t)tile * ex.E + e) & ((1u << (t & 31)) - 1u));
}

__global__ void __launch_bounds__(kThreads) expand_kernel(DedupArgs a, const uint4* __restrict__ dx,
                                                          const float* __restrict__ dscale,
                                                          int nvec, int nblk,
                                                          uint4* __restrict__ recv_x,
                                                          float* __restrict__ recv_scale,
                                                          int32_t* __restrict__ recv_src)
{
    griddep_wait();
    __shared__ int s_row[32];
    __shared__ int s_n;
    const int total = __ldg(a.rank_off + a.R);
    for (int q = blockIdx.x; q < total; q += gridDim.x) {
        const uint4* src = dx + (size_t)q * nvec;
        // the pass loop is uniform across the CTA (it holds barriers)
        for (int pass = 0; pass < nvec; pass += kUnroll * kThreads) {
            const int v0 = pass + threadIdx.x;
            uint4 buf[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int v = v0 + u * kThreads;
                if (v < nvec) buf[u] = __ldg(src + v);
            }
            if (pass == 0 && threadIdx.x < 32) {
                const int lane = threadIdx.x;
                const int r = row_rank(a.rank_off, a.R, q, lane);
                const int t = __ldg(a.dsrc + q);
                const bool has = lane < a.L && ((__ldg(a.dmask + q) >> lane) & 1u);
                const unsigned b = __ballot_sync(kFull, has);
                if (has) {
                    const int er = expert_row(a.ex, t, r * a.L + lane);
                    s_row[__popc(b & ((1u << lane) - 1u))] = er;
                    if (recv_src) recv_src[er] = t;
                }
                if (lane == 0) s_n = __popc(b);
            }
            __syncthreads();
            const int n = s_n;
            for (int i = 0; i < n; ++i) {
                uint4* dst = recv_x + (size_t)s_row[i] * nvec;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int v = v0 + u * kThreads;
                    if (v < nvec) dst[v] = buf[u];
                }
                if (pass == 0 && dscale)
                    for (int c = threadIdx.x; c < nblk; c += kThreads)
                        recv_scale[(size_t)s_row[i] * nblk + c] = __ldg(dscale + (size_t)q * nblk + c);
            }
            __syncthreads();
        }
    }
}

// One CTA per token: the token's k expert-output rows are read once and each
// rank's pairs (in j order) are reduced into that rank's dedup row -- the
// same partials the ranks would form from their own rows, without a chain of
// lookups from dedup row back to token before the gathers can start.
// Register budget: as the combine kernel, enough CTAs per SM to keep many
// tokens' gathered rows in flight.
constexpr int partial_min_ctas(int kmax)
{
    return kmax <= 2 ? 12 : (kmax <= 4 ? 10 : (kmax <= 8 ? 8 : (kmax <= 16 ? 4 : 2)));
}

template <int KMAX>  // k <= KMAX
__global__ void __launch_bounds__(kThreads, partial_min_ctas(KMAX)) combine_partial_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ row,
    const int32_t* __restrict__ drow, const float* __restrict__ w, int T, int k, int E, int L,
    const uint4* __restrict__ y, int nvec, uint4* __restrict__ partial)
{
    griddep_wait();
    __shared__ int s_row[KMAX];   // expert row of pair j (-1: none)
    __shared__ float s_w[KMAX];
    __shared__ int s_lead[KMAX];  // first pair of j's rank (-1: pair without a row)
    __shared__ int s_q[KMAX];     // dedup row when pair j leads its rank, else -1
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            const unsigned lower = (1u << lane) - 1u;
            int e = -2 - lane;
            if (lane < k) e = __ldg(idx + (size_t)t * k + lane);
            const unsigned peers = __match_any_sync(kFull, e);
            const bool valid = lane < k && e >= 0 && e < E && (peers & lower) == 0u;
            const unsigned rpeers = __match_any_sync(kFull, valid ? e / L : -100 - lane);
            if (lane < KMAX) {
                const bool in = lane < k;
                s_row[lane] = valid ? __ldg(row + (size_t)t * k + lane) : -1;
                s_w[lane] = in ? __ldg(w + (size_t)t * k + lane) : 0.f;
                s_lead[lane] = valid ? __ffs(rpeers) - 1 : -1;
                s_q[lane] = in ? __ldg(drow + (size_t)t * k + lane) : -1;
            }
        }
        __syncthreads();
        int rr[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) rr[j] = s_row[j];
        for (int v = threadIdx.x; v < nvec; v += kThreads) {
            uint4 val[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (rr[j] >= 0) val[j] = __ldcs(y + (size_t)rr[j] * nvec + v);  // read once
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                const int q = s_q[j];  // block-uniform: the bookkeeping stays in shared memory
                if (q < 0) continue;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = j; i < KMAX; ++i)
                    if (s_lead[i] == j) acc8(acc, s_w[i], val[i]);
                partial[(size_t)q * nvec + v] = pack8(acc);
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_expand(const DedupArgs& a, const void* dx, const float* dscale, int row_bytes,
                          int nblk, void* recv_x, float* recv_scale, int32_t* recv_src,
                          int max_rows, int sm_count, cudaStream_t s)
{
    if (max_rows <= 0) return cudaSuccess;
    (void)sm_count;
    const int blocks = max_rows;  // one CTA per possible dedup row (the rest exit)
    return launch_pdl(expand_kernel, dim3(blocks), dim3(kThreads), s, a, (const uint4*)dx, dscale,
                      row_bytes / 16, dscale ? nblk : 0, (uint4*)recv_x, recv_scale, recv_src);
}

cudaError_t launch_combine_partial(const RowArgs& ex, const int32_t* row, const int32_t* drow,
                                   int L, const float* w, const void* y, int H, void* partial,
                                   int sm_count, cudaStream_t s)
{
    const int T = ex.T, k = ex.k;
    if (T <= 0) return cudaSuccess;
    const int blocks = T < sm_count * 16 ? T : sm_count * 16;
    const uint4* yy = (const uint4*)y;
    uint4* pp = (uint4*)partial;
    const int nvec = H / 8;
#define MOEEP_PARTIAL(KM)                                                                   \
    return launch_pdl(combine_partial_kernel<KM>, dim3(blocks), dim3(kThreads), s, ex.idx, row, \
                      drow, w, T, k, ex.E, L, yy, nvec, pp)
    if (k <= 1) MOEEP_PARTIAL(1);
    if (k <= 2) MOEEP_PARTIAL(2);
    if (k <= 4) MOEEP_PARTIAL(4);
    if (k <= 8) MOEEP_PARTIAL(8);
    if (k <= 16) MOEEP_PARTIAL(16);
    MOEEP_PARTIAL(32);
#undef MOEEP_PARTIAL
}

}  // namespace moeep
