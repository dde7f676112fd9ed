// Node-level layout for two-hop dispatch, and the routing statistics.
//
// "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": high-throughput dispatch
// sends a token once to every remote node holding one of its experts (to the
// GPU in the same position, over RDMA), and that GPU forwards it over NVLink to
// the GPUs that hold the experts.  With experts in contiguous blocks,
// gpu = e / (E/R) and node = gpu / (R/N).  This builds, from the handle's
// routing:
//   - node rows, node-major with tokens ascending (the same counting layout as
//     the expert layout, at node granularity: the last CTA's column scan in
//     layout_dev.cuh), each row carrying the mask of the node's GPUs to
//     forward to;
//   - the statistics the page's simulation prints: nodes touched per token
//     (own node included) and cross-node copies per expert, per distinct GPU
//     and per distinct node, relative to the source node src_node.
// One warp per token: lanes < k hold the token's experts; match_any groups
// lanes by GPU and by node, ballots count the leaders.  Repeated or invalid
// expert ids are skipped (only a repeat's first occurrence counts).
#include "layout_dev.cuh"

namespace moeep {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;

struct TokenNodes {
    int node;          // node of this lane's expert (unique negative when invalid)
    uint32_t mask;     // GPUs of `node` that hold one of the token's experts
    bool valid;        // the lane holds a counted expert
    bool node_leader;  // first counted lane of its node
    bool gpu_leader;   // first counted lane of its GPU
};

__device__ __forceinline__ TokenNodes token_nodes(const NodeArgs& a, int t, int lane)
{
    TokenNodes r;
    int e = -2 - lane;  // lanes >= k: distinct values that match nothing
    if (lane < a.k) e = __ldg(a.idx + (size_t)t * a.k + lane);
    const unsigned lower = (1u << lane) - 1u;
    const unsigned peers = __match_any_sync(kFull, e);
    r.valid = lane < a.k && e >= 0 && e < a.E && !(peers & lower);
    const int gpu = r.valid ? e / a.L : -1000 - lane;
    r.node = r.valid ? gpu / a.gpn : -1000 - lane;
    const unsigned gp = __match_any_sync(kFull, gpu);
    const unsigned np = __match_any_sync(kFull, r.node);
    r.gpu_leader = r.valid && !(gp & lower);
    r.node_leader = r.valid && !(np & lower);
    const uint32_t bit = r.valid ? 1u << (gpu % a.gpn) : 0u;
    uint32_t m = 0u;
    for (int j = 0; j < a.k; ++j) {
        const uint32_t b = __shfl_sync(kFull, bit, j);
        if ((np >> j) & 1u) m |= b;
    }
    r.mask = m;
    return r;
}

__global__ void __launch_bounds__(kThreads) node_bits_kernel(NodeArgs a, LayoutArgs la,
                                                             unsigned long long* stats)
{
    griddep_wait();
    __shared__ uint32_t s_word[kMaxExperts];
    __shared__ int s_scratch[kTailSmemInts];
    __shared__ unsigned long long s_stats[4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int n = tid; n < a.N; n += blockDim.x) s_word[n] = 0u;
    if (tid < 4) s_stats[tid] = 0ull;
    __syncthreads();
    const int t0 = blockIdx.x * kTileTokens;
    unsigned st[4] = {0u, 0u, 0u, 0u};
    for (int tl = warp; tl < kTileTokens; tl += kThreads / 32) {
        const int t = t0 + tl;
        if (t >= a.T) break;
        const TokenNodes r = token_nodes(a, t, lane);
        const bool remote = r.valid && r.node != a.src;
        st[0] += __popc(__ballot_sync(kFull, r.node_leader));
        st[1] += __popc(__ballot_sync(kFull, remote));
        st[2] += __popc(__ballot_sync(kFull, r.gpu_leader && remote));
        st[3] += __popc(__ballot_sync(kFull, r.node_leader && remote));
        if (r.node_leader) atomicOr(&s_word[r.node], 1u << tl);
    }
    if (lane == 0)
        for (int q = 0; q < 4; ++q) atomicAdd(&s_stats[q], (unsigned long long)st[q]);
    __syncthreads();
    if (stats && tid < 4) atomicAdd(stats + tid, s_stats[tid]);
    for (int n = tid; n < a.N; n += blockDim.x) {
        const uint32_t wd = s_word[n];
        la.tile_word[(size_t)blockIdx.x * a.N + n] = wd;
        la.tile_cnt[tile_cnt_index(blockIdx.x, n, a.N)] = (uint8_t)__popc(wd);
    }
    griddep_launch_dependents();
    finish_layout_if_last(la, s_scratch);
}

__global__ void __launch_bounds__(kThreads) node_rows_kernel(NodeArgs a, const uint32_t* tile_word,
                                                             const uint8_t* tile_cnt,
                                                             const int32_t* grp_base,
                                                             const int32_t* node_off,
                                                             int32_t* node_src, uint32_t* node_mask)
{
    griddep_wait();
    const int lane = threadIdx.x & 31, wpc = blockDim.x >> 5;
    for (int t = blockIdx.x * wpc + (threadIdx.x >> 5); t < a.T; t += gridDim.x * wpc) {
        const TokenNodes r = token_nodes(a, t, lane);
        if (!r.node_leader) continue;
        const int tile = t / kTileTokens;
        const int row = __ldg(node_off + r.node) +
                        pairs_before_tile(tile_cnt, grp_base, a.N, r.node, tile) +
                        __popc(__ldg(tile_word + (size_t)tile * a.N + r.node) & ((1u << (t & 31)) - 1u));
        node_src[row] = t;
        node_mask[row] = r.mask;
    }
}

}  // namespace

cudaError_t launch_node_layout(const NodeArgs& a, const LayoutArgs& la, unsigned long long* stats,
                               int32_t* node_src, uint32_t* node_mask, int sm_count, cudaStream_t s)
{
    if (a.T <= 0) return cudaSuccess;
    cudaError_t e = launch_pdl(node_bits_kernel, dim3(la.ntiles), dim3(kThreads), s, a,
                               tail_planned(la, kThreads), stats);
    if (e != cudaSuccess || !node_src) return e;  // no node_src: the layout only
    int blocks = (a.T + 7) / 8;
    if (blocks > sm_count * 8) blocks = sm_count * 8;
    return launch_pdl(node_rows_kernel, dim3(blocks), dim3(kThreads), s, a,
                      (const uint32_t*)la.tile_word, (const uint8_t*)la.tile_cnt,
                      (const int32_t*)la.grp_base, (const int32_t*)la.off, node_src, node_mask);
}

}  // namespace moeep
