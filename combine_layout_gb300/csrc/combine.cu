// Combine: gather each token's k expert-output rows back to token order and
// reduce them with the gate weights.
//
// "NCCL EP 论文解读", item "核心功能函数": combine collects the tokens and reduces
// them to the original order, un-permuting with the routing state stored in
// the handle.  "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": what comes
// back is the weighted sum of the expert outputs, kept in BF16.
//
// out[t][h] = bf16_rn(fma(w_{k-1}, y_{k-1}, ... fma(w_1, y_1, fma(w_0, y_0, 0)))),
// fp32 accumulation in fixed j order, so results do not depend on scheduling
// (w == nullptr: every weight 1, a plain sum -- the source-side stage of the
// per-rank dedup combine, which adds each rank's partial row).
// HBM-bound: k gathered row reads and one row write per token; a CTA takes
// one token at a time, every thread issuing the loads of all k rows for its
// 16-byte slice before accumulating.  The rows are read with the streaming
// (evict-first) policy: each is read once, and the bench step measured
// 179.5 -> 171.2 us with it (the lines the dispatch left dirty in L2 are
// then not pushed out by rows that are never read again).  Tokens are taken
// from the last to the first: when the rows were written token by token just
// before (the dispatch's own output, read back by identity experts, or any
// token-major producer), the last tokens' rows are the ones still in L2, and
// they are read before the stream of other rows evicts them (4096 x 7168,
// k = 8: the dispatch + combine step 164.6 -> 157.0 us; 8192 x 4096, k = 2:
// 68.0 -> 64.4 us).  Rows written expert by expert (an expert GEMM) have no
// such order, and the walk then makes no difference (the FP8 workload's
// separate expert-output buffer: 137.3 us either way).
#include "bf16x8.cuh"
#include "common.cuh"

namespace moeep {
namespace {

constexpr int kThreads = 128;

// Register budget per row count: enough CTAs per SM to keep the gathered rows
// of many tokens in flight (k <= 8: 64 registers, 8 CTAs -- measured on the
// bench shape 6.64 TB/s vs 6.29 TB/s with 5 CTAs; k <= 2: 40 registers).
constexpr int combine_min_ctas(int kmax)
{
    return kmax <= 2 ? 12 : (kmax <= 4 ? 10 : (kmax <= 8 ? 8 : (kmax <= 16 ? 4 : 2)));
}

template <int KMAX>
__global__ void __launch_bounds__(kThreads, combine_min_ctas(KMAX)) combine_kernel(
    const uint4* __restrict__ y, int T, int k, int nvec, TokenSplit split,
    const int32_t* __restrict__ row, const float* __restrict__ w, uint4* __restrict__ out,
    SendSignal sig)
{
    griddep_wait();
    __shared__ int s_row[KMAX];
    __shared__ float s_w[KMAX];
    const int items = split_items(split, T);
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        int t, vb, ve;  // token t's vectors [vb, ve)
        split_item(split, it, nvec, t, vb, ve);
        t = T - 1 - t;  // last token first (see above)
        if (threadIdx.x < k) {
            s_row[threadIdx.x] = row[(size_t)t * k + threadIdx.x];
            s_w[threadIdx.x] = w ? w[(size_t)t * k + threadIdx.x] : 1.f;
        }
        __syncthreads();
        int r[KMAX];
        float wj[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            r[j] = j < k ? s_row[j] : -1;
            wj[j] = j < k ? s_w[j] : 0.f;
        }
        for (int v = vb + threadIdx.x; v < ve; v += kThreads) {
            uint4 val[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (r[j] >= 0) val[j] = __ldcs(y + (size_t)r[j] * nvec + v);  // read once
            float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (r[j] >= 0) acc8(a, wj[j], val[j]);
            out[(size_t)t * nvec + v] = pack8(a);
        }
        __syncthreads();
    }
    send_arrive(sig);
}

}  // namespace

cudaError_t launch_combine(const void* y, int T, int H, int k, const int32_t* row, const float* w,
                           void* out, int sm_count, cudaStream_t s, const SendSignal& sig)
{
    if (T <= 0 && !sig.signal) return cudaSuccess;
    if (T < 0) T = 0;
    const int nvec = H / 8;
    // one CTA per token (or per token slice in small batches), at most 16
    // per SM, grid-stride beyond (small tokens then amortise the CTA launch)
    // -- except for rows of 256 vectors or more when there are at least twice
    // that many tokens or a sliced tail: then one CTA per item, so the
    // hardware balances the tail instead of a fixed token stride (measured:
    // 16384 tokens x 7168, step 518.3 -> 510.7 us; 8192 x 4096, 69.6 -> 68.4
    // us; 4096 x 7168 with its last 456 tokens in 7 slices, combine 76.4 ->
    // 74.2 us).  A send-only launch with no tokens still runs one CTA, for
    // the signal.
    // tail slices of at most 128 vectors (one pass per thread), from 4 tokens
    // per SM
    TokenSplit split = (nvec % 16 == 0 && T > 0)
                           ? token_split(T, nvec / 16, sm_count, 8, 4 * sm_count)
                           : TokenSplit{T, 1, 1};
    int nsplit = split.nsa;
    if (nsplit > 1) {
        // a small batch: slices of at most one pass (kThreads vectors), so no
        // thread waits for its rows twice, while the CTAs still fit in one
        // wave of resident CTAs
        const int units = nvec / 16, resident = sm_count * combine_min_ctas(k <= 8 ? 8 : 32);
        for (int d = nsplit; d <= units; ++d) {
            if (units % d != 0 || nvec / d > kThreads) continue;
            if ((int64_t)T * d <= resident) nsplit = d;
            break;
        }
        split = TokenSplit{T, nsplit, 1};
    }
    const int items = split_items(split, T);
    const int cap = sm_count * 16;
    const bool tail = split.th < T;  // sliced tail: one CTA per item
    int blocks = (nvec / nsplit >= 256 && (tail || items >= 2 * cap)) ? items
                                                                      : (items < cap ? items : cap);
    if (blocks < 1) blocks = 1;
    const uint4* yy = (const uint4*)y;
    uint4* oo = (uint4*)out;
#define MOEEP_COMBINE(KM)                                                                      \
    return launch_pdl(combine_kernel<KM>, dim3(blocks), dim3(kThreads), s, yy, T, k, nvec,     \
                      split, row, w, oo, sig)
    if (k <= 1) MOEEP_COMBINE(1);
    if (k <= 2) MOEEP_COMBINE(2);
    if (k <= 4) MOEEP_COMBINE(4);
    if (k <= 8) MOEEP_COMBINE(8);
    if (k <= 16) MOEEP_COMBINE(16);
    MOEEP_COMBINE(32);
#undef MOEEP_COMBINE
}

}  // namespace moeep
