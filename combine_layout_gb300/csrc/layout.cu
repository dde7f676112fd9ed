// Row map: the receive row of every (token, j) pair, from the finished layout
// (see layout_dev.cuh).  Dispatch computes and stores the same rows itself;
// this kernel serves a combine or a layout copy that comes without a dispatch.
// Also the one-CTA finish of a deferred layout (counts and offsets from the
// tile words) for consumers that come before any dispatch.
#include "layout_dev.cuh"

namespace moeep {
namespace {

__global__ void __launch_bounds__(256) rowmap_kernel(RowArgs a, int32_t* __restrict__ row)
{
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int wpc = blockDim.x >> 5;
    for (int t = blockIdx.x * wpc + (threadIdx.x >> 5); t < a.T; t += gridDim.x * wpc) {
        uint32_t m = 0u;
        const int r = token_pair_row(a, t, lane, &m);
        if (lane < a.k) row[(size_t)t * a.k + lane] = r;
    }
}

// A deferred layout's counts and offsets, when something needs them before
// (or without) a dispatch: one CTA.
__global__ void __launch_bounds__(128) finish_words_kernel(LayoutArgs a)
{
    griddep_wait();
    finish_layout_from_words<128>(a, nullptr);
}

}  // namespace

cudaError_t launch_finish_words(const LayoutArgs& la, cudaStream_t s)
{
    return launch_pdl(finish_words_kernel, dim3(1), dim3(128), s, la);
}

cudaError_t launch_rowmap(const RowArgs& ra, int32_t* row, int sm_count, cudaStream_t s)
{
    if (ra.T <= 0) return cudaSuccess;
    int blocks = (ra.T + 7) / 8;
    if (blocks > sm_count * 8) blocks = sm_count * 8;
    return launch_pdl(rowmap_kernel, dim3(blocks), dim3(256), s, ra, row);
}

}  // namespace moeep
