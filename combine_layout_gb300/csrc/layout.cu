// Row map: the receive row of every (token, j) pair, from the finished layout
// (see layout_dev.cuh).  Dispatch computes and stores the same rows itself;
// this kernel serves a combine or a layout copy that comes without a dispatch.
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

}  // namespace

cudaError_t launch_rowmap(const RowArgs& ra, int32_t* row, int sm_count, cudaStream_t s)
{
    if (ra.T <= 0) return cudaSuccess;
    int blocks = (ra.T + 7) / 8;
    if (blocks > sm_count * 8) blocks = sm_count * 8;
    return launch_pdl(rowmap_kernel, dim3(blocks), dim3(256), s, ra, row);
}

}  // namespace moeep
