// Routing + layout without any device allocation, for callers that cannot
// call cudaMalloc: a host that hands the library only pre-placed buffers (a
// caching allocator or memory pool that owns all device memory, an embedded
// runtime with a fixed memory plan).  moe_ep_route needs a handle, and
// moe_ep_create_handle allocates its workspace; this entry point instead keeps
// the layout's scratch -- the per-tile expert bitmaps and counts, the column
// prefix and the arrival counter -- in one file-scope device array of fixed
// size, which every GPU that loads the library holds until the process exits.
//
// The scratch array is shared by every call on a device and keeps the last
// call's contents.  The arrival counter, the only part that must start at
// zero, is cleared (cudaMemsetAsync, no allocation) at the start of every call.
// Calls whose work overlaps on the GPU (concurrent streams) race on the array:
// order them on one stream or serialise them.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"

namespace moeep {
namespace {

// Capacity: ceil(T / 32) * E <= kStaticCells tile-expert cells
// (for example T = 8192 tokens with E = 256 experts).
constexpr int kStaticCells = 65536;
constexpr size_t kWordBytes = sizeof(uint32_t) * kStaticCells;               // tile words
// group bases: ceil(ntiles / 16) * E <= kStaticCells / 16 + E
constexpr size_t kBaseBytes = sizeof(int32_t) * (kStaticCells / 16 + kMaxExperts);
constexpr size_t kCntBytes = (size_t)kStaticCells + 16 * (size_t)kMaxExperts; // byte counts, last group padded
constexpr size_t kDoneBytes = 256;                                           // arrival counter
constexpr size_t kScratchBytes = kWordBytes + kBaseBytes + kCntBytes + kDoneBytes;  // 346.25 KiB

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device, looked up once
// per device (with that device current) and then reused for the life of the
// process: it belongs to the device's primary context, so it is stale after
// cudaDeviceReset (the header tells callers not to use the entry point then).
int scratch_for_current_device(unsigned char** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_EP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_route_scratch) != cudaSuccess || !ptr) return MOE_EP_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
    return MOE_EP_OK;
}

}  // namespace
}  // namespace moeep

using namespace moeep;

extern "C" MOE_EP_API int moe_ep_route_layout_static(
    const float* scores, int num_tokens, int experts, int ranks, int mode, int slots,
    const moe_ep_route_opts_t* opts, int32_t* topk_idx, float* topk_w, int32_t* row, int32_t* cnt,
    int32_t* off, int32_t* rcnt, int32_t* roff, moe_ep_stream_t stream)
{
    const int T = num_tokens;
    if (!opts || !scores || !cnt || !off || !rcnt || !roff) return MOE_EP_ERR_INVALID;
    if (mode != MOE_EP_LL && mode != MOE_EP_HT) return MOE_EP_ERR_INVALID;
    if (experts < 1 || experts > kMaxExperts || ranks < 1 || experts % ranks != 0)
        return MOE_EP_ERR_INVALID;
    const int k = opts->topk;
    if (T < 0 || k < 1 || k > kMaxTopk || k > experts) return MOE_EP_ERR_INVALID;
    if (T > 0 && (!topk_idx || !row)) return MOE_EP_ERR_INVALID;
    if (mode == MOE_EP_LL && (slots < 1 || (int64_t)experts * slots > INT32_MAX))
        return MOE_EP_ERR_INVALID;
    if (mode == MOE_EP_LL && T > slots) return MOE_EP_ERR_OVERFLOW;
    if ((int64_t)T * k > INT32_MAX) return MOE_EP_ERR_INVALID;
    const int ntiles = (T + kTileTokens - 1) / kTileTokens;
    if ((int64_t)ntiles * experts > kStaticCells) return MOE_EP_ERR_OVERFLOW;  // beyond the scratch

    RouteParams p;
    p.E = experts;
    p.G = opts->num_groups;
    p.kg = opts->topk_groups;
    p.k = k;
    p.wmode = opts->weight_mode;
    if (p.G < 1 || p.G > kMaxGroups || experts % p.G != 0) return MOE_EP_ERR_INVALID;
    if (p.kg < 1 || p.kg > p.G) return MOE_EP_ERR_INVALID;
    if (p.wmode < MOE_EP_W_SOFTMAX_TOPK || p.wmode > MOE_EP_W_SCORE_NORM) return MOE_EP_ERR_INVALID;
    p.gs = experts / p.G;
    if ((int64_t)p.kg * p.gs < k) return MOE_EP_ERR_INVALID;
    p.limit = (p.G > 1 && p.kg < p.G) ? 1 : 0;
    p.m = opts->group_topk > 0 ? opts->group_topk : (k + p.kg - 1) / p.kg;
    if (p.limit && (p.m < 1 || p.m > kMaxGroupTopk || p.m > p.gs)) return MOE_EP_ERR_INVALID;
    p.lpg = 1;
    p.lpg_log2 = 0;
    while (p.lpg * 2 * p.G <= 32) {
        p.lpg *= 2;
        p.lpg_log2 += 1;
    }
    p.epl = (p.gs + p.lpg - 1) / p.lpg;
    if (p.epl > kMaxExpertsPerLane) return MOE_EP_ERR_INVALID;
    p.vec4 = (p.epl % 4 == 0 && p.gs == p.lpg * p.epl && experts % 4 == 0 &&
              ((uintptr_t)scores & 15u) == 0) ? 1 : 0;

    unsigned char* base = nullptr;
    int st = scratch_for_current_device(&base);
    if (st != MOE_EP_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;

    LayoutArgs la;
    la.tile_word = reinterpret_cast<uint32_t*>(base);
    la.grp_base = reinterpret_cast<int32_t*>(base + kWordBytes);
    la.tile_cnt = base + kWordBytes + kBaseBytes;
    la.done = reinterpret_cast<unsigned*>(base + kWordBytes + kBaseBytes + kCntBytes);
    la.cnt = cnt;
    la.off = off;
    la.rcnt = rcnt;
    la.roff = roff;
    la.E = experts;
    la.R = ranks;
    la.ntiles = ntiles;
    la.host_out = nullptr;
    la.seq = 0u;
    la.align = 1;

    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(int32_t) * (size_t)experts, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(off, 0, sizeof(int32_t) * (size_t)(experts + 1), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(rcnt, 0, sizeof(int32_t) * (size_t)ranks, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(roff, 0, sizeof(int32_t) * (size_t)(ranks + 1), s);
        return e == cudaSuccess ? MOE_EP_OK : MOE_EP_ERR_CUDA;
    }
    // the arrival counter must start at zero; everything else is overwritten
    if (cudaMemsetAsync(la.done, 0, sizeof(unsigned), s) != cudaSuccess) return MOE_EP_ERR_CUDA;
    if (launch_route(scores, T, p, topk_idx, topk_idx, topk_w, la, s) != cudaSuccess)
        return MOE_EP_ERR_CUDA;

    RowArgs ra;
    ra.idx = topk_idx;
    ra.tile_word = la.tile_word;
    ra.tile_cnt = la.tile_cnt;
    ra.grp_base = la.grp_base;
    ra.off = off;
    ra.T = T;
    ra.k = k;
    ra.E = experts;
    ra.S = slots;
    ra.mode = mode;
    ra.G = 1;
    ra.ncols = experts;
    ra.mask = nullptr;
    ra.off_out = nullptr;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MOE_EP_ERR_CUDA;
    if (launch_rowmap(ra, row, sms, s) != cudaSuccess) return MOE_EP_ERR_CUDA;
    return MOE_EP_OK;
}
