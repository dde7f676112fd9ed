// C ABI of libmoeep: groups, handles, argument checks and kernel launches.
// The operations follow "NCCL EP 论文解读", item "核心功能函数" (group, handle,
// dispatch, combine, receive-count query); see include/moe_ep.h for the
// contract of every call.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <chrono>
#include <new>

#include "common.cuh"

using namespace moeep;

struct moe_ep_group {
    int mode, E, R, L, S, H;
    int device, sm_count;
    int handles;                  // live handles
    volatile unsigned* err_host;  // [kErrSlots], mapped pinned memory
    unsigned* err_dev;            // device alias of err_host
};

struct moe_ep_handle {
    moe_ep_group* g;
    int max_topk;
    int ntiles_max;
    // device workspace
    uint32_t* tile_word;  // [ntiles_max][E]
    uint8_t* tile_cnt;    // [ngroups_max][E][16]
    int32_t* grp_base;    // [ngroups_max][E]
    int32_t* cnt;         // [E]
    int32_t* off;         // [E+1]
    int32_t* rcnt;        // [R]
    int32_t* roff;        // [R+1]
    int32_t* row;         // [max_tokens * max_topk]
    int32_t* idx;         // [max_tokens * max_topk], copy of the routing
    unsigned* done;       // layout CTA counter
    // node-level layout workspace (nodes <= ranks)
    uint32_t* ntile_word;  // [ntiles_max][R]
    uint8_t* ntile_cnt;    // [ngroups_max][R][16]
    int32_t* ngrp_base;    // [ngroups_max][R]
    unsigned* ndone;
    // per-rank dedup layout workspace (columns = ranks)
    uint32_t* rtile_word;  // [ntiles_max][R]
    uint8_t* rtile_cnt;    // [ngroups_max][R][16]
    int32_t* rgrp_base;    // [ngroups_max][R]
    unsigned* rdone;
    int32_t* rk_cnt;       // [R] tokens per destination rank
    int32_t* rk_off;       // [R+1]
    int32_t* drow;         // [max_tokens * max_topk] dedup row of each pair (-1: not its rank's first)
    int dedup_ready;       // the dedup layout and row map belong to the last route
    // counts published by the layout for the receive-count query (mapped
    // pinned memory): off[E+1], rcnt[R], cnt[E], then the sequence number of
    // the route that wrote them
    int32_t* host_counts;
    int32_t* host_counts_dev;  // device alias
    unsigned seq;              // sequence number of the last HT route
    // state of the last route
    int routed;
    int rows_ready;       // row[] written for the last route
    int words_only;       // the last route's layout is deferred: tile words only (small LL batch)
    int layout_pending;   // ... and its counts and offsets are not computed yet
    int T, k;
    int64_t host_total;   // total rows known on the host (-1: not queried)
    int align;            // HT expert blocks padded to a multiple of align rows
    int x_early;          // x is complete before the route (moe_ep_set_x_before_route)
    int captured;         // the last route was recorded into a CUDA graph (stream capture)
    // send-only operations (staged execution): the send kernels' CTA arrival
    // counter and the signal their last CTA adds 1 to (device workspace), the
    // event recorded after the last send, and the sends not yet completed
    unsigned* send_arrive;
    unsigned* send_signal;
    cudaEvent_t sent;
    unsigned pending;
};

namespace {

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_EP_OK : MOE_EP_ERR_CUDA; }

// Limit of the receive wait that moe_ep_complete enqueues: its sends are
// ordered before it, so in correct use the first poll succeeds.
constexpr uint64_t kCompleteWaitNs = 200ull * 1000 * 1000;
// Largest limit moe_ep_wait_signal accepts.
constexpr int64_t kMaxWaitNs = 10ll * 1000 * 1000 * 1000;

inline int check_group(const moe_ep_group* g)
{
    if (!g) return MOE_EP_ERR_INVALID;
    if (g->err_host[kErrTimeout]) return MOE_EP_ERR_TIMEOUT;
    for (int i = 0; i < kErrSlots; ++i)
        if (g->err_host[i]) return MOE_EP_ERR_DEVICE;
    return MOE_EP_OK;
}

// Next 256-byte-aligned piece of a handle's single device allocation.
template <typename T>
T* carve(char*& cur, size_t count)
{
    T* p = reinterpret_cast<T*>(cur);
    size_t bytes = (sizeof(T) * count + 255) & ~(size_t)255;
    cur += bytes;
    return p;
}

// Dedup rows a route can need: one per (token, destination rank).
int64_t dedup_capacity(const moe_ep_handle* h)
{
    const int k = h->k, R = h->g->R;
    return (int64_t)h->T * (k < R ? k : R);
}

int64_t required_rows(const moe_ep_handle* h)
{
    const moe_ep_group* g = h->g;
    if (g->mode == MOE_EP_LL) return (int64_t)g->E * g->S;
    if (h->host_total >= 0) return h->host_total;
    return (int64_t)h->T * h->k + (int64_t)g->E * (h->align - 1);
}

LayoutArgs layout_args(const moe_ep_handle* h, int T)
{
    LayoutArgs a;
    a.tile_word = h->tile_word;
    a.tile_cnt = h->tile_cnt;
    a.grp_base = h->grp_base;
    a.cnt = h->cnt;
    a.off = h->off;
    a.rcnt = h->rcnt;
    a.roff = h->roff;
    a.done = h->done;
    a.E = h->g->E;
    a.R = h->g->R;
    a.ntiles = (T + kTileTokens - 1) / kTileTokens;
    a.host_out = nullptr;
    a.seq = 0u;
    a.align = h->align;
    return a;
}

RowArgs row_args(const moe_ep_handle* h)
{
    RowArgs a;
    a.idx = h->idx;
    a.tile_word = h->tile_word;
    a.tile_cnt = h->tile_cnt;
    a.grp_base = h->grp_base;
    a.off = h->off;
    a.T = h->T;
    a.k = h->k;
    a.E = h->g->E;
    a.S = h->g->S;
    a.mode = h->g->mode;
    a.G = 1;
    a.ncols = a.E;
    a.mask = nullptr;
    a.off_out = nullptr;
    a.from_words = h->words_only;
    return a;
}

// The counts and offsets of a deferred layout, before a consumer that reads
// them without a dispatch having produced them.
int ensure_counts(moe_ep_handle* h, cudaStream_t s)
{
    if (!h->layout_pending) return MOE_EP_OK;
    LayoutArgs la = layout_args(h, h->T);
    la.deferred = 1;
    int st = cuda_status(launch_finish_words(la, s));
    if (st == MOE_EP_OK) h->layout_pending = 0;
    return st;
}

int ensure_rows(moe_ep_handle* h, cudaStream_t s)
{
    if (h->rows_ready) return MOE_EP_OK;
    int st = cuda_status(launch_rowmap(row_args(h), h->row, h->g->sm_count, s));
    if (st == MOE_EP_OK) h->rows_ready = 1;
    return st;
}

}  // namespace

extern "C" {

const char* moe_ep_status_string(int status)
{
    switch (status) {
        case MOE_EP_OK: return "ok";
        case MOE_EP_ERR_INVALID: return "invalid argument";
        case MOE_EP_ERR_OVERFLOW: return "more tokens than max_tokens";
        case MOE_EP_ERR_CUDA: return "CUDA runtime error";
        case MOE_EP_ERR_DEVICE: return "device-error word set";
        case MOE_EP_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
        default: return "unknown status";
    }
}

int moe_ep_create_group(moe_ep_group_t* out, int mode, int experts, int ranks, int max_tokens,
                        int hidden)
{
    if (!out) return MOE_EP_ERR_INVALID;
    *out = nullptr;
    if (mode != MOE_EP_LL && mode != MOE_EP_HT) return MOE_EP_ERR_INVALID;
    if (experts < 1 || experts > kMaxExperts || ranks < 1 || experts % ranks != 0)
        return MOE_EP_ERR_INVALID;
    if (max_tokens < 1 || hidden < 8 || hidden % 8 != 0) return MOE_EP_ERR_INVALID;
    // row ids are int32: every receive row index must fit
    if ((int64_t)experts * max_tokens > INT32_MAX || (int64_t)max_tokens * kMaxTopk > INT32_MAX)
        return MOE_EP_ERR_INVALID;

    moe_ep_group* g = new (std::nothrow) moe_ep_group();
    if (!g) return MOE_EP_ERR_INVALID;
    g->mode = mode;
    g->E = experts;
    g->R = ranks;
    g->L = experts / ranks;
    g->S = max_tokens;
    g->H = hidden;
    if (cudaGetDevice(&g->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&g->sm_count, cudaDevAttrMultiProcessorCount, g->device) !=
            cudaSuccess) {
        delete g;
        return MOE_EP_ERR_CUDA;
    }
    void* hp = nullptr;
    if (cudaHostAlloc(&hp, sizeof(unsigned) * kErrSlots, cudaHostAllocMapped) != cudaSuccess) {
        delete g;
        return MOE_EP_ERR_CUDA;
    }
    memset(hp, 0, sizeof(unsigned) * kErrSlots);
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, hp, 0) != cudaSuccess) {
        cudaFreeHost(hp);
        delete g;
        return MOE_EP_ERR_CUDA;
    }
    g->err_host = (volatile unsigned*)hp;
    g->err_dev = (unsigned*)dp;
    *out = g;
    return MOE_EP_OK;
}

int moe_ep_destroy_group(moe_ep_group_t g)
{
    if (!g) return MOE_EP_ERR_INVALID;
    if (g->handles != 0) return MOE_EP_ERR_INVALID;
    cudaError_t e = cudaDeviceSynchronize();
    cudaFreeHost((void*)g->err_host);
    delete g;
    return cuda_status(e);
}

int moe_ep_create_handle(moe_ep_group_t g, int max_topk, moe_ep_handle_t* out)
{
    if (!g || !out || max_topk < 1 || max_topk > kMaxTopk || max_topk > g->E)
        return MOE_EP_ERR_INVALID;
    *out = nullptr;
    moe_ep_handle* h = new (std::nothrow) moe_ep_handle();
    if (!h) return MOE_EP_ERR_INVALID;
    h->g = g;
    h->max_topk = max_topk;
    h->ntiles_max = (g->S + kTileTokens - 1) / kTileTokens;
    const size_t nt = (size_t)h->ntiles_max * g->E;
    // one allocation, carved in this order, each piece 256-byte aligned
    const size_t ntn = (size_t)h->ntiles_max * g->R;
    const size_t cstride = ((size_t)h->ntiles_max + 15) / 16 * 16;
    const size_t ngrp = cstride / 16;
    const size_t counts[23] = {nt, ngrp * g->E, (size_t)g->E, (size_t)g->E + 1, (size_t)g->R,
                               (size_t)g->R + 1, (size_t)g->S * max_topk, (size_t)g->S * max_topk, 1,
                               (size_t)g->E * cstride / 4,
                               ntn, (size_t)g->R * cstride / 4, ngrp * g->R, 1,
                               ntn, (size_t)g->R * cstride / 4, ngrp * g->R, 1, (size_t)g->R,
                               (size_t)g->R + 1, (size_t)g->S * max_topk, 1, 1};
    size_t bytes = 0;
    for (size_t c : counts) bytes += (sizeof(int32_t) * c + 255) & ~(size_t)255;
    void* base = nullptr;
    if (cudaMalloc(&base, bytes) != cudaSuccess) {
        delete h;
        return MOE_EP_ERR_CUDA;
    }
    char* cur = (char*)base;
    h->tile_word = carve<uint32_t>(cur, counts[0]);
    h->grp_base = carve<int32_t>(cur, counts[1]);
    h->cnt = carve<int32_t>(cur, counts[2]);
    h->off = carve<int32_t>(cur, counts[3]);
    h->rcnt = carve<int32_t>(cur, counts[4]);
    h->roff = carve<int32_t>(cur, counts[5]);
    h->row = carve<int32_t>(cur, counts[6]);
    h->idx = carve<int32_t>(cur, counts[7]);
    h->done = carve<unsigned>(cur, counts[8]);
    h->tile_cnt = carve<uint8_t>(cur, (size_t)g->E * cstride);
    h->ntile_word = carve<uint32_t>(cur, ntn);
    h->ntile_cnt = carve<uint8_t>(cur, (size_t)g->R * cstride);
    h->ngrp_base = carve<int32_t>(cur, counts[12]);
    h->ndone = carve<unsigned>(cur, 1);
    h->rtile_word = carve<uint32_t>(cur, counts[14]);
    h->rtile_cnt = carve<uint8_t>(cur, (size_t)g->R * cstride);
    h->rgrp_base = carve<int32_t>(cur, counts[16]);
    h->rdone = carve<unsigned>(cur, 1);
    h->rk_cnt = carve<int32_t>(cur, counts[18]);
    h->rk_off = carve<int32_t>(cur, counts[19]);
    h->drow = carve<int32_t>(cur, counts[20]);
    h->send_arrive = carve<unsigned>(cur, 1);
    h->send_signal = carve<unsigned>(cur, 1);
    if (cudaMemset(base, 0, bytes) != cudaSuccess) {
        cudaFree(base);
        delete h;
        return MOE_EP_ERR_CUDA;
    }
    void* hs = nullptr;
    void* hs_dev = nullptr;
    const size_t stage_bytes = sizeof(int32_t) * (size_t)(g->E + 1 + g->R + g->E + 1);
    if (cudaHostAlloc(&hs, stage_bytes, cudaHostAllocMapped) != cudaSuccess) {
        cudaFree(base);
        delete h;
        return MOE_EP_ERR_CUDA;
    }
    if (cudaHostGetDevicePointer(&hs_dev, hs, 0) != cudaSuccess) {
        cudaFreeHost(hs);
        cudaFree(base);
        delete h;
        return MOE_EP_ERR_CUDA;
    }
    memset(hs, 0, stage_bytes);
    h->host_counts = (int32_t*)hs;
    h->host_counts_dev = (int32_t*)hs_dev;
    h->seq = 0u;
    if (cudaEventCreateWithFlags(&h->sent, cudaEventDisableTiming) != cudaSuccess) {
        cudaFreeHost(hs);
        cudaFree(base);
        delete h;
        return MOE_EP_ERR_CUDA;
    }
    h->pending = 0;
    h->routed = 0;
    h->rows_ready = 0;
    h->words_only = 0;
    h->layout_pending = 0;
    h->dedup_ready = 0;
    h->host_total = -1;
    h->align = 1;
    h->x_early = 0;
    h->captured = 0;
    g->handles += 1;
    *out = h;
    return MOE_EP_OK;
}

int moe_ep_destroy_handle(moe_ep_handle_t h)
{
    if (!h) return MOE_EP_ERR_INVALID;
    cudaError_t e = cudaDeviceSynchronize();
    cudaFree(h->tile_word);  // start of the single allocation
    cudaFreeHost(h->host_counts);
    cudaEventDestroy(h->sent);
    h->g->handles -= 1;
    delete h;
    return cuda_status(e);
}

int moe_ep_route(moe_ep_handle_t h, const float* scores, int num_tokens,
                 const moe_ep_route_opts_t* opts, int32_t* topk_idx, float* topk_w,
                 moe_ep_stream_t stream)
{
    if (!h || !opts) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    const int T = num_tokens, k = opts->topk;
    if (T < 0 || k < 1 || k > h->max_topk || k > g->E) return MOE_EP_ERR_INVALID;
    if (T > g->S) return MOE_EP_ERR_OVERFLOW;
    if (T > 0 && !topk_idx) return MOE_EP_ERR_INVALID;
    cudaStream_t s = (cudaStream_t)stream;
    // a route recorded into a CUDA graph publishes its counts with the
    // sequence number of the capture on every replay (see the query)
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        cap = cudaStreamCaptureStatusNone;
    }
    LayoutArgs la = layout_args(h, T);
    // LL batches of at most kDeferMaxTiles tiles: no serial tail after the
    // router; the dispatch's first CTA finishes the counts and offsets
    la.deferred = (g->mode == MOE_EP_LL && T > 0 && la.ntiles <= kDeferMaxTiles) ? 1 : 0;
    if (g->mode == MOE_EP_HT && T > 0) {
        // the layout publishes the counts for the receive-count query
        la.host_out = h->host_counts_dev;
        la.seq = h->seq + 1u;
    }

    if (T == 0) {
        // no pairs: counts and offsets are zero
        cudaError_t e = cudaMemsetAsync(h->cnt, 0, sizeof(int32_t) * (size_t)g->E, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(h->off, 0, sizeof(int32_t) * (size_t)(g->E + 1), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(h->rcnt, 0, sizeof(int32_t) * (size_t)g->R, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(h->roff, 0, sizeof(int32_t) * (size_t)(g->R + 1), s);
        st = cuda_status(e);
    } else if (scores) {
        RouteParams p;
        p.E = g->E;
        p.G = opts->num_groups;
        p.kg = opts->topk_groups;
        p.k = k;
        p.wmode = opts->weight_mode;
        if (p.G < 1 || p.G > kMaxGroups || g->E % p.G != 0) return MOE_EP_ERR_INVALID;
        if (p.kg < 1 || p.kg > p.G) return MOE_EP_ERR_INVALID;
        if (p.wmode < MOE_EP_W_SOFTMAX_TOPK || p.wmode > MOE_EP_W_SCORE_NORM) return MOE_EP_ERR_INVALID;
        p.gs = g->E / p.G;
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
        p.vec4 = (p.epl % 4 == 0 && p.gs == p.lpg * p.epl && g->E % 4 == 0 &&
                  ((uintptr_t)scores & 15u) == 0) ? 1 : 0;
        st = cuda_status(launch_route(scores, T, p, topk_idx, h->idx, topk_w, la, s));
    } else {
        st = cuda_status(launch_layout_bits(topk_idx, T, k, h->idx, la, g->err_dev, s));
    }
    if (st != MOE_EP_OK) return st;
    if (la.host_out) h->seq = la.seq;
    h->routed = 1;
    h->captured = (cap == cudaStreamCaptureStatusActive) ? 1 : 0;
    h->rows_ready = 0;
    h->words_only = la.deferred;
    h->layout_pending = la.deferred;
    h->dedup_ready = 0;
    h->T = T;
    h->k = k;
    h->host_total = -1;
    return MOE_EP_OK;
}

int moe_ep_get_num_recv_tokens(moe_ep_handle_t h, int64_t* total, int32_t* per_rank,
                               int32_t* per_expert, moe_ep_stream_t stream)
{
    if (!h || !total) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!h->routed) return MOE_EP_ERR_INVALID;
    if (g->mode == MOE_EP_LL) {
        *total = (int64_t)g->E * g->S;
        if (per_rank)
            for (int r = 0; r < g->R; ++r) per_rank[r] = g->L * g->S;
        if (per_expert)
            for (int e = 0; e < g->E; ++e) per_expert[e] = g->S;
        return MOE_EP_OK;
    }
    // HT: the layout kernel publishes off[] and rcnt[] into mapped host memory
    // and then its route's sequence number; wait for that number only (not for
    // the rest of the stream), checking the stream now and then for errors.
    cudaStream_t s = (cudaStream_t)stream;
    const int E = g->E, R = g->R;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        cap = cudaStreamCaptureStatusNone;
    }
    if (cap == cudaStreamCaptureStatusActive) return MOE_EP_ERR_INVALID;  // a host wait
    if (h->T > 0 && h->captured) {
        // every replay of the captured route publishes the same sequence
        // number, so it cannot tell one replay's counts from the last one's:
        // wait for the stream (the replays on it) instead
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_EP_ERR_CUDA;
        const volatile unsigned* seq_word =
            reinterpret_cast<const volatile unsigned*>(h->host_counts + E + 1 + R + E);
        if (__atomic_load_n(seq_word, __ATOMIC_ACQUIRE) != h->seq) return MOE_EP_ERR_INVALID;
    } else if (h->T > 0) {
        volatile unsigned* seq_word = reinterpret_cast<volatile unsigned*>(h->host_counts + E + 1 + R + E);
        const auto t0 = std::chrono::steady_clock::now();
        for (uint64_t it = 1;; ++it) {
            if (__atomic_load_n(seq_word, __ATOMIC_ACQUIRE) == h->seq) break;
            if ((it & 4095u) == 0u) {
                const cudaError_t q = cudaStreamQuery(s);
                if (q != cudaSuccess && q != cudaErrorNotReady) return MOE_EP_ERR_CUDA;
                const bool idle = (q == cudaSuccess);
                const bool late = std::chrono::steady_clock::now() - t0 > std::chrono::seconds(10);
                if (idle || late) {
                    // everything on `stream` is done (or taking long): finish the
                    // device's work, then the words must be there
                    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_EP_ERR_CUDA;
                    if (__atomic_load_n(seq_word, __ATOMIC_ACQUIRE) != h->seq) return MOE_EP_ERR_CUDA;
                    break;
                }
            }
        }
    }
    st = check_group(g);
    if (st != MOE_EP_OK) return st;
    const int32_t* off = h->host_counts;
    const int64_t tot = (h->T > 0) ? off[E] : 0;
    *total = tot;
    h->host_total = tot;
    if (per_rank)
        for (int r = 0; r < R; ++r) per_rank[r] = (h->T > 0) ? off[E + 1 + r] : 0;
    if (per_expert)
        for (int x = 0; x < E; ++x) per_expert[x] = (h->T > 0) ? off[E + 1 + R + x] : 0;
    return MOE_EP_OK;
}

}  // extern "C"

namespace {

// moe_ep_dispatch, and with sig the send of moe_ep_dispatch_send.
int dispatch_impl(moe_ep_handle_t h, const void* x, int fp8, void* recv_x, float* recv_scale,
                  int32_t* recv_src, int32_t* recv_cnt, int64_t recv_rows, cudaStream_t stream,
                  const SendSignal& sig)
{
    if (!h) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!h->routed) return MOE_EP_ERR_INVALID;
    if (recv_rows < required_rows(h)) return MOE_EP_ERR_INVALID;
    if (h->T > 0 && (!x || !recv_x || !aligned16(x) || !aligned16(recv_x)))
        return MOE_EP_ERR_INVALID;
    if (fp8) {
        if (g->H % 128 != 0) return MOE_EP_ERR_INVALID;
        if (h->T > 0 && (!recv_scale || ((uintptr_t)recv_scale & 3u))) return MOE_EP_ERR_INVALID;
    }
    if (recv_src && ((uintptr_t)recv_src & 3u)) return MOE_EP_ERR_INVALID;
    if (recv_cnt && ((uintptr_t)recv_cnt & 3u)) return MOE_EP_ERR_INVALID;
    LayoutArgs fin = layout_args(h, h->T);
    RowArgs ra = row_args(h);
    ra.sig = sig;
    st = cuda_status(launch_dispatch(ra, x, g->H, fp8, h->row, recv_x, recv_scale, recv_src,
                                     h->cnt, recv_cnt, g->sm_count, stream,
                                     h->layout_pending ? &fin : nullptr, h->x_early));
    if (st == MOE_EP_OK) {
        h->rows_ready = 1;
        h->layout_pending = 0;
    }
    return st;
}

// moe_ep_combine, and with sig the send of moe_ep_combine_send.
int combine_impl(moe_ep_handle_t h, const void* y, const float* topk_w, void* out,
                 int64_t recv_rows, cudaStream_t stream, const SendSignal& sig)
{
    if (!h) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!h->routed) return MOE_EP_ERR_INVALID;
    if (recv_rows < required_rows(h)) return MOE_EP_ERR_INVALID;
    if (h->T > 0) {
        if (!y || !topk_w || !out || !aligned16(y) || !aligned16(out) || ((uintptr_t)topk_w & 3u))
            return MOE_EP_ERR_INVALID;
        // out must not overlap y
        const char* yb = (const char*)y;
        const char* ye = yb + (size_t)recv_rows * g->H * 2;
        const char* ob = (const char*)out;
        const char* oe = ob + (size_t)h->T * g->H * 2;
        if (ob < ye && yb < oe) return MOE_EP_ERR_INVALID;
    }
    st = ensure_rows(h, stream);
    if (st != MOE_EP_OK) return st;
    return cuda_status(launch_combine(y, h->T, g->H, h->k, h->row, topk_w, out, g->sm_count,
                                      stream, sig));
}

// The send kernels of one handle run in issue order: a send waits (on the
// device) for the handle's previous send, wherever it was enqueued.
int before_send(moe_ep_handle_t h, cudaStream_t send_stream, SendSignal* sig)
{
    if (!h) return MOE_EP_ERR_INVALID;
    int st = check_group(h->g);
    if (st != MOE_EP_OK) return st;
    if (h->pending && cudaStreamWaitEvent(send_stream, h->sent, 0) != cudaSuccess)
        return MOE_EP_ERR_CUDA;
    sig->arrive = h->send_arrive;
    sig->signal = h->send_signal;
    return MOE_EP_OK;
}

int after_send(moe_ep_handle_t h, cudaStream_t send_stream)
{
    if (cudaEventRecord(h->sent, send_stream) != cudaSuccess) return MOE_EP_ERR_CUDA;
    h->pending += 1;
    return MOE_EP_OK;
}

}  // namespace

extern "C" {

int moe_ep_dispatch(moe_ep_handle_t h, const void* x, int fp8, void* recv_x, float* recv_scale,
                    int32_t* recv_src, int32_t* recv_cnt, int64_t recv_rows,
                    moe_ep_stream_t stream)
{
    return dispatch_impl(h, x, fp8, recv_x, recv_scale, recv_src, recv_cnt, recv_rows,
                         (cudaStream_t)stream, SendSignal{});
}

int moe_ep_combine(moe_ep_handle_t h, const void* y, const float* topk_w, void* out,
                   int64_t recv_rows, moe_ep_stream_t stream)
{
    return combine_impl(h, y, topk_w, out, recv_rows, (cudaStream_t)stream, SendSignal{});
}

int moe_ep_dispatch_send(moe_ep_handle_t h, const void* x, int fp8, void* recv_x,
                         float* recv_scale, int32_t* recv_src, int32_t* recv_cnt,
                         int64_t recv_rows, moe_ep_stream_t send_stream)
{
    SendSignal sig;
    cudaStream_t s = (cudaStream_t)send_stream;
    int st = before_send(h, s, &sig);
    if (st == MOE_EP_OK)
        st = dispatch_impl(h, x, fp8, recv_x, recv_scale, recv_src, recv_cnt, recv_rows, s, sig);
    return st == MOE_EP_OK ? after_send(h, s) : st;
}

int moe_ep_combine_send(moe_ep_handle_t h, const void* y, const float* topk_w, void* out,
                        int64_t recv_rows, moe_ep_stream_t send_stream)
{
    SendSignal sig;
    cudaStream_t s = (cudaStream_t)send_stream;
    int st = before_send(h, s, &sig);
    if (st == MOE_EP_OK) st = combine_impl(h, y, topk_w, out, recv_rows, s, sig);
    return st == MOE_EP_OK ? after_send(h, s) : st;
}

int moe_ep_complete(moe_ep_handle_t h, moe_ep_stream_t stream)
{
    if (!h) return MOE_EP_ERR_INVALID;
    int st = check_group(h->g);
    if (st != MOE_EP_OK) return st;
    if (!h->pending) return MOE_EP_OK;
    cudaStream_t s = (cudaStream_t)stream;
    // order the receive after the sends (no kernel waits for one that may not
    // be running), then check on the device that every send has signalled
    if (cudaStreamWaitEvent(s, h->sent, 0) != cudaSuccess) return MOE_EP_ERR_CUDA;
    st = cuda_status(launch_wait_signal(h->send_signal, h->pending, kCompleteWaitNs,
                                        h->g->err_dev, s));
    if (st == MOE_EP_OK) h->pending = 0;
    return st;
}

int moe_ep_signal_add(moe_ep_group_t g, uint32_t* signal, uint32_t value, moe_ep_stream_t stream)
{
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!signal || ((uintptr_t)signal & 3u)) return MOE_EP_ERR_INVALID;
    return cuda_status(launch_signal_add(signal, value, (cudaStream_t)stream));
}

int moe_ep_wait_signal(moe_ep_group_t g, uint32_t* signal, uint32_t expected, int64_t timeout_ns,
                       moe_ep_stream_t stream)
{
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!signal || ((uintptr_t)signal & 3u) || timeout_ns <= 0 || timeout_ns > kMaxWaitNs)
        return MOE_EP_ERR_INVALID;
    return cuda_status(launch_wait_signal(signal, expected, (uint64_t)timeout_ns, g->err_dev,
                                          (cudaStream_t)stream));
}

int moe_ep_set_row_align(moe_ep_handle_t h, int align)
{
    if (!h || align < 1 || align > 1024 || (align & (align - 1)) != 0) return MOE_EP_ERR_INVALID;
    if (h->g->mode != MOE_EP_HT && align != 1) return MOE_EP_ERR_INVALID;
    h->align = align;
    return MOE_EP_OK;
}

int moe_ep_set_x_before_route(moe_ep_handle_t h, int on)
{
    if (!h || (on != 0 && on != 1)) return MOE_EP_ERR_INVALID;
    h->x_early = on;
    return MOE_EP_OK;
}

int moe_ep_dequant(moe_ep_handle_t h, const void* recv_q, const float* recv_scale, void* y,
                   int64_t recv_rows, moe_ep_stream_t stream)
{
    if (!h) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!h->routed) return MOE_EP_ERR_INVALID;
    if (g->H % 128 != 0) return MOE_EP_ERR_INVALID;
    if (recv_rows < required_rows(h)) return MOE_EP_ERR_INVALID;
    if (h->T == 0) return MOE_EP_OK;
    if (!recv_q || !recv_scale || !y || !aligned16(recv_q) || !aligned16(y) ||
        ((uintptr_t)recv_scale & 3u))
        return MOE_EP_ERR_INVALID;
    st = ensure_counts(h, (cudaStream_t)stream);
    if (st != MOE_EP_OK) return st;
    return cuda_status(launch_dequant(h->cnt, h->off, g->E, g->S, g->mode, g->H,
                                      (const uint8_t*)recv_q, recv_scale, y,
                                      (int64_t)h->T * h->k, g->sm_count, g->err_dev,
                                      (cudaStream_t)stream));
}

int moe_ep_node_layout(moe_ep_handle_t h, int num_nodes, int src_node, int32_t* node_cnt,
                       int32_t* node_off, int32_t* node_src, uint32_t* node_mask,
                       int64_t node_rows, int64_t* stats, moe_ep_stream_t stream)
{
    if (!h) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!h->routed) return MOE_EP_ERR_INVALID;
    const int N = num_nodes;
    if (N < 1 || N > g->R || g->R % N != 0 || g->R / N > 32 || src_node < 0 || src_node >= N)
        return MOE_EP_ERR_INVALID;
    if (!node_cnt || !node_off) return MOE_EP_ERR_INVALID;
    const int T = h->T, k = h->k;
    if (T > 0 && (!node_src || !node_mask)) return MOE_EP_ERR_INVALID;
    if (node_rows < (int64_t)T * (k < N ? k : N)) return MOE_EP_ERR_INVALID;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (stats) e = cudaMemsetAsync(stats, 0, 4 * sizeof(int64_t), s);
    if (e == cudaSuccess && T == 0) {
        e = cudaMemsetAsync(node_cnt, 0, sizeof(int32_t) * (size_t)N, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(node_off, 0, sizeof(int32_t) * (size_t)(N + 1), s);
        return cuda_status(e);
    }
    if (e != cudaSuccess) return MOE_EP_ERR_CUDA;
    NodeArgs a;
    a.idx = h->idx;
    a.T = T;
    a.k = k;
    a.E = g->E;
    a.L = g->L;
    a.gpn = g->R / N;
    a.N = N;
    a.src = src_node;
    LayoutArgs la;
    la.tile_word = h->ntile_word;
    la.tile_cnt = h->ntile_cnt;
    la.grp_base = h->ngrp_base;
    la.cnt = node_cnt;
    la.off = node_off;
    la.rcnt = node_cnt;  // one "rank" per node: the same sums
    la.roff = node_off;
    la.done = h->ndone;
    la.E = N;
    la.R = N;
    la.ntiles = (T + kTileTokens - 1) / kTileTokens;
    la.host_out = nullptr;
    la.seq = 0u;
    la.align = 1;
    return cuda_status(launch_node_layout(a, la, reinterpret_cast<unsigned long long*>(stats),
                                          node_src, node_mask, g->sm_count, s));
}

int moe_ep_dispatch_dedup(moe_ep_handle_t h, const void* x, int fp8, void* drecv_x,
                          float* drecv_scale, int32_t* drecv_src, uint32_t* drecv_mask,
                          int32_t* rank_cnt, int32_t* rank_off, int64_t drecv_rows,
                          moe_ep_stream_t stream)
{
    if (!h) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!h->routed || g->mode != MOE_EP_HT || g->L > 32) return MOE_EP_ERR_INVALID;
    if (drecv_rows < dedup_capacity(h)) return MOE_EP_ERR_INVALID;
    if (h->T > 0 && (!x || !drecv_x || !aligned16(x) || !aligned16(drecv_x)))
        return MOE_EP_ERR_INVALID;
    if (fp8) {
        if (g->H % 128 != 0) return MOE_EP_ERR_INVALID;
        if (h->T > 0 && (!drecv_scale || ((uintptr_t)drecv_scale & 3u))) return MOE_EP_ERR_INVALID;
    }
    if (((uintptr_t)drecv_src & 3u) || ((uintptr_t)drecv_mask & 3u) ||
        ((uintptr_t)rank_cnt & 3u) || ((uintptr_t)rank_off & 3u))
        return MOE_EP_ERR_INVALID;
    cudaStream_t s = (cudaStream_t)stream;
    const int T = h->T;
    cudaError_t e = cudaSuccess;
    if (T == 0) {
        e = cudaMemsetAsync(h->rk_cnt, 0, sizeof(int32_t) * g->R, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(h->rk_off, 0, sizeof(int32_t) * (g->R + 1), s);
    } else {
        // the layout over ranks: the node layout with one "GPU" per expert and
        // one "node" per rank (GPU mask bits = local experts)
        NodeArgs na;
        na.idx = h->idx;
        na.T = T;
        na.k = h->k;
        na.E = g->E;
        na.L = 1;
        na.gpn = g->L;
        na.N = g->R;
        na.src = 0;
        LayoutArgs la;
        la.tile_word = h->rtile_word;
        la.tile_cnt = h->rtile_cnt;
        la.grp_base = h->rgrp_base;
        la.cnt = h->rk_cnt;
        la.off = h->rk_off;
        la.rcnt = h->rk_cnt;  // one "rank" per column: the same sums
        la.roff = h->rk_off;
        la.done = h->rdone;
        la.E = g->R;
        la.R = g->R;
        la.ntiles = (T + kTileTokens - 1) / kTileTokens;
        la.host_out = nullptr;
        la.seq = 0u;
        la.align = 1;
        e = launch_node_layout(na, la, nullptr, nullptr, nullptr, g->sm_count, s);
        if (e == cudaSuccess) {
            RowArgs ra;
            ra.idx = h->idx;
            ra.tile_word = h->rtile_word;
            ra.tile_cnt = h->rtile_cnt;
            ra.grp_base = h->rgrp_base;
            ra.off = h->rk_off;
            ra.T = T;
            ra.k = h->k;
            ra.E = g->E;
            ra.S = g->S;
            ra.mode = MOE_EP_HT;
            ra.G = g->L;
            ra.ncols = g->R;
            ra.mask = drecv_mask;
            ra.off_out = rank_off;
            e = launch_dispatch(ra, x, g->H, fp8, h->drow, drecv_x, drecv_scale, drecv_src,
                                h->rk_cnt, rank_cnt, g->sm_count, s, nullptr, h->x_early);
        }
    }
    if (T == 0) {
        if (e == cudaSuccess && rank_cnt) e = cudaMemsetAsync(rank_cnt, 0, sizeof(int32_t) * g->R, s);
        if (e == cudaSuccess && rank_off)
            e = cudaMemsetAsync(rank_off, 0, sizeof(int32_t) * (g->R + 1), s);
    }
    if (e != cudaSuccess) return MOE_EP_ERR_CUDA;
    h->dedup_ready = 1;
    return MOE_EP_OK;
}

int moe_ep_expand(moe_ep_handle_t h, const void* drecv_x, const float* drecv_scale,
                  const int32_t* drecv_src, const uint32_t* drecv_mask, int fp8, void* recv_x,
                  float* recv_scale, int32_t* recv_src, int64_t recv_rows, moe_ep_stream_t stream)
{
    if (!h) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!h->dedup_ready) return MOE_EP_ERR_INVALID;
    if (recv_rows < required_rows(h)) return MOE_EP_ERR_INVALID;
    if (h->T == 0) return MOE_EP_OK;
    if (!drecv_x || !drecv_src || !drecv_mask || !recv_x || !aligned16(drecv_x) ||
        !aligned16(recv_x) || ((uintptr_t)drecv_src & 3u) || ((uintptr_t)drecv_mask & 3u) ||
        ((uintptr_t)recv_src & 3u))
        return MOE_EP_ERR_INVALID;
    if (fp8 && (g->H % 128 != 0 || !drecv_scale || !recv_scale ||
                ((uintptr_t)drecv_scale & 3u) || ((uintptr_t)recv_scale & 3u)))
        return MOE_EP_ERR_INVALID;
    DedupArgs a;
    a.ex = row_args(h);
    a.rank_off = h->rk_off;
    a.dsrc = drecv_src;
    a.dmask = drecv_mask;
    a.R = g->R;
    a.L = g->L;
    const int row_bytes = fp8 ? g->H : 2 * g->H;
    return cuda_status(launch_expand(a, drecv_x, fp8 ? drecv_scale : nullptr, row_bytes,
                                     g->H / 128, recv_x, fp8 ? recv_scale : nullptr, recv_src,
                                     (int)dedup_capacity(h), g->sm_count, (cudaStream_t)stream));
}

int moe_ep_combine_dedup(moe_ep_handle_t h, const void* y, const float* topk_w,
                         const int32_t* drecv_src, void* partial, void* out, int64_t recv_rows,
                         int64_t drecv_rows, moe_ep_stream_t stream)
{
    if (!h) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    int st = check_group(g);
    if (st != MOE_EP_OK) return st;
    if (!h->dedup_ready) return MOE_EP_ERR_INVALID;
    if (recv_rows < required_rows(h) || drecv_rows < dedup_capacity(h)) return MOE_EP_ERR_INVALID;
    if (h->T == 0) return MOE_EP_OK;
    if (!y || !topk_w || !drecv_src || !partial || !out || !aligned16(y) || !aligned16(partial) ||
        !aligned16(out) || ((uintptr_t)topk_w & 3u) || ((uintptr_t)drecv_src & 3u))
        return MOE_EP_ERR_INVALID;
    // the partial rows must not overlap y or out
    const size_t rb = (size_t)g->H * 2;
    const char* pb = (const char*)partial;
    const char* pe = pb + (size_t)drecv_rows * rb;
    const char* yb = (const char*)y;
    const char* ye = yb + (size_t)recv_rows * rb;
    const char* ob = (const char*)out;
    const char* oe = ob + (size_t)h->T * rb;
    if ((pb < ye && yb < pe) || (pb < oe && ob < pe) || (ob < ye && yb < oe))
        return MOE_EP_ERR_INVALID;
    cudaStream_t s = (cudaStream_t)stream;
    st = ensure_rows(h, s);
    if (st != MOE_EP_OK) return st;
    st = cuda_status(launch_combine_partial(row_args(h), h->row, h->drow, g->L, topk_w, y, g->H,
                                            partial, g->sm_count, s));
    if (st != MOE_EP_OK) return st;
    // the source adds its ranks' partial rows: weights 1, dedup row map
    return cuda_status(launch_combine(partial, h->T, g->H, h->k, h->drow, nullptr, out,
                                      g->sm_count, s));
}

int moe_ep_copy_layout(moe_ep_handle_t h, int32_t* cnt, int32_t* off, int32_t* rcnt, int32_t* roff,
                       int32_t* row, moe_ep_stream_t stream)
{
    if (!h) return MOE_EP_ERR_INVALID;
    if (!h->routed) return MOE_EP_ERR_INVALID;
    moe_ep_group* g = h->g;
    cudaStream_t s = (cudaStream_t)stream;
    if (row && h->T > 0) {
        int st = ensure_rows(h, s);
        if (st != MOE_EP_OK) return st;
    }
    int st = ensure_counts(h, s);
    if (st != MOE_EP_OK) return st;
    cudaError_t e = cudaSuccess;
    if (cnt && e == cudaSuccess)
        e = cudaMemcpyAsync(cnt, h->cnt, sizeof(int32_t) * g->E, cudaMemcpyDefault, s);
    if (off && e == cudaSuccess)
        e = cudaMemcpyAsync(off, h->off, sizeof(int32_t) * (g->E + 1), cudaMemcpyDefault, s);
    if (rcnt && e == cudaSuccess)
        e = cudaMemcpyAsync(rcnt, h->rcnt, sizeof(int32_t) * g->R, cudaMemcpyDefault, s);
    if (roff && e == cudaSuccess)
        e = cudaMemcpyAsync(roff, h->roff, sizeof(int32_t) * (g->R + 1), cudaMemcpyDefault, s);
    if (row && e == cudaSuccess && h->T > 0)
        e = cudaMemcpyAsync(row, h->row, sizeof(int32_t) * (size_t)h->T * h->k, cudaMemcpyDefault,
                            s);
    return cuda_status(e);
}

int moe_ep_get_device_errors(moe_ep_group_t g, uint32_t* bits)
{
    if (!g || !bits) return MOE_EP_ERR_INVALID;
    uint32_t b = 0;
    if (g->err_host[kErrRange]) b |= MOE_EP_DEVERR_EXPERT_RANGE;
    if (g->err_host[kErrDuplicate]) b |= MOE_EP_DEVERR_DUPLICATE;
    if (g->err_host[kErrTimeout]) b |= MOE_EP_DEVERR_TIMEOUT;
    *bits = b;
    return MOE_EP_OK;
}

int moe_ep_clear_device_errors(moe_ep_group_t g)
{
    if (!g) return MOE_EP_ERR_INVALID;
    for (int i = 0; i < kErrSlots; ++i) g->err_host[i] = 0u;
    return MOE_EP_OK;
}

}  // extern "C"
