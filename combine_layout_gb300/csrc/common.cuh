// Internal declarations shared by the libmoeep translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_ep.h"

namespace moeep {

// Layout tiles hold 32 tokens so that one expert's presence in a tile is one
// 32-bit word (bit i = token tile*32 + i chose that expert).
constexpr int kTileTokens = 32;
// Tiles per group of the layout's byte counts.
constexpr int kGroupTiles = 16;
// The most tiles of a deferred LL layout (LayoutArgs.deferred): its
// consumers sum the earlier tiles' words directly, two loads at a time.
constexpr int kDeferMaxTiles = 8;
constexpr int kMaxTopk = 32;
constexpr int kMaxGroups = 32;
constexpr int kMaxGroupTopk = 4;
constexpr int kMaxExpertsPerLane = 16;
constexpr int kMaxExperts = 512;

// Slots of the device-error word array (each written with a plain store).
constexpr int kErrSlots = 4;
constexpr int kErrRange = 0;
constexpr int kErrDuplicate = 1;
constexpr int kErrTimeout = 2;  // a bounded wait inside a kernel gave up

// Every kernel of the library is launched with programmatic stream
// serialization: its CTAs may become resident while the kernel before it on
// the stream is still finishing (launch latency and that kernel's tail
// overlap), and each kernel executes griddep_wait() before its first global
// memory access, which returns once the kernels before it have completed and
// their writes are visible (the one exception: the bf16 dispatch's token
// loads when the caller declared x complete before the route).  Kernels that
// produce a layout signal their dependents as soon as every CTA has written
// its tile (the grid's last CTA then finishes the layout while the next
// kernel's CTAs are being placed).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_smem(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                       Args... args)
{
    return launch_pdl_smem(kernel, grid, block, 0, s, args...);
}

#ifdef __CUDACC__
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// Completion signal of a send-only dispatch or combine ("NCCL EP 论文解读",
// item "send_only与双buffer": the send and the receive are separate kernels).
// arrive counts the CTAs of the send kernel that have finished (the last one
// resets it to 0); signal counts the sends that have landed and that no
// receive has consumed yet.  Both null: not a send-only launch.
struct SendSignal {
    unsigned* arrive = nullptr;
    unsigned* signal = nullptr;
};

#ifdef __CUDACC__
// Called once by every CTA of a send kernel, with all its threads, after its
// last store.  The barrier orders the CTA's stores before thread 0's arrival
// (an atomic add with acquire-release semantics at GPU scope); the last CTA
// to arrive has acquired every other CTA's stores and publishes them all
// with its release add on the signal.
__device__ __forceinline__ void send_arrive(const SendSignal& sig)
{
    if (!sig.signal) return;  // uniform across the grid
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(sig.arrive)
                     : "memory");
        if (prev == gridDim.x - 1) {
            // the next send kernel starts after this grid has completed
            *sig.arrive = 0u;
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(sig.signal) : "memory");
        }
    }
}
#endif

struct RouteParams {
    int E;      // experts
    int G;      // routing groups (nodes)
    int kg;     // groups kept
    int m;      // scores summed per group
    int k;      // experts per token
    int wmode;  // moe_ep_weight_mode_t
    int gs;     // experts per group
    int lpg;    // lanes per group (power of two, lpg * G <= 32)
    int lpg_log2;
    int epl;    // experts held per lane
    int limit;  // 1 when some groups are banned
    int vec4;   // 1 when every lane's experts can be read as float4
};

// Where the layout lives (the handle's workspace).
struct LayoutArgs {
    uint32_t* tile_word;  // [ntiles][E]
    uint8_t* tile_cnt;    // [ngroups][E][16], popc of tile_word (groups of 16 tiles)
    int32_t* grp_base;    // [ngroups][E], pairs before each group of 16 tiles
    int32_t* cnt;         // [E]
    int32_t* off;         // [E+1]
    int32_t* rcnt;        // [R]
    int32_t* roff;        // [R+1]
    unsigned* done;       // CTAs finished (reset to 0 by the last one)
    int E, R, ntiles;
    int align;            // expert blocks padded to a multiple of align rows (1: none)
    // Work split of the last CTA, set on the host for the launch's block size
    // (tail_planned in layout_dev.cuh): experts per rank, column-pass columns,
    // parts and groups per part, experts per prefix thread, prefix threads,
    // threads that take part at all.
    int L, cols, parts, rg, per, nact, nwork;
    // 1: the producers wrote only tile_word (a tile's word assembled from the
    // bytes of several CTAs); the last CTA derives tile_cnt from the words
    // and writes it.  Only with ntiles <= 32 (at most two groups).
    int cnt_from_words = 0;
    // 1: the producers write only tile_word and skip the last-CTA tail; the
    // layout's consumers rank pairs from the words (RowArgs.from_words) and
    // the first of them finishes cnt / off / rcnt / roff
    // (finish_layout_from_words).  LL layouts of at most kDeferMaxTiles
    // tiles only.
    int deferred = 0;
    // Optional publication of the counts to the host (mapped pinned memory,
    // device alias): off[E+1], rcnt[R], cnt[E], then the sequence number
    // `seq`, written last, after a system-scope fence.  nullptr: none.
    int32_t* host_out;
    unsigned seq;
};

// What placing a pair into its receive row needs.  Columns of the layout are
// blocks of G consecutive experts (G = 1: experts; G = E/R: ranks, one row
// per (token, rank) at the token's first pair on that rank).
struct RowArgs {
    const int32_t* idx;        // handle copy of topk_idx [T][k]
    const uint32_t* tile_word;
    const uint8_t* tile_cnt;
    const int32_t* grp_base;
    const int32_t* off;
    int T, k, E, S, mode;
    int G;                     // experts per column
    int ncols;                 // E / G
    uint32_t* mask;            // G > 1: per row, bit l = local expert l of the token (may be null)
    int32_t* off_out;          // dispatch: copy of off[0 .. ncols] (may be null)
    int from_words = 0;        // 1: rank pairs from the tile words alone (deferred LL layout)
    SendSignal sig;            // dispatch: set for a send-only launch
};

// What the receiver side of the per-rank dedup path needs: the expert layout
// (G = 1) and the dedup rows' ranks, tokens and local-expert masks.
struct DedupArgs {
    RowArgs ex;
    const int32_t* rank_off;  // [R+1]
    const int32_t* dsrc;      // [dedup rows] token
    const uint32_t* dmask;    // [dedup rows] bit l: local expert l of the row's rank
    int R, L;
};

// What the node-level layout needs.
struct NodeArgs {
    const int32_t* idx;  // handle copy of topk_idx [T][k]
    int T, k, E;
    int L;               // experts per GPU (rank)
    int gpn;             // GPUs per node
    int N;               // nodes
    int src;             // source node
};

// Router: one warp per token, one 32-token tile per CTA.  Writes topk_idx
// (caller's and the handle's copy), topk_w, the tile words and byte counts,
// and -- in the last CTA to finish -- grp_base, cnt, off, rcnt, roff.
cudaError_t launch_route(const float* scores, int T, const RouteParams& p, int32_t* topk_idx,
                         int32_t* idx_copy, float* topk_w, const LayoutArgs& la, cudaStream_t s);

// Same layout from caller-made topk_idx, with validity checks.
cudaError_t launch_layout_bits(const int32_t* topk_idx, int T, int k, int32_t* idx_copy,
                               const LayoutArgs& la, volatile unsigned* err, cudaStream_t s);

// Row map row[t][j] (dispatch writes it itself; this serves combine or a
// layout copy that comes without a dispatch).
cudaError_t launch_rowmap(const RowArgs& ra, int32_t* row, int sm_count, cudaStream_t s);

// Counts and offsets of a deferred layout (la.deferred) from its tile words:
// one CTA (the dispatch does the same in its first CTA).
cudaError_t launch_finish_words(const LayoutArgs& la, cudaStream_t s);

// Column slices per token for small batches: the smallest divisor of
// `units` (equal slices of a row) that puts about two CTAs on every SM;
// 1 when the tokens alone do.
int slices_for(int T, int units, int sm_count);

// Work items of a token-parallel kernel (one CTA per item): tokens [0, th)
// in nsa equal column slices each, tokens [th, T) in nsb.  Small batches:
// th = T and nsa = slices_for (enough items to fill the GPU).  Large
// batches: nsa = 1 and the last few hundred tokens in nsb short slices, so
// the launch's last wave is made of short items and the SMs run out of work
// at nearly the same time (one CTA per whole token leaves SMs idle for up to
// a token's duration at the end).  Rows are split in units of 16 vectors.
struct TokenSplit {
    int th;
    int nsa;
    int nsb;
};

__host__ __device__ inline int split_items(const TokenSplit& s, int T)
{
    return s.th * s.nsa + (T - s.th) * s.nsb;
}

// The split for T tokens of `units` 16-vector units each, the tail's slices
// at most max_slice_units long; no sliced tail below min_tokens tokens.
TokenSplit token_split(int T, int units, int sm_count, int max_slice_units, int min_tokens);

#ifdef __CUDACC__
// Token and vector range [vb, ve) of work item b (nvec vectors per row).
__device__ __forceinline__ void split_item(const TokenSplit& s, int b, int nvec, int& t, int& vb,
                                           int& ve)
{
    int sl, ns;
    if (b < s.th * s.nsa) {
        ns = s.nsa;
        t = b / ns;
        sl = b - t * ns;
    } else {
        ns = s.nsb;
        const int q = b - s.th * s.nsa;
        const int u = q / ns;
        sl = q - u * ns;
        t = s.th + u;
    }
    const int ch = nvec / ns;
    vb = sl * ch;
    ve = vb + ch;
}
#endif

// Dispatch pack: x bf16 [T][H] -> receive rows (bf16 copy or FP8 + scales).
// Also writes the row map and recv_src, and copies cnt into recv_cnt -- or,
// with fin != nullptr (a deferred layout), its first CTA finishes the
// layout's counts and offsets from the tile words and writes recv_cnt.
// early: x was complete before the layout's producer started, so each bf16
// CTA reads its first token before waiting for that producer (the FP8
// kernels read after the wait: measured no faster with the early read).
cudaError_t launch_dispatch(const RowArgs& ra, const void* x, int H, int fp8, int32_t* row,
                            void* recv_x, float* recv_scale, int32_t* recv_src,
                            const int32_t* cnt, int32_t* recv_cnt, int sm_count, cudaStream_t s,
                            const LayoutArgs* fin = nullptr, int early = 0);

// Node-level layout (node counts, offsets, rows with GPU masks) and the
// routing statistics (stats may be null; otherwise 4 sums, accumulated).
// node_src == nullptr: the layout (counts, offsets, tile words) only.
cudaError_t launch_node_layout(const NodeArgs& a, const LayoutArgs& la, unsigned long long* stats,
                               int32_t* node_src, uint32_t* node_mask, int sm_count, cudaStream_t s);

// Receive-side dequantisation of the rows the layout defines:
// y = bf16_rn(float(q) * scale) (fp32 product).
// err: the group's device-error word (kErrTimeout is latched there if a
// bounded wait of the TMA-staged variant gives up).
// max_rows: an upper bound of the defined rows (sizes the grid).
cudaError_t launch_dequant(const int32_t* cnt, const int32_t* off, int E, int S, int mode, int H,
                           const uint8_t* q, const float* scale, void* y, int64_t max_rows,
                           int sm_count, unsigned* err, cudaStream_t s);

// Per-rank dedup, receiver side: copy every dedup row to the HT rows of its
// local experts (row_bytes per row, nblk scales per row when dscale is set),
// and the per-rank BF16 partial weighted sums.  max_rows bounds the grid;
// the kernels read the number of dedup rows from rank_off[R].
cudaError_t launch_expand(const DedupArgs& a, const void* dx, const float* dscale, int row_bytes,
                          int nblk, void* recv_x, float* recv_scale, int32_t* recv_src,
                          int max_rows, int sm_count, cudaStream_t s);
// The partials: for each token (ex.idx, ex.T, ex.k, ex.E), its pairs' expert
// rows row[t][j], dedup rows drow[t][j] (the first pair of each rank), L
// experts per rank.
cudaError_t launch_combine_partial(const RowArgs& ex, const int32_t* row, const int32_t* drow,
                                   int L, const float* w, const void* y, int H, void* partial,
                                   int sm_count, cudaStream_t s);

// Combine: out[t] = bf16(sum_j w[t][j] * y[row[t][j]]) (w == nullptr: weights 1).
// sig: set for a send-only launch (then a grid is launched even for T = 0, so
// the signal still arrives).
cudaError_t launch_combine(const void* y, int T, int H, int k, const int32_t* row, const float* w,
                           void* out, int sm_count, cudaStream_t s,
                           const SendSignal& sig = SendSignal{});

// Receive side of a send-only operation: one thread waits (at most limit_ns,
// and a bounded number of polls) until *signal >= expected, then subtracts
// expected; when the bound passes first it latches err[kErrTimeout].
cudaError_t launch_wait_signal(uint32_t* signal, uint32_t expected, uint64_t limit_ns,
                               unsigned* err, cudaStream_t s);
// *signal += value with release semantics at GPU scope, after the work before
// it on the stream.
cudaError_t launch_signal_add(uint32_t* signal, uint32_t value, cudaStream_t s);

}  // namespace moeep
