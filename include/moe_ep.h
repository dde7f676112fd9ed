/*
 * moe_ep.h -- C ABI of libmoeep: MoE expert-parallel token dispatch and combine
 * on one GPU (sm_103a), destination ranks being logical partitions of the GPU's
 * own memory.
 *
 * The calls follow the statement of the problem on "NCCL EP 论文解读" (lpnh.cn),
 * item "核心功能函数": a group holds the resources shared across operations, a
 * handle holds one forward pass's routing state created from topk_idx, dispatch
 * sends tokens to their experts, combine gathers them back into the original
 * token order and reduces them, and a receive-count query serves buffer sizing.
 * The two algorithm modes are those of item "算法模式" and of
 * "NVSHMEM 与 DeepEP：GPU 发起的通信" (anrans.github.io), sections "高吞吐模式" (HT)
 * and "低延迟模式" (LL).
 *
 * Conventions for every call:
 *  - Pointers marked "device" must point to memory the current CUDA device can
 *    access; "host" pointers are ordinary host memory.  The caller owns every
 *    buffer passed in or out; the library owns only the workspace of groups
 *    and handles, allocated once at creation (nothing is allocated per call).
 *  - Every call is asynchronous on the given stream except where stated.  A
 *    NULL stream is the legacy default stream.
 *  - bf16 buffers are passed as void* holding IEEE bfloat16 bit patterns;
 *    fp8 buffers hold OCP e4m3fn bytes.  All integers are int32 unless stated.
 *  - Every call returns a moe_ep_status_t.  Argument and capacity errors are
 *    found on the host before any launch.  Invalid data found on the device
 *    (an expert id out of range, an expert repeated within a token) never
 *    causes an out-of-bounds access: the pair is dropped and a bit is latched
 *    in the group's device-error word, which is visible to the host without a
 *    synchronisation once the kernel has finished; while it is set every call
 *    on the group returns MOE_EP_ERR_DEVICE (MOE_EP_ERR_TIMEOUT when a
 *    bounded wait gave up) until moe_ep_clear_device_errors.
 *    Kernels never trap and never wait on a kernel that may still be
 *    running: the only waits are on a CTA's own bulk copies and on signal
 *    words whose producers are ordered before the waiting kernel, each
 *    bounded.
 *  - A handle's workspace is reused by each moe_ep_route call: use one handle
 *    per forward pass in flight (for instance one per layer).
 */
#ifndef MOE_EP_H
#define MOE_EP_H

#include <stdint.h>

#if defined(__GNUC__)
#define MOE_EP_API __attribute__((visibility("default")))
#else
#define MOE_EP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* moe_ep_stream_t;

typedef enum {
    MOE_EP_LL = 0, /* low latency: fixed worst-case slots, no count exchange */
    MOE_EP_HT = 1  /* high throughput: dense 2D receive layout, counts known after one sync */
} moe_ep_mode_t;

typedef enum {
    MOE_EP_OK = 0,
    MOE_EP_ERR_INVALID = 1,  /* bad argument, shape or alignment */
    MOE_EP_ERR_OVERFLOW = 2, /* more tokens than the group's max_tokens (LL slots) */
    MOE_EP_ERR_CUDA = 3,     /* a CUDA runtime call or launch failed */
    MOE_EP_ERR_DEVICE = 4,   /* device-error word set (see moe_ep_get_device_errors) */
    MOE_EP_ERR_TIMEOUT = 5   /* device-error word holds MOE_EP_DEVERR_TIMEOUT: a
                                bounded wait inside a kernel gave up */
} moe_ep_status_t;

/* Bits of the device-error word. */
#define MOE_EP_DEVERR_EXPERT_RANGE 1u /* a topk_idx entry outside [-1, experts) */
#define MOE_EP_DEVERR_DUPLICATE 2u    /* an expert repeated within one token */
#define MOE_EP_DEVERR_TIMEOUT 4u      /* a bounded wait inside a kernel gave up (the
                                         kernel latched it, skipped the rest of its
                                         work and returned; outputs are incomplete) */

typedef enum {
    MOE_EP_W_SOFTMAX_TOPK = 0,   /* w_j = softmax over the k selected scores */
    MOE_EP_W_SOFTMAX_RENORM = 1, /* softmax over all experts, renormalised over the k */
    MOE_EP_W_SCORE_NORM = 2      /* w_j = s_j / sum of the k selected scores */
} moe_ep_weight_mode_t;

typedef struct moe_ep_group* moe_ep_group_t;
typedef struct moe_ep_handle* moe_ep_handle_t;

/* Routing options ("NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": keep the
 * best topk_groups nodes by the sum of each node's group_topk best expert
 * scores, then take the topk best experts among them). */
typedef struct {
    int topk;        /* k, experts per token, 1..32 */
    int num_groups;  /* G, routing groups (nodes); experts split into G contiguous blocks; 1 = no limit */
    int topk_groups; /* groups kept per token, 1..G */
    int group_topk;  /* scores summed per group, 1..4; 0 = ceil(topk / topk_groups) */
    int weight_mode; /* moe_ep_weight_mode_t */
} moe_ep_route_opts_t;

/* Create a communication group ("核心功能函数": ncclEpCreateGroup picks the
 * algorithm mode, the expert count, the maximum tokens per rank and the buffer
 * sizes).  experts E are split over `ranks` R logical ranks in contiguous blocks
 * of L = E / R ("Moe模型": E experts placed blockwise over N ranks); rank r
 * belongs to no physical device other than the current one.  max_tokens bounds
 * the tokens of one forward; in LL mode it is also the slot count S per
 * (rank, local expert) ("低延迟模式": num_max_dispatch_tokens_per_rank).
 * hidden H is the token width in elements, a multiple of 8 (128 for FP8).
 * Synchronous.  Allocates the group's device-error word on the current device.
 * Errors: MOE_EP_ERR_INVALID for E % R != 0, E > 512, non-positive sizes,
 * H % 8 != 0; MOE_EP_ERR_CUDA if the device cannot be queried or allocated. */
MOE_EP_API int moe_ep_create_group(moe_ep_group_t* out, int mode, int experts, int ranks, int max_tokens,
                        int hidden);
/* Frees the group.  Its handles must have been destroyed first
 * (MOE_EP_ERR_INVALID otherwise).  Synchronous (waits for the device). */
MOE_EP_API int moe_ep_destroy_group(moe_ep_group_t g);

/* Create a routing handle ("核心功能函数": ncclEpCreateHandle, one per forward
 * pass, shared by the matching dispatch and combine).  Allocates, once, the
 * device workspace for max_tokens x max_topk pairs: per-tile expert bitmaps,
 * column prefixes, counts, offsets and the row map.  Synchronous. */
MOE_EP_API int moe_ep_create_handle(moe_ep_group_t g, int max_topk, moe_ep_handle_t* out);
MOE_EP_API int moe_ep_destroy_handle(moe_ep_handle_t h);

/* Route num_tokens tokens and lay out their (token, j) pairs.
 * scores   device fp32 [T][E] row-major, or NULL: then topk_idx is an input
 *          (routing made by the caller) and topk_w is not touched.
 * topk_idx device int32 [T][k]: output (or input when scores == NULL).  Row t
 *          lists token t's experts best first (score descending, lower index
 *          on ties).  As an input, -1 masks a pair (it gets no row).
 * topk_w   device fp32 [T][k], output weights per opts->weight_mode; may be NULL.
 * Layout (HT): expert e's pairs occupy receive rows [off[e], off[e+1]) in
 * ascending token order, i.e. rows are ordered by (rank, local expert, token)
 * ("算法模式": deterministic order, per-expert counts mark the boundaries).
 * Layout (LL): pair (t, j) with expert e = r * L + l goes to slot
 * s = #(earlier tokens of e) of row e * S + s, i.e. [r][l][s] of the
 * [R][L][S][H] receive buffer ("Tensor Layouts": 3D expert-major).
 * Errors: MOE_EP_ERR_OVERFLOW if num_tokens > max_tokens; MOE_EP_ERR_INVALID
 * for bad options (k > max_topk, E % G, G > 32, kg * E / G < k, ...). */
MOE_EP_API int moe_ep_route(moe_ep_handle_t h, const float* scores, int num_tokens,
                 const moe_ep_route_opts_t* opts, int32_t* topk_idx, float* topk_w,
                 moe_ep_stream_t stream);

/* Receive-token query ("核心功能函数": ncclEpHandleGetNumRecvTokens, used for
 * buffer sizing).  HT: returns the total receive rows and, if non-NULL, the
 * per-rank [R] and per-expert [E] counts on the host -- the one host
 * synchronisation of HT mode ("高吞吐模式": the CPU must learn the receive size).
 * The layout of moe_ep_route publishes these counts into mapped host memory
 * itself, so the call waits (host-side) for that layout only, not for work
 * queued after it (a dispatch or combine already launched keeps running); on
 * an error or a stall of more than 10 s it falls back to synchronising the
 * device.  `stream` is only used for that check.  HT forward recorded into a
 * CUDA graph (the handle's last moe_ep_route was called during a stream
 * capture): every replay publishes the counts under the same sequence number,
 * so the call synchronises `stream` -- pass the stream the graph is replayed
 * on -- and returns the counts of the last replay that completed on it
 * (MOE_EP_ERR_INVALID if none has run yet).  Called while `stream` is being
 * captured (a host wait cannot be recorded): MOE_EP_ERR_INVALID.  LL: returns the fixed
 * capacity without any synchronisation ("低延迟模式": no count exchange):
 * total = E * S, per_rank[r] = L * S, per_expert[e] = S.
 * total, per_rank, per_expert: host pointers (per_rank/per_expert may be NULL). */
MOE_EP_API int moe_ep_get_num_recv_tokens(moe_ep_handle_t h, int64_t* total, int32_t* per_rank,
                               int32_t* per_expert, moe_ep_stream_t stream);

/* Dispatch ("核心功能函数": ncclEpDispatch; "通信模式": read the token, write it to
 * the buffer, quantise in-kernel when FP8 is on).  Every pair with a row gets a
 * copy of its token.
 * x          device bf16 [T][H] (16-byte aligned).
 * fp8 == 0:  recv_x device bf16 [recv_rows][H]; recv_scale unused (may be NULL).
 * fp8 != 0:  recv_x device e4m3 [recv_rows][H]; recv_scale device fp32
 *            [recv_rows][H/128]: per block of 128 elements of one token,
 *            scale = amax / 448 (1 when amax == 0) and q = e4m3(x / scale),
 *            IEEE fp32 division, round to nearest even, saturating
 *            ("高吞吐模式": FP8 with one scale per 128 elements).
 * recv_src   device int32 [recv_rows] or NULL: source token of each written row.
 * recv_cnt   device int32 [E] or NULL: per-expert receive counts
 *            ("Tensor Layouts": _RECV_EXPERT_COUNTER_DEVICE).
 * recv_rows  rows the receive buffers hold: at least T * k (HT; or the total of
 *            the last moe_ep_get_num_recv_tokens) or E * S (LL).  Rows not
 *            named by the layout are left untouched (LL's unused slots are
 *            never cleared).
 * Errors: MOE_EP_ERR_INVALID for misaligned pointers, H % 128 != 0 with fp8,
 * recv_rows too small, or no preceding moe_ep_route on the handle. */
MOE_EP_API int moe_ep_dispatch(moe_ep_handle_t h, const void* x, int fp8, void* recv_x, float* recv_scale,
                    int32_t* recv_src, int32_t* recv_cnt, int64_t recv_rows,
                    moe_ep_stream_t stream);

/* Combine ("核心功能函数": ncclEpCombine gathers the tokens back and reduces them
 * to the original order using the handle's routing state; "高吞吐模式": the
 * result is the BF16 weighted sum of the expert outputs).
 * out[t][h] = bf16_rn( sum over j = 0..k-1 with a row of w[t][j] * y[row(t,j)][h] ),
 * an fp32 fused multiply-add chain in j order, rounded once to nearest even.
 * y       device bf16 in the receive layout [recv_rows][H] (16-byte aligned).
 * topk_w  device fp32 [T][k].
 * out     device bf16 [T][H] (16-byte aligned); must not overlap y.
 * Errors as for dispatch. */
MOE_EP_API int moe_ep_combine(moe_ep_handle_t h, const void* y, const float* topk_w, void* out,
                   int64_t recv_rows, moe_ep_stream_t stream);

/* Staged execution ("NCCL EP 论文解读", items "核心功能函数" and "send_only与双
 * buffer": with send_only a dispatch or combine only starts its transfer and
 * returns, ncclEpComplete later finishes the receive, and two micro-batches on
 * two handles -- double buffers -- overlap one's transfer with the other's
 * expert computation; "低延迟模式" on the DeepEP page: the LL hook).
 * moe_ep_dispatch_send / moe_ep_combine_send: the same work as moe_ep_dispatch
 * / moe_ep_combine, enqueued on `send_stream`; the send kernel's last CTA, once
 * every CTA's stores are done, adds 1 to the handle's device signal word
 * ("设备API GIN": SignalAdd), and the handle records an event after it.  A
 * handle's sends run in issue order (each waits, on the device, for the
 * previous one).  moe_ep_complete: the receive -- makes `stream` wait (on the
 * device, no host synchronisation) for the handle's last send, then enqueues a
 * one-thread kernel that checks the signal word holds the number of sends
 * since the last complete and takes that number off it ("WaitOnSignal"), so
 * the word is ready for the next micro-batch, also across CUDA-graph replays.
 * Because of the event join the check's first poll succeeds in correct use;
 * its wait is bounded (200 ms): if the signal is short it latches
 * MOE_EP_DEVERR_TIMEOUT and the group's next call returns MOE_EP_ERR_TIMEOUT.
 * A no-op if the handle has no send since its last complete.  With LL mode
 * (no host synchronisation anywhere) route, sends, completes and combines can
 * be captured into a CUDA graph (capture the sends and their complete in the
 * same graph). */
MOE_EP_API int moe_ep_dispatch_send(moe_ep_handle_t h, const void* x, int fp8, void* recv_x,
                                    float* recv_scale, int32_t* recv_src, int32_t* recv_cnt,
                                    int64_t recv_rows, moe_ep_stream_t send_stream);
MOE_EP_API int moe_ep_combine_send(moe_ep_handle_t h, const void* y, const float* topk_w,
                                   void* out, int64_t recv_rows, moe_ep_stream_t send_stream);
MOE_EP_API int moe_ep_complete(moe_ep_handle_t h, moe_ep_stream_t stream);

/* Device signal words ("NCCL EP 论文解读", item "设备API GIN": SignalAdd adds to a
 * signal word, WaitOnSignal waits until it reaches an expected value) -- the
 * primitives under moe_ep_complete, for a caller's own producers and consumers.
 * signal: device uint32 (4-byte aligned), owned by the caller, starting at 0.
 * moe_ep_signal_add: after the work before it on `stream`, *signal += value
 * with release semantics at GPU scope (one thread of a one-CTA kernel).
 * moe_ep_wait_signal: a one-thread kernel on `stream` polls *signal (acquire)
 * until it is >= expected, then subtracts expected; if timeout_ns (1 .. 10^10)
 * pass first, it latches MOE_EP_DEVERR_TIMEOUT in g's device-error word,
 * leaves *signal alone and returns, and g's next call returns
 * MOE_EP_ERR_TIMEOUT.  The producers of the signal must be ordered before the
 * wait on the GPU (the same stream, or an event the stream waits for): the
 * wait checks that their signals arrived, it does not stand in for that
 * ordering -- one GPU never guarantees that a kernel still queued elsewhere
 * runs while another waits for it.  Errors: MOE_EP_ERR_INVALID for a null or
 * misaligned signal or a limit outside the range. */
MOE_EP_API int moe_ep_signal_add(moe_ep_group_t g, uint32_t* signal, uint32_t value,
                                 moe_ep_stream_t stream);
MOE_EP_API int moe_ep_wait_signal(moe_ep_group_t g, uint32_t* signal, uint32_t expected,
                                  int64_t timeout_ns, moe_ep_stream_t stream);

/* Pad every HT expert block of the receive layout to a multiple of `align`
 * rows (a power of two, 1..1024; 1 = dense, the default) for the routes that
 * follow: expert e's rows become off[e] .. off[e] + cnt[e] with off[e] a
 * multiple of align, so a grouped GEMM takes whole row tiles per expert
 * ("NCCL EP 论文解读", "Tensor Layouts": the expert-major layout feeds the GEMM
 * directly).  Padding rows are never written.  The receive-count query then
 * returns total = off[E] (the rows to allocate) and the actual per-rank and
 * per-expert counts; before a query, dispatch and combine require
 * T * k + E * (align - 1) receive rows.  LL layouts are slot-aligned already:
 * only align = 1 is accepted in LL mode.  Host only, no synchronisation. */
MOE_EP_API int moe_ep_set_row_align(moe_ep_handle_t h, int align);

/* Declare (on = 1) that for every dispatch on this handle the tokens x were
 * complete before the moe_ep_route that made the handle's layout was
 * enqueued, on the same stream -- as in an MoE layer, where x is the input of
 * the gate that produces the scores.  A bf16 dispatch (moe_ep_dispatch,
 * moe_ep_dispatch_send, moe_ep_dispatch_dedup) then reads each CTA's first
 * token while the router is still finishing the layout, instead of after it
 * (FP8 dispatch is unaffected).  Results are the same either way; with on = 1
 * and an x written after the route was enqueued (for instance by a kernel
 * launched between the route and the dispatch) the dispatch may read stale
 * tokens.  Default 0.
 * Host only, no synchronisation. */
MOE_EP_API int moe_ep_set_x_before_route(moe_ep_handle_t h, int on);

/* Receive-side dequantisation of an FP8 dispatch: for every row the last
 * route's layout defines (HT: expert blocks without their padding; LL: slots
 * below each expert's count), y[row] = bf16_rn(float(q[row]) * scale), the
 * product in fp32, one scale per 128 elements -- the bf16 expert-major input
 * of an expert GEMM.  Rows the layout does not define are left untouched.
 * recv_q device e4m3 [recv_rows][H] (16-byte aligned), recv_scale device fp32
 * [recv_rows][H/128], y device bf16 [recv_rows][H] (16-byte aligned, may not
 * overlap recv_q).  No host synchronisation: the rows are enumerated on the
 * device from the counts.  Errors: MOE_EP_ERR_INVALID for H % 128 != 0,
 * misaligned pointers, too few rows, or no preceding moe_ep_route.  Large
 * batches stage rows in shared memory with bulk copies whose waits are
 * bounded: a wait that gives up latches MOE_EP_DEVERR_TIMEOUT (the rows of
 * that CTA are then incomplete), reported by the group's next call. */
MOE_EP_API int moe_ep_dequant(moe_ep_handle_t h, const void* recv_q, const float* recv_scale,
                              void* y, int64_t recv_rows, moe_ep_stream_t stream);

/* Node-level layout of the last route, for two-hop dispatch ("NVSHMEM 与 DeepEP：
 * GPU 发起的通信", section "高吞吐模式": a token is sent once to every remote node
 * that holds one of its experts -- to the GPU in the same position -- which
 * forwards it over NVLink to the GPUs holding the experts).  The R ranks form
 * num_nodes nodes of R / num_nodes GPUs (contiguous), GPU g of node n being
 * rank n * (R / num_nodes) + g.
 * node_cnt  device int32 [N]: tokens touching node n.
 * node_off  device int32 [N+1]: exclusive prefix of node_cnt.
 * node_src  device int32 [node_rows]: token of each node row; rows are
 *           node-major with tokens ascending.
 * node_mask device uint32 [node_rows]: bit g set when GPU g of the row's node
 *           holds one of the token's experts (the forwarding set).
 * node_rows capacity of node_src / node_mask: at least T * min(k, N).
 * stats     device int64 [4] or NULL, overwritten: sums over tokens of (0) nodes
 *           touched, own node included; cross-node copies (1) per expert,
 *           (2) per distinct GPU, (3) per distinct node, src_node being the
 *           source GPU's node -- the quantities of the page's routing simulation.
 * Masked (-1), invalid and repeated expert ids are skipped as in the layout.
 * Errors: MOE_EP_ERR_INVALID for N not dividing R, R / N > 32, src_node
 * outside [0, N), too small node_rows, or no preceding moe_ep_route. */
MOE_EP_API int moe_ep_node_layout(moe_ep_handle_t h, int num_nodes, int src_node,
                                  int32_t* node_cnt, int32_t* node_off, int32_t* node_src,
                                  uint32_t* node_mask, int64_t node_rows, int64_t* stats,
                                  moe_ep_stream_t stream);

/* Per-rank dedup dispatch (HT mode): one copy of a token per destination rank
 * holding at least one of its experts, instead of one per expert -- the
 * page's copies by destination GPU ("NVSHMEM 与 DeepEP：GPU 发起的通信", section
 * "高吞吐模式", routing simulation: "按目标卡去重"), the receive format of DeepEP's
 * normal mode.  Rows are rank-major with tokens ascending; each carries its
 * token and the mask of the rank's local experts it must reach.
 * x           device bf16 [T][H] (16-byte aligned), as moe_ep_dispatch.
 * fp8         0: drecv_x bf16 [drecv_rows][H]; 1: drecv_x e4m3 [drecv_rows][H]
 *             with drecv_scale fp32 [drecv_rows][H/128] (the same per-128
 *             quantisation as moe_ep_dispatch).
 * drecv_src   device int32 [drecv_rows]: token of each dedup row (or NULL).
 * drecv_mask  device uint32 [drecv_rows]: bit l set when local expert l of the
 *             row's rank (expert r * E/R + l) is one of the token's experts
 *             (or NULL).
 * rank_cnt    device int32 [R] (or NULL): dedup rows per rank.
 * rank_off    device int32 [R+1] (or NULL): exclusive prefix; rank_off[R] is
 *             the number of dedup rows.
 * drecv_rows  capacity: at least T * min(k, R).
 * The handle keeps the rank layout and the dedup row of every (token, pair)
 * for moe_ep_expand and moe_ep_combine_dedup; the next moe_ep_route clears it.
 * Masked (-1), invalid and repeated expert ids are skipped as in the layout.
 * Errors: MOE_EP_ERR_INVALID in LL mode, for E/R > 32, too small drecv_rows,
 * misaligned pointers, or no preceding moe_ep_route. */
MOE_EP_API int moe_ep_dispatch_dedup(moe_ep_handle_t h, const void* x, int fp8, void* drecv_x,
                                     float* drecv_scale, int32_t* drecv_src,
                                     uint32_t* drecv_mask, int32_t* rank_cnt, int32_t* rank_off,
                                     int64_t drecv_rows, moe_ep_stream_t stream);

/* Receiver side of the dedup dispatch: every dedup row is copied, bytes as
 * they are (bf16, or e4m3 with its scales), to the expert-major HT receive
 * row of each local expert in its mask -- the rows moe_ep_dispatch writes, so
 * recv_x / recv_scale / recv_src equal the direct dispatch's output bit for
 * bit.  Inputs are the outputs of the last moe_ep_dispatch_dedup on this
 * handle (drecv_x, drecv_scale when fp8, drecv_src, drecv_mask); recv_x etc.
 * as moe_ep_dispatch (recv_src may be NULL), recv_rows at least what
 * moe_ep_dispatch requires.  No host synchronisation: the number of dedup
 * rows is read on the device.  Errors: MOE_EP_ERR_INVALID without a
 * preceding moe_ep_dispatch_dedup for the current route, for misaligned or
 * missing buffers, or too few rows. */
MOE_EP_API int moe_ep_expand(moe_ep_handle_t h, const void* drecv_x, const float* drecv_scale,
                             const int32_t* drecv_src, const uint32_t* drecv_mask, int fp8,
                             void* recv_x, float* recv_scale, int32_t* recv_src,
                             int64_t recv_rows, moe_ep_stream_t stream);

/* Combine over the dedup rows, in two stages ("NVSHMEM 与 DeepEP", "高吞吐模式":
 * combine sends back BF16 weighted sums of the expert outputs).  Receiver
 * side: each dedup row (token t, rank r) gets
 *   partial = bf16_rn( fma chain in j order over t's valid pairs j on rank r
 *                      of topk_w[t][j] * y[row(t, j)] )   (fp32);
 * source side: out[t] = bf16_rn( sum of t's partial rows, fp32, in the order of
 * the pairs that carry them ).
 * y       device bf16 [recv_rows][H] in the expert-major HT layout (16-byte
 *         aligned), as moe_ep_combine.
 * topk_w  device fp32 [T][k].
 * drecv_src the dedup rows' tokens from moe_ep_dispatch_dedup.
 * partial device bf16 [drecv_rows][H] (16-byte aligned), written: the rows the
 *         ranks send back.
 * out     device bf16 [T][H] (16-byte aligned).  partial, y and out must not
 *         overlap.
 * Errors: MOE_EP_ERR_INVALID without a preceding moe_ep_dispatch_dedup for the
 * current route, for misaligned, missing or overlapping buffers, or too few
 * rows. */
MOE_EP_API int moe_ep_combine_dedup(moe_ep_handle_t h, const void* y, const float* topk_w,
                                    const int32_t* drecv_src, void* partial, void* out,
                                    int64_t recv_rows, int64_t drecv_rows,
                                    moe_ep_stream_t stream);

/* Copy the handle's layout to caller buffers (device or host pointers; NULL
 * skips an item): cnt [E], off [E+1], rcnt [R], roff [R+1], row [T][k] with -1
 * for pairs without a row.  Asynchronous for device destinations; host
 * destinations must be pinned for the copy to be asynchronous. */
MOE_EP_API int moe_ep_copy_layout(moe_ep_handle_t h, int32_t* cnt, int32_t* off, int32_t* rcnt,
                       int32_t* roff, int32_t* row, moe_ep_stream_t stream);

/* Routing + layout that allocates nothing, for callers that cannot allocate
 * device memory themselves or through the library: a host whose memory pool or
 * fixed memory plan owns every device byte and hands the library only
 * pre-placed buffers.  (The source pages have no counterpart: there every
 * rank allocates its communication buffers at group creation.)
 * Computes what moe_ep_route followed by moe_ep_copy_layout computes on a
 * handle of the same mode, experts, ranks and slots, with the same options
 * and the default row alignment of 1 (dense HT expert blocks; there is no
 * alignment argument):
 * topk_idx [T][k], topk_w [T][k] (may be NULL), row [T][k], cnt [E],
 * off [E+1], rcnt [R], roff [R+1], all device buffers owned by the caller.
 * The layout's scratch lives in one static device array of 346.25 KiB that every
 * GPU loading the library holds until exit; it is never allocated or freed.
 * Capacity: ceil(num_tokens / 32) * experts <= 65536 (e.g. 8192 tokens with
 * 256 experts); larger sizes return MOE_EP_ERR_OVERFLOW without launching.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and keeps it for the life of the
 * process; make that first call before any stream capture, and do not call
 * this entry point again after cudaDeviceReset (or any teardown of the
 * device's primary context): the kept address would be stale.  Every call
 * shares the array: calls whose work overlaps on the GPU (different streams
 * without ordering) race; calls on one stream do not.
 * mode: MOE_EP_LL or MOE_EP_HT; slots: S for LL (>= num_tokens), ignored for HT.
 * Asynchronous on `stream`. */
MOE_EP_API int moe_ep_route_layout_static(const float* scores, int num_tokens, int experts,
                                          int ranks, int mode, int slots,
                                          const moe_ep_route_opts_t* opts, int32_t* topk_idx,
                                          float* topk_w, int32_t* row, int32_t* cnt, int32_t* off,
                                          int32_t* rcnt, int32_t* roff, moe_ep_stream_t stream);

/* Read (host, no synchronisation) / clear the group's device-error word. */
MOE_EP_API int moe_ep_get_device_errors(moe_ep_group_t g, uint32_t* bits);
MOE_EP_API int moe_ep_clear_device_errors(moe_ep_group_t g);

/* Static description of a status code. */
MOE_EP_API const char* moe_ep_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif
