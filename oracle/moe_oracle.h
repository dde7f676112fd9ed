/*
 * moe_oracle.h -- plain, slow, single-threaded CPU oracle for MoE expert-parallel
 * dispatch / combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
 * baseline / reference leg of the benchmark may load this library.  The product
 * (libmoeep) shares no code, header, table or constant with it.
 *
 * Every function follows a passage of the source pages:
 *   "NVSHMEM 与 DeepEP：GPU 发起的通信" (anrans.github.io ai-infra-handbooks,
 *       section "高吞吐模式" for node-limited routing, the expert -> GPU -> node
 *       placement and FP8 with one fp32 scale per 128 elements; section
 *       "低延迟模式" for the fixed LL slots),
 *   "NCCL EP 论文解读" (lpnh.cn, items "核心功能函数", "算法模式", "Tensor Layouts"
 *       for the HT 2D / LL 3D expert-major layouts and the combine that
 *       un-permutes and reduces back to token order).
 * Readings of points the pages leave open are stated next to each function.
 *
 * Status codes returned by the functions below.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_ERR_INVALID = 1, ORC_ERR_OVERFLOW = 2 };
enum { ORC_MODE_LL = 0, ORC_MODE_HT = 1 };
enum { ORC_W_SOFTMAX_TOPK = 0, ORC_W_SOFTMAX_RENORM = 1, ORC_W_SCORE_NORM = 2 };

/* bf16 <-> binary64. bf16 -> double is exact; double -> bf16 rounds once,
 * to nearest, ties to even. */
double   orc_bf16_to_double(uint16_t b);
uint16_t orc_bf16_from_double(double v);

/* OCP e4m3fn (bias 7, largest finite 448, no infinity, NaN = S.1111.111). */
double   orc_e4m3_to_double(uint8_t code);
/* Round to nearest, ties to even; finite magnitudes beyond 448 (and infinities)
 * saturate to +-448; NaN -> 0x7F with the sign kept. */
uint8_t  orc_e4m3_from_float(float v);
void     orc_e4m3_from_float_array(const float* v, int64_t n, uint8_t* out);

/* Quantise one token row of H bf16 values (H % 128 == 0): per block of 128,
 * amax = max |x|, scale = amax / 448 (fp32 division; 1 when amax == 0),
 * q = e4m3(x / scale) with fp32 division. */
int orc_quant_row(const uint16_t* x, int H, uint8_t* q, float* scale);

/* Node-limited (grouped) top-k routing, then the gate weights.
 * scores [T][E] fp32; E experts in G contiguous groups (nodes) of E/G.
 * If 1 < G and kg < G: group score = the exact sum of the group's m largest
 * scores (m <= 2: exact, as a binary64 two-sum; m > 2: summed in ascending
 * order in binary64); the G - kg groups with the lowest group score are banned
 * (on equal score the higher index is banned first).
 * The k best allowed experts are taken by (score desc, index asc).
 * A NaN score ranks as -infinity; -0 is the score +0.
 * weight_mode: ORC_W_SOFTMAX_TOPK   softmax over the k selected scores,
 *              ORC_W_SOFTMAX_RENORM softmax over all E, renormalised over the k
 *                                   (both in binary64),
 *              ORC_W_SCORE_NORM     s_j / sum of the k selected s, in fp32: the
 *                                   sum in j order (best first), one rounding
 *                                   per addition, then one division per weight.
 * Outputs topk_idx [T][k] int32 and topk_w [T][k] (binary64 storage; the
 * score-normalised weights are fp32 values). */
int orc_route(const float* scores, int64_t T, int E, int G, int kg, int m, int k,
              int weight_mode, int32_t* topk_idx, double* topk_w);

/* Per-expert counting and prefix layout of the (token, j) pairs.
 * topk_idx [T][k]: -1 = masked (no row); ids outside [-1, E) or an expert
 * repeated within a token are invalid: the pair gets no row and the call
 * returns ORC_ERR_INVALID.
 * Outputs: cnt [E], off [E+1] (exclusive prefix of cnt), rcnt [R] (sum of the
 * L = E/R experts of rank r), roff [R+1], row [T][k]:
 *   HT: row = off[e] + (number of earlier pairs (t', j') < (t, j) with expert e)
 *   LL: row = e * S + that same in-expert rank (slot), slot < S else overflow. */
int orc_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int mode, int S,
               int32_t* cnt, int32_t* off, int32_t* rcnt, int32_t* roff, int32_t* row);

/* The same layout with every HT expert block padded to a multiple of `align`
 * rows (so a grouped GEMM takes whole row tiles per expert; "NCCL EP 论文解读",
 * "Tensor Layouts": the expert-major layout feeds the GEMM directly):
 * off[e+1] = off[e] + roundup(cnt[e], align); rows off[e] + rank; roff[r] =
 * off[r * L]; cnt and rcnt stay the actual counts.  align = 1 is orc_layout. */
int orc_layout_aligned(const int32_t* topk_idx, int64_t T, int k, int E, int R, int mode, int S,
                       int align, int32_t* cnt, int32_t* off, int32_t* rcnt, int32_t* roff,
                       int32_t* row);

/* Dequantise FP8 receive rows to bf16: y = bf16_rn(float(q) * scale), the
 * product rounded to fp32 first (fp32 dequantisation, bf16 storage).
 * q [nrows][H] e4m3, scale [nrows][H/128], y [nrows][H] bf16 bits; only the
 * rows listed in `rows` (nlist entries) are written. */
int orc_dequant_rows(const uint8_t* q, const float* scale, int64_t nrows, int H,
                     const int64_t* rows, int64_t nlist, uint16_t* y);

/* Node-level layout for two-hop dispatch ("NVSHMEM 与 DeepEP：GPU 发起的通信",
 * section "高吞吐模式": a token goes once to every remote node that holds one of
 * its experts, to the GPU in the same position, which forwards it over NVLink
 * to the GPUs that hold the experts).  Experts are placed in contiguous
 * blocks: gpu = e / (E/R), node = gpu / (R/N).
 * Outputs: node_cnt [N] tokens touching node n, node_off [N+1], and per node
 * row (node-major, tokens ascending) node_src = token, node_mask = bit g set
 * when local GPU g of that node holds one of the token's experts.
 * stats [4] (sums over tokens; -1 / invalid ids skipped, repeated experts
 * counted once): distinct nodes touched (own node included), cross-node copies
 * sent per expert, per distinct GPU, per distinct node -- the quantities of the
 * page's routing simulation, with src_node as "own node". */
int orc_node_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int N, int src_node,
                    int32_t* node_cnt, int32_t* node_off, int32_t* node_src, uint32_t* node_mask,
                    int64_t* stats);

/* Dispatch: every (t, j) with row r >= 0 receives token t.
 * fp8 == 0: recv_x is bf16 [nrows][H] and recv_scale is unused.
 * fp8 != 0: recv_x is e4m3 [nrows][H], recv_scale fp32 [nrows][H/128].
 * recv_src [nrows] int32 gets t.  Rows never named by row[] are not touched. */
int orc_dispatch(const uint16_t* x, int64_t T, int H, int k, const int32_t* row, int64_t nrows,
                 int fp8, void* recv_x, float* recv_scale, int32_t* recv_src);

/* Combine: out[t] = bf16_rn( sum_j w[t][j] * y[row[t][j]] ), accumulated in
 * binary64 in j order; masked pairs (row < 0) contribute nothing.
 * tokens == NULL: all T tokens, out is [T][H]; otherwise the ntok listed tokens,
 * out is [ntok][H]. */
int orc_combine(const uint16_t* y, int64_t nrows, int H, const int32_t* row, const float* w,
                int64_t T, int k, const int64_t* tokens, int64_t ntok, uint16_t* out);

/* Per-rank dedup layout (HT): one row per (token, destination rank holding at
 * least one of the token's experts) -- the page's "按目标卡去重" (dedup by
 * destination GPU) in the routing simulation of "NVSHMEM 与 DeepEP：GPU 发起的通信",
 * section "高吞吐模式": a token goes once to every rank that needs it.  Experts in
 * contiguous blocks of L = E/R (rank = e / L), L <= 32.  Rows rank-major,
 * tokens ascending.  Outputs: rank_cnt [R], rank_off [R+1], drow [T][k] = the
 * row of pair (t, j) when j is the first valid pair of t on its rank, else -1;
 * dsrc [rows] = token, dmask [rows] = bit l set when local expert l of the
 * row's rank is one of the token's experts.  Invalid and repeated expert ids
 * are skipped as in orc_layout (status ORC_ERR_INVALID when any is seen). */
int orc_rank_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int32_t* rank_cnt,
                    int32_t* rank_off, int32_t* drow, int32_t* dsrc, uint32_t* dmask);

/* Receiver-side expansion of dedup rows into the expert-major HT layout: every
 * dedup row q of rank r (token t = dsrc[q]) is copied, payload bytes as they
 * are (row_bytes per row; FP8 scales nscale floats per row when dscale is not
 * NULL), to the expert rows of the local experts in dmask[q], ascending:
 * expert e = r*L + l, row = row[t][j] for the pair (t, j) with topk_idx = e.
 * recv_src of every written row gets t. */
int orc_expand(const uint8_t* dx, const float* dscale, int64_t nd, int64_t row_bytes, int nscale,
               const int32_t* dsrc, const uint32_t* dmask, const int32_t* rank_off, int R, int E,
               const int32_t* topk_idx, const int32_t* row, int64_t T, int k, int64_t nrows,
               uint8_t* recv_x, float* recv_scale, int32_t* recv_src);

/* Combine over dedup rows, in two stages.  Stage 1 (receiver side): each
 * dedup row (t, r) gets partial = bf16_rn( sum over the token's valid pairs j
 * on rank r, in j order, of w[t][j] * y[row[t][j]] ) -- the BF16 weighted sum
 * of the rank's expert outputs that combine sends back ("NVSHMEM 与 DeepEP",
 * "高吞吐模式": combine returns BF16 weighted sums).  Stage 2 (source side):
 * out[t] = bf16_rn( exact sum of the token's partials ).  Sums in binary64.
 * tokens / ntok as orc_combine; partial [nd][H] may be NULL. */
int orc_combine_dedup(const uint16_t* y, int64_t nrows, int H, const int32_t* topk_idx,
                      const int32_t* row, const float* w, int64_t T, int k, int E, int R,
                      const int32_t* drow, int64_t nd, const int64_t* tokens, int64_t ntok,
                      uint16_t* partial, uint16_t* out);

#ifdef __cplusplus
}
#endif
#endif
