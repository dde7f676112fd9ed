/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for MoE expert-parallel
 * routing, layout, dispatch (optionally FP8) and combine.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg, never by the product library.
 * It shares no code with the CUDA path.  Build: gcc -O2 -ffp-contract=off
 * (no fast-math), so every fp32 / binary64 operation below is one IEEE
 * operation, rounded to nearest.
 *
 * Sources (see moe_oracle.h for the full list):
 *  - "NVSHMEM 与 DeepEP：GPU 发起的通信", section "高吞吐模式": node-limited routing
 *    (keep 4 nodes by the sum of each node's two best expert scores, then pick 8
 *    experts among them), contiguous expert -> GPU -> node placement, FP8
 *    dispatch with one fp32 scale per 128 elements, BF16 combine of the
 *    weighted sum of expert outputs.
 *  - same page, section "低延迟模式": fixed slots per (local expert, source).
 *  - "NCCL EP 论文解读", items "算法模式" and "Tensor Layouts": HT 2D output
 *    [total_recv_tokens x hidden] in deterministic order with per-expert counts,
 *    LL 3D expert-major output; "核心功能函数": combine un-permutes with the
 *    routing state of the handle and reduces back to token order.
 *
 * parity pins: every function here is pinned by tests under tests/ (page
 * statistics, brute force, closed forms, hand-worked FP8 cases).
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* bf16                                                                       */
/* ------------------------------------------------------------------------- */

static float bits_to_float(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t float_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

double orc_bf16_to_double(uint16_t b) { return (double)bits_to_float((uint32_t)b << 16); }

static float bf16_to_float(uint16_t b) { return bits_to_float((uint32_t)b << 16); }

/* Round a binary64 value to the nearest bf16 (8 significant bits, exponent
 * range of fp32, subnormal spacing 2^-133), ties to even, in one step. */
uint16_t orc_bf16_from_double(double v)
{
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                /* spacing of bf16 values near a */
    if (q < -133) q = -133;       /* subnormal range */
    double n = ldexp(a, -q);      /* exact: a / 2^q */
    double fl = floor(n);
    double rem = n - fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    double r = ldexp(fl, q);
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;   /* overflow -> inf */
    uint32_t u = float_to_bits((float)r);             /* exact */
    return sign | (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------- */
/* e4m3fn                                                                     */
/* ------------------------------------------------------------------------- */

double orc_e4m3_to_double(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9)          /* m/8 * 2^-6 */
                        : ldexp((double)(8 + m), e - 10); /* (1+m/8) * 2^(e-7) */
    return s ? -v : v;
}

uint8_t orc_e4m3_from_float(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0;
    if (isnan(v)) return sign | 0x7F;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;   /* saturate to the largest finite value */
    /* Largest non-negative code whose value is <= a (codes 0..0x7E are
     * ordered by value). */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (orc_e4m3_to_double((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
    }
    double below = orc_e4m3_to_double((uint8_t)lo);
    double above = orc_e4m3_to_double((uint8_t)(lo + 1));  /* lo + 1 <= 0x7E */
    double dl = a - below, du = above - a;                 /* both exact */
    int c;
    if (dl < du) c = lo;
    else if (du < dl) c = lo + 1;
    else c = (lo & 1) ? lo + 1 : lo;                       /* tie: even code */
    return sign | (uint8_t)c;
}

void orc_e4m3_from_float_array(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_from_float(v[i]);
}

int orc_quant_row(const uint16_t* x, int H, uint8_t* q, float* scale)
{
    if (H <= 0 || H % 128 != 0) return ORC_ERR_INVALID;
    for (int b = 0; b < H / 128; ++b) {
        const uint16_t* xb = x + (int64_t)b * 128;
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float a = fabsf(bf16_to_float(xb[i]));
            if (a > amax) amax = a;
        }
        float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;   /* fp32 division */
        scale[b] = s;
        for (int i = 0; i < 128; ++i) {
            float r = bf16_to_float(xb[i]) / s;            /* fp32 division */
            q[(int64_t)b * 128 + i] = orc_e4m3_from_float(r);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* routing                                                                    */
/* ------------------------------------------------------------------------- */

/* v + lo is the exact value (lo = 0 unless a node score needs it) */
typedef struct { double v; double lo; int i; } scored;

/* (value descending, index ascending) */
static int by_value_desc(const void* pa, const void* pb)
{
    const scored* a = (const scored*)pa;
    const scored* b = (const scored*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

/* (exact value ascending, index descending): the first entries are the ones
 * to ban.  (v, lo) pairs with lo the rounding error of v order like v + lo. */
static int by_value_asc_index_desc(const void* pa, const void* pb)
{
    const scored* a = (const scored*)pa;
    const scored* b = (const scored*)pb;
    if (a->v < b->v) return -1;
    if (a->v > b->v) return 1;
    if (a->lo < b->lo) return -1;
    if (a->lo > b->lo) return 1;
    return (a->i < b->i) - (a->i > b->i);
}

static int double_asc(const void* pa, const void* pb)
{
    double a = *(const double*)pa, b = *(const double*)pb;
    return (a > b) - (a < b);
}

int orc_route(const float* scores, int64_t T, int E, int G, int kg, int m, int k,
              int weight_mode, int32_t* topk_idx, double* topk_w)
{
    if (T < 0 || E <= 0 || G <= 0 || E % G != 0 || kg < 1 || kg > G || k < 1 || k > E)
        return ORC_ERR_INVALID;
    const int gs = E / G;
    const int limit = (G > 1 && kg < G);
    if ((int64_t)kg * gs < k) return ORC_ERR_INVALID;
    if (limit && (m < 1 || m > gs)) return ORC_ERR_INVALID;
    if (weight_mode < ORC_W_SOFTMAX_TOPK || weight_mode > ORC_W_SCORE_NORM) return ORC_ERR_INVALID;

    char* allowed = (char*)malloc((size_t)E);
    double* tmp = (double*)malloc(sizeof(double) * (size_t)gs);
    scored* nodes = (scored*)malloc(sizeof(scored) * (size_t)G);
    scored* cand = (scored*)malloc(sizeof(scored) * (size_t)E);
    float* sv = (float*)malloc(sizeof(float) * (size_t)E);

    for (int64_t t = 0; t < T; ++t) {
        const float* s_in = scores + t * E;
        for (int e = 0; e < E; ++e) {
            allowed[e] = 1;
            sv[e] = isnan(s_in[e]) ? -INFINITY : s_in[e];   /* NaN ranks as -infinity */
            if (sv[e] == 0.0f) sv[e] = 0.0f;                 /* -0 is the score 0 */
        }
        const float* s = sv;

        /* Step 1 (node limit): score every node by the sum of its m best
         * expert scores, then ban the G - kg lowest-scoring nodes. */
        if (limit) {
            for (int n = 0; n < G; ++n) {
                for (int i = 0; i < gs; ++i) tmp[i] = (double)s[n * gs + i];
                qsort(tmp, (size_t)gs, sizeof(double), double_asc);
                /* node score: the exact sum of the node's m best scores */
                double sum = 0.0, lo = 0.0;
                if (m <= 2) {
                    /* two fp32 values: hi + lo = exact sum (Knuth's two-sum) */
                    double a = tmp[gs - 1], b = (m == 2) ? tmp[gs - 2] : 0.0;
                    sum = b + a;
                    if (isfinite(sum)) {
                        double bb = sum - a;
                        lo = (a - (sum - bb)) + (b - bb);
                    }
                } else {
                    for (int i = gs - m; i < gs; ++i) sum += tmp[i];   /* ascending order */
                }
                if (isnan(sum)) { sum = -INFINITY; lo = 0.0; }      /* inf + -inf ranks lowest */
                nodes[n].v = sum;
                nodes[n].lo = (lo == 0.0) ? 0.0 : lo;
                nodes[n].i = n;
            }
            qsort(nodes, (size_t)G, sizeof(scored), by_value_asc_index_desc);
            for (int b = 0; b < G - kg; ++b) {
                int n = nodes[b].i;
                for (int i = 0; i < gs; ++i) allowed[n * gs + i] = 0;
            }
        }

        /* Step 2: the k best allowed experts, best first. */
        int nc = 0;
        for (int e = 0; e < E; ++e)
            if (allowed[e]) { cand[nc].v = (double)s[e]; cand[nc].lo = 0.0; cand[nc].i = e; ++nc; }
        qsort(cand, (size_t)nc, sizeof(scored), by_value_desc);
        for (int j = 0; j < k; ++j) topk_idx[t * k + j] = cand[j].i;

        /* Step 3: gate weights.  Score-normalised: the selected scores are
         * fp32 values; their sum is taken in fp32, one rounding per addition,
         * in j order (best first), and each weight is one fp32 division -- a
         * definition with a single correctly rounded answer.  The softmax
         * rules go through exp and are computed in binary64. */
        double* w = topk_w + t * k;
        if (weight_mode == ORC_W_SCORE_NORM) {
            float den = 0.0f;
            for (int j = 0; j < k; ++j) den = den + (float)cand[j].v;
            for (int j = 0; j < k; ++j) w[j] = (double)((float)cand[j].v / den);
        } else if (weight_mode == ORC_W_SOFTMAX_TOPK) {
            double mx = cand[0].v, den = 0.0;
            for (int j = 0; j < k; ++j) den += exp(cand[j].v - mx);
            for (int j = 0; j < k; ++j) w[j] = exp(cand[j].v - mx) / den;
        } else {
            double mx = (double)s[0];
            for (int e = 1; e < E; ++e) if ((double)s[e] > mx) mx = (double)s[e];
            double z = 0.0;
            for (int e = 0; e < E; ++e) z += exp((double)s[e] - mx);
            double sel = 0.0;
            for (int j = 0; j < k; ++j) { w[j] = exp(cand[j].v - mx) / z; sel += w[j]; }
            for (int j = 0; j < k; ++j) w[j] = w[j] / sel;
        }
    }
    free(allowed); free(tmp); free(nodes); free(cand); free(sv);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* layout                                                                     */
/* ------------------------------------------------------------------------- */

/* 1 = the pair gets a row, 0 = masked (-1), -1 = invalid input */
static int pair_kind(const int32_t* idx_row, int j, int E)
{
    int32_t e = idx_row[j];
    if (e == -1) return 0;
    if (e < -1 || e >= E) return -1;
    for (int jj = 0; jj < j; ++jj)
        if (idx_row[jj] == e) return -1;   /* repeated expert within the token */
    return 1;
}

int orc_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int mode, int S,
               int32_t* cnt, int32_t* off, int32_t* rcnt, int32_t* roff, int32_t* row)
{
    return orc_layout_aligned(topk_idx, T, k, E, R, mode, S, 1, cnt, off, rcnt, roff, row);
}

int orc_layout_aligned(const int32_t* topk_idx, int64_t T, int k, int E, int R, int mode, int S,
                       int align, int32_t* cnt, int32_t* off, int32_t* rcnt, int32_t* roff,
                       int32_t* row)
{
    if (T < 0 || k < 1 || E < 1 || R < 1 || E % R != 0 || align < 1) return ORC_ERR_INVALID;
    if (mode != ORC_MODE_LL && mode != ORC_MODE_HT) return ORC_ERR_INVALID;
    if (mode == ORC_MODE_LL && S < 1) return ORC_ERR_INVALID;
    const int L = E / R;
    int status = ORC_OK;

    /* Pass 1: tokens bound for every expert. */
    for (int e = 0; e < E; ++e) cnt[e] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int kind = pair_kind(topk_idx + t * k, j, E);
            if (kind < 0) status = ORC_ERR_INVALID;
            if (kind == 1) cnt[topk_idx[t * k + j]] += 1;
        }
    off[0] = 0;
    for (int e = 0; e < E; ++e) off[e + 1] = off[e] + (cnt[e] + align - 1) / align * align;
    for (int r = 0; r < R; ++r) {
        rcnt[r] = 0;
        for (int l = 0; l < L; ++l) rcnt[r] += cnt[r * L + l];
    }
    for (int r = 0; r <= R; ++r) roff[r] = off[r * L];

    /* Pass 2: each pair's place, tokens of one expert in ascending order. */
    int32_t* cursor = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int64_t p = t * k + j;
            if (pair_kind(topk_idx + t * k, j, E) != 1) { row[p] = -1; continue; }
            int e = topk_idx[p];
            int rank = cursor[e]++;
            if (mode == ORC_MODE_HT) {
                row[p] = off[e] + rank;
            } else if (rank < S) {
                row[p] = e * S + rank;
            } else {
                row[p] = -1;
                status = ORC_ERR_OVERFLOW;
            }
        }
    free(cursor);
    return status;
}

/* ------------------------------------------------------------------------- */
/* dequantisation                                                             */
/* ------------------------------------------------------------------------- */

int orc_dequant_rows(const uint8_t* q, const float* scale, int64_t nrows, int H,
                     const int64_t* rows, int64_t nlist, uint16_t* y)
{
    if (H <= 0 || H % 128 != 0) return ORC_ERR_INVALID;
    const int nb = H / 128;
    for (int64_t i = 0; i < nlist; ++i) {
        const int64_t r = rows[i];
        if (r < 0 || r >= nrows) return ORC_ERR_INVALID;
        for (int h = 0; h < H; ++h) {
            const float v = (float)orc_e4m3_to_double(q[r * H + h]);   /* exact */
            const float p = v * scale[r * nb + h / 128];                /* fp32 product */
            y[r * H + h] = orc_bf16_from_double((double)p);             /* one bf16 rounding */
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* node-level (two-hop) layout                                                */
/* ------------------------------------------------------------------------- */

int orc_node_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int N, int src_node,
                    int32_t* node_cnt, int32_t* node_off, int32_t* node_src, uint32_t* node_mask,
                    int64_t* stats)
{
    if (T < 0 || k < 1 || E < 1 || R < 1 || E % R != 0 || N < 1 || R % N != 0 || N > 64 ||
        R / N > 32 || src_node < 0 || src_node >= N)
        return ORC_ERR_INVALID;
    const int L = E / R, GPN = R / N;
    uint32_t* mask = (uint32_t*)calloc((size_t)N, sizeof(uint32_t));
    for (int n = 0; n < N; ++n) node_cnt[n] = 0;
    for (int q = 0; q < 4; ++q) stats[q] = 0;
    /* pass 1: per token, the GPUs it needs on every node; counts and statistics */
    for (int64_t t = 0; t < T; ++t) {
        for (int n = 0; n < N; ++n) mask[n] = 0;
        for (int j = 0; j < k; ++j) {
            if (pair_kind(topk_idx + t * k, j, E) != 1) continue;
            int e = topk_idx[t * k + j];
            int gpu = e / L, n = gpu / GPN;
            mask[n] |= 1u << (gpu % GPN);
            if (n != src_node) stats[1] += 1;                 /* per expert */
        }
        for (int n = 0; n < N; ++n) {
            if (!mask[n]) continue;
            node_cnt[n] += 1;
            stats[0] += 1;                                     /* nodes touched */
            if (n != src_node) {
                stats[3] += 1;                                 /* per node */
                for (int g = 0; g < GPN; ++g) stats[2] += (mask[n] >> g) & 1u;   /* per GPU */
            }
        }
    }
    node_off[0] = 0;
    for (int n = 0; n < N; ++n) node_off[n + 1] = node_off[n] + node_cnt[n];
    /* pass 2: rows, node-major, tokens ascending */
    int32_t* cursor = (int32_t*)calloc((size_t)N, sizeof(int32_t));
    for (int64_t t = 0; t < T; ++t) {
        for (int n = 0; n < N; ++n) mask[n] = 0;
        for (int j = 0; j < k; ++j) {
            if (pair_kind(topk_idx + t * k, j, E) != 1) continue;
            int gpu = topk_idx[t * k + j] / L;
            mask[gpu / GPN] |= 1u << (gpu % GPN);
        }
        for (int n = 0; n < N; ++n) {
            if (!mask[n]) continue;
            int r = node_off[n] + cursor[n]++;
            node_src[r] = (int32_t)t;
            node_mask[r] = mask[n];
        }
    }
    free(cursor);
    free(mask);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* dispatch                                                                   */
/* ------------------------------------------------------------------------- */

int orc_dispatch(const uint16_t* x, int64_t T, int H, int k, const int32_t* row, int64_t nrows,
                 int fp8, void* recv_x, float* recv_scale, int32_t* recv_src)
{
    if (T < 0 || H <= 0 || k < 1) return ORC_ERR_INVALID;
    if (fp8 && H % 128 != 0) return ORC_ERR_INVALID;
    const int nb = H / 128;
    uint8_t* q = fp8 ? (uint8_t*)malloc((size_t)H) : NULL;
    float* sc = fp8 ? (float*)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1)) : NULL;
    int status = ORC_OK;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* xt = x + t * H;
        if (fp8) orc_quant_row(xt, H, q, sc);
        for (int j = 0; j < k; ++j) {
            int64_t r = row[t * k + j];
            if (r < 0) continue;
            if (r >= nrows) { status = ORC_ERR_INVALID; continue; }
            if (fp8) {
                memcpy((uint8_t*)recv_x + r * H, q, (size_t)H);
                memcpy(recv_scale + r * nb, sc, sizeof(float) * (size_t)nb);
            } else {
                memcpy((uint16_t*)recv_x + r * H, xt, sizeof(uint16_t) * (size_t)H);
            }
            recv_src[r] = (int32_t)t;
        }
    }
    free(q); free(sc);
    return status;
}

/* ------------------------------------------------------------------------- */
/* combine                                                                    */
/* ------------------------------------------------------------------------- */

int orc_combine(const uint16_t* y, int64_t nrows, int H, const int32_t* row, const float* w,
                int64_t T, int k, const int64_t* tokens, int64_t ntok, uint16_t* out)
{
    if (T < 0 || H <= 0 || k < 1) return ORC_ERR_INVALID;
    int64_t n = tokens ? ntok : T;
    int status = ORC_OK;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) { status = ORC_ERR_INVALID; continue; }
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t r = row[t * k + j];
                if (r < 0) continue;
                if (r >= nrows) { status = ORC_ERR_INVALID; continue; }
                acc += (double)w[t * k + j] * orc_bf16_to_double(y[r * H + h]);
            }
            out[i * H + h] = orc_bf16_from_double(acc);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------- */
/* per-rank dedup layout, expansion and two-stage combine                     */
/* ------------------------------------------------------------------------- */

int orc_rank_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int32_t* rank_cnt,
                    int32_t* rank_off, int32_t* drow, int32_t* dsrc, uint32_t* dmask)
{
    if (T < 0 || k < 1 || E < 1 || R < 1 || E % R != 0 || E / R > 32) return ORC_ERR_INVALID;
    const int L = E / R;
    int status = ORC_OK;
    uint32_t* m = (uint32_t*)calloc((size_t)R, sizeof(uint32_t));
    for (int r = 0; r < R; ++r) rank_cnt[r] = 0;
    /* pass 1: ranks each token needs */
    for (int64_t t = 0; t < T; ++t) {
        for (int r = 0; r < R; ++r) m[r] = 0;
        for (int j = 0; j < k; ++j) {
            int kind = pair_kind(topk_idx + t * k, j, E);
            if (kind < 0) status = ORC_ERR_INVALID;
            if (kind != 1) continue;
            int e = topk_idx[t * k + j];
            m[e / L] |= 1u << (e % L);
        }
        for (int r = 0; r < R; ++r)
            if (m[r]) rank_cnt[r] += 1;
    }
    rank_off[0] = 0;
    for (int r = 0; r < R; ++r) rank_off[r + 1] = rank_off[r] + rank_cnt[r];
    /* pass 2: rows rank-major, tokens ascending; the pair map names each
     * token's row on a rank at the first valid pair on that rank */
    int32_t* cursor = (int32_t*)calloc((size_t)R, sizeof(int32_t));
    for (int64_t t = 0; t < T; ++t) {
        for (int r = 0; r < R; ++r) m[r] = 0;
        for (int j = 0; j < k; ++j) {
            if (pair_kind(topk_idx + t * k, j, E) != 1) continue;
            int e = topk_idx[t * k + j];
            m[e / L] |= 1u << (e % L);
        }
        for (int j = 0; j < k; ++j) drow[t * k + j] = -1;
        for (int j = 0; j < k; ++j) {
            if (pair_kind(topk_idx + t * k, j, E) != 1) continue;
            int r = topk_idx[t * k + j] / L;
            int first = 1;
            for (int jj = 0; jj < j; ++jj)
                if (pair_kind(topk_idx + t * k, jj, E) == 1 && topk_idx[t * k + jj] / L == r)
                    first = 0;
            if (!first) continue;
            int q = rank_off[r] + cursor[r]++;
            drow[t * k + j] = q;
            dsrc[q] = (int32_t)t;
            dmask[q] = m[r];
        }
    }
    free(cursor);
    free(m);
    return status;
}

int orc_expand(const uint8_t* dx, const float* dscale, int64_t nd, int64_t row_bytes, int nscale,
               const int32_t* dsrc, const uint32_t* dmask, const int32_t* rank_off, int R, int E,
               const int32_t* topk_idx, const int32_t* row, int64_t T, int k, int64_t nrows,
               uint8_t* recv_x, float* recv_scale, int32_t* recv_src)
{
    if (R < 1 || E % R != 0 || E / R > 32 || row_bytes < 1 || rank_off[R] > nd)
        return ORC_ERR_INVALID;
    const int L = E / R;
    for (int r = 0; r < R; ++r)
        for (int64_t q = rank_off[r]; q < rank_off[r + 1]; ++q) {
            const int64_t t = dsrc[q];
            if (t < 0 || t >= T) return ORC_ERR_INVALID;
            for (int l = 0; l < L; ++l) {
                if (!((dmask[q] >> l) & 1u)) continue;
                const int e = r * L + l;
                int64_t er = -1;
                for (int j = 0; j < k && er < 0; ++j)
                    if (pair_kind(topk_idx + t * k, j, E) == 1 && topk_idx[t * k + j] == e)
                        er = row[t * k + j];
                if (er < 0 || er >= nrows) return ORC_ERR_INVALID;
                memcpy(recv_x + er * row_bytes, dx + q * row_bytes, (size_t)row_bytes);
                if (dscale)
                    memcpy(recv_scale + er * nscale, dscale + q * nscale, sizeof(float) * (size_t)nscale);
                recv_src[er] = (int32_t)t;
            }
        }
    return ORC_OK;
}

int orc_combine_dedup(const uint16_t* y, int64_t nrows, int H, const int32_t* topk_idx,
                      const int32_t* row, const float* w, int64_t T, int k, int E, int R,
                      const int32_t* drow, int64_t nd, const int64_t* tokens, int64_t ntok,
                      uint16_t* partial, uint16_t* out)
{
    if (T < 0 || H <= 0 || k < 1 || R < 1 || E % R != 0) return ORC_ERR_INVALID;
    const int L = E / R;
    const int64_t n = tokens ? ntok : T;
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    int status = ORC_OK;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) { status = ORC_ERR_INVALID; continue; }
        for (int h = 0; h < H; ++h) acc[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            const int64_t q = drow[t * k + j];
            if (q < 0) continue;              /* not the first pair of its rank */
            if (q >= nd) { status = ORC_ERR_INVALID; continue; }
            const int r = topk_idx[t * k + j] / L;
            for (int h = 0; h < H; ++h) {
                /* stage 1: this rank's weighted sum, rounded to bf16 once */
                double p = 0.0;
                for (int jj = 0; jj < k; ++jj) {
                    if (pair_kind(topk_idx + t * k, jj, E) != 1) continue;
                    if (topk_idx[t * k + jj] / L != r) continue;
                    const int64_t er = row[t * k + jj];
                    if (er < 0 || er >= nrows) { status = ORC_ERR_INVALID; continue; }
                    p += (double)w[t * k + jj] * orc_bf16_to_double(y[er * H + h]);
                }
                const uint16_t pb = orc_bf16_from_double(p);
                if (partial) partial[q * H + h] = pb;
                /* stage 2: the source adds the ranks' partials */
                acc[h] += orc_bf16_to_double(pb);
            }
        }
        for (int h = 0; h < H; ++h) out[i * H + h] = orc_bf16_from_double(acc[h]);
    }
    free(acc);
    return status;
}
