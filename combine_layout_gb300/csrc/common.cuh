// Internal declarations shared by the libmoeep translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_ep.h"

namespace moeep {

// Layout tiles hold 32 tokens so that one expert's presence in a tile is one
// 32-bit word (bit i = token tile*32 + i chose that expert).
constexpr int kTileTokens = 32;
constexpr int kMaxTopk = 32;
constexpr int kMaxGroups = 32;
constexpr int kMaxGroupTopk = 4;
constexpr int kMaxExpertsPerLane = 16;
constexpr int kMaxExperts = 512;

// Slots of the device-error word array (each written with a plain store).
constexpr int kErrSlots = 4;
constexpr int kErrRange = 0;
constexpr int kErrDuplicate = 1;

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
};

// Router: one warp per token, one 32-token tile per CTA.  Writes topk_idx,
// topk_w and the tile's expert bitmap words tile_word[tile][E].
cudaError_t launch_route(const float* scores, int T, const RouteParams& p, int32_t* topk_idx,
                         float* topk_w, uint32_t* tile_word, cudaStream_t s);

// Bitmap words for caller-made topk_idx, with validity checks.
cudaError_t launch_layout_bits(const int32_t* topk_idx, int T, int k, int E, uint32_t* tile_word,
                               volatile unsigned* err, cudaStream_t s);

// Column prefix over tiles: tile_base[tile][e] and cnt[e].
cudaError_t launch_layout_scan(const uint32_t* tile_word, int ntiles, int E, int32_t* tile_base,
                               int32_t* cnt, cudaStream_t s);

// Offsets (off, rcnt, roff, total) and the row map row[t][j].
cudaError_t launch_rowmap(const int32_t* topk_idx, int T, int k, int E, int R, int mode, int S,
                          const uint32_t* tile_word, const int32_t* tile_base, const int32_t* cnt,
                          int32_t* off, int32_t* rcnt, int32_t* roff, int32_t* row,
                          int sm_count, cudaStream_t s);

// Dispatch pack: x bf16 [T][H] -> receive rows (bf16 copy or FP8 + scales).
cudaError_t launch_dispatch(const void* x, int T, int H, int k, int fp8, const int32_t* row,
                            void* recv_x, float* recv_scale, int32_t* recv_src,
                            const int32_t* cnt, int32_t* recv_cnt, int E, int sm_count,
                            cudaStream_t s);

// Combine: out[t] = bf16(sum_j w[t][j] * y[row[t][j]]).
cudaError_t launch_combine(const void* y, int T, int H, int k, const int32_t* row, const float* w,
                           void* out, int sm_count, cudaStream_t s);

}  // namespace moeep
