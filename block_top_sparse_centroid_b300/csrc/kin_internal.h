// Host-side declarations shared by the translation units of libkin.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kin.h"

namespace kin {

// Centroid (mean key) of the listed pages: kernel launch.
cudaError_t launch_centroids(kin_dtype dtype, int head_dim, int num_kv_heads,
                             const void *k_pages, int64_t num_pages, const int32_t *page_ids,
                             int64_t n, void *centroids, int32_t *err, cudaStream_t stream);

struct ScoreParams {
  const void *q;             // [B, H*G, d]
  const void *centroids;     // [P, H, d]
  const int32_t *block_table;
  const int32_t *seq_lens;
  float *scores;             // [B*H, max_blocks]
  int32_t *sel;              // [B*H, top_k]
  int32_t *err;
  int64_t num_pages;
  int batch, num_kv_heads, group, max_blocks, top_k;
  int chunk;                 // candidate blocks scored per CTA
};
cudaError_t launch_score(kin_dtype dtype, int head_dim, const ScoreParams &p,
                         cudaStream_t stream);
cudaError_t launch_select(const ScoreParams &p, cudaStream_t stream);

struct AttnParams {
  const void *q;             // [B, H*G, d]
  const void *k_pages;       // [P, H, 16, d]
  const void *v_pages;
  const int32_t *block_table;
  const int32_t *seq_lens;
  const int32_t *sel;        // [B*H, sel_stride] kept logical blocks, or NULL = every block
  void *out;                 // [B, H*G, d]
  float *lse;                // [B, H*G] or NULL
  void *cent_out;            // centroid table written when append_final is set
  float *part_o;             // [B*H, max_splits, G, d] unnormalised partial outputs
  float *part_ml;            // [B*H, max_splits, G, 2] (running max in log2 units, sum)
  int32_t *counters;         // [B*H] split arrivals (cleared before the kernel starts)
  int32_t *err;
  int64_t num_pages;
  int batch, num_kv_heads, group, max_blocks, sel_stride;
  int items_per_split;       // blocks handled by one CTA
  int max_splits;
  int append_final;
  float sm_scale;
};
// fp32 caches: CUDA-core split-KV attention (grid = max_splits x rows).
cudaError_t launch_attention_f32(int head_dim, const AttnParams &p, cudaStream_t stream);

// bf16 caches: one persistent, warp-specialised kernel for score + select + attention
// (+ final-block append).  Work items, handed out in this order by a global counter:
//   score items   (sequence b, head range hr, chunk c): scores of candidate blocks
//                 [c * score_chunk, (c + 1) * score_chunk) for heads [hr * HS, hr * HS + HS)
//   select items  (sequence b, head range hr): top-k selection of those rows
//   attention     (row = b * H + h, split): attention over one split of the kept list
struct FusedParams {
  const __nv_bfloat16 *q;          // [B, H*G, d]
  const __nv_bfloat16 *centroids;  // [P, H, d] first centroid code (the fp32 mean in bf16)
  const __nv_bfloat16 *cent_lo;    // [P, H, d] second code (the rounding residual in bf16)
  __nv_bfloat16 *cent_out;         // both planes written when append_final is set
  __nv_bfloat16 *cent_lo_out;
  const int32_t *block_table;      // [B, max_blocks]
  const int32_t *seq_lens;         // [B]
  void *out;                       // [B, H*G, d]
  float *lse;                      // [B, H*G] or NULL
  float *scores;                   // [B*H, max_blocks]
  int32_t *sel;                    // [B*H, top_k] kept lists the attention reads (workspace)
  int32_t *sel_out;                // [B*H, top_k] the caller's copy, ascending, or NULL
  float *part_o;                   // [B*H, splits_per_row, G, d]
  float *part_ml;                  // [B*H, splits_per_row, G, 2]
  int32_t *work_next;              // work-queue head
  int32_t *score_cnt;              // [B * head_ranges] finished score items
  int32_t *attn_cnt;               // [B*H] split arrivals
  int32_t *ready;                  // [B*H] selection published
  uint32_t *bound;                 // [B*H] score error bound of the row (fp32 bits, max)
  int32_t *exit_cnt;               // CTAs finished (self_clean only)
  int32_t *counters;               // all of the above counters, n_counters words
  int n_counters;
  int self_clean;                  // the last CTA to finish zeroes the counters
  int32_t *err;
  int64_t num_pages;
  int batch, num_kv_heads, group, max_blocks;
  int top_k;                       // 0 = dense decode (every block, no scoring)
  int heads_per_range, head_ranges;  // HS = min(H, 32) heads per score / select item
  int score_chunk, chunks_per_seq;   // candidate blocks per score item, items per range
  int items_per_split, splits_per_row;
  int n_score_items, n_select_items, n_attn_items;
  // Queue order: round r holds the score items of sequence r, the select items of
  // sequence r - lag_select and the attention items of sequence r - lag_attn (each part
  // only when that sequence exists), so that streaming scores and attention overlap.
  int lag_select, lag_attn;
  int coop_select;                 // select items are single rows, selected by all consumer warps
  int append_final;
  int shared_prefix_blocks;        // leading logical blocks read with the evict-last policy
  float sm_scale;
};
// Token-level top-k decode (bf16 caches): score every token, select the top_k per row,
// attend over the kept tokens (token_topk.cu).
struct TokenParams {
  const __nv_bfloat16 *q;          // [B, H*G, d]
  const __nv_bfloat16 *k_pages;    // [P, H, 16, d]
  const __nv_bfloat16 *v_pages;
  const int32_t *block_table;      // [B, max_blocks]
  const int32_t *seq_lens;         // [B]
  void *out;                       // [B, H*G, d]
  float *lse;                      // [B, H*G] or NULL
  float *scores;                   // [B*H, score_stride] token scores
  int64_t score_stride;            // 16 * max_blocks
  int32_t *gather;                 // [B*H, top_k] kept tokens' rows of the [P*H*16, d] view
  int32_t *sel_out;                // [B*H, top_k] kept positions ascending, or NULL
  float *part_o, *part_ml;         // split partials [B*H, splits, G, d] and [.., G, 2]
  int32_t *counters;               // [B*H] split arrivals (zero between calls)
  int32_t *err;
  int64_t num_pages;
  int batch, num_kv_heads, group, max_blocks;
  int top_k;                       // tokens kept per row
  int splits, tokens_per_split;    // attention CTAs per row and kept tokens each
  float sm_scale;
};
cudaError_t launch_token_score(int head_dim, const TokenParams &p, cudaStream_t stream);
cudaError_t launch_token_select(const TokenParams &p, cudaStream_t stream);
cudaError_t launch_token_attn(int head_dim, const TokenParams &p, cudaStream_t stream);
// Kept tokens one attention CTA takes per pass (its warps' tiles); splits are multiples.
int token_tile_tokens();

cudaError_t launch_fused(int head_dim, const FusedParams &p, const CUtensorMap *kmap,
                         const CUtensorMap *vmap, cudaStream_t stream);
// Largest score chunk the fused kernel accepts (candidate blocks per score item).
int fused_max_score_chunk();

// Tiling facts the host needs for workspace sizing and split planning.
int attention_warps();

// Record a one-line reason for kin_last_error() and return `s`.
kin_status set_error(kin_status s, const char *fmt, ...);

}  // namespace kin
