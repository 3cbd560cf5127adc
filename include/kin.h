/*
 * kin.h -- block top-k (centroid-scored) sparse decode attention on B300 (sm_103a).
 *
 * The method: every 16-token key block of a paged KV cache is summarised by its mean
 * key vector (its centroid); for one decode step, the blocks of each (sequence, KV head)
 * row are scored by the dot product of that centroid with the query heads of the GQA
 * group, summed over the group; the top-k blocks are kept and softmax attention runs
 * over the kept blocks' keys and values only.  Sources:
 *   - block top-k ranks key blocks by their mean key vectors and keeps the k best
 *     blocks of each GQA query group -- Pith review of "Kinetics: Rethinking Test-Time
 *     Scaling Laws", section "What carries the argument" (block top-k as the sparse
 *     replacement of the quadratic KV term in the eFLOPs cost model C_TTS);
 *   - block = KV page of 16 tokens, k counted in pages, one decoder layer of paged
 *     decode, dense decode as the comparison -- Kinetics README, section "Benchmark
 *     Block TopK Attention throughput" (--page_size 16 --topk_page 64).
 * Readings where the pages are silent (identical in the library and in its tests):
 *   - the group score is the SUM over the group's query heads of q_g . c_j;
 *   - the final block (holding the current token, possibly partial) is always kept and
 *     counts toward k; it is never scored; with nb <= k blocks every block is kept;
 *   - equal scores go to the lower block index;
 *   - sm_scale multiplies q.k inside the softmax; scoring is scale-free.
 *
 * Conventions for every entry point:
 *   - All pointers inside the structs are DEVICE pointers (cudaMalloc'd or torch
 *     tensors on the current device) unless stated otherwise; the structs themselves
 *     live in host memory and are read during the call only.
 *   - The library allocates no memory and never synchronises: all work is enqueued on
 *     the given stream (a cudaStream_t; NULL = the legacy default stream) and runs
 *     asynchronously.  The caller owns every buffer and keeps it alive until the
 *     stream reaches the enqueued work.
 *   - Every call runs on the device that holds the cache's pages (it makes that device
 *     current while it enqueues) and leaves the calling thread's current device as it
 *     found it, on every return path.
 *   - Arguments are validated on the host before anything is enqueued; a bad argument
 *     returns a status and enqueues nothing.  kin_last_error() gives a one-line reason.
 *   - Errors only the device can see (a block-table entry outside [0, num_pages), a
 *     seq_len outside [1, 16 * max_blocks]) are OR-ed into *err_flag (KIN_DEVERR_*
 *     bits) when err_flag is non-NULL; the offending block or row is skipped (a skipped
 *     row gets zero output and lse = -inf).  Kernels never trap and never wait without
 *     bound.
 *   - Layout: K and V pages are [num_pages, num_kv_heads, 16, head_dim], contiguous,
 *     row-major; query head q_h uses KV head h / G with G = num_q_heads / num_kv_heads
 *     (query heads of one group are consecutive).
 *   - Supported: head_dim in {64, 128}; G in 1..16; dtype f32 or bf16 (the same for Q,
 *     K, V, centroids and O).  Anything else returns KIN_ERR_UNSUPPORTED.
 */
#ifndef KIN_H
#define KIN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KIN_API __attribute__((visibility("default")))
#else
#define KIN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kin_stream_t; /* same type as cudaStream_t */

typedef enum {
  KIN_OK = 0,
  KIN_ERR_INVALID_ARG = 1, /* NULL where required, negative size, bad shape        */
  KIN_ERR_UNSUPPORTED = 2, /* head_dim / group / dtype / size outside the set above */
  KIN_ERR_WORKSPACE = 3,   /* workspace missing or smaller than kin_workspace_size  */
  KIN_ERR_CUDA = 4         /* a CUDA runtime or driver call failed at enqueue time  */
} kin_status;

typedef enum { KIN_F32 = 0, KIN_BF16 = 1 } kin_dtype;

/* Bits OR-ed into *err_flag by the kernels. */
#define KIN_DEVERR_PAGE_ID 1 /* a block-table or page-list entry outside [0, num_pages) */
#define KIN_DEVERR_SEQ_LEN 2 /* a seq_len outside [1, 16 * max_blocks]                 */
#define KIN_DEVERR_TIMEOUT 4 /* a bounded wait gave up: for a copy, for another CTA's
                                result (scores published, a selection released) or for
                                a shared counter; the kernel then winds down            */

/* A paged KV cache of one attention layer (caller-owned device memory). */
typedef struct {
  kin_dtype dtype;
  int32_t num_kv_heads;   /* H, >= 1                                                  */
  int32_t head_dim;       /* d, 64 or 128                                             */
  int32_t page_size;      /* tokens per page == tokens per block; must be 16          */
  int64_t num_pages;      /* P; num_pages * num_kv_heads * 16 must stay below 2^31    */
  const void *k_pages;    /* [P, H, 16, d], 16-byte aligned                           */
  const void *v_pages;    /* [P, H, 16, d], 16-byte aligned                           */
} kin_kv_cache;

/* One decode step over a batch of sequences. */
typedef struct {
  int32_t batch;          /* B >= 1                                                   */
  int32_t num_q_heads;    /* H * G                                                    */
  int32_t max_blocks;     /* columns of block_table, 1..16384                          */
  int32_t top_k;          /* k >= 1 blocks kept per (sequence, KV head); ignored by dense */
  float sm_scale;         /* softmax scale (> 0), e.g. 1/sqrt(d)                      */
  const void *q;          /* [B, H*G, d]                                              */
  const int32_t *block_table; /* [B, max_blocks] physical page of logical block j      */
  const int32_t *seq_lens;    /* [B] tokens incl. the current one; nb = ceil(L/16)     */
  void *centroids;        /* block centroids (kin_centroids_build): fp32 caches [P, H, d];
                             bf16 caches [2, P, H, d] (plane 0: the fp32 mean rounded to
                             bf16, plane 1: its rounding residual rounded to bf16).  Read
                             by block top-k; rows of complete final blocks written when
                             flags has KIN_DECODE_APPEND_FINAL; unused by dense otherwise */
  void *out;              /* [B, H*G, d] attention output                              */
  float *lse;             /* optional [B, H*G]: natural-log sum of exp(sm_scale * q.k)  */
  int32_t *sel_blocks;    /* optional [B, H, top_k]: kept logical blocks, ascending,
                             -1 padded when nb < k (block top-k only)                   */
  float *scores;          /* optional [B, H, max_blocks]: group scores of blocks
                             0..nb-2 of rows with nb > k (other entries untouched); for
                             bf16 caches computed from plane 0 of the centroids          */
  void *workspace;        /* scratch of kin_workspace_size() bytes, 256-byte aligned.
                             Zero-fill it once before its first use (cudaMemset); after
                             that only decode calls may write it: every call leaves its
                             counter area zero again, so calls of any shapes can share it
                             without a clearing launch.  Calls that may overlap on the GPU
                             (other streams) must not share a workspace                  */
  size_t workspace_bytes;
  int32_t *err_flag;      /* optional device int; KIN_DEVERR_* bits are OR-ed in       */
  int32_t flags;          /* KIN_DECODE_* bits, 0 for none                             */
  int32_t shared_prefix_blocks; /* 0..max_blocks: the leading logical blocks whose pages
                             every sequence of the batch shares (a Best-of-N prompt).
                             Block top-k and dense decode then keep those pages' K, V and
                             centroid rows in L2 for the whole step (evict-last copies,
                             every other copy streams evict-first), so that HBM serves
                             each shared page once per step however many sequences read
                             it.  A hint: results are identical for any value; 0 = none.
                             Ignored by kin_token_topk_decode                           */
} kin_decode_args;

/* Decode flag: when a sequence's final block is complete (seq_len a multiple of 16: the
 * current token completed its page), also write that page's centroid into
 * args->centroids, with the arithmetic of kin_centroids_append.  This is the append a
 * decode step needs for later steps (the final block itself is never scored), done from
 * the keys the attention already stages on chip, so it costs no extra HBM read. */
#define KIN_DECODE_APPEND_FINAL 1

/* Human-readable name of a status. Never NULL. */
KIN_API const char *kin_status_str(kin_status s);

/* One-line description of the last failed call on this host thread ("" if none). */
KIN_API const char *kin_last_error(void);

/* Bytes of workspace that kin_blocktopk_decode (mode 0), kin_dense_decode (mode 1) or
 * kin_token_topk_decode (mode 2) needs for these shapes (pointers inside the structs are
 * not read).  Calls of different modes may share one workspace sized for the largest. */
KIN_API kin_status kin_workspace_size(const kin_kv_cache *cache, const kin_decode_args *args,
                              int32_t mode, size_t *bytes);

/* Centroid (mean key) of every listed page, for every KV head:
 *   c[p, h, :] = (sum_{t<16} K[p, h, t, :]) / 16
 * summed in fp32 in ascending t.  Blocks are ranked by this mean key -- Pith review,
 * "What carries the argument".  fp32 caches store c in centroids[p, h, :].  bf16 caches
 * store two bf16 codes per element: centroids[0, p, h, :] = bf16(c) (round-to-nearest-
 * even) and centroids[1, p, h, :] = bf16(c - bf16(c)) (the difference is exact in fp32),
 * whose sum is c to about 2^-16 of its size.  Block scores are streamed from plane 0;
 * plane 1 settles the candidates whose plane-0 scores lie too close to the cut to rank
 * them as the fp32 mean would.
 * page_ids: device int32[n] physical page ids (pages must hold 16 valid tokens), or
 * NULL for all pages 0..num_pages-1 (then n must equal num_pages).  centroids: device
 * [num_pages, H, d] (fp32) or [2, num_pages, H, d] (bf16); only the listed pages' rows
 * are written.  Ids outside [0, num_pages) are skipped and flagged in *err_flag
 * (optional). */
KIN_API kin_status kin_centroids_build(const kin_kv_cache *cache, const int32_t *page_ids, int64_t n,
                               void *centroids, int32_t *err_flag, kin_stream_t stream);

/* Same arithmetic as kin_centroids_build for the pages a decode step just completed
 * (a page whose 16th token was written).  n may be 0 (nothing is enqueued). */
KIN_API kin_status kin_centroids_append(const kin_kv_cache *cache, const int32_t *page_ids, int32_t n,
                                void *centroids, int32_t *err_flag, kin_stream_t stream);

/* One block top-k decode step: for every sequence b and KV head h with
 * nb = ceil(seq_lens[b] / 16) blocks:
 *   score   s_j = sum_g q[b, hG+g, :] . c[block_table[b, j], h, :],  j < nb-1
 *   select  S = {nb-1} + the k-1 largest s_j (ties to lower j); all blocks if nb <= k
 *   attend  out[b, hG+g, :] = softmax over the valid tokens of S of sm_scale * q.k, applied to V
 * with c the fp32 block mean.  Pith review, "What carries the argument"; Kinetics README,
 * "Benchmark Block TopK Attention throughput".  Needs args->centroids built for every
 * complete block that can be scored (all blocks but the final one of each sequence).
 * bf16 caches: every candidate is scored with plane 0 of the centroids (fp32
 * arithmetic); with E a bound on that score's distance from the fp32-mean score over the
 * row, candidates more than 2E above (below) the k-th score are kept (dropped), and
 * those in between are re-scored with both planes before the cut is made.  The kept set
 * is therefore the fp32-mean ranking's, up to rankings that the two planes cannot
 * separate (score differences of about 2^-16 of the scores' size).  args->scores holds
 * the plane-0 scores.  Outputs are undefined when the call sets KIN_DEVERR_TIMEOUT. */
KIN_API kin_status kin_blocktopk_decode(const kin_kv_cache *cache, const kin_decode_args *args,
                                kin_stream_t stream);

/* Dense paged decode over every block (the comparison baseline): the attend step of
 * kin_blocktopk_decode with S = all blocks.  args->top_k, centroids, sel_blocks and
 * scores are ignored. */
KIN_API kin_status kin_dense_decode(const kin_kv_cache *cache, const kin_decode_args *args,
                            kin_stream_t stream);

/* One token-level ("oracle") top-k decode step, the exact-selection upper bound that
 * block top-k approximates (scime summary of "Kinetics: Rethinking Test-Time Scaling
 * Laws", "Key results"; Pith review of the paper, "assumptions").  For every sequence b
 * and KV head h with L = seq_lens[b] tokens and B = args->top_k (tokens, not blocks):
 *   score   s_t = sum_g q[b, hG+g, :] . K[t, h, :]  for every t < L  (fp32)
 *   select  T = the B largest s_t, ties to the lower position; every token if L <= B
 *   attend  out[b, hG+g, :] = softmax over T of sm_scale * q.k, applied to V
 * No token is forced in.  Reads every key of every row once (three kernels: score,
 * select, attend).  bf16 caches only (KIN_ERR_UNSUPPORTED otherwise); args->flags must be
 * 0 and args->centroids is not read.  args->sel_blocks, optional, is [B, H, top_k]: the
 * kept token positions ascending, -1 padded when L < top_k.  args->scores, optional, is
 * [B, H, 16 * max_blocks]: s_t of positions t < L (other entries untouched).  The
 * workspace (kin_workspace_size mode 2) follows the rules of kin_decode_args.workspace;
 * kin_decode_timed mode 2 records events[1] after scoring and events[2] after
 * selection. */
KIN_API kin_status kin_token_topk_decode(const kin_kv_cache *cache, const kin_decode_args *args,
                                         kin_stream_t stream);

/* kin_blocktopk_decode for callers that cannot allocate device memory -- e.g. a server
 * that gives all GPU memory to its KV-cache pool at start-up and allows no allocation
 * afterwards, or a loop that must not let cudaMalloc/cudaFree synchronise the device.
 * The paper has no counterpart: this is a property of the library, not of the method.
 * Identical work and results; args->workspace / workspace_bytes are ignored and the
 * scratch is instead a 32 MiB array inside the library, which every GPU that loads the
 * library keeps until the process exits.  Shapes whose kin_workspace_size exceeds 32 MiB
 * return KIN_ERR_WORKSPACE.  The first call on a device looks up the array's device
 * address (with that device current); make that first call before any stream capture.
 * All calls share the one array, which starts zero-filled and keeps the previous call's
 * contents (every call leaves its counter area zero), so calls that may overlap on the
 * GPU -- other streams, other host threads -- race and must not be issued. */
KIN_API kin_status kin_blocktopk_decode_static(const kin_kv_cache *cache,
                                               const kin_decode_args *args,
                                               kin_stream_t stream);

/* Measurement variant of kin_blocktopk_decode (mode 0), kin_dense_decode (mode 1) or
 * kin_token_topk_decode (mode 2):
 * identical work, plus cudaEventRecord of the caller's events on `stream`: events[0]
 * before the step, events[3] after its last kernel (and, for calls that clear their
 * counters with memsets, after the clearing).  Modes 0 and 1 on bf16 caches run one
 * kernel, and events[1] and events[2] are recorded right before it; on fp32 caches, and in
 * mode 2, events[1] follows scoring and events[2] selection (dense: both right after
 * events[0]).  events: host array of 4 created
 * cudaEvent_t handles.  Used to time a step's kernels without a profiler.  While `stream`
 * is being captured into a CUDA graph the records are made with cudaEventRecordExternal,
 * so that they become event-record nodes and every replay of the graph timestamps its
 * kernels. */
KIN_API kin_status kin_decode_timed(const kin_kv_cache *cache, const kin_decode_args *args,
                                    int32_t mode, void *const *events, kin_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KIN_H */
