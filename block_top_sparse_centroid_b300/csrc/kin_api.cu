// C-ABI entry points of libkin: argument validation, workspace layout, split planning,
// TMA descriptor encoding and kernel launches.  Every call validates on the host first
// and enqueues nothing when it returns an error.  No call allocates or synchronises.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "kin_common.cuh"
#include "kin_internal.h"
#include <algorithm>

namespace kin {
namespace {

thread_local char g_last_error[512] = "";

kin_status fail(kin_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

kin_status ok() {
  g_last_error[0] = '\0';
  return KIN_OK;
}

kin_status cuda_fail(cudaError_t e, const char *what) {
  return fail(KIN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Split planning is a pure function of the shapes (never of the device), so the
// workspace size and the launch always agree.  The bf16 kernel runs one CTA per SM of a
// B300 (148); the plan splits a row's kept list only when there are fewer than two rows
// per CTA (every split past the first costs a partial write and a merge), and aims at
// about three score items per CTA.  Measured: on the 256 rows of the 32-sequence,
// 32K-context workload two splits per row are 4 % faster than one (rows finish their
// selection at different times, and shorter attention items fill the gaps); 2 or 4 score
// items per CTA instead of 3 change no workload by more than the run-to-run spread.
constexpr int kPlanSMs = 148;
#ifndef KIN_PLAN_ATTN_ITEMS
#define KIN_PLAN_ATTN_ITEMS 2
#endif
constexpr int kAttnItemsPerCta = KIN_PLAN_ATTN_ITEMS;
constexpr int kScoreItemsPerCta = 3;
constexpr int kMaxItemsPerSplit = 256;
constexpr int kMaxBlocksLimit = 16384;
constexpr int kHeadsPerRange = 32;

struct Plan {
  int rows, group, max_items, items_per_split, max_splits;
  int score_chunk;      // candidate blocks per score CTA (fp32) or score item (bf16)
  int heads_per_range, head_ranges, chunks_per_seq;   // bf16 score / select items
};

Plan make_plan(const kin_kv_cache *c, const kin_decode_args *a, int mode) {
  Plan pl{};
  pl.rows = a->batch * c->num_kv_heads;
  pl.group = a->num_q_heads / c->num_kv_heads;
  pl.max_items = mode == 0 ? (a->top_k < a->max_blocks ? a->top_k : a->max_blocks) : a->max_blocks;
  const int warps = attention_warps();
  const int target = kPlanSMs * kAttnItemsPerCta;
  int splits = (target + pl.rows - 1) / pl.rows;
  const int max_useful = (pl.max_items + 2 * warps - 1) / (2 * warps);  // >= 2 blocks per warp
  if (splits > max_useful) splits = max_useful;
  if (splits < 1) splits = 1;
  int ips = (pl.max_items + splits - 1) / splits;
  ips = (ips + warps - 1) / warps * warps;
  if (ips > kMaxItemsPerSplit) ips = kMaxItemsPerSplit;
  pl.items_per_split = ips;
  pl.max_splits = (pl.max_items + ips - 1) / ips;
  pl.heads_per_range = c->num_kv_heads < kHeadsPerRange ? c->num_kv_heads : kHeadsPerRange;
  pl.head_ranges = (c->num_kv_heads + pl.heads_per_range - 1) / pl.heads_per_range;
  if (c->dtype == KIN_BF16) {
    // Score items: chunks of the candidate blocks (all but the final block) of one
    // (sequence, head range), a multiple of the pages one ring stage holds.
    const int pps = 32 / pl.heads_per_range;
    const long long cand = static_cast<long long>(a->batch) * pl.head_ranges * (a->max_blocks - 1);
    long long chunk = (cand + kPlanSMs * kScoreItemsPerCta - 1) / (kPlanSMs * kScoreItemsPerCta);
    if (chunk < 2 * pps) chunk = 2 * pps;
    chunk = (chunk + pps - 1) / pps * pps;
    const int cap = fused_max_score_chunk() / pps * pps;
    if (chunk > cap) chunk = cap;
    pl.score_chunk = static_cast<int>(chunk);
    const int n = a->max_blocks - 1;
    pl.chunks_per_seq = mode == 0 && n > 0 ? (n + pl.score_chunk - 1) / pl.score_chunk : 0;
  } else {
    // fp32 score kernel: about 8 CTAs per SM over all candidate blocks, 64..1024 per CTA.
    const long long cand = static_cast<long long>(pl.rows) * a->max_blocks;
    long long chunk = (cand + kPlanSMs * 8 - 1) / (kPlanSMs * 8);
    chunk = (chunk + 63) / 64 * 64;
    if (chunk < 64) chunk = 64;
    if (chunk > 1024) chunk = 1024;
    pl.score_chunk = static_cast<int>(chunk);
  }
  return pl;
}

// The counters of one decode call: the work-queue head, CTAs finished, score arrivals per
// (sequence, head range), split arrivals, ready flags and score error bounds per row.  They sit at the start
// of the workspace, in an area of at least kCounterWords words that no other region
// uses, and are zero between calls: a bf16 call whose counters fit in that area leaves
// them zero itself (the last CTA of its kernel clears them), so it needs no clearing
// launch; any other call clears its counters before its kernels and after them.
constexpr size_t kCounterWords = 16384;
struct Counters {
  size_t work_next, exit_cnt, score_cnt, attn_cnt, ready, bound, count;
};
Counters counter_layout(const kin_decode_args *a, const Plan &pl) {
  Counters k{};
  k.work_next = 0;
  k.exit_cnt = 1;
  k.score_cnt = 2;
  k.attn_cnt = k.score_cnt + static_cast<size_t>(a->batch) * pl.head_ranges;
  k.ready = k.attn_cnt + pl.rows;
  k.bound = k.ready + pl.rows;
  k.count = k.bound + pl.rows;
  return k;
}

struct Layout {
  size_t counters, counter_bytes, part_ml, part_o, scores, sel, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Layout make_layout(const kin_kv_cache *c, const kin_decode_args *a, const Plan &pl, int mode) {
  Layout L{};
  size_t off = 0;
  L.counters = off;
  L.counter_bytes = sizeof(int32_t) * counter_layout(a, pl).count;
  off = align256(off + std::max(L.counter_bytes, sizeof(int32_t) * kCounterWords));
  L.part_ml = off;
  off = align256(off + sizeof(float) * 2 * static_cast<size_t>(pl.rows) * pl.max_splits * pl.group);
  L.part_o = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(pl.rows) * pl.max_splits * pl.group *
                           c->head_dim);
  L.scores = off;
  if (mode == 0) off = align256(off + sizeof(float) * static_cast<size_t>(pl.rows) * a->max_blocks);
  L.sel = off;
  if (mode == 0) off = align256(off + sizeof(int32_t) * static_cast<size_t>(pl.rows) * a->top_k);
  L.total = off;
  return L;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kin_status check_cache_shape(const kin_kv_cache *c) {
  if (c == nullptr) return fail(KIN_ERR_INVALID_ARG, "cache is NULL");
  if (c->dtype != KIN_F32 && c->dtype != KIN_BF16)
    return fail(KIN_ERR_UNSUPPORTED, "dtype %d is not f32 (0) or bf16 (1)", static_cast<int>(c->dtype));
  if (c->page_size != kBlock)
    return fail(KIN_ERR_UNSUPPORTED, "page_size %d: only 16-token pages are supported", c->page_size);
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(KIN_ERR_UNSUPPORTED, "head_dim %d: only 64 and 128 are supported", c->head_dim);
  if (c->num_kv_heads < 1) return fail(KIN_ERR_INVALID_ARG, "num_kv_heads %d < 1", c->num_kv_heads);
  if (c->num_pages < 1) return fail(KIN_ERR_INVALID_ARG, "num_pages %lld < 1", (long long)c->num_pages);
  if (c->num_pages * c->num_kv_heads * kBlock >= (1LL << 31))
    return fail(KIN_ERR_UNSUPPORTED, "num_pages * num_kv_heads * 16 must be below 2^31");
  return ok();
}

kin_status check_cache(const kin_kv_cache *c) {
  kin_status s = check_cache_shape(c);
  if (s != KIN_OK) return s;
  if (c->k_pages == nullptr || c->v_pages == nullptr)
    return fail(KIN_ERR_INVALID_ARG, "k_pages / v_pages is NULL");
  if (!aligned16(c->k_pages) || !aligned16(c->v_pages))
    return fail(KIN_ERR_INVALID_ARG, "k_pages / v_pages must be 16-byte aligned");
  return ok();
}

kin_status check_args(const kin_kv_cache *c, const kin_decode_args *a, int mode) {
  if (a == nullptr) return fail(KIN_ERR_INVALID_ARG, "args is NULL");
  if (a->batch < 1) return fail(KIN_ERR_INVALID_ARG, "batch %d < 1", a->batch);
  if (a->num_q_heads < 1 || a->num_q_heads % c->num_kv_heads != 0)
    return fail(KIN_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of num_kv_heads %d",
                a->num_q_heads, c->num_kv_heads);
  const int G = a->num_q_heads / c->num_kv_heads;
  if (G > 16) return fail(KIN_ERR_UNSUPPORTED, "group size %d > 16", G);
  if (a->max_blocks < 1 || a->max_blocks > kMaxBlocksLimit)
    return fail(KIN_ERR_UNSUPPORTED, "max_blocks %d outside 1..%d", a->max_blocks, kMaxBlocksLimit);
  if ((mode == 0 || mode == 2) && a->top_k < 1)
    return fail(KIN_ERR_INVALID_ARG, "top_k %d < 1", a->top_k);
  if (mode == 2 && c->dtype != KIN_BF16)
    return fail(KIN_ERR_UNSUPPORTED, "token top-k decode needs a bf16 cache");
  if (mode == 2 && a->flags != 0)
    return fail(KIN_ERR_INVALID_ARG, "token top-k decode takes no flags (0x%x)",
                static_cast<unsigned>(a->flags));
  if (!(a->sm_scale > 0.f) || a->sm_scale == INFINITY)
    return fail(KIN_ERR_INVALID_ARG, "sm_scale must be a positive finite number");
  if (a->q == nullptr || a->block_table == nullptr || a->seq_lens == nullptr || a->out == nullptr)
    return fail(KIN_ERR_INVALID_ARG, "q / block_table / seq_lens / out must not be NULL");
  if (!aligned16(a->q)) return fail(KIN_ERR_INVALID_ARG, "q must be 16-byte aligned");
  if ((a->flags & ~KIN_DECODE_APPEND_FINAL) != 0)
    return fail(KIN_ERR_INVALID_ARG, "unknown flags 0x%x", static_cast<unsigned>(a->flags));
  if (a->shared_prefix_blocks < 0 || a->shared_prefix_blocks > a->max_blocks)
    return fail(KIN_ERR_INVALID_ARG, "shared_prefix_blocks %d outside 0..max_blocks (%d)",
                a->shared_prefix_blocks, a->max_blocks);
  if (mode == 0 || (a->flags & KIN_DECODE_APPEND_FINAL) != 0) {
    if (a->centroids == nullptr) return fail(KIN_ERR_INVALID_ARG, "centroids must not be NULL");
    if (!aligned16(a->centroids)) return fail(KIN_ERR_INVALID_ARG, "centroids must be 16-byte aligned");
  }
  return ok();
}

kin_status check_workspace(const kin_decode_args *a, const Layout &L) {
  if (a->workspace == nullptr)
    return fail(KIN_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", L.total);
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
    return fail(KIN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (a->workspace_bytes < L.total)
    return fail(KIN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", a->workspace_bytes, L.total);
  return ok();
}

// --- TMA descriptors -----------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// The page pool as a bf16 tensor of P*H*16 rows of d columns, copied one page of one head
// (16 rows) per TMA with the 128-byte swizzle: rows are split into 64-column halves of
// 128 bytes, and a page lands in shared memory as [d/64 halves][16 rows][64 columns].
// d = 64: a 2-D view (64 columns, rows), box {64, 16}.  d = 128: a 3-D view (64 columns,
// rows, 2 halves) with strides (256 B, 128 B), box {64, 16, 2}, so one copy moves the
// whole page in that same layout.
kin_status encode_page_map(CUtensorMap *map, const kin_kv_cache *c, const void *base) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(KIN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t rows = static_cast<cuuint64_t>(c->num_pages) * c->num_kv_heads * kBlock;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(c->head_dim) * 2;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r;
  if (c->head_dim == 128) {
    const cuuint64_t dims[3] = {64, rows, 2};
    const cuuint64_t strides[2] = {row_bytes, 128};
    const cuuint32_t box[3] = {64, kBlock, 2};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[2] = {64, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {64, kBlock};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return fail(KIN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return KIN_OK;
}

// Makes the device that holds the cache current for the duration of one call (the
// caller's framework may have another device current) and puts the caller's device back
// when the call returns, on every path.
class DeviceScope {
 public:
  DeviceScope() = default;
  DeviceScope(const DeviceScope &) = delete;
  DeviceScope &operator=(const DeviceScope &) = delete;
  ~DeviceScope() {
    if (prev_ >= 0) cudaSetDevice(prev_);
  }
  kin_status enter(const void *ptr) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
      return fail(KIN_ERR_INVALID_ARG, "cache pages are not device memory");
    int cur = -1;
    e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (cur != attr.device) {
      e = cudaSetDevice(attr.device);
      if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
      prev_ = cur;
    }
    return KIN_OK;
  }

 private:
  int prev_ = -1;   // the caller's device, when the call switched away from it
};

// Inside a stream capture the events become event-record nodes of the graph, so that a
// replayed graph still timestamps its kernels.
kin_status record(void *const *events, int i, cudaStream_t stream) {
  if (events == nullptr) return KIN_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  cudaEvent_t ev = static_cast<cudaEvent_t>(events[i]);
  e = cs == cudaStreamCaptureStatusActive
          ? cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal)
          : cudaEventRecord(ev, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  return KIN_OK;
}

// Token top-k: attention CTAs per row (splits) so that about three per SM run at once,
// each taking a multiple of one pass of its warps' 16-token tiles.
struct TokenPlan {
  int rows, group, keep_max, tokens_per_split, splits;
};

TokenPlan make_token_plan(const kin_kv_cache *c, const kin_decode_args *a) {
  TokenPlan tp{};
  tp.rows = a->batch * c->num_kv_heads;
  tp.group = a->num_q_heads / c->num_kv_heads;
  const long long cap = static_cast<long long>(kBlock) * a->max_blocks;
  tp.keep_max = static_cast<int>(a->top_k < cap ? a->top_k : cap);
  const int tile = token_tile_tokens();
  const int max_useful = (tp.keep_max + tile - 1) / tile;
  int splits = (3 * kPlanSMs + tp.rows - 1) / tp.rows;
  if (splits > max_useful) splits = max_useful;
  if (splits < 1) splits = 1;
  int tps = (tp.keep_max + splits - 1) / splits;
  tps = (tps + tile - 1) / tile * tile;
  tp.tokens_per_split = tps;
  tp.splits = (tp.keep_max + tps - 1) / tps;
  return tp;
}

struct TokenLayout {
  size_t counters, part_ml, part_o, scores, gather, total;
};

TokenLayout make_token_layout(const kin_kv_cache *c, const kin_decode_args *a, const TokenPlan &tp) {
  TokenLayout L{};
  size_t off = 0;
  L.counters = off;
  off = align256(off + sizeof(int32_t) * static_cast<size_t>(tp.rows));
  L.part_ml = off;
  off = align256(off + sizeof(float) * 2 * static_cast<size_t>(tp.rows) * tp.splits * tp.group);
  L.part_o = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(tp.rows) * tp.splits * tp.group *
                           c->head_dim);
  L.scores = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(tp.rows) * kBlock * a->max_blocks);
  L.gather = off;
  off = align256(off + sizeof(int32_t) * static_cast<size_t>(tp.rows) * a->top_k);
  L.total = off;
  return L;
}

kin_status run_token_decode(const kin_kv_cache *c, const kin_decode_args *a, cudaStream_t stream,
                            void *const *events = nullptr) {
  kin_status s = check_cache(c);
  if (s != KIN_OK) return s;
  s = check_args(c, a, 2);
  if (s != KIN_OK) return s;
  const TokenPlan tp = make_token_plan(c, a);
  const TokenLayout L = make_token_layout(c, a, tp);
  if (a->workspace == nullptr)
    return fail(KIN_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", L.total);
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
    return fail(KIN_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (a->workspace_bytes < L.total)
    return fail(KIN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", a->workspace_bytes, L.total);
  if (events != nullptr && (events[0] == nullptr || events[1] == nullptr ||
                            events[2] == nullptr || events[3] == nullptr))
    return fail(KIN_ERR_INVALID_ARG, "events must hold 4 created CUDA events");
  DeviceScope scope;
  s = scope.enter(c->k_pages);
  if (s != KIN_OK) return s;
  uint8_t *ws = static_cast<uint8_t *>(a->workspace);
  TokenParams p{};
  p.q = static_cast<const __nv_bfloat16 *>(a->q);
  p.k_pages = static_cast<const __nv_bfloat16 *>(c->k_pages);
  p.v_pages = static_cast<const __nv_bfloat16 *>(c->v_pages);
  p.block_table = a->block_table;
  p.seq_lens = a->seq_lens;
  p.out = a->out;
  p.lse = a->lse;
  p.scores = a->scores != nullptr ? a->scores : reinterpret_cast<float *>(ws + L.scores);
  p.score_stride = static_cast<int64_t>(kBlock) * a->max_blocks;
  p.gather = reinterpret_cast<int32_t *>(ws + L.gather);
  p.sel_out = a->sel_blocks;
  p.part_o = reinterpret_cast<float *>(ws + L.part_o);
  p.part_ml = reinterpret_cast<float *>(ws + L.part_ml);
  p.counters = reinterpret_cast<int32_t *>(ws + L.counters);
  p.err = a->err_flag;
  p.num_pages = c->num_pages;
  p.batch = a->batch;
  p.num_kv_heads = c->num_kv_heads;
  p.group = tp.group;
  p.max_blocks = a->max_blocks;
  p.top_k = a->top_k;
  p.splits = tp.splits;
  p.tokens_per_split = tp.tokens_per_split;
  p.sm_scale = a->sm_scale;
  if ((s = record(events, 0, stream)) != KIN_OK) return s;
  cudaError_t e = launch_token_score(c->head_dim, p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "token score kernel launch");
  if ((s = record(events, 1, stream)) != KIN_OK) return s;
  e = launch_token_select(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "token select kernel launch");
  if ((s = record(events, 2, stream)) != KIN_OK) return s;
  e = launch_token_attn(c->head_dim, p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "token attention kernel launch");
  if ((s = record(events, 3, stream)) != KIN_OK) return s;
  return ok();
}

kin_status run_decode(const kin_kv_cache *c, const kin_decode_args *a, int mode,
                      cudaStream_t stream, void *const *events = nullptr) {
  kin_status s = check_cache(c);
  if (s != KIN_OK) return s;
  s = check_args(c, a, mode);
  if (s != KIN_OK) return s;
  const Plan pl = make_plan(c, a, mode);
  const Layout L = make_layout(c, a, pl, mode);
  s = check_workspace(a, L);
  if (s != KIN_OK) return s;
  if (events != nullptr && (events[0] == nullptr || events[1] == nullptr ||
                            events[2] == nullptr || events[3] == nullptr))
    return fail(KIN_ERR_INVALID_ARG, "events must hold 4 created CUDA events");
  DeviceScope scope;
  s = scope.enter(c->k_pages);
  if (s != KIN_OK) return s;
  uint8_t *ws = static_cast<uint8_t *>(a->workspace);
  int32_t *cnt = reinterpret_cast<int32_t *>(ws + L.counters);
  const Counters ck = counter_layout(a, pl);
  float *scores = a->scores != nullptr ? a->scores : reinterpret_cast<float *>(ws + L.scores);
  int32_t *sel = a->sel_blocks != nullptr ? a->sel_blocks : reinterpret_cast<int32_t *>(ws + L.sel);
  const int append = (a->flags & KIN_DECODE_APPEND_FINAL) != 0;
  const bool self_clean = c->dtype == KIN_BF16 && ck.count <= kCounterWords;
  if ((s = record(events, 0, stream)) != KIN_OK) return s;
  if (!self_clean) {
    cudaError_t me = cudaMemsetAsync(cnt, 0, L.counter_bytes, stream);
    if (me != cudaSuccess) return cuda_fail(me, "cudaMemsetAsync of the workspace counters");
  }
  // After the kernels of a call that does not clear its own counters.
  auto clear_after = [&]() -> kin_status {
    if (self_clean) return KIN_OK;
    cudaError_t me = cudaMemsetAsync(cnt, 0, L.counter_bytes, stream);
    return me == cudaSuccess ? KIN_OK : cuda_fail(me, "cudaMemsetAsync of the workspace counters");
  };

  if (c->dtype == KIN_BF16) {
    CUtensorMap kmap, vmap;
    s = encode_page_map(&kmap, c, c->k_pages);
    if (s != KIN_OK) return s;
    s = encode_page_map(&vmap, c, c->v_pages);
    if (s != KIN_OK) return s;
    FusedParams fp{};
    fp.q = static_cast<const __nv_bfloat16 *>(a->q);
    // the centroid table of a bf16 cache: plane 0 (first codes), then plane 1 (residuals)
    const int64_t plane = c->num_pages * c->num_kv_heads * c->head_dim;
    fp.centroids = static_cast<const __nv_bfloat16 *>(a->centroids);
    fp.cent_lo = fp.centroids == nullptr ? nullptr : fp.centroids + plane;
    fp.cent_out = static_cast<__nv_bfloat16 *>(a->centroids);
    fp.cent_lo_out = fp.cent_out == nullptr ? nullptr : fp.cent_out + plane;
    fp.block_table = a->block_table;
    fp.seq_lens = a->seq_lens;
    fp.out = a->out;
    fp.lse = a->lse;
    fp.scores = scores;
    fp.sel = reinterpret_cast<int32_t *>(ws + L.sel);   // the attention's kept lists
    fp.sel_out = a->sel_blocks;
    fp.part_o = reinterpret_cast<float *>(ws + L.part_o);
    fp.part_ml = reinterpret_cast<float *>(ws + L.part_ml);
    fp.work_next = cnt + ck.work_next;
    fp.score_cnt = cnt + ck.score_cnt;
    fp.attn_cnt = cnt + ck.attn_cnt;
    fp.ready = cnt + ck.ready;
    fp.bound = reinterpret_cast<uint32_t *>(cnt + ck.bound);
    fp.exit_cnt = cnt + ck.exit_cnt;
    fp.counters = cnt;
    fp.n_counters = static_cast<int>(ck.count);
    fp.self_clean = self_clean ? 1 : 0;
    fp.err = a->err_flag;
    fp.num_pages = c->num_pages;
    fp.batch = a->batch;
    fp.num_kv_heads = c->num_kv_heads;
    fp.group = pl.group;
    fp.max_blocks = a->max_blocks;
    fp.top_k = mode == 0 ? a->top_k : 0;
    fp.heads_per_range = pl.heads_per_range;
    fp.head_ranges = pl.head_ranges;
    fp.score_chunk = pl.score_chunk;
    fp.chunks_per_seq = pl.chunks_per_seq;
    fp.items_per_split = pl.items_per_split;
    fp.splits_per_row = pl.max_splits;
    fp.n_score_items = mode == 0 ? a->batch * pl.head_ranges * pl.chunks_per_seq : 0;
    // With up to two rows per CTA, a row's selection is on the critical path (there is too
    // little other attention work to hide it), so all consumer warps of a CTA select one
    // row, one row per select item: ~4-5 us for 2047 candidates instead of ~17 us for a
    // warp alone.  With more rows the cheaper one-warp-per-row selection of a whole head
    // range per item wins.  Measured with the in-selection re-scoring: 256 rows of 32K
    // tokens 9 % faster cooperative than one warp per row; 2048 rows of 3K-17K tokens 21 %
    // slower.
    fp.coop_select = pl.rows <= 2 * kPlanSMs ? 1 : 0;
    fp.n_select_items = mode == 0 ? a->batch * (fp.coop_select ? c->num_kv_heads : pl.head_ranges) : 0;
    fp.n_attn_items = pl.rows * pl.max_splits;
    // Queue lags in rounds (one sequence per round).  At the start every CTA takes an item
    // and prefetches the next, so the first two waves of the queue (2 x 148 items) start
    // at once: a select item comes about two waves of score items after its sequence's
    // score items, and an attention item about two waves of score and select items after
    // its select, so that both normally find what they wait for done.
    if (mode == 0) {
      const int s_per = fp.n_score_items / a->batch, sel_per = fp.n_select_items / a->batch;
      const int span = 2 * kPlanSMs;
      fp.lag_select = s_per > 0 ? (span + s_per - 1) / s_per : 0;
      fp.lag_attn = fp.lag_select + (span + s_per + sel_per - 1) / (s_per + sel_per);
      if (pl.rows <= kPlanSMs) {
        // No more rows than CTAs: every row's selection runs on a CTA of its own anyway, so
        // the queue takes all score items, then all select items, then all attention items
        // (measured: 16 sequences of 8K-32K tokens 12 % faster than interleaved, 8
        // sequences 6 %).
        fp.lag_select = a->batch;
        fp.lag_attn = 2 * a->batch;
      }
    } else {
      fp.lag_select = fp.lag_attn = 0;
    }

    fp.append_final = append;
    fp.shared_prefix_blocks = a->shared_prefix_blocks;
    fp.sm_scale = a->sm_scale;
    // One launch: score, select and attention items through one work queue, so the
    // scoring of later rows overlaps the attention of earlier ones.
    if ((s = record(events, 1, stream)) != KIN_OK) return s;
    if ((s = record(events, 2, stream)) != KIN_OK) return s;
    const FusedParams f2 = fp;
    cudaError_t e = launch_fused(c->head_dim, f2, &kmap, &vmap, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fused decode kernel launch");
    if ((s = clear_after()) != KIN_OK) return s;
    if ((s = record(events, 3, stream)) != KIN_OK) return s;
    return ok();
  }

  // fp32: standalone score, select and CUDA-core attention kernels.
  const int32_t *kept = nullptr;
  if (mode == 0) {
    ScoreParams sp{};
    sp.q = a->q;
    sp.centroids = a->centroids;
    sp.block_table = a->block_table;
    sp.seq_lens = a->seq_lens;
    sp.scores = scores;
    sp.sel = sel;
    sp.err = a->err_flag;
    sp.num_pages = c->num_pages;
    sp.batch = a->batch;
    sp.num_kv_heads = c->num_kv_heads;
    sp.group = pl.group;
    sp.max_blocks = a->max_blocks;
    sp.top_k = a->top_k;
    sp.chunk = pl.score_chunk;
    cudaError_t e = launch_score(c->dtype, c->head_dim, sp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "score kernel launch");
    if ((s = record(events, 1, stream)) != KIN_OK) return s;
    e = launch_select(sp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "select kernel launch");
    if ((s = record(events, 2, stream)) != KIN_OK) return s;
    kept = sel;
  } else {
    if ((s = record(events, 1, stream)) != KIN_OK) return s;
    if ((s = record(events, 2, stream)) != KIN_OK) return s;
  }
  AttnParams ap{};
  ap.q = a->q;
  ap.k_pages = c->k_pages;
  ap.v_pages = c->v_pages;
  ap.block_table = a->block_table;
  ap.seq_lens = a->seq_lens;
  ap.sel = kept;
  ap.out = a->out;
  ap.lse = a->lse;
  ap.cent_out = a->centroids;
  ap.part_o = reinterpret_cast<float *>(ws + L.part_o);
  ap.part_ml = reinterpret_cast<float *>(ws + L.part_ml);
  ap.counters = cnt + ck.attn_cnt;
  ap.err = a->err_flag;
  ap.num_pages = c->num_pages;
  ap.batch = a->batch;
  ap.num_kv_heads = c->num_kv_heads;
  ap.group = pl.group;
  ap.max_blocks = a->max_blocks;
  ap.sel_stride = mode == 0 ? a->top_k : 0;
  ap.items_per_split = pl.items_per_split;
  ap.max_splits = pl.max_splits;
  ap.append_final = append;
  ap.sm_scale = a->sm_scale;
  cudaError_t e = launch_attention_f32(c->head_dim, ap, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
  if ((s = clear_after()) != KIN_OK) return s;
  if ((s = record(events, 3, stream)) != KIN_OK) return s;
  return ok();
}

kin_status run_centroids(const kin_kv_cache *c, const int32_t *page_ids, int64_t n,
                         void *centroids, int32_t *err, cudaStream_t stream) {
  kin_status s = check_cache(c);
  if (s != KIN_OK) return s;
  if (n < 0) return fail(KIN_ERR_INVALID_ARG, "n %lld < 0", (long long)n);
  if (centroids == nullptr) return fail(KIN_ERR_INVALID_ARG, "centroids is NULL");
  if (!aligned16(centroids)) return fail(KIN_ERR_INVALID_ARG, "centroids must be 16-byte aligned");
  if (page_ids == nullptr && n != c->num_pages)
    return fail(KIN_ERR_INVALID_ARG, "page_ids is NULL but n (%lld) != num_pages (%lld)",
                (long long)n, (long long)c->num_pages);
  if (n == 0) return ok();
  DeviceScope scope;
  s = scope.enter(c->k_pages);
  if (s != KIN_OK) return s;
  cudaError_t e = launch_centroids(c->dtype, c->head_dim, c->num_kv_heads, c->k_pages,
                                   c->num_pages, page_ids, n, centroids, err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "centroid kernel launch");
  return ok();
}

}  // namespace

kin_status set_error(kin_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

}  // namespace kin

extern "C" {

const char *kin_status_str(kin_status s) {
  switch (s) {
    case KIN_OK: return "KIN_OK";
    case KIN_ERR_INVALID_ARG: return "KIN_ERR_INVALID_ARG";
    case KIN_ERR_UNSUPPORTED: return "KIN_ERR_UNSUPPORTED";
    case KIN_ERR_WORKSPACE: return "KIN_ERR_WORKSPACE";
    case KIN_ERR_CUDA: return "KIN_ERR_CUDA";
  }
  return "KIN_ERR_UNKNOWN";
}

const char *kin_last_error(void) { return kin::g_last_error; }

kin_status kin_workspace_size(const kin_kv_cache *cache, const kin_decode_args *args, int32_t mode,
                              size_t *bytes) {
  using namespace kin;
  if (bytes == nullptr) return fail(KIN_ERR_INVALID_ARG, "bytes is NULL");
  if (mode < 0 || mode > 2) return fail(KIN_ERR_INVALID_ARG, "mode %d is not 0, 1 or 2", mode);
  kin_status s = check_cache_shape(cache);
  if (s != KIN_OK) return s;
  if (args == nullptr) return fail(KIN_ERR_INVALID_ARG, "args is NULL");
  if (args->batch < 1 || args->num_q_heads < 1 || args->max_blocks < 1 ||
      args->max_blocks > kMaxBlocksLimit || args->num_q_heads % cache->num_kv_heads != 0 ||
      args->num_q_heads / cache->num_kv_heads > 16 || (mode != 1 && args->top_k < 1))
    return fail(KIN_ERR_INVALID_ARG, "bad shapes for workspace sizing");
  if (mode == 2) {
    *bytes = make_token_layout(cache, args, make_token_plan(cache, args)).total;
    return ok();
  }
  const Plan pl = make_plan(cache, args, mode);
  *bytes = make_layout(cache, args, pl, mode).total;
  return ok();
}

kin_status kin_centroids_build(const kin_kv_cache *cache, const int32_t *page_ids, int64_t n,
                               void *centroids, int32_t *err_flag, kin_stream_t stream) {
  return kin::run_centroids(cache, page_ids, n, centroids, err_flag,
                            reinterpret_cast<cudaStream_t>(stream));
}

kin_status kin_centroids_append(const kin_kv_cache *cache, const int32_t *page_ids, int32_t n,
                                void *centroids, int32_t *err_flag, kin_stream_t stream) {
  using namespace kin;
  if (n > 0 && page_ids == nullptr) return fail(KIN_ERR_INVALID_ARG, "page_ids is NULL");
  return kin::run_centroids(cache, page_ids, n, centroids, err_flag,
                            reinterpret_cast<cudaStream_t>(stream));
}

kin_status kin_blocktopk_decode(const kin_kv_cache *cache, const kin_decode_args *args,
                                kin_stream_t stream) {
  return kin::run_decode(cache, args, 0, reinterpret_cast<cudaStream_t>(stream));
}

kin_status kin_dense_decode(const kin_kv_cache *cache, const kin_decode_args *args,
                            kin_stream_t stream) {
  return kin::run_decode(cache, args, 1, reinterpret_cast<cudaStream_t>(stream));
}

kin_status kin_token_topk_decode(const kin_kv_cache *cache, const kin_decode_args *args,
                                 kin_stream_t stream) {
  return kin::run_token_decode(cache, args, reinterpret_cast<cudaStream_t>(stream));
}

kin_status kin_decode_timed(const kin_kv_cache *cache, const kin_decode_args *args, int32_t mode,
                            void *const *events, kin_stream_t stream) {
  using namespace kin;
  if (mode < 0 || mode > 2) return fail(KIN_ERR_INVALID_ARG, "mode %d is not 0, 1 or 2", mode);
  if (events == nullptr) return fail(KIN_ERR_INVALID_ARG, "events is NULL");
  if (mode == 2) return kin::run_token_decode(cache, args, reinterpret_cast<cudaStream_t>(stream), events);
  return kin::run_decode(cache, args, mode, reinterpret_cast<cudaStream_t>(stream), events);
}

}  // extern "C"
