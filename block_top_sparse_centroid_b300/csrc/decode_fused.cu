// One persistent, warp-specialised kernel for a whole bf16 decode step: group scoring,
// top-k block selection and split-KV attention, plus the centroid append of complete
// final blocks.
//
// Block top-k ranks key blocks by their mean key vectors and keeps the k best blocks of
// each GQA query group (Pith review of "Kinetics: Rethinking Test-Time Scaling Laws",
// "What carries the argument"); blocks are 16-token pages and k counts pages (Kinetics
// README, "Benchmark Block TopK Attention throughput").
//
// One CTA per SM: kProducers producer warps and 4 or 8 consumer warps around a ring of
// shared-memory stages (128 KB with 8 consumer warps, 160 KB with 4).  HBM needs well over
// 100 KB in flight per SM to run near its peak, and one thread issues a page's copies only
// every few hundred cycles, so four producer warps run ahead of the consumers across work
// items, bounded only by the ring (and, for attention pages, by a short L2 prefetch).
//
// Work items, handed out by a global counter (queue order: see queue_item):
//   score items   (sequence, head range, chunk of candidate blocks).  The producers copy
//                 each candidate's centroid rows for the head range (one contiguous
//                 [heads, d] run per page) into the ring with bulk copies; the consumers
//                 form s_j = (sum_g q_g) . c_j and store it.  The last consumer warp to
//                 finish the item publishes it with an arrival count per (sequence, head
//                 range).
//   select items  (sequence, head range), one consumer warp per row; or, when there are
//                 no more rows than CTAs, a single row selected by all consumer warps
//                 together.  After the row's score items have published, the m-th largest
//                 score key is built bit by bit over keys held in registers (a radix
//                 select over L2 for rows too long for that), the kept list is written
//                 ascending (equal scores to the lower block index, the final block last)
//                 and the row's ready flag released.  A CTA holds at most two unfinished
//                 select items.
//   attention     (row, split of the kept list).  The producer waits for the row's ready
//                 flag, reads the split's kept blocks and their pages, and stages each
//                 page's K and V (one TMA tiled copy each, 128-byte swizzle).  Producer
//                 q stages pages q, q + kProducers, ... for its pipeline's consumer warps,
//                 which compute S^T = K Q^T and O^T += V^T P^T with mma.m16n8k16 (bf16 in,
//                 fp32 accumulate) and an online softmax; the warps' states are combined
//                 in shared memory and the row's splits merged by the last split to
//                 arrive (attn_common.cuh).
// Every wait is bounded (a timeout sets KIN_DEVERR_TIMEOUT) and none can deadlock: every
// item comes after everything it waits for in the queue (score items wait for nothing but
// their own copies, select items for their row's score items, attention items for their
// row's selection), and a CTA takes items in queue order, so the unfinished item with the
// smallest queue index can always progress.  The last CTA to finish zeroes the workspace
// counters for the next call.
#include <atomic>
#include <type_traits>

#include "attn_common.cuh"
#include "kin_internal.h"

namespace kin {
namespace {

constexpr int kProducers = 4;                       // producer warps = ring pipelines
// L2 prefetch distance of each producer in its own attention pages.  When the producer
// issues page l it also prefetches the K and V tiles of page l + kPrefetchPages, which then
// stream from HBM while the producer waits for a free ring stage.  Measured over distances
// 1..20 (distance 0 is no prefetch): 1-3 are equally best, 12 and more lose again (L2
// pressure); at 2, dense decode is 15 % and block top-k 5-12 % faster than without.  A like
// prefetch of the centroid rows of score items (4 stages ahead) made them slower.
constexpr int kPrefetchPages = 2;
constexpr int kMaxRingBytes = 160 * 1024;
constexpr int kMaxStages = kMaxRingBytes / (64 * 64);  // stages at d = 64
constexpr int kDescs = 8;                           // descriptor slots producer -> consumers
constexpr int kMaxScoreChunk = 256;                 // candidate blocks per score item
constexpr int kHeadsPerRange = 32;                  // KV heads per score / select item
constexpr int kScoreSlots = 16;                     // score-item arrival counters (> kDescs)
// Consumer scratch: the combine buffers of an attention item, the group-summed queries
// of a score item, or the histograms of the selections (never at once).
constexpr int kScratchBytes = 34 * 1024;
static_assert(kScratchBytes >= 8 * 8 * (128 + 2) * 4, "combine buffers, 8 warps x 8 heads");
static_assert(kScratchBytes >= 4 * 16 * (128 + 2) * 4, "combine buffers, 4 warps x 16 heads");
static_assert(kScratchBytes >= kHeadsPerRange * 128 * 4, "group-summed queries, shared");
static_assert(kScratchBytes >= 8 * 8 * 128 * 4, "group-summed queries, one copy per warp");

// Launch shape for a head dimension D and NT n-tiles of 8 query heads (NT = 1: groups
// of up to 8 query heads, NT = 2: up to 16).  kCW consumer warps (threads 0 .. 32 kCW - 1)
// and kProducers producer warps after them; consumer warp w takes its pages from
// pipeline w % kProducers, alternating with the other consumers of that pipeline.
template <int D, int NT>
struct Cfg {
  static constexpr int kCW = NT == 1 ? 8 : 4;
  static constexpr int kCThreads = kCW * 32;
  static constexpr int kAllThreads = (kCW + kProducers) * 32;
  static constexpr int kPPC = kCW / kProducers;    // consumers per pipeline
  static constexpr int kQMax = 8 * NT;
  using Bar = GroupBarrier<kCThreads>;
  static_assert(kCW * kQMax * (D + 2) * 4 <= kScratchBytes, "combine buffers");
  static_assert(kCW * 256 * 4 <= kScratchBytes, "selection histograms");
};

// The ring is split into one sub-ring per consumer warp.  Producer q stages the pages
// (or score stages) q, q + kProducers, ... of every item, handing them in turn to its
// consumer warps q, q + kProducers, ... (kPPC of them); each goes through that consumer's
// sub-ring.  So every sub-ring has a single producer and a single consumer, both walk it
// in the same order, and neither can get two laps ahead of the other (which the parity
// waits of an mbarrier could not tell apart).
template <int D, int NT>
struct Ring {
  static constexpr int kStageBytes = BfTile<D>::kStageBytes;   // K + V page of one head
  static constexpr int kBytes = NT == 1 ? 128 * 1024 : kMaxRingBytes;
  static constexpr int kStages = kBytes / kStageBytes;         // 16 / 32 or 20 / 40
  static constexpr int kPer = kStages / Cfg<D, NT>::kCW;       // stages per consumer
  static_assert(kStages <= kMaxStages && kStages % Cfg<D, NT>::kCW == 0, "stage arrays");
  // shared-memory stage of consumer w's n-th page (or score stage), and its phase
  __device__ static __forceinline__ int slot(int w, uint32_t n) { return w * kPer + n % kPer; }
  __device__ static __forceinline__ uint32_t phase(uint32_t n) { return (n / kPer) & 1u; }
};


// Score items of up to 8 heads and groups of up to 8 query heads (NT = 1) get their raw q
// rows staged by a bulk copy into one of two slots, so that no consumer waits on a global
// load of q (a dependent load costs microseconds while HBM is saturated).
constexpr int kQSlotBytes = 8 * 8 * 128 * 2;
template <int NT>
constexpr int q_stage_bytes() { return NT == 1 ? 2 * kQSlotBytes : 0; }

template <int D, int NT>
constexpr size_t fused_smem_bytes() {
  // 1024: alignment of the ring base
  return 1024 + Ring<D, NT>::kBytes + kScratchBytes + q_stage_bytes<NT>();
}

enum : int { kDescEnd = 0, kDescScore = 1, kDescSelect = 2, kDescAttn = 3, kDescEmptyRow = 4 };
enum : int { kAttnEveryBlock = 1, kAttnAppendLast = 2 };

// A work item as the producer hands it to the consumers.
struct Desc {
  int kind;
  int first;   // score: staged q slot (0 / 1), or -1 when q is read from global memory
  int count;   // stages of the item (attention: pages)
  int row;     // score / select: sequence b; attention / empty row: b * H + h
  int x0;      // score / select: first head h0; attention: split
  int x1;      // score: first candidate j0; select: candidates n; attention: splits
  int x2;      // score / select: heads in the range; attention: kAttn* flags
  int x3;      // tokens L of the sequence
#ifdef KIN_TRACE_CYCLES
  int item;
#endif
};

struct FusedShared {
  uint64_t full[kMaxStages];    // stage filled (producer arrival + copy bytes)
  uint64_t empty[kMaxStages];   // stage consumed (one consumer warp)
  uint64_t dfull[kDescs];       // descriptor written
  uint64_t dempty[kDescs];      // descriptor read by every consumer warp
  uint64_t qfull[2];            // staged q rows landed
  uint64_t qempty[2];           // staged q rows read by every consumer warp
  int4 meta[kMaxStages];        // attention: {page, ntok}; score: {j of first page, pages, valid mask}
  Desc desc[kDescs];
  int plist[kProducers][kMaxScoreChunk];  // producers: pages of the current score item
  int score_arrive[16];         // consumers: warps done with a score item (kScoreSlots)
  int flag;                     // consumers: last-arriver flag of the split merge
  int sel_done;                 // consumers: select items finished (read by the queue leader)
  int sel_ok;                   // consumers: the current select item's scores arrived
  int last_cta;                 // this CTA finished last (clears the counters)
  int abort;                    // set after a wait of this CTA timed out
};

// Bounded mbarrier wait.  After any wait of the CTA has timed out (a broken protocol),
// later waits give up within a few hundred polls, so the CTA winds down quickly instead
// of timing out wait by wait.  The waits that hand out work descriptors (deliver = true)
// are the exception: they never take that shortcut and have a 16 times longer bound,
// because every warp of the CTA must see the same items in the same order (the consumer
// warps' group barriers inside an item are reached by all of them only then), and after a
// timeout the queue leader still delivers every descriptor promptly (its other waits end
// early).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, FusedShared &sh,
                                         int32_t *err, bool deliver = false) {
  const uint32_t addr = smem_u32(bar);
  const uint32_t tries = deliver ? 16u * kMaxWaitTries : kMaxWaitTries;
  for (uint32_t i = 0; i < tries; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if (!deliver && (i & 255u) == 255u && *reinterpret_cast<volatile int *>(&sh.abort) != 0)
      return false;
  }
  *reinterpret_cast<volatile int *>(&sh.abort) = 1;
  flag_error(err, KIN_DEVERR_TIMEOUT);
  return false;
}

// Bounded wait until *flag >= target (acquire).  Same abort rule as wait_bar.
__device__ __forceinline__ bool wait_flag(const int32_t *flag, int target, FusedShared &sh,
                                          int32_t *err) {
  for (uint32_t i = 0; i < kMaxWaitTries; ++i) {
    if (ld_acquire_gpu(flag) >= target) return true;
    if ((i & 255u) == 255u && *reinterpret_cast<volatile int *>(&sh.abort) != 0) return false;
    __nanosleep(64);
  }
  *reinterpret_cast<volatile int *>(&sh.abort) = 1;
  flag_error(err, KIN_DEVERR_TIMEOUT);
  return false;
}

// wait_flag returning the value seen (the last one read when the wait gives up).
__device__ __forceinline__ int wait_flag_value(const int32_t *flag, int target, FusedShared &sh,
                                               int32_t *err) {
  int v = 0;
  for (uint32_t i = 0; i < kMaxWaitTries; ++i) {
    v = ld_acquire_gpu(flag);
    if (v >= target) return v;
    if ((i & 255u) == 255u && *reinterpret_cast<volatile int *>(&sh.abort) != 0) return v;
    __nanosleep(64);
  }
  *reinterpret_cast<volatile int *>(&sh.abort) = 1;
  flag_error(err, KIN_DEVERR_TIMEOUT);
  return v;
}

// Bounded wait until the shared counter *cnt >= target.  Same abort rule as wait_bar.
__device__ __forceinline__ bool wait_shared_count(const int *cnt, int target, FusedShared &sh,
                                                  int32_t *err) {
  for (uint32_t i = 0; i < kMaxWaitTries; ++i) {
    if (*reinterpret_cast<const volatile int *>(cnt) >= target) return true;
    if ((i & 255u) == 255u && *reinterpret_cast<volatile int *>(&sh.abort) != 0) return false;
    __nanosleep(32);
  }
  *reinterpret_cast<volatile int *>(&sh.abort) = 1;
  flag_error(err, KIN_DEVERR_TIMEOUT);
  return false;
}

// Optional cycle counters per (CTA, warp) for tuning (compile with -DKIN_TRACE_CYCLES;
// off in the library build).  Lane 0 of each warp accumulates clock64() deltas into slots.
#ifdef KIN_TRACE_CYCLES
constexpr int kTraceCtas = 160, kTraceWarps = 12, kTraceSlots = 20;
__device__ unsigned long long g_trace[kTraceCtas * kTraceWarps * kTraceSlots];
// Per-thread accumulators (registers / local memory), flushed once per warp at exit.
struct TraceAcc {
  long long v[kTraceSlots];
};
__device__ __forceinline__ void trace_flush(const TraceAcc &t) {
  if ((threadIdx.x & 31) == 0 && blockIdx.x < kTraceCtas)
    for (int i = 0; i < kTraceSlots; ++i)
      g_trace[(blockIdx.x * kTraceWarps + (threadIdx.x >> 5)) * kTraceSlots + i] += t.v[i];
}
#define KIN_TRACE_DECL TraceAcc tr_ = {};
#define KIN_TRACE_PARAM , TraceAcc &tr_
#define KIN_TRACE_ARG , tr_
#define KIN_TRACE_FLUSH trace_flush(tr_)
#define KIN_TIC(name) const long long name = clock64()
#define KIN_TOC(slot, name) (tr_.v[slot] += clock64() - (name))
#define KIN_COUNT(slot, n) (tr_.v[slot] += (n))
// Per-item timeline: {cta, fetched, ready seen, consume begin, consume end, kind} in
// globaltimer nanoseconds, for the first kTraceItems work items.
constexpr int kTraceItems = 1 << 16;
__device__ unsigned long long g_items[kTraceItems * 8];
__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define KIN_ITEM_STAMP(item, field, value) \
  do { if ((item) >= 0 && (item) < kTraceItems) g_items[(item) * 8 + (field)] = (value); } while (0)
#else
#define KIN_ITEM_STAMP(item, field, value) do {} while (0)
#define KIN_TRACE_DECL
#define KIN_TRACE_PARAM
#define KIN_TRACE_ARG
#define KIN_TRACE_FLUSH
#define KIN_TIC(v)
#define KIN_TOC(slot, v)
#define KIN_COUNT(slot, n)
#endif
// producer slots
enum { kTrTotal = 0, kTrPWaitEmpty = 1, kTrPIssue = 2, kTrPMeta = 3, kTrPReady = 4, kTrPPush = 5,
       kTrPPages = 6, kTrPItems = 7, kTrPNext = 8 };
// consumer slots
enum { kTrCWaitFull = 1, kTrCPage = 2, kTrCDesc = 3, kTrCEpilogue = 4, kTrCScore = 5,
       kTrCSelect = 6, kTrCPages = 7, kTrCItems = 8, kTrCQ = 9, kTrCScoreQ = 10,
       kTrCScoreWait = 11, kTrCEpiBar = 12, kTrCSelWait = 13, kTrCScoreComp = 14,
       kTrCSelComp = 15, kTrCSelKeys = 16, kTrCSelPass = 17 };

__device__ __forceinline__ uint32_t score_key(float s) {
  // order-preserving 32-bit key: -0 and +0 equal, NaN below every number (branch-free)
  const uint32_t u = __float_as_uint(s + 0.0f);
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return s != s ? 0u : k;
}

// The score of a key (inverse of score_key for keys of numbers).
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ----------------------------------------------------------------------------------
// Selection.  The kernel scores every candidate with the first centroid code (bf16), which
// is what it can stream at full bandwidth; the reference ranking is by the fp32 mean.  With
// E >= |s - s*| for every candidate of the row (p.bound) and a threshold T that at most m
// scores exceed and at least m reach (the m-th largest score, or a smaller value at which
// exactly m scores are >= T, where the search stops early), a candidate with s > T + 2E is
// in the top m by s* as well (only candidates with s > T, at most m of them counting
// itself, can beat it), and one with s < T - 2E is out (every candidate with s >= T, at
// least m of them, beats it).  The candidates in between ("ambiguous") are
// re-scored with both codes, s + qs . c2, which is the score of the fp32 mean to about
// 2^-16 of its size, and the m - (number in) best of them are kept, equal scores to the
// lower block index.  The selection runs on modified keys: in -> kKeyIn, out -> 0,
// ambiguous -> the key of the re-scored value, so that one top-m search over them yields
// the kept list.  Keys of real scores are >= 2, padding slots 0.
// ----------------------------------------------------------------------------------
constexpr uint32_t kKeyIn = 0xffffffffu;   // above the key of every number (+inf: 0xff800000)
// Ambiguous candidates a row's selection re-scores in shared memory (more: the long-row path).
constexpr int kAmbCapWarp = 256;

struct Window {
  uint32_t lo, hi;   // in: key > hi; ambiguous: lo <= key <= hi; out: key < lo
  bool refine;       // ambiguous candidates are re-scored (else they tie, lower index first)
};

// The window around the m-th largest key t for the row bound E.  Without a usable bound (a
// non-finite T or E) the window is t itself: candidates tied at t, taken in index order.
__device__ __forceinline__ Window make_window(uint32_t t, float E) {
  const float T = key_score(t);
  if (t < 2u || !(fabsf(T) <= 3.0e38f) || !(E >= 0.f && E <= 1.0e37f)) return Window{t, t, false};
  const float e2 = 2.f * E;
  return Window{max(score_key(__fadd_rd(T, -e2)), 2u), score_key(__fadd_ru(T, e2)), true};
}

// What the re-scoring of a row's ambiguous candidates needs.
struct RefineCtx {
  const __nv_bfloat16 *c2;     // second centroid code of KV head h: page p at c2 + p * stride
  const int32_t *trow;         // block-table row of the sequence
  int64_t stride;              // H * D
  int64_t num_pages;
  const float *qs;             // group-summed query of the row, fp32 [D] (shared memory)
};

// Key of the re-scored candidate j with first-code score s: s + qs . c2_j, computed by LPC
// consecutive lanes (each one D / LPC slice of the dimensions; every lane of the group
// returns the key).  All loads of a lane are issued before any is used.
template <int D, int LPC>
__device__ __forceinline__ uint32_t refined_key(const RefineCtx &rc, int j, float s, int lane) {
  constexpr int kChunks = D / 8 / LPC;   // 16-byte chunks per lane
  const int part = lane % LPC;
  const int pg = __ldg(rc.trow + j);
  float corr = 0.f;
  if (pg >= 0 && pg < rc.num_pages) {
    const uint4 *src = reinterpret_cast<const uint4 *>(rc.c2 + pg * rc.stride) + part * kChunks;
    uint4 raw[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) raw[c] = __ldcg(src + c);
    const float *qs = rc.qs + part * kChunks * 8;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      float f[8];
      Elem<__nv_bfloat16>::unpack(raw[c], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) corr = fmaf(qs[8 * c + k], f[k], corr);
    }
  }
#pragma unroll
  for (int o = 1; o < LPC; o <<= 1) corr += __shfl_xor_sync(0xffffffffu, corr, o);
  return max(score_key(s + corr), 2u);
}

// Group-summed query of KV head h (sum over g in order, fp32) into qs[0..D), by one warp:
// lane l sums dimensions [l D / 32, (l + 1) D / 32), one vector load per query head; the
// loop is unrolled so that several heads' loads are in flight at once.
template <int D>
__device__ __forceinline__ void group_query(const __nv_bfloat16 *qg, int G, float *qs, int lane) {
  constexpr int kPer = D / 32;                     // 4 (D = 128) or 2 (D = 64)
  using Raw = typename std::conditional<kPer == 4, uint2, uint32_t>::type;
  auto unpack = [](const Raw &r, float (&f)[kPer]) {
    if constexpr (kPer == 4) {
      f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x); f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    } else {
      f[0] = bf16_lo(r); f[1] = bf16_hi(r);
    }
  };
  const Raw *src = reinterpret_cast<const Raw *>(qg + lane * kPer);
  float acc[kPer];
  unpack(__ldg(src), acc);
#pragma unroll 4
  for (int g = 1; g < G; ++g) {
    float f[kPer];
    unpack(__ldg(src + g * (D / kPer)), f);
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] += f[i];
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) qs[lane * kPer + i] = acc[i];
}

// m-th largest of the keys held in registers by one warp (lane l: slots i, candidate
// l + 32 i; 0 = padding or out): t, and whether exactly m keys are >= t.  Built bit by bit
// from the highest bit where the nonzero keys differ: a bit stays set when at least m keys
// are >= the candidate prefix; the search stops once exactly m keys are >= the prefix (those
// are the m largest, and nothing outside them ties with anything inside).
template <int KPL>
__device__ __forceinline__ uint32_t bits_threshold(const uint32_t (&key)[KPL], int m, bool &exact) {
  uint32_t all_and = 0xffffffffu, all_or = 0u;
  int nz = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    all_and &= key[i] != 0u ? key[i] : 0xffffffffu;
    all_or |= key[i];
    nz += key[i] != 0u ? 1 : 0;
  }
  all_and = __reduce_and_sync(0xffffffffu, all_and);
  all_or = __reduce_or_sync(0xffffffffu, all_or);
  nz = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(nz)));
  const uint32_t diff = all_and ^ all_or;
  const int top = diff == 0u ? 0 : 32 - __clz(diff);   // bits [0, top) undecided
  uint32_t t = top == 32 ? 0u : (all_and & (0xffffffffu << top));
  // keys >= t: every nonzero key shares the bits above `top` (t = 0 only while the search
  // runs: the callers have more than m nonzero keys, so the last bit sets t >= 1)
  int cnt_t = nz;
#pragma unroll 1
  for (int b = top - 1; b >= 0 && cnt_t != m; --b) {
    const uint32_t cand = t | (1u << b);
    int c0 = 0, c1 = 0;
#pragma unroll
    for (int i = 0; i + 1 < KPL; i += 2) {
      c0 += key[i] >= cand ? 1 : 0;
      c1 += key[i + 1] >= cand ? 1 : 0;
    }
    const int c = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c0 + c1)));
    if (c >= m) {
      t = cand;
      cnt_t = c;
    }
  }
  exact = cnt_t == m;
  return t;
}

// Index-order compaction of the m kept candidates: every key > t, plus (exact: the keys
// equal to t too; else the first m - count(key > t) keys equal to t in index order).
// jbase: candidate index of slot 0 of lane 0; out[pos0 ..] receives the warp's kept
// candidates, eq0 equal keys are already taken by earlier warps, take_eq in total.
template <int KPL>
__device__ __forceinline__ void bits_emit(const uint32_t (&key)[KPL], uint32_t t, bool exact,
                                          int take_eq, int pos0, int eq0, int m, int jbase,
                                          int32_t *out, int lane) {
  const unsigned lt = (1u << lane) - 1u;
  int written = pos0, eq_seen = eq0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {   // unrolled: key[] stays in registers
    unsigned km = __ballot_sync(0xffffffffu, exact ? key[i] >= t : key[i] > t);
    if (!exact) {
      const unsigned eqm = __ballot_sync(0xffffffffu, key[i] == t);
      const int eq_here = __popc(eqm);
      int eq_take = take_eq - eq_seen;
      if (eq_take >= eq_here) {
        km |= eqm;
      } else if (eq_take > 0) {   // the first eq_take of this slot
        unsigned msk = eqm;
        for (; eq_take > 0; --eq_take) {
          const unsigned low = msk & (0u - msk);
          km |= low;
          msk ^= low;
        }
      }
      eq_seen += eq_here;
    }
    const int pos = written + __popc(km & lt);
    if (((km >> lane) & 1u) && pos < m) out[pos] = jbase + lane + 32 * i;
    written += __popc(km);
  }
}

// Classify the warp's register keys against the window: for every slot i, the ballots of
// its in and ambiguous candidates go to bal[i] and bal[KPL + i] (shared memory, written by
// lane 0), so that the later passes over the candidates run as short loops over the
// ballots instead of long unrolled code over the registers.  Returns the warp's counts.
template <int KPL>
__device__ __forceinline__ void classify(const uint32_t (&key)[KPL], const Window &w,
                                         uint32_t *bal, int &n_in, int &n_amb, int lane) {
  int a = 0, b = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const unsigned bi = __ballot_sync(0xffffffffu, key[i] > w.hi);
    const unsigned ba = __ballot_sync(0xffffffffu, key[i] >= w.lo && key[i] <= w.hi);
    if (lane == 0) {
      bal[i] = bi;
      bal[KPL + i] = ba;
    }
    a += __popc(bi);
    b += __popc(ba);
  }
  n_in = a;
  n_amb = b;
  __syncwarp();
}

// classify for one warp that also writes, in the same pass, the certain candidates to
// out[0 .. n_in) (ascending) and the ambiguous ones with their first-code scores to
// lst[0 .. min(n_amb, cap)) (ascending).
template <int KPL>
__device__ __forceinline__ void classify_emit(const uint32_t (&key)[KPL], const Window &w,
                                              uint32_t *bal, int32_t *out, int2 *lst, int cap,
                                              int &n_in, int &n_amb, int lane) {
  const unsigned lt = (1u << lane) - 1u;
  int a = 0, b = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const bool is_in = key[i] > w.hi, is_amb = key[i] >= w.lo && key[i] <= w.hi;
    const unsigned bi = __ballot_sync(0xffffffffu, is_in);
    const unsigned ba = __ballot_sync(0xffffffffu, is_amb);
    if (lane == 0) {
      bal[i] = bi;
      bal[KPL + i] = ba;
    }
    if (is_in) out[a + __popc(bi & lt)] = lane + 32 * i;
    const int rank = b + __popc(ba & lt);
    if (is_amb && rank < cap) lst[rank] = make_int2(lane + 32 * i, __float_as_int(key_score(key[i])));
    a += __popc(bi);
    b += __popc(ba);
  }
  n_in = a;
  n_amb = b;
  __syncwarp();
}

// The same writes for the warps of a cooperative selection, from their class ballots:
// this warp's certain candidates go to out[in0 ..], its ambiguous ones to lst[amb0 ..].
template <int KPL>
__device__ __forceinline__ void emit_in_and_list(const uint32_t (&key)[KPL], const uint32_t *bal,
                                                 int in0, int amb0, int jbase, int32_t *out,
                                                 int2 *lst, int cap, int lane) {
  const unsigned lt = (1u << lane) - 1u;
  int a = in0, b = amb0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const unsigned bi = bal[i], ba = bal[KPL + i];
    const int j = jbase + lane + 32 * i;
    if ((bi >> lane) & 1u) out[a + __popc(bi & lt)] = j;
    const int rank = b + __popc(ba & lt);
    if (((ba >> lane) & 1u) && rank < cap) lst[rank] = make_int2(j, __float_as_int(key_score(key[i])));
    a += __popc(bi);
    b += __popc(ba);
  }
}

// Choose r of the na listed ambiguous candidates (ranks 0 .. na - 1, in index order) by
// one warp: the r largest re-scored keys lr[rank * KS], equal keys to the lower rank.  Sets
// lf[rank] (1 = kept) for every rank.  KA keys per lane: na <= 32 KA.
template <int KA, int KS = 1>
__device__ __forceinline__ void choose_amb(const uint32_t *lr, int na, int r, uint8_t *lf,
                                           int lane) {
  uint32_t key[KA];
#pragma unroll
  for (int i = 0; i < KA; ++i) key[i] = lane + 32 * i < na ? lr[(lane + 32 * i) * KS] : 0u;
  bool exact;
  const uint32_t t = bits_threshold<KA>(key, r, exact);
  int take_eq = 0;
  if (!exact) {
    int g = 0;
#pragma unroll
    for (int i = 0; i < KA; ++i) g += key[i] > t ? 1 : 0;
    take_eq = r - static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(g)));
  }
  const unsigned lt = (1u << lane) - 1u;
  int eq_seen = 0;
#pragma unroll
  for (int i = 0; i < KA; ++i) {
    const bool eq = !exact && key[i] == t;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const bool keep = exact ? key[i] >= t : (key[i] > t || (eq && eq_seen + __popc(eqm & lt) < take_eq));
    if (lane + 32 * i < na) lf[lane + 32 * i] = keep ? 1 : 0;
    eq_seen += __popc(eqm);
  }
}

// Index-order compaction from the class ballots (classify): the in candidates (take_in),
// and the ambiguous ones that are chosen (take_amb; lf[rank] != 0, or when lf is NULL the
// first amb_limit of them in index order).  Ranks of this warp's ambiguous candidates start at rank0; its emitted candidates
// go to out[pos0 ..] (at most up to out[m - 1]).
__device__ __forceinline__ void emit_class(const uint32_t *bal, int nslots, const uint8_t *lf,
                                           bool take_in, bool take_amb, int rank0, int pos0,
                                           int m, int jbase, int32_t *out, int lane,
                                           int amb_limit = 0x7fffffff) {
  const unsigned lt = (1u << lane) - 1u;
  int base = rank0, written = pos0;
  for (int i = 0; i < nslots; ++i) {
    const unsigned bi = bal[i], ba = bal[nslots + i];
    const bool a = ((ba >> lane) & 1u) != 0;
    const int rank = base + __popc(ba & lt);
    const bool keep = (take_in && ((bi >> lane) & 1u) != 0) ||
                      (take_amb && a && (lf == nullptr ? rank < amb_limit : lf[rank] != 0));
    const unsigned km = __ballot_sync(0xffffffffu, keep);
    const int pos = written + __popc(km & lt);
    if (keep && pos < m) out[pos] = jbase + lane + 32 * i;
    written += __popc(km);
    base += __popc(ba);
  }
}

#ifndef KIN_RK_ROWS
#define KIN_RK_ROWS 16   // candidate rows per re-scoring batch of one warp (no spill at d = 128)
#endif
// Pages of the listed ambiguous candidates lst[e].x into pg[e] (-1: outside the table or
// an invalid page id), e = ti, ti + nthr, ...; several loads in flight per thread.
__device__ __forceinline__ void list_pages(const int2 *lst, int n, const int32_t *trow,
                                           int max_blocks, int64_t num_pages, int *pg, int ti,
                                           int nthr) {
#pragma unroll 4
  for (int e = ti; e < n; e += nthr) {
    const int j = lst[e].x;
    const int pp = j >= 0 && j < max_blocks ? __ldg(trow + j) : -1;
    pg[e] = pp >= 0 && pp < num_pages ? pp : -1;
  }
}

// Re-scored keys of the listed ambiguous candidates lst[e] = (j, first-code score bits),
// e in batches of KIN_RK_ROWS starting at e_begin, e_step apart (one warp): lst[e].y becomes the
// key of s + qs . c2_j.  Each candidate row is read by D / 8 lanes, one 16-byte chunk each
// (lane chunk c: dimensions 8c .. 8c + 7, whose qs values the lane keeps in registers),
// and all loads of a batch are issued before any is used, so a batch costs one memory
// latency.
template <int D>
__device__ __forceinline__ void refine_keys(int2 *lst, const int *pg, int n, int e_begin,
                                            int e_step, const __nv_bfloat16 *c2, int64_t stride,
                                            const float *qs, int lane) {
  constexpr int kLpr = D / 8;        // lanes per candidate row
  constexpr int kRpi = 32 / kLpr;    // rows per warp-wide load
  constexpr int kNld = KIN_RK_ROWS / kRpi;    // loads per lane per batch
  const int c = lane % kLpr, sub = lane / kLpr;
  float qv[8];
  {
    const float4 a = *reinterpret_cast<const float4 *>(qs + 8 * c);
    const float4 b = *reinterpret_cast<const float4 *>(qs + 8 * c + 4);
    qv[0] = a.x; qv[1] = a.y; qv[2] = a.z; qv[3] = a.w;
    qv[4] = b.x; qv[5] = b.y; qv[6] = b.z; qv[7] = b.w;
  }
#pragma unroll 1
  for (int e0 = e_begin; e0 < n; e0 += e_step) {
    uint4 raw[kNld];
#pragma unroll
    for (int k = 0; k < kNld; ++k) {
      const int e = e0 + k * kRpi + sub;
      const int pgv = e < n ? pg[e] : -1;
      raw[k] = pgv >= 0 ? __ldcg(reinterpret_cast<const uint4 *>(c2 + pgv * stride) + c)
                        : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kNld; ++k) {
      float f[8];
      Elem<__nv_bfloat16>::unpack(raw[k], f);
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) part = fmaf(qv[i], f[i], part);
#pragma unroll
      for (int o = 1; o < kLpr; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      const int e = e0 + k * kRpi + sub;
      if (c == 0 && e < n)
        lst[e].y = static_cast<int>(max(score_key(__int_as_float(lst[e].y) + part), 2u));
    }
  }
}

// The chosen ambiguous candidates (lf[e] != 0) in index order into dst[0 .. r), one warp.
__device__ __forceinline__ void append_chosen(const int2 *lst, const uint8_t *lf, int n, int r,
                                              int32_t *dst, int lane) {
  const unsigned lt = (1u << lane) - 1u;
  int written = 0;
  for (int e0 = 0; e0 < n; e0 += 32) {
    const int e = e0 + lane;
    const bool pick = e < n && lf[e] != 0;
    const unsigned km = __ballot_sync(0xffffffffu, pick);
    const int at = written + __popc(km & lt);
    if (pick && at < r) dst[at] = lst[e].x;
    written += __popc(km);
  }
}

// Kept lists are released in two phases (the row's ready word): first the candidates that
// are in for certain (positions 0 .. n_in - 1, ascending) and the final block (position m),
// ready word n_in + 1, as soon as they are classified; then, once the ambiguous ones are
// re-scored, the chosen ones (positions n_in .. m - 1, ascending), ready word kReadyAll.
// The attention streams the first part meanwhile.  A selection with no ambiguous
// candidate to re-score releases kReadyAll at once.  The caller's copy (sel_out) is
// ascending.
constexpr int kReadyAll = 1 << 30;

// Scratch of one selecting warp (or of the CTA in a cooperative selection).
struct SelScratch {
  float *qs;      // [D] group-summed query of the row
  uint32_t *bal;  // [2 * slots] class ballots of the warp (cooperative: per warp)
  int *hist;      // [256] radix histograms (rows too long for the registers)
  int *xs;        // [128] cross-warp partial sums (cooperative selection)
  int2 *lst;      // [kAmbCapWarp] listed ambiguous candidates (block, score bits / key)
  int *pg;        // [kAmbCapWarp] their pages
  uint8_t *lf;    // [kAmbCapWarp] chosen flags
};

template <int D>
__device__ void warp_select_long(const float *srow, int n, int m, int nb, float E,
                                 const RefineCtx &rc, const __nv_bfloat16 *qg, int G,
                                 const SelScratch &ss, int32_t *out, int lane);

// Kept blocks of one row by one warp, keys in registers: lane l holds candidates
// j = l + 32 i, i < KPL (n <= 32 KPL).  Writes the kept list out[0 .. m] (the final block
// nb - 1 at out[m]), releasing the certain candidates before it re-scores the ambiguous
// ones (lst, this warp's shared memory); returns true (the row is settled).
template <int KPL, int D>
__device__ bool warp_select_bits(const float *srow, int n, int m, int nb, float E,
                                 const RefineCtx &rc, const __nv_bfloat16 *qg, int G,
                                 const SelScratch &ss, int32_t *out, int32_t *out_user,
                                 int32_t *ready, int2 *lst, int lane KIN_TRACE_PARAM) {
  KIN_TIC(t_k);
  uint32_t key[KPL];
  const int nv = n > lane ? (n - lane + 31) / 32 : 0;   // this lane's candidates
  {
    float sv[KPL];   // every load issued before any is used
#pragma unroll
    for (int i = 0; i < KPL; ++i) sv[i] = i < nv ? __ldcg(srow + lane + 32 * i) : 0.f;
    group_query<D>(qg, G, ss.qs, lane);   // for the re-scoring; its loads overlap these
#pragma unroll
    for (int i = 0; i < KPL; ++i) key[i] = i < nv ? max(score_key(sv[i]), 2u) : 0u;
  }
  KIN_TOC(kTrCSelKeys, t_k);
  if (lane == 0) {
    out[m] = nb - 1;
    if (out_user != nullptr) out_user[m] = nb - 1;
  }
  if (m == 0) return true;
  KIN_TIC(t_p);
  bool exact;
  const uint32_t t = bits_threshold<KPL>(key, m, exact);
  const Window w = make_window(t, E);
  int n_in, n_amb;
  classify_emit<KPL>(key, w, ss.bal, out, lst, kAmbCapWarp, n_in, n_amb, lane);
  const int r = m - n_in;
  bool complete = true;
  if (n_amb == r || r == 0 || !w.refine) {
    // every ambiguous candidate kept, none, or a tie at the cut without a usable bound
    // (equal scores: the first r in index order)
    emit_class(ss.bal, KPL, nullptr, true, true, 0, 0, m, 0, out, lane, r);
    if (out_user != nullptr) emit_class(ss.bal, KPL, nullptr, true, true, 0, 0, m, 0, out_user, lane, r);
  } else if (n_amb > kAmbCapWarp) {
    // more ambiguous candidates than the list holds (clustered scores): the exact
    // selection that re-reads the row instead of holding it
    warp_select_long<D>(srow, n, m, nb, E, rc, qg, G, ss, out, lane);
    __syncwarp();
    if (out_user != nullptr)
      for (int i = lane; i <= m; i += 32) out_user[i] = out[i];
  } else {
    // the certain ones are in place: release them, then re-score the listed ambiguous
    // candidates (their pages from the block table, then their second codes: two memory
    // latencies per 32 of them), choose r and append them
    __syncwarp();
    if (lane == 0) st_release_gpu(ready, n_in + 1);
    list_pages(lst, n_amb, rc.trow, n, rc.num_pages, ss.pg, lane, 32);
    __syncwarp();
    refine_keys<D>(lst, ss.pg, n_amb, 0, KIN_RK_ROWS, rc.c2, rc.stride, ss.qs, lane);
    __syncwarp();
    const uint32_t *lr = reinterpret_cast<const uint32_t *>(lst) + 1;
    if (n_amb <= 64)
      choose_amb<2, 2>(lr, n_amb, r, ss.lf, lane);
    else
      choose_amb<kAmbCapWarp / 32, 2>(lr, n_amb, r, ss.lf, lane);
    __syncwarp();
    append_chosen(lst, ss.lf, n_amb, r, out + n_in, lane);
    if (out_user != nullptr) emit_class(ss.bal, KPL, ss.lf, true, true, 0, 0, m, 0, out_user, lane);
  }
  KIN_TOC(kTrCSelPass, t_p);
  return complete;
}

// Selection of one row by all NW consumer warps: warp w holds candidates
// j = w 32 KPL + 32 i + lane (i < KPL), keys in registers; n <= NW 32 KPL.  The same steps
// as warp_select_bits, with each count summed over the warps through shared memory (a
// per-warp partial, double-buffered by parity, one consumer-group barrier per sum).  The
// kept list is written in index order: each warp offsets its own compaction by the counts
// of the warps before it.
template <int KPL, int NW, int D, typename Bar>
__device__ bool cta_select_row(const float *srow, int n, int m, int nb, float E,
                               const RefineCtx &rc, const __nv_bfloat16 *qg, int G,
                               const SelScratch &ss, int32_t *out, int32_t *out_user,
                               int32_t *ready, int2 *lst) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int jbase = w * 32 * KPL;
  uint32_t key[KPL];
  {
    float sv[KPL];
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int j = jbase + lane + 32 * i;
      sv[i] = j < n ? __ldcg(srow + j) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < KPL; ++i) key[i] = jbase + lane + 32 * i < n ? max(score_key(sv[i]), 2u) : 0u;
  }
  if (w == 0) group_query<D>(qg, G, ss.qs, lane);   // published by the first CTA sum's barrier
  int *xs = ss.xs;
  int par = 0;
  // sum of v over the consumer warps (v must be warp-uniform); *before = the sum over the
  // warps before this one
  auto cta_sum = [&](int v, int *before) -> int {
    if (lane == 0) xs[par * NW + w] = v;
    Bar::sync();
    int s = 0, b = 0;
#pragma unroll
    for (int u = 0; u < NW; ++u) {
      const int x = xs[par * NW + u];
      s += x;
      b += u < w ? x : 0;
    }
    par ^= 1;
    if (before != nullptr) *before = b;
    return s;
  };
  // m-th largest key over the CTA (same bit search as bits_threshold)
  auto threshold = [&](bool &exact) -> uint32_t {
    uint32_t a = 0xffffffffu, o = 0u;
    int nz = 0;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      a &= key[i] != 0u ? key[i] : 0xffffffffu;
      o |= key[i];
      nz += key[i] != 0u ? 1 : 0;
    }
    a = __reduce_and_sync(0xffffffffu, a);
    o = __reduce_or_sync(0xffffffffu, o);
    nz = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(nz)));
    if (lane == 0) {
      xs[64 + w] = static_cast<int>(a);
      xs[64 + NW + w] = static_cast<int>(o);
    }
    const int nz_all = cta_sum(nz, nullptr);   // its barrier also publishes a and o
    uint32_t all_and = 0xffffffffu, all_or = 0u;
#pragma unroll
    for (int u = 0; u < NW; ++u) {
      all_and &= static_cast<uint32_t>(xs[64 + u]);
      all_or |= static_cast<uint32_t>(xs[64 + NW + u]);
    }
    const uint32_t diff = all_and ^ all_or;
    const int top = diff == 0u ? 0 : 32 - __clz(diff);
    uint32_t t = top == 32 ? 0u : (all_and & (0xffffffffu << top));
    int cnt_t = nz_all;
#pragma unroll 1
    for (int b = top - 1; b >= 0 && cnt_t != m; --b) {
      const uint32_t cand = t | (1u << b);
      int c0 = 0, c1 = 0;
#pragma unroll
      for (int i = 0; i + 1 < KPL; i += 2) {
        c0 += key[i] >= cand ? 1 : 0;
        c1 += key[i + 1] >= cand ? 1 : 0;
      }
      const int cw = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(c0 + c1)));
      const int c = cta_sum(cw, nullptr);
      if (c >= m) {
        t = cand;
        cnt_t = c;
      }
    }
    Bar::sync();   // xs[64 ..] is rewritten by the next search
    exact = cnt_t == m;
    return t;
  };
  if (threadIdx.x == 0) {
    out[m] = nb - 1;
    if (out_user != nullptr) out_user[m] = nb - 1;
  }
  if (m == 0) return true;
  bool exact;
  const uint32_t t = threshold(exact);
  const Window win = make_window(t, E);
  uint32_t *bal = ss.bal + w * 2 * KPL;   // this warp's class ballots
  int n_in_w, n_amb_w;
  classify<KPL>(key, win, bal, n_in_w, n_amb_w, lane);
  int in_before;
  const int n_in = cta_sum(n_in_w, &in_before);
  int amb_before;
  const int n_amb = cta_sum(n_amb_w, &amb_before);
  const int r = m - n_in;
  if (n_amb == r || r == 0 || !win.refine) {
    // every ambiguous candidate kept, none, or a tie without a usable bound: the first r
    // in index order; this warp's kept ones follow the earlier warps'
    const int take_before = min(amb_before, r);
    emit_class(bal, KPL, nullptr, true, true, amb_before, in_before + take_before, m, jbase, out,
               lane, r);
    if (out_user != nullptr)
      emit_class(bal, KPL, nullptr, true, true, amb_before, in_before + take_before, m, jbase,
                 out_user, lane, r);
    return true;
  }
  if (n_amb > kAmbCapWarp) {
    // more ambiguous candidates than the list holds: warp 0 selects the row exactly,
    // re-reading it from L2
    if (w == 0) {
      warp_select_long<D>(srow, n, m, nb, E, rc, qg, G, ss, out, lane);
      __syncwarp();
      if (out_user != nullptr)
        for (int i = lane; i <= m; i += 32) out_user[i] = out[i];
    }
    return true;
  }
  emit_in_and_list<KPL>(key, bal, in_before, amb_before, jbase, out, lst, kAmbCapWarp, lane);
  // the certain ones in place: release them; the ambiguous ones listed: every warp
  // re-scores KIN_RK_ROWS of them at a time (one memory latency after the page lookup),
  // warp 0 chooses r and appends them, every warp merges its part of the caller's
  // ascending copy
  Bar::sync();
  if (threadIdx.x == 0) st_release_gpu(ready, n_in + 1);
  list_pages(lst, n_amb, rc.trow, n, rc.num_pages, ss.pg, threadIdx.x, NW * 32);
  Bar::sync();
  refine_keys<D>(lst, ss.pg, n_amb, KIN_RK_ROWS * w, KIN_RK_ROWS * NW, rc.c2, rc.stride, ss.qs, lane);
  Bar::sync();
  if (w == 0) {
    const uint32_t *lr = reinterpret_cast<const uint32_t *>(lst) + 1;
    if (n_amb <= 64)
      choose_amb<2, 2>(lr, n_amb, r, ss.lf, lane);
    else
      choose_amb<kAmbCapWarp / 32, 2>(lr, n_amb, r, ss.lf, lane);
    __syncwarp();
    append_chosen(lst, ss.lf, n_amb, r, out + n_in, lane);
  }
  Bar::sync();
  if (out_user != nullptr) {
    int cb = 0;   // chosen among the ambiguous candidates of the warps before this one
    for (int e = lane; e < amb_before; e += 32) cb += ss.lf[e] != 0 ? 1 : 0;
    cb = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(cb)));
    emit_class(bal, KPL, ss.lf, true, true, amb_before, in_before + cb, m, jbase, out_user, lane);
  }
  return true;
}

// Kept blocks of one row by one warp for rows too long for the registers: radix select
// (8-bit digits, shared histogram) that re-reads the row from L2 on every pass, first on
// the first-code keys (for the window), then on the modified keys, whose ambiguous
// candidates are re-scored wherever a pass meets them.
template <int D>
__device__ void warp_select_long(const float *srow, int n, int m, int nb, float E,
                                 const RefineCtx &rc, const __nv_bfloat16 *qg, int G,
                                 const SelScratch &ss, int32_t *out, int lane) {
  int *hist = ss.hist;
  // m-th largest key of key_at(0 .. n) (keys >= 1 where counted) and how many keys equal
  // to it are kept
  auto radix = [&](auto key_at, uint32_t &thr, int &take_eq) {
    uint32_t prefix = 0u, mask = 0u;
    int remaining = m;               // keys still to take at or below the current prefix
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = lane; i < 256; i += 32) hist[i] = 0;
      __syncwarp();
      for (int j = lane; j < n; j += 32) {
        const uint32_t key = key_at(j);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncwarp();
      int c[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[lane * 8 + i];
        tot += c[i];
      }
      int incl = tot;                // keys in this lane's digits and all higher ones
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      const int above_lane = incl - tot;
      const bool mine = above_lane < remaining && remaining <= incl;
      int digit = 0, above = 0;
      if (mine) {
        int run = above_lane;
        for (int i = 7; i >= 0; --i) {
          if (run + c[i] >= remaining) {
            digit = lane * 8 + i;
            above = run;
            break;
          }
          run += c[i];
        }
      }
      const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
      digit = __shfl_sync(0xffffffffu, digit, src);
      above = __shfl_sync(0xffffffffu, above, src);
      remaining -= above;
      prefix |= static_cast<uint32_t>(digit) << shift;
      mask |= 255u << shift;
      __syncwarp();
    }
    thr = prefix;
    take_eq = remaining;
  };
  auto first_key = [&](int j) -> uint32_t { return max(score_key(__ldcg(srow + j)), 2u); };
  if (m > 0) {
    uint32_t t;
    int take_eq;
    radix(first_key, t, take_eq);
    const Window w = make_window(t, E);
    int n_in = 0, n_amb = 0;
    for (int j = lane; j < n; j += 32) {
      const uint32_t k = first_key(j);
      n_in += k > w.hi ? 1 : 0;
      n_amb += (k >= w.lo && k <= w.hi) ? 1 : 0;
    }
    n_in = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(n_in)));
    n_amb = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(n_amb)));
    if (w.refine && n_amb != m - n_in) group_query<D>(qg, G, const_cast<float *>(rc.qs), lane);
    __syncwarp();
    const bool every_amb = n_amb == m - n_in;
    auto mod_key = [&](int j) -> uint32_t {
      const float s = __ldcg(srow + j);
      const uint32_t k = max(score_key(s), 2u);
      if (k > w.hi) return kKeyIn;
      if (k < w.lo) return 0u;
      if (every_amb) return kKeyIn;
      return w.refine ? refined_key<D, 1>(rc, j, s, lane) : 2u;
    };
    radix(mod_key, t, take_eq);
    const unsigned lt = (1u << lane) - 1u;
    int written = 0, eq_seen = 0;
    for (int base = 0; base < n; base += 32) {
      const int j = base + lane;
      const uint32_t key = j < n ? mod_key(j) : 0u;
      const bool gt = j < n && key > t;
      const bool eq = j < n && key == t;
      const unsigned eqm = __ballot_sync(0xffffffffu, eq);
      const bool keep = gt || (eq && eq_seen + __popc(eqm & lt) < take_eq);
      const unsigned km = __ballot_sync(0xffffffffu, keep);
      const int pos = written + __popc(km & lt);
      if (keep && pos < m) out[pos] = j;
      written += __popc(km);
      eq_seen += __popc(eqm);
    }
  }
  if (lane == 0) out[m] = nb - 1;
}

// The kept list of a row whose selection could not run (its scores never arrived): the
// first m candidates and the final block, so that the attention reads valid pages.  Only
// written after a timeout, which the error flag reports.
__device__ __forceinline__ void fallback_kept(int m, int nb, int32_t *out, int ti, int nthr) {
  for (int i = ti; i <= m; i += nthr) out[i] = i < m ? i : nb - 1;
}

// ----------------------------------------------------------------------------------
// Producer warps.  One thread issues one page's copies every few hundred cycles (barrier
// wait, byte-count arrival, TMA issue), so kProducers warps share the work: producer q
// stages the pages (attention) or ring stages (scores) i = q, q + kProducers, ... of every
// item, which consumer warp q then processes.  Producer 0 also runs the work queue: it
// turns items into descriptors.  In each warp lane 0 does the barrier and copy work and
// the other lanes help read block tables and kept lists.
// ----------------------------------------------------------------------------------

// Work queue order.  Round r (0 <= r < batch + lag_attn) holds, in this order, the score
// items of sequence r, the select items of sequence r - lag_select and the attention items
// of sequence r - lag_attn, each part only when that sequence exists.  Every item still
// comes after everything it waits for (lag_attn >= lag_select >= 0), so a CTA that takes items in queue order
// never waits on an item that no CTA has taken; the lags let the score streaming of later
// sequences overlap the attention of earlier ones.
enum : int { kItemScore = 0, kItemSelect = 1, kItemAttn = 2 };
struct QueueItem {
  int kind;    // kItem*
  int local;   // index among the items of its kind, in sequence-major order
};

__device__ __forceinline__ int queue_before(const FusedParams &p, int r) {   // items in rounds < r
  const int B = p.batch;
  const int s_per = p.n_score_items / B, sel_per = p.n_select_items / B;
  const int a_per = p.n_attn_items / B;
  return s_per * min(max(r, 0), B) + sel_per * min(max(r - p.lag_select, 0), B) +
         a_per * min(max(r - p.lag_attn, 0), B);
}

__device__ QueueItem queue_item(const FusedParams &p, int i) {
  const int B = p.batch;
  const int s_per = p.n_score_items / B, sel_per = p.n_select_items / B;
  const int a_per = p.n_attn_items / B;
  int lo = 0, hi = B + p.lag_attn;   // the last round r in [lo, hi) with queue_before(r) <= i
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (queue_before(p, mid) <= i) lo = mid; else hi = mid;
  }
  int off = i - queue_before(p, lo);
  if (lo < B) {
    if (off < s_per) return QueueItem{kItemScore, lo * s_per + off};
    off -= s_per;
  }
  const int ss = lo - p.lag_select;
  if (ss >= 0 && ss < B) {
    if (off < sel_per) return QueueItem{kItemSelect, ss * sel_per + off};
    off -= sel_per;
  }
  return QueueItem{kItemAttn, (lo - p.lag_attn) * a_per + off};
}

// The descriptor of work item `qi`; false when the item has nothing to do (an empty chunk or split, a row kept whole).
template <int D>
__device__ bool make_desc(const FusedParams &p, QueueItem qi, Desc &d) {
  const int H = p.num_kv_heads, HS = p.heads_per_range;
  const int item = qi.local;
  if (qi.kind == kItemScore) {
    const int per_seq = p.head_ranges * p.chunks_per_seq;
    const int b = item / per_seq, r = item % per_seq;
    const int hr = r / p.chunks_per_seq, chunk = r % p.chunks_per_seq;
    const int L = __ldg(p.seq_lens + b);
    if (L < 1 || L > kBlock * p.max_blocks) return false;     // flagged by attention
    const int nb = (L + kBlock - 1) / kBlock;
    if (nb <= p.top_k) return false;                            // every block kept
    const int j0 = chunk * p.score_chunk;
    if (j0 >= nb - 1) return false;
    const int npg = min(nb - 1, j0 + p.score_chunk) - j0;
    const int h0 = hr * HS, hs = min(HS, H - h0);
    const int pps = BfTile<D>::kStageBytes / (hs * D * 2);    // pages per stage
    d = Desc{kDescScore, 0, (npg + pps - 1) / pps, b, h0, j0, hs, L};
    return true;
  }
  if (qi.kind == kItemSelect) {
    const int it = item;
    const int per_seq = p.coop_select ? H : p.head_ranges;
    const int b = it / per_seq, r = it % per_seq;
    const int L = __ldg(p.seq_lens + b);
    if (L < 1 || L > kBlock * p.max_blocks) return false;
    const int nb = (L + kBlock - 1) / kBlock;
    if (nb <= p.top_k) return false;
    if (p.coop_select) {   // one row (head r), all consumer warps; first = 1 marks it
      d = Desc{kDescSelect, 1, 0, b, r, nb - 1, 1, L};
    } else {               // head range r, one warp per row
      const int h0 = r * HS;
      d = Desc{kDescSelect, 0, 0, b, h0, nb - 1, min(HS, H - h0), L};
    }
    return true;
  }
  const int a = item;
  const int row = a / p.splits_per_row, split = a % p.splits_per_row;
  const int L = __ldg(p.seq_lens + row / H);
  if (L < 1 || L > kBlock * p.max_blocks) {
    if (split != 0) return false;
    d = Desc{kDescEmptyRow, 0, 0, row, 0, 1, 0, L};
    return true;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  const bool every_block = p.top_k == 0 || nb <= p.top_k;
  const int n_items = p.top_k == 0 ? nb : min(nb, p.top_k);
  const int splits = (n_items + p.items_per_split - 1) / p.items_per_split;
  if (split >= splits) return false;
  const int cnt = min(n_items, (split + 1) * p.items_per_split) - split * p.items_per_split;
  const int flags = (every_block ? kAttnEveryBlock : 0) |
                    ((p.append_final != 0 && (L % kBlock) == 0 && split == splits - 1)
                         ? kAttnAppendLast : 0);
  d = Desc{kDescAttn, 0, cnt, row, split, splits, flags, L};
  return true;
}

template <int D, int NT>
__device__ void producer(const FusedParams &p, const CUtensorMap *kmap, const CUtensorMap *vmap,
                         uint8_t *ring, uint8_t *qstage, FusedShared &sh) {
  KIN_TRACE_DECL
  using R = Ring<D, NT>;
  using C = Cfg<D, NT>;
  const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) - C::kCW;
  const bool leader = q == 0;
  // Every copy streams (evict-first), except the pages of the leading blocks that all
  // sequences share (a Best-of-N prompt), which stay in L2 for the step's other readers.
  const uint64_t policy = l2_policy_evict_first();
  const uint64_t keep_policy = l2_policy_evict_last();
  const int shared_j = p.shared_prefix_blocks;
  const int H = p.num_kv_heads;
  const int total = p.n_score_items + p.n_select_items + p.n_attn_items;
  uint32_t pos[C::kPPC] = {};  // sub-ring position of each of the pipeline's consumers
  uint32_t nd = 0;            // descriptors read (and, by the leader, pushed)
  uint32_t nq = 0;            // leader: score items whose q rows it staged
  int sel_taken = 0;          // leader: select items taken (compared with sh.sel_done)
  int next = 0;
  if (leader && lane == 0) next = atomicAdd(p.work_next, 1);

  // Lane 0: claim the next stage of the sub-ring of consumer q + kProducers cc and post
  // what will land there.  The j-th page (score stage) of an item in this pipeline goes
  // to consumer cc = j % kPPC: a fixed function of the item, so that the partition of an
  // item's pages among warps, and with it every rounding, is the same on every call.
  auto claim = [&](int cc, int4 meta, uint32_t bytes) {
    const uint32_t n = pos[cc];
    const int s = R::slot(q + kProducers * cc, n);
    KIN_TIC(t0);
    wait_bar(&sh.empty[s], R::phase(n) ^ 1u, sh, p.err);
    KIN_TOC(kTrPWaitEmpty, t0);
    sh.meta[s] = meta;
    if (bytes != 0)
      mbar_arrive_expect_tx(&sh.full[s], bytes);
    else
      mbar_arrive(&sh.full[s]);
    return s;
  };

  KIN_TIC(t_start);
#pragma unroll 1
  while (true) {
    if (leader) {
      // Next item with work (END once the queue is exhausted), pushed as a descriptor.
      Desc d{kDescEnd, 0, 0, 0, 0, 0, 0, 0};
      KIN_TIC(t_next);
      while (true) {
        const int item = __shfl_sync(0xffffffffu, next, 0);
        if (item >= total) break;
        const QueueItem qi = queue_item(p, item);
        const bool is_select = qi.kind == kItemSelect;
        sel_taken += is_select ? 1 : 0;
        if (lane == 0) {
          // A CTA holds at most two unfinished select items: a run of selections queued
          // behind one another in one CTA would hold back every row they release.
          if (sel_taken >= 2) wait_shared_count(&sh.sel_done, sel_taken - 1, sh, p.err);
          next = atomicAdd(p.work_next, 1);   // prefetch the one after
        }
        const bool ok = make_desc<D>(p, qi, d);
        if (is_select && !ok) --sel_taken;   // a row kept whole: no descriptor, no selection
        if (ok) {
#ifdef KIN_TRACE_CYCLES
          d.item = item;
          if (lane == 0) {
            KIN_ITEM_STAMP(item, 0, blockIdx.x);
            KIN_ITEM_STAMP(item, 1, gtime());
          }
#endif
          break;
        }
      }
      KIN_TOC(kTrPNext, t_next);
      if (d.kind == kDescScore) {
        d.first = -1;
        if (NT == 1 && d.x2 <= 8) {   // q rows [b, h0 G .. (h0 + hs) G) are contiguous
          const int qslot = static_cast<int>(nq & 1u);
          d.first = qslot;
          if (lane == 0) {
            const uint32_t bytes = static_cast<uint32_t>(d.x2) * p.group * D * 2;
            wait_bar(&sh.qempty[qslot], ((nq >> 1) & 1u) ^ 1u, sh, p.err);
            mbar_arrive_expect_tx(&sh.qfull[qslot], bytes);
            bulk_load(qstage + qslot * kQSlotBytes,
                      p.q + (static_cast<int64_t>(d.row) * H * p.group + d.x0 * p.group) * D, bytes,
                      &sh.qfull[qslot], policy);
          }
          ++nq;
        }
      }
      if (lane == 0) {
        const int slot = nd % kDescs;
        KIN_TIC(t0);
        wait_bar(&sh.dempty[slot], ((nd / kDescs) & 1u) ^ 1u, sh, p.err, true);
        KIN_TOC(kTrPPush, t0);
        sh.desc[slot] = d;
        mbar_arrive(&sh.dfull[slot]);
      }
      __syncwarp();
    }
    const int slot = nd % kDescs;
    if (!wait_bar(&sh.dfull[slot], (nd / kDescs) & 1u, sh, p.err, true)) break;
    const Desc d = sh.desc[slot];
    ++nd;
    if (d.kind == kDescScore) {
      // Ring stages t = q, q + kProducers, ... of the chunk: pps pages' centroid rows each.
      const int b = d.row, h0 = d.x0, j0 = d.x1, hs = d.x2, L = d.x3;
      const int npg = min((L + kBlock - 1) / kBlock - 1, j0 + p.score_chunk) - j0;
      const int pps = R::kStageBytes / (hs * D * 2);
      const uint32_t row_bytes = static_cast<uint32_t>(hs) * D * 2;
      int *plist = sh.plist[q];
      const int32_t *trow = p.block_table + static_cast<int64_t>(b) * p.max_blocks + j0;
      KIN_TIC(t_meta);
      // All loads issued before any is used: one memory latency, not one per 32 pages.
      int pgs[kMaxScoreChunk / 32];
#pragma unroll
      for (int k = 0; k < kMaxScoreChunk / 32; ++k) {
        const int i = lane + 32 * k;
        pgs[k] = i < npg ? __ldg(trow + i) : -1;
      }
#pragma unroll
      for (int k = 0; k < kMaxScoreChunk / 32; ++k) {
        const int i = lane + 32 * k;
        if (i < npg) {
          int pg = pgs[k];
          if (pg < 0 || pg >= p.num_pages) {
            if (q == 0) flag_error(p.err, KIN_DEVERR_PAGE_ID);
            pg = -1;
          }
          plist[i] = pg;
        }
      }
      __syncwarp();
      KIN_TOC(kTrPMeta, t_meta);
      for (int t = q, j = 0; t < d.count; t += kProducers, ++j) {
        KIN_TIC(t_issue);
        const int cc = j % C::kPPC;
        const int pa = t * pps, pb = min(npg, pa + pps);
        const int pg = lane < pb - pa ? plist[pa + lane] : -1;
        const uint32_t vmask = __ballot_sync(0xffffffffu, pg >= 0);
        int s = 0;
        if (lane == 0)
          s = claim(cc, make_int4(j0 + pa, pb - pa, static_cast<int>(vmask), 0), __popc(vmask) * row_bytes);
        s = __shfl_sync(0xffffffffu, s, 0);
        ++pos[cc];
        if (pg >= 0)
          bulk_load(ring + s * R::kStageBytes + lane * row_bytes,
                    p.centroids + (static_cast<int64_t>(pg) * H + h0) * D, row_bytes, &sh.full[s],
                    j0 + pa + lane < shared_j ? keep_policy : policy);
        KIN_TOC(kTrPIssue, t_issue);
      }
    } else if (d.kind == kDescAttn) {
      // Pages i = q, q + kProducers, ... of the split: lane l reads page
      // i = base + l * kProducers, then the pages are staged in order.
      const int row = d.row, L = d.x3, cnt = d.count;
      const int b = row / H;
      const int nb = (L + kBlock - 1) / kBlock;
      const bool every_block = (d.x2 & kAttnEveryBlock) != 0;
      const int i0 = d.x0 * p.items_per_split;
      // entries [0, ready_v - 1) and the final block (entry top_k - 1) may be read once
      // the row's ready word is ready_v; all of them at kReadyAll
      int ready_v = kReadyAll;
      if (!every_block && q < cnt) {
        KIN_TIC(t0);
        if (lane == 0) ready_v = wait_flag_value(p.ready + row, 1, sh, p.err);
        ready_v = __shfl_sync(0xffffffffu, ready_v, 0);
        __syncwarp();   // the lanes read the kept list after lane 0's acquire
        KIN_TOC(kTrPReady, t0);
#ifdef KIN_TRACE_CYCLES
        if (lane == 0 && q == 0) KIN_ITEM_STAMP(d.item, 2, gtime());
#endif
      }
      const int32_t *srow = p.sel + static_cast<int64_t>(row) * p.top_k;
      const int32_t *trow = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
      const int32_t ybase = (row % H) * kBlock;
      for (int base = q; base < cnt; base += 32 * kProducers) {
        KIN_TIC(t_meta);
        if (ready_v < kReadyAll) {
          // this batch reads entries i0 + base .. i0 + base + 31 kProducers
          const int e_lo = i0 + base, e_hi = i0 + min(cnt - 1, base + 31 * kProducers);
          if (e_lo < p.top_k - 1 && e_hi >= ready_v - 1) {
            if (lane == 0) ready_v = wait_flag_value(p.ready + row, kReadyAll, sh, p.err);
            ready_v = __shfl_sync(0xffffffffu, ready_v, 0);
            __syncwarp();
          }
        }
        const int i = base + lane * kProducers;
        int page = -1, ntok = 0, jblk = -1;
        if (i < cnt) {
          const int j = every_block ? i0 + i : __ldcg(srow + i0 + i);
          jblk = j;
          if (j >= 0 && j < nb) {
            const int pg = __ldg(trow + j);
            if (pg >= 0 && pg < p.num_pages) {
              page = pg;
              ntok = min(kBlock, L - kBlock * j);
            } else {
              flag_error(p.err, KIN_DEVERR_PAGE_ID);
            }
          }
        }
        KIN_TOC(kTrPMeta, t_meta);
        const int n_here = min(32, (cnt - base + kProducers - 1) / kProducers);
        // L2 prefetch of the K and V tiles kPrefetchPages of this producer's pages ahead of
        // the copy into the ring: lane l holds page l of the batch.
        auto prefetch_page = [&]() {
          if (page < 0) return;
          const int32_t y = page * H * kBlock + ybase;
          if (D == 128) {
            tma_prefetch_3d(kmap, 0, y, 0);
            tma_prefetch_3d(vmap, 0, y, 0);
          } else {
            tma_prefetch_2d(kmap, 0, y);
            tma_prefetch_2d(vmap, 0, y);
          }
        };
        if (lane < kPrefetchPages) prefetch_page();
        for (int l = 0; l < n_here; ++l) {
          KIN_TIC(t_issue);
          if (lane == l + kPrefetchPages) prefetch_page();
          const int pg = __shfl_sync(0xffffffffu, page, l);
          const int nt = __shfl_sync(0xffffffffu, ntok, l);
          const int jb = __shfl_sync(0xffffffffu, jblk, l);
          const bool shared = jb >= 0 && jb < shared_j;
          int s = 0;
          const int cc = ((base - q) / kProducers + l) % C::kPPC;
          if (lane == 0) s = claim(cc, make_int4(pg, nt, 0, 0), pg >= 0 ? R::kStageBytes : 0u);
          s = __shfl_sync(0xffffffffu, s, 0);
          ++pos[cc];
          if (pg >= 0 && lane < 2) {   // lane 0: K, lane 1: V; one copy per page each
            uint8_t *dst = ring + s * R::kStageBytes + (lane ? BfTile<D>::kKBytes : 0);
            const CUtensorMap *map = lane ? vmap : kmap;
            const uint64_t pol = shared ? keep_policy : policy;
            if (D == 128)
              tma_load_3d(dst, map, 0, pg * H * kBlock + ybase, 0, &sh.full[s], pol);
            else
              tma_load_2d(dst, map, 0, pg * H * kBlock + ybase, &sh.full[s], pol);
          }
          KIN_TOC(kTrPIssue, t_issue);
          KIN_COUNT(kTrPPages, 1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.dempty[slot]);
    if (d.kind == kDescEnd) break;
    KIN_COUNT(kTrPItems, 1);
  }
  KIN_TOC(kTrTotal, t_start);
  KIN_TRACE_FLUSH;
  // Leave no copy in flight: wait (bounded) for the last use of each stage of the sub-rings
  // this warp fills.  Their consumers normally saw them all complete; this matters only
  // after a timeout.
  if (lane == 0) {
    for (int cc = 0; cc < C::kPPC; ++cc) {
      const uint32_t n = pos[cc];
      for (uint32_t j = 0; j < static_cast<uint32_t>(R::kPer) && j < n; ++j) {
        const uint32_t last = j + ((n - 1 - j) / R::kPer) * R::kPer;
        if (!mbar_wait(&sh.full[R::slot(q + kProducers * cc, last)], R::phase(last))) {
          flag_error(p.err, KIN_DEVERR_TIMEOUT);
          break;
        }
      }
    }
  }
  __syncwarp();
}

// ----------------------------------------------------------------------------------
// Consumer warps (threads 0 .. 32 kCW - 1; Cfg::Bar syncs exactly them).  Consumer warp w
// belongs to pipeline q = w % kProducers as its c = w / kProducers-th consumer: of the
// pipeline's pages (score stages) j = 0, 1, ... of an item it takes those with
// j % kPPC == c, and finds them at its own sub-ring position n.
// ----------------------------------------------------------------------------------
// Score of the centroids of one ring stage ([pages][hs heads][d], at most 32 centroids):
// lane l owns dimensions [l * kPer, l * kPer + kPer) of every centroid (conflict-free
// shared reads), and a butterfly over the 32 partial sums leaves centroid c's score in
// lane c.  QS > 0: the range has QS heads and the lane's slice of the group-summed queries
// sits in registers (qr[h][i], loaded once per item); QS = 0: any number of heads, the
// queries are read from shared memory (qs[h * D + dim]) for each centroid.  Loads are
// unconditional (stale shared memory is harmless), so the unrolled loop issues them back
// to back; invalid centroids are masked after the products.
template <int D>
struct QRegs {
  float v[8][D / 32];
};

template <int D, int QS>
__device__ __forceinline__ float stage_scores(const uint8_t *stage, const QRegs<D> &qr,
                                              const float *qs, int hs, int nc, uint32_t vmask,
                                              int lane, float &hb) {
  constexpr int kPer = D / 32;
  const uint8_t *own = stage + lane * (D * 2);   // centroid `lane`'s row of the stage
  const float *qown = qs + (lane % hs) * D;       // the group-summed query of its head
  stage += lane * kPer * 2;
  qs += lane * kPer;
  auto unpack = [&](int cc, float (&f)[kPer]) {
    if constexpr (kPer == 4) {
      const uint2 raw = *reinterpret_cast<const uint2 *>(stage + cc * (D * 2));
      f[0] = bf16_lo(raw.x); f[1] = bf16_hi(raw.x); f[2] = bf16_lo(raw.y); f[3] = bf16_hi(raw.y);
    } else {
      const uint32_t raw = *reinterpret_cast<const uint32_t *>(stage + cc * (D * 2));
      f[0] = bf16_lo(raw); f[1] = bf16_hi(raw);
    }
  };
  // bit cc: centroid cc of the stage is scored (present and its page valid)
  uint32_t vm = 0u;
  {
    int hh = 0, pi = 0;
#pragma unroll
    for (int cc = 0; cc < 32; ++cc) {
      const int page = QS > 0 ? cc / QS : pi;
      vm |= static_cast<uint32_t>(cc < nc && ((vmask >> page) & 1u)) << cc;
      if constexpr (QS == 0) {
        if (++hh == hs) {
          hh = 0;
          ++pi;
        }
      }
    }
  }
  auto valid = [&](int cc) { return ((vm >> cc) & 1u) != 0; };
  // 32 partial sums, one per centroid, reduced so that lane c ends with centroid c's sum
  auto butterfly = [&](float (&v)[32]) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int k = 0; k < o; ++k) {
        const float send = upper ? v[k] : v[k + o];
        const float keep = upper ? v[k + o] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    return v[0];
  };
  float v[32];
  int hh = 0;
#pragma unroll
  for (int cc = 0; cc < 32; ++cc) {
    float f[kPer], qv[kPer];
    unpack(cc, f);
    if constexpr (QS > 0) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) qv[i] = qr.v[cc % QS][i];
    } else if constexpr (kPer == 4) {
      const float4 q4 = *reinterpret_cast<const float4 *>(qs + hh * D);
      qv[0] = q4.x; qv[1] = q4.y; qv[2] = q4.z; qv[3] = q4.w;
    } else {
      const float2 q2 = *reinterpret_cast<const float2 *>(qs + hh * D);
      qv[0] = q2.x; qv[1] = q2.y;
    }
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc = fmaf(qv[i], f[i], acc);
    v[cc] = valid(cc) ? acc : 0.f;
    if constexpr (QS == 0) {
      if (++hh == hs) hh = 0;
    }
  }
  const float score = butterfly(v);
  // lane c: sum_i |qs_i| |c1_i| of centroid c (row_bound) from its own row, 16-byte
  // chunks in an order rotated by the lane (rows are 2 D bytes apart, so 8 consecutive
  // lanes read 8 distinct bank groups)
  float acc_b = 0.f;
  if (valid(lane)) {
#pragma unroll 4
    for (int c = 0; c < D / 8; ++c) {
      const int cr = (c + lane) & (D / 8 - 1);
      float f[8];
      Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4 *>(own + cr * 16), f);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc_b = fmaf(fabsf(qown[8 * cr + k]), fabsf(f[k]), acc_b);
    }
  }
  hb = acc_b;
  return score;
}

// Score of the centroids of one ring stage for ranges of exactly 8 heads: four lanes per
// centroid.  Lane l serves head l / 4 of every page of the stage and dimensions
// [(l % 4) D / 4, (l % 4 + 1) D / 4) of it, so its slice of the group-summed query (D / 4
// values, qv) stays in registers for the whole item; a page is 4 x 16-byte reads, D / 4
// products and a two-step shuffle sum per lane.  The lane reads its 16-byte chunks in a
// rotated order (chunk c at position (c + rot) mod D / 32) so that every 8-lane phase of a
// read touches 8 distinct bank groups; qv is stored in the same order.  Returns nothing:
// lanes l % 4 == 0 store the scores of head l / 4.
template <int D>
struct QSlice {
  float v[D / 4];
};

template <int D>
__device__ __forceinline__ int h8_rot(int lane) {
  return D == 128 ? (lane >> 1) & 3 : (lane >> 2) & 1;
}

template <int D>
__device__ __forceinline__ void load_qslice(const float *qs, int lane, QSlice<D> &qv) {
  constexpr int kCh = D / 32;   // 16-byte chunks (8 dims) per lane
  const int head = lane >> 2, part = lane & 3, rot = h8_rot<D>(lane);
  const float *src = qs + head * D + part * (D / 4);
#pragma unroll
  for (int c = 0; c < kCh; ++c) {
    const float *cp = src + ((c + rot) & (kCh - 1)) * 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) qv.v[c * 8 + k] = cp[k];
  }
}

template <int D>
__device__ __forceinline__ void stage_scores_h8(const uint8_t *stage, const QSlice<D> &qv, int np,
                                                uint32_t vmask, float *srow_base, int64_t sstride,
                                                int jst, int lane, float &hb_max) {
  constexpr int kCh = D / 32;
  const int head = lane >> 2, part = lane & 3, rot = h8_rot<D>(lane);
  const uint8_t *base = stage + head * (D * 2) + part * (D / 4) * 2;
  float acc[4], nrm[4];
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {   // pages of the stage (loads unconditional)
    const uint8_t *row = base + pp * 8 * (D * 2);
    float a0 = 0.f, a1 = 0.f, n0 = 0.f, n1 = 0.f;
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(row + ((c + rot) & (kCh - 1)) * 16);
      float f[8];
      f[0] = bf16_lo(raw.x); f[1] = bf16_hi(raw.x); f[2] = bf16_lo(raw.y); f[3] = bf16_hi(raw.y);
      f[4] = bf16_lo(raw.z); f[5] = bf16_hi(raw.z); f[6] = bf16_lo(raw.w); f[7] = bf16_hi(raw.w);
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        a0 = fmaf(qv.v[c * 8 + k], f[k], a0);
        a1 = fmaf(qv.v[c * 8 + k + 1], f[k + 1], a1);
        n0 = fmaf(fabsf(qv.v[c * 8 + k]), fabsf(f[k]), n0);
        n1 = fmaf(fabsf(qv.v[c * 8 + k + 1]), fabsf(f[k + 1]), n1);
      }
    }
    acc[pp] = a0 + a1;
    nrm[pp] = n0 + n1;
  }
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {
    acc[pp] += __shfl_xor_sync(0xffffffffu, acc[pp], 1);
    acc[pp] += __shfl_xor_sync(0xffffffffu, acc[pp], 2);
    nrm[pp] += __shfl_xor_sync(0xffffffffu, nrm[pp], 1);
    nrm[pp] += __shfl_xor_sync(0xffffffffu, nrm[pp], 2);
  }
  if (part == 0) {
    float *dst = srow_base + head * sstride + jst;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const bool valid = pp < np && ((vmask >> pp) & 1u);
      if (pp < np) __stcg(dst + pp, valid ? acc[pp] : -INFINITY);
      if (valid) hb_max = fmaxf(hb_max, nrm[pp]);
    }
  }
}

// Upper bound of |s - s*| for every candidate of a row, where s is the group score the
// kernel computes from the first centroid code c1 (bf16) and s* the exact score of the
// fp32 mean c.  c1_i is c_i rounded to nearest with 8 significant bits, so for a normal
// c1_i in [2^e, 2^(e+1)] the error |c_i - c1_i| is at most half a unit in the last place
// of c_i's binade, <= 2^(e-8) <= 2^-8 |c1_i|; hence |s - s*| <= 2^-8 hb with
// hb = sum_i |qs_i| |c1_i|, which the score stage sums per centroid (one multiply-add per
// element, the absolute values being operand modifiers).  fp32 rounding of the score's
// products and sums, of hb and of qs itself stays below 2^-15 hb for d <= 128 and G <= 16.
// kBoundScale = 2^-8 + 2^-12 covers both.  A zero or subnormal c1_i is off by at most
// 2^-134, which the 1e-30 |qs|_1 term covers.  (Summing 2^e instead of |c1_i| gives a
// bound up to half as large, but costs a mask per element: measured slower.)
constexpr float kBoundScale = 0.00415039062f;   // 2^-8 + 2^-12, exact in fp32
__device__ __forceinline__ float row_bound(float qn1, float hb) {
  return kBoundScale * hb + 1e-30f * qn1;
}

// The warp's ring stages of one score item (stages t = q, q + kProducers, ... of the item,
// those with j % kPPC == c): wait for each, score its centroids, store them, free it.  Also
// raises each row's error bound (p.bound) to cover the centroids this warp scored.
template <int D, int NT, int QS>
__device__ __forceinline__ void score_stages(const FusedParams &p, const Desc &d, uint8_t *ring,
                                             const float *qs, FusedShared &sh, uint32_t &n
                                             KIN_TRACE_PARAM) {
  using R = Ring<D, NT>;
  using C = Cfg<D, NT>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q = warp % kProducers, c = warp / kProducers;
  const int H = p.num_kv_heads;
  const int b = d.row, h0 = d.x0, hs = d.x2;
  QRegs<D> qr;
  QSlice<D> qv;
  float qn1 = 0.f;           // |qs|_1 of the lane's head
  float hbm = -1.f;          // largest hb (row_bound) of the centroids the lane scored (-1: none)
  int head;                  // the lane's head within the range
  if constexpr (QS == 8) {
    load_qslice<D>(qs, lane, qv);
#pragma unroll
    for (int i = 0; i < D / 4; ++i) qn1 += fabsf(qv.v[i]);
    qn1 += __shfl_xor_sync(0xffffffffu, qn1, 1);
    qn1 += __shfl_xor_sync(0xffffffffu, qn1, 2);
    head = lane >> 2;
  } else {
    if constexpr (QS > 0) {
#pragma unroll
      for (int hh = 0; hh < QS; ++hh)
#pragma unroll
        for (int i = 0; i < D / 32; ++i) qr.v[hh][i] = qs[hh * D + lane * (D / 32) + i];
    }
    head = lane % hs;
    for (int i = 0; i < D; ++i) qn1 += fabsf(qs[head * D + i]);
  }
  for (int t = q, j = 0; t < d.count; t += kProducers, ++j) {
    if (j % C::kPPC != c) continue;
    const int s = R::slot(warp, n);
    KIN_TIC(t_w);
    const bool ok = wait_bar(&sh.full[s], R::phase(n), sh, p.err);
    ++n;
    KIN_TOC(kTrCScoreWait, t_w);
    KIN_TIC(t_sc);
    const int4 meta = sh.meta[s];
    const int jst = meta.x, np = meta.y;
    const uint32_t vmask = static_cast<uint32_t>(meta.z);
    const int nc = ok ? np * hs : 0;
    if constexpr (QS == 8) {
      stage_scores_h8<D>(ring + s * R::kStageBytes, qv, ok ? np : 0, vmask,
                         p.scores + static_cast<int64_t>(b * H + h0) * p.max_blocks, p.max_blocks,
                         jst, lane, hbm);
    } else {
      float hb;
      const float score = stage_scores<D, QS>(ring + s * R::kStageBytes, qr, qs, hs, nc, vmask, lane, hb);
      if (lane < nc) {
        const int pl = lane / hs, hl = lane % hs;
        const bool valid = ((vmask >> pl) & 1u) != 0;
        __stcg(p.scores + static_cast<int64_t>(b * H + h0 + hl) * p.max_blocks + jst + pl,
               valid ? score : -INFINITY);
        if (valid) hbm = fmaxf(hbm, hb);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
    KIN_TOC(kTrCScoreComp, t_sc);
  }
  // bounds are non-negative, so their fp32 bit patterns order like the values
  if (hbm >= 0.f) atomicMax(p.bound + b * H + h0 + head, __float_as_uint(row_bound(qn1, hbm)));
}

template <int D, int NT>
__device__ void consume_score(const FusedParams &p, const Desc &d, uint8_t *ring, float *qsum,
                              const uint8_t *qstage, FusedShared &sh, uint32_t &n, uint32_t &nqs,
                              uint32_t &nsc KIN_TRACE_PARAM) {
  using R = Ring<D, NT>;
  using C = Cfg<D, NT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.num_kv_heads, G = p.group;
  const int b = d.row, h0 = d.x0, hs = d.x2;
  // Group-summed queries of the range's heads (fp32, summed over g in order).  With up to
  // 8 heads each warp builds its own copy in its slice of the scratch and needs no CTA
  // barrier; with more, the consumer warps build one shared copy.
  const bool private_q = hs <= 8;
  float *qs = private_q ? qsum + warp * 8 * D : qsum;
  KIN_TIC(t_q);
  if (d.first >= 0) {
    // q rows staged in shared memory: each warp sums its own copy, then frees the slot.
    const int qslot = d.first;
    const bool ok = wait_bar(&sh.qfull[qslot], (nqs >> 1) & 1u, sh, p.err);
    ++nqs;
    const __nv_bfloat16 *qraw = reinterpret_cast<const __nv_bfloat16 *>(qstage + qslot * kQSlotBytes);
    for (int x = lane; x < hs * (D / 8); x += 32) {
      const int hh = x / (D / 8), c8 = (x % (D / 8)) * 8;
      float acc[8], f[8];
      Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4 *>(qraw + (hh * G) * D + c8), acc);
      for (int g = 1; g < G; ++g) {
        Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4 *>(qraw + (hh * G + g) * D + c8), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += f[i];
      }
      float4 *dst = reinterpret_cast<float4 *>(qs + hh * D + c8);
      dst[0] = ok ? make_float4(acc[0], acc[1], acc[2], acc[3]) : make_float4(0.f, 0.f, 0.f, 0.f);
      dst[1] = ok ? make_float4(acc[4], acc[5], acc[6], acc[7]) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.qempty[qslot]);
  } else {
    // q from global memory: the consumer warps build one shared copy.
    for (int x = tid; x < hs * (D / 8); x += C::kCThreads) {
      const int hh = x / (D / 8), c8 = (x % (D / 8)) * 8;
      const __nv_bfloat16 *qp = p.q + (static_cast<int64_t>(b) * H * G + (h0 + hh) * G) * D + c8;
      float acc[8], f[8];
      Elem<__nv_bfloat16>::unpack(__ldg(reinterpret_cast<const uint4 *>(qp)), acc);
      for (int g = 1; g < G; ++g) {
        Elem<__nv_bfloat16>::unpack(__ldg(reinterpret_cast<const uint4 *>(qp + g * D)), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += f[i];
      }
      float4 *dst = reinterpret_cast<float4 *>(qsum + hh * D + c8);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    C::Bar::sync();
    qs = qsum;
  }
  KIN_TOC(kTrCScoreQ, t_q);
  // The warp's stages of the item, with the queries in registers for ranges of up to 8
  // heads (the lane's slice: hs x D / 32 values).
  switch (hs) {
    case 8: score_stages<D, NT, 8>(p, d, ring, qs, sh, n KIN_TRACE_ARG); break;
    case 4: score_stages<D, NT, 4>(p, d, ring, qs, sh, n KIN_TRACE_ARG); break;
    case 2: score_stages<D, NT, 2>(p, d, ring, qs, sh, n KIN_TRACE_ARG); break;
    case 1: score_stages<D, NT, 1>(p, d, ring, qs, sh, n KIN_TRACE_ARG); break;
    default: score_stages<D, NT, 0>(p, d, ring, qs, sh, n KIN_TRACE_ARG); break;
  }
  // Publish the item: every consumer warp counts itself in at CTA scope (release /
  // acquire), and the last one publishes all warps' scores at GPU scope (its fence is
  // cumulative), so one warp per item pays the fence and none waits for the others.
  // Counters are reused every kScoreSlots score items; the descriptor ring keeps the
  // warps of a CTA fewer than kDescs items apart, so a counter is back to zero first.
  __syncwarp();
  if (lane == 0) {
    int32_t *cnt = &sh.score_arrive[nsc % kScoreSlots];
    if (atom_add_acq_rel_cta_shared(cnt, 1) == C::kCW - 1) {
      *cnt = 0;
      fence_acq_rel_gpu();
      red_add_relaxed_gpu(p.score_cnt + b * p.head_ranges + h0 / p.heads_per_range, 1);
    }
  }
  ++nsc;
  if (d.first < 0) C::Bar::sync();   // the shared group-summed queries are reused next item
}

// Selection scratch: per selecting warp (one warp per row) kSelWarpBytes of the consumer
// scratch; a cooperative selection uses the start of it for the whole CTA.
constexpr int kSelWarpBytes = 4096;
static_assert(8 * kSelWarpBytes <= kScratchBytes, "per-warp selection scratch");
static_assert(kSelWarpBytes % 16 == 0, "aligned per-warp regions");

template <int D>
__device__ __forceinline__ SelScratch sel_scratch(uint8_t *base, bool coop) {
  SelScratch ss;
  ss.xs = reinterpret_cast<int *>(base);                          // 128 ints
  ss.qs = reinterpret_cast<float *>(base + 512);                  // D floats
  ss.hist = reinterpret_cast<int *>(base + 512 + D * 4);          // 256 ints
  // class ballots: one warp: 2 x 64 slots in the xs area (a one-warp selection uses no
  // cross-warp sums); cooperative: 8 warps x 2 x 16 slots after the histogram
  ss.bal = coop ? reinterpret_cast<uint32_t *>(base + 512 + D * 4 + 1024)
                : reinterpret_cast<uint32_t *>(base);
  // ambiguous candidates of the row: one warp: the list after the histogram, pages and
  // then chosen flags in the histogram area (each dead by the time the next is written);
  // cooperative: each after the class ballots
  ss.lst = reinterpret_cast<int2 *>(base + (coop ? 4096 : 2048));
  ss.pg = coop ? reinterpret_cast<int *>(base + 6144) : ss.hist;
  ss.lf = coop ? base + 7168 : reinterpret_cast<uint8_t *>(ss.hist);
  return ss;
}
static_assert(512 + 128 * 4 + 1024 <= 2048 && 2048 + kAmbCapWarp * 8 <= kSelWarpBytes,
              "per-warp ambiguous list");
static_assert(512 + 128 * 4 + 1024 + 8 * 2 * 16 * 4 <= 4096 && 7168 + kAmbCapWarp <= kScratchBytes,
              "cooperative ambiguous list");
static_assert(512 + 128 * 4 + 1024 <= kSelWarpBytes, "per-warp selection scratch");
static_assert(2 * 64 * 4 <= 512, "per-warp class ballots in the xs area");
static_assert(512 + 128 * 4 + 1024 + 8 * 2 * 16 * 4 <= kScratchBytes, "cooperative selection scratch");

template <int D, int NT>
__device__ void consume_select(const FusedParams &p, const Desc &d, uint8_t *scratch,
                               FusedShared &sh KIN_TRACE_PARAM) {
  using C = Cfg<D, NT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.num_kv_heads, G = p.group;
  const int b = d.row, h0 = d.x0, n = d.x1, hs = d.x2;
  const int nb = n + 1;
  const int m = p.top_k - 1;
  const int32_t *trow = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
  KIN_TIC(t_sw);
  if (tid == 0) {
    // Wait until every score item (chunk) of this (sequence, head range) has published.
    const int32_t *cnt = p.score_cnt + b * p.head_ranges + h0 / p.heads_per_range;
    const int expected = (n + p.score_chunk - 1) / p.score_chunk;
    sh.sel_ok = wait_flag(cnt, expected, sh, p.err) ? 1 : 0;
  }
  C::Bar::sync();
  const bool ok = *reinterpret_cast<volatile int *>(&sh.sel_ok) != 0;
  KIN_TOC(kTrCSelWait, t_sw);
  if (d.first == 1) {   // one row, all consumer warps
    KIN_TIC(t_sel);
    constexpr int NW = C::kCW;
    const int row = b * H + h0;
    const float *srow = p.scores + static_cast<int64_t>(row) * p.max_blocks;
    int32_t *out = p.sel + static_cast<int64_t>(row) * p.top_k;
    int32_t *out_user = p.sel_out == nullptr ? nullptr : p.sel_out + static_cast<int64_t>(row) * p.top_k;
    const SelScratch ss = sel_scratch<D>(scratch, true);
    const float E = __uint_as_float(__ldcg(p.bound + row));
    const RefineCtx rc{p.cent_lo + h0 * D, trow, static_cast<int64_t>(H) * D, p.num_pages, ss.qs};
    const __nv_bfloat16 *qg = p.q + (static_cast<int64_t>(b) * H * G + h0 * G) * D;
    using Bar = typename C::Bar;
    int32_t *ready = p.ready + row;
    int2 *lst = ss.lst;
    bool complete = true;
    if (!ok) {
      fallback_kept(m, nb, out, tid, C::kCThreads);
      if (out_user != nullptr) fallback_kept(m, nb, out_user, tid, C::kCThreads);
    } else if (n <= NW * 32 * 2) {
      complete = cta_select_row<2, NW, D, Bar>(srow, n, m, nb, E, rc, qg, G, ss, out, out_user, ready, lst);
    } else if (n <= NW * 32 * 4) {
      complete = cta_select_row<4, NW, D, Bar>(srow, n, m, nb, E, rc, qg, G, ss, out, out_user, ready, lst);
    } else if (n <= NW * 32 * 8) {
      complete = cta_select_row<8, NW, D, Bar>(srow, n, m, nb, E, rc, qg, G, ss, out, out_user, ready, lst);
    } else if (n <= NW * 32 * 16) {
      complete = cta_select_row<16, NW, D, Bar>(srow, n, m, nb, E, rc, qg, G, ss, out, out_user, ready, lst);
    } else if (warp == 0) {   // longer rows: one warp, radix select over L2
      warp_select_long<D>(srow, n, m, nb, E, rc, qg, G, ss, out, lane);
      __syncwarp();
      if (out_user != nullptr)
        for (int i = lane; i <= m; i += 32) out_user[i] = out[i];
    }
    C::Bar::sync();
    if (tid == 0 && complete) st_release_gpu(ready, kReadyAll);
    KIN_TOC(kTrCSelComp, t_sel);
    C::Bar::sync();   // the scratch is reused by the next item
    if (tid == 0) *reinterpret_cast<volatile int *>(&sh.sel_done) += 1;
    return;
  }
  const SelScratch ss = sel_scratch<D>(scratch + warp * kSelWarpBytes, false);
  KIN_TIC(t_sel);
  for (int hh = warp; hh < hs; hh += C::kCW) {
    const int h = h0 + hh;
    const int row = b * H + h;
    const float *srow = p.scores + static_cast<int64_t>(row) * p.max_blocks;
    int32_t *out = p.sel + static_cast<int64_t>(row) * p.top_k;
    int32_t *out_user = p.sel_out == nullptr ? nullptr : p.sel_out + static_cast<int64_t>(row) * p.top_k;
    int32_t *ready = p.ready + row;
    const float E = __uint_as_float(__ldcg(p.bound + row));
    const RefineCtx rc{p.cent_lo + h * D, trow, static_cast<int64_t>(H) * D, p.num_pages, ss.qs};
    const __nv_bfloat16 *qg = p.q + (static_cast<int64_t>(b) * H * G + h * G) * D;
    int2 *lst = ss.lst;
    bool complete = true;
    if (!ok) {
      fallback_kept(m, nb, out, lane, 32);
      if (out_user != nullptr) fallback_kept(m, nb, out_user, lane, 32);
    } else if (n <= 32 * 16) {
      complete = warp_select_bits<16, D>(srow, n, m, nb, E, rc, qg, G, ss, out, out_user, ready, lst, lane KIN_TRACE_ARG);
    } else if (n <= 32 * 32) {
      complete = warp_select_bits<32, D>(srow, n, m, nb, E, rc, qg, G, ss, out, out_user, ready, lst, lane KIN_TRACE_ARG);
    } else if (n <= 32 * 64) {
      complete = warp_select_bits<64, D>(srow, n, m, nb, E, rc, qg, G, ss, out, out_user, ready, lst, lane KIN_TRACE_ARG);
    } else {
      warp_select_long<D>(srow, n, m, nb, E, rc, qg, G, ss, out, lane);
      __syncwarp();
      if (out_user != nullptr)
        for (int i = lane; i <= m; i += 32) out_user[i] = out[i];
    }
    __syncwarp();
    if (lane == 0 && complete) st_release_gpu(ready, kReadyAll);
    __syncwarp();
  }
  KIN_TOC(kTrCSelComp, t_sel);
  C::Bar::sync();   // the scratch is reused by the next item
  if (tid == 0) *reinterpret_cast<volatile int *>(&sh.sel_done) += 1;
}

template <int D, int NT>
__device__ void consume_attention(const FusedParams &p, const Desc &d, uint8_t *ring,
                                  uint8_t *scratch, FusedShared &sh,
                                  uint32_t &n KIN_TRACE_PARAM) {
  using R = Ring<D, NT>;
  using Tile = BfTile<D>;
  using C = Cfg<D, NT>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = warp % kProducers, c = warp / kProducers;
  const int H = p.num_kv_heads, G = p.group;
  const int row = d.row, split = d.x0, splits = d.x1, flags = d.x2, L = d.x3, cnt = d.count;
  const int b = row / H, h = row % H;
  const EmitCtx ec{p.out, p.lse, p.part_o, p.part_ml, p.attn_cnt, p.splits_per_row, G, H};
  if (p.top_k > 0 && p.sel_out != nullptr && (flags & kAttnEveryBlock) && split == 0) {
    // no selection ran for this row: its kept list is every block, -1 padded
    const int nb = (L + kBlock - 1) / kBlock;
    int32_t *srow = p.sel_out + static_cast<int64_t>(row) * p.top_k;
    for (int i = tid; i < p.top_k; i += C::kCThreads) srow[i] = i < nb ? i : -1;
  }
  KIN_TIC(t_q);
  uint32_t qb[D / 16][NT][2];
  load_qT_frags<D, NT>(qb, p.q + (static_cast<int64_t>(b) * H * G + h * G) * D, G, lane);
  KIN_TOC(kTrCQ, t_q);
  const float scale_log2 = p.sm_scale * kLog2e;
  const bool append = (flags & kAttnAppendLast) != 0;
  WarpSoftmaxT<D, NT> st;
  st.init();
  for (int i = q, j = 0; i < cnt; i += kProducers, ++j) {
    if (j % C::kPPC != c) continue;
    const int s = R::slot(warp, n);
    KIN_TIC(t_w);
    const bool ok = wait_bar(&sh.full[s], R::phase(n), sh, p.err);
    ++n;
    KIN_TOC(kTrCWaitFull, t_w);
    KIN_TIC(t_pg);
    const int4 meta = sh.meta[s];
    const int page = meta.x, ntok = meta.y;
    bool wrote = false;
    if (ok && ntok > 0) {
      uint8_t *stage = ring + s * R::kStageBytes;
      if (ntok < kBlock) {
        // Stale slots of a partial final page may hold anything (even NaN): zero their
        // V rows so that P = 0 times V stays 0.
        uint8_t *vrow = stage + Tile::kKBytes;
        for (int e = lane; e < (kBlock - ntok) * Tile::kBoxes * 8; e += 32) {
          const int t = ntok + e / (Tile::kBoxes * 8);
          const int rem = e % (Tile::kBoxes * 8);
          *reinterpret_cast<uint4 *>(vrow + (rem / 8) * Tile::kBoxBytes + t * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        wrote = true;
        __syncwarp();
      } else if (append && i == cnt - 1) {
        // The final block just became complete: its centroid (fp32 sum over the 16
        // tokens in order, times 1/16) from the staged keys.
        constexpr int kPer = D / 32;
        float acc[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
#pragma unroll
        for (int t = 0; t < kBlock; ++t) {
          const uint8_t *src = stage + swz_offset(t, lane * kPer);
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const float x = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(src)[k]);
            acc[k] = t == 0 ? x : __fadd_rn(acc[k], x);
          }
        }
        // both codes: the mean rounded to bf16, and its rounding residual rounded to bf16
        const int64_t off = (static_cast<int64_t>(page) * H + h) * D + lane * kPer;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const float mean = __fmul_rn(acc[k], 1.0f / kBlock);
          const __nv_bfloat16 c1 = __float2bfloat16_rn(mean);
          p.cent_out[off + k] = c1;
          p.cent_lo_out[off + k] = __float2bfloat16_rn(__fsub_rn(mean, __bfloat162float(c1)));
        }
      }
      const uint32_t sK = smem_u32(stage);
      st.page(qb, sK, sK + Tile::kKBytes, ntok, scale_log2, lane);
    }
    // generic-proxy writes to the stage must be ordered before the next TMA into it
    if (wrote) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
    KIN_TOC(kTrCPage, t_pg);
    KIN_COUNT(kTrCPages, 1);
  }
  KIN_TIC(t_ep);
  float *wm = reinterpret_cast<float *>(scratch);
  float *wl = wm + C::kCW * C::kQMax;
  float *wo = wl + C::kCW * C::kQMax;
  C::Bar::sync();   // the scratch may still hold the previous item's data
  KIN_TOC(kTrCEpiBar, t_ep);
  st.store(wm + warp * C::kQMax, wl + warp * C::kQMax, wo + warp * C::kQMax * D, lane, G);
  C::Bar::sync();
  combine_and_emit<__nv_bfloat16, D, C::kCW, C::kQMax, C::kCThreads, typename C::Bar>(
      ec, row, b, h, split, splits, wm, wl, wo, &sh.flag);
  KIN_TOC(kTrCEpilogue, t_ep);
}

template <int D, int NT>
__device__ void consumer(const FusedParams &p, uint8_t *ring, uint8_t *scratch,
                         const uint8_t *qstage, FusedShared &sh) {
  using C = Cfg<D, NT>;
  KIN_TRACE_DECL
  uint32_t n = 0;   // this warp's own pages / score stages so far (its sub-ring position)
  uint32_t nqs = 0;  // score items with staged q rows so far
  uint32_t nsc = 0;  // score items so far
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t nd = 0;
  KIN_TIC(t_start);
#pragma unroll 1
  while (true) {
    const int slot = nd % kDescs;
    KIN_TIC(t_d);
    const bool got = wait_bar(&sh.dfull[slot], (nd / kDescs) & 1u, sh, p.err, true);
    KIN_TOC(kTrCDesc, t_d);
    if (!got) break;
    const Desc d = sh.desc[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.dempty[slot]);
    ++nd;
    if (d.kind == kDescEnd) break;
    KIN_COUNT(kTrCItems, 1);
#ifdef KIN_TRACE_CYCLES
    if (tid == 0) {
      KIN_ITEM_STAMP(d.item, 3, gtime());
      KIN_ITEM_STAMP(d.item, 5, d.kind);
    }
#endif
    if (d.kind == kDescScore) {
      KIN_TIC(t0);
      consume_score<D, NT>(p, d, ring, reinterpret_cast<float *>(scratch), qstage, sh, n, nqs, nsc KIN_TRACE_ARG);
      KIN_TOC(kTrCScore, t0);
    } else if (d.kind == kDescSelect) {
      KIN_TIC(t0);
      consume_select<D, NT>(p, d, scratch, sh KIN_TRACE_ARG);
      KIN_TOC(kTrCSelect, t0);
    } else if (d.kind == kDescAttn) {
      consume_attention<D, NT>(p, d, ring, scratch, sh, n KIN_TRACE_ARG);
    } else {   // kDescEmptyRow: a sequence whose length is out of range
      const int H = p.num_kv_heads;
      const int b = d.row / H, h = d.row % H;
      const EmitCtx ec{p.out, p.lse, p.part_o, p.part_ml, p.attn_cnt, p.splits_per_row, p.group, H};
      write_empty_row<__nv_bfloat16, D, C::kCThreads>(ec, b, h);
      if (tid == 0 && h == 0) flag_error(p.err, KIN_DEVERR_SEQ_LEN);
      if (p.top_k > 0 && p.sel_out != nullptr) {
        int32_t *srow = p.sel_out + static_cast<int64_t>(d.row) * p.top_k;
        for (int i = tid; i < p.top_k; i += C::kCThreads) srow[i] = -1;
      }
    }
#ifdef KIN_TRACE_CYCLES
    if (tid == 0) KIN_ITEM_STAMP(d.item, 4, gtime());
#endif
  }
  KIN_TOC(kTrTotal, t_start);
  KIN_TRACE_FLUSH;
}

template <int D, int NT>
__global__ void __launch_bounds__(Cfg<D, NT>::kAllThreads, 1)
    fused_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const FusedParams p) {
  using C = Cfg<D, NT>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FusedShared sh;
  uint8_t *ring = align1024(smem_raw);
  uint8_t *scratch = ring + Ring<D, NT>::kBytes;
  uint8_t *qstage = scratch + kScratchBytes;   // q_stage_bytes<NT>(), 16-byte aligned
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < Ring<D, NT>::kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int i = 0; i < kDescs; ++i) {
      mbar_init(&sh.dfull[i], 1);
      mbar_init(&sh.dempty[i], C::kCW + kProducers);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.qfull[i], 1);
      mbar_init(&sh.qempty[i], C::kCW);
    }
    for (int i = 0; i < kScoreSlots; ++i) sh.score_arrive[i] = 0;
    sh.sel_done = 0;
    sh.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if ((tid >> 5) >= C::kCW)
    producer<D, NT>(p, &kmap, &vmap, ring, qstage, sh);
  else
    consumer<D, NT>(p, ring, scratch, qstage, sh);
  if (p.self_clean) {
    // Leave the counters zero for the next call.  Each CTA counts itself out after all of
    // its threads are done with the counters (barrier, then a cumulative GPU-scope fence);
    // the CTA that counts out last has seen every other CTA's counter updates and clears.
    // Every wait is bounded, so every CTA gets here, after a timeout too.
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      sh.last_cta = atomicAdd(p.exit_cnt, 1) == static_cast<int>(gridDim.x) - 1;
      __threadfence();
    }
    __syncthreads();
    if (sh.last_cta)
      for (int i = tid; i < p.n_counters; i += C::kAllThreads) p.counters[i] = 0;
  }
}

template <int D, int NT>
cudaError_t launch_d(const FusedParams &p, const CUtensorMap *kmap, const CUtensorMap *vmap,
                     cudaStream_t stream) {
  using C = Cfg<D, NT>;
  const size_t smem = fused_smem_bytes<D, NT>();
  // The shared-memory attribute is per device: set it, and look up the resident CTAs, once
  // per device (racing host threads set the same values).
  constexpr int kMaxDevices = 64;
  static std::atomic<int> resident[kMaxDevices];   // SMs x CTAs per SM, 0 = not yet known
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int ctas = dev >= 0 && dev < kMaxDevices ? resident[dev].load(std::memory_order_acquire) : 0;
  if (ctas == 0) {
    e = cudaFuncSetAttribute(fused_decode_kernel<D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int sms = 0, occupancy = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occupancy, fused_decode_kernel<D, NT>,
                                                      C::kAllThreads, smem);
    if (e != cudaSuccess) return e;
    ctas = sms * (occupancy < 1 ? 1 : occupancy);
    if (dev >= 0 && dev < kMaxDevices) resident[dev].store(ctas, std::memory_order_release);
  }
  const int total = p.n_score_items + p.n_select_items + p.n_attn_items;
  const int grid = min(total, ctas);
  if (grid <= 0) return cudaSuccess;
  fused_decode_kernel<D, NT><<<grid, C::kAllThreads, smem, stream>>>(*kmap, *vmap, p);
  return cudaGetLastError();
}

}  // namespace

int fused_max_score_chunk() { return kMaxScoreChunk; }

#ifdef KIN_TRACE_CYCLES
// Copy out (and clear) the cycle counters: [CTA][warp][slot], 160 x 12 x 20 words.
cudaError_t trace_take(unsigned long long *host, size_t words) {
  const size_t n = sizeof(g_trace) / sizeof(g_trace[0]);
  cudaError_t e = cudaMemcpyFromSymbol(host, g_trace, (words < n ? words : n) * 8);
  if (e != cudaSuccess) return e;
  static unsigned long long zeros[sizeof(g_trace) / sizeof(g_trace[0])];
  return cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros));
}
// Copy out (and clear) the per-item timeline: [item][8] words.
cudaError_t trace_items_take(unsigned long long *host, size_t words) {
  const size_t n = sizeof(g_items) / sizeof(g_items[0]);
  cudaError_t e = cudaMemcpyFromSymbol(host, g_items, (words < n ? words : n) * 8);
  if (e != cudaSuccess) return e;
  void *addr = nullptr;
  e = cudaGetSymbolAddress(&addr, g_items);
  if (e != cudaSuccess) return e;
  return cudaMemset(addr, 0, sizeof(g_items));
}
#endif

cudaError_t launch_fused(int head_dim, const FusedParams &p, const CUtensorMap *kmap,
                         const CUtensorMap *vmap, cudaStream_t stream) {
  if (p.group <= 8)
    return head_dim == 128 ? launch_d<128, 1>(p, kmap, vmap, stream)
                           : launch_d<64, 1>(p, kmap, vmap, stream);
  return head_dim == 128 ? launch_d<128, 2>(p, kmap, vmap, stream)
                         : launch_d<64, 2>(p, kmap, vmap, stream);
}

}  // namespace kin
