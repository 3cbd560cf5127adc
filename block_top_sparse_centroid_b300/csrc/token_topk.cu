// Token-level ("oracle") top-k decode for bf16 caches: three kernels on one stream.
//
// Oracle top-k attention keeps, for each query group, the keys with the largest exact
// scores q . k -- the perfect-selection upper bound that block top-k approximates with
// mean keys of 16-token pages (scime summary of "Kinetics: Rethinking Test-Time Scaling
// Laws", "Key results"; Pith review of the paper, "assumptions" and "What carries the
// argument").  Per (sequence b, KV head h) row with L = seq_lens[b] tokens and budget B:
//   score   s_t = sum_g q[b, hG+g, :] . K[t, h, :]   for every t < L   (fp32)
//   select  the B largest s_t, ties to the lower position; every t when L <= B
//   attend  out[b, hG+g, :] = softmax over the kept t of sm_scale * q.k, applied to V
//
// token_score_kernel streams every key of every row once (the step's dominant bytes, so
// it is a plain HBM stream: 16-byte loads, two pages in flight per warp, many CTAs per SM)
// and writes one fp32 score per token.  token_select_kernel (one CTA per row) finds the
// B-th largest score by a radix select over order-preserving 32-bit keys read back from
// L2 and writes the kept positions ascending, with each one's row in the [P*H*16, d] view
// of the page pool.  token_attn_kernel gathers the kept tokens' K and V rows with 16-byte
// asynchronous copies into the same swizzled 16-token tiles the block decode stages by
// TMA, so the tensor-core page step and the split merge of the block decode serve it
// unchanged; splits of a row merge through the last-arriving CTA.
#include "attn_common.cuh"
#include "kin_common.cuh"
#include "kin_internal.h"

namespace kin {
namespace {

constexpr int kTsThreads = 256;   // score kernel: 8 warps
constexpr int kTsWarps = kTsThreads / 32;
constexpr int kTsPages = 32;      // pages per score CTA (a multiple of 2 kTsWarps)
constexpr int kTselThreads = 512; // select kernel
constexpr int kTaWarps = 4;       // attention kernel
constexpr int kTaThreads = kTaWarps * 32;
constexpr int kTaStages = 2;      // gathered 16-token tiles in flight per warp
constexpr int kTaOffChunk = 2048; // kept tokens whose rows a CTA stages in shared memory at once
static_assert(kTsPages % (2 * kTsWarps) == 0, "two pages per warp per step");

template <int D>
constexpr size_t token_attn_smem() {
  return 1024 + static_cast<size_t>(kTaWarps) * kTaStages * BfTile<D>::kStageBytes;
}
static_assert(kTaWarps * 16 * 128 * 4 <= kTaWarps * kTaStages * 2 * 2 * 16 * 128,
              "the combine buffers fit in the stage memory they reuse");

__device__ __forceinline__ uint32_t token_key(float s) {
  // order-preserving 32-bit key: -0 and +0 equal, NaN below every number
  if (s != s) return 0u;
  const uint32_t u = __float_as_uint(s + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------------------- score
template <int D>
__global__ void __launch_bounds__(kTsThreads) token_score_kernel(TokenParams p) {
  constexpr int kCpt = D / 8;             // 16-byte chunks per token row
  constexpr int kTpl = 32 / kCpt;         // tokens one warp-wide load covers
  constexpr int kLoads = kBlock / kTpl;   // loads per lane per page
  __shared__ float qs[D];
  __shared__ int pages[kTsPages];
  const int row = blockIdx.y;
  const int H = p.num_kv_heads, G = p.group;
  const int b = row / H, h = row % H;
  const int L = p.seq_lens[b];
  if (L < 1 || L > kBlock * p.max_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && h == 0) flag_error(p.err, KIN_DEVERR_SEQ_LEN);
    return;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  const int j0 = blockIdx.x * kTsPages;
  if (j0 >= nb) return;
  const int np = min(nb - j0, kTsPages);
  // The group-summed query (fp32, ascending g) and the chunk's pages, one load each.
  const __nv_bfloat16 *qrow = p.q + (static_cast<int64_t>(b) * H * G + h * G) * D;
  for (int x = threadIdx.x; x < D / 8; x += kTsThreads) {
    float acc[8], f[8];
    Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4 *>(qrow + 8 * x), acc);
    for (int g = 1; g < G; ++g) {
      Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4 *>(qrow + g * D + 8 * x), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) qs[8 * x + i] = acc[i];
  }
  if (threadIdx.x < np) {
    const int pg = p.block_table[static_cast<int64_t>(b) * p.max_blocks + j0 + threadIdx.x];
    const bool ok = pg >= 0 && pg < p.num_pages;
    if (!ok) flag_error(p.err, KIN_DEVERR_PAGE_ID);
    pages[threadIdx.x] = ok ? pg : -1;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = lane % kCpt, sub = lane / kCpt;
  float qv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) qv[i] = qs[8 * c + i];
  float *srow = p.scores + static_cast<int64_t>(row) * p.score_stride;
  const __nv_bfloat16 *kp = p.k_pages;
  // pages i = warp, warp + kTsWarps, ... of the chunk, two per step (all loads first)
  for (int i = warp; i < np; i += 2 * kTsWarps) {
    uint4 raw[2][kLoads];
    int pg[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int ii = i + u * kTsWarps;
      pg[u] = ii < np ? pages[ii] : -1;
      const __nv_bfloat16 *base =
          kp + (static_cast<int64_t>(pg[u] < 0 ? 0 : pg[u]) * H + h) * kBlock * D + c * 8;
#pragma unroll
      for (int k = 0; k < kLoads; ++k)
        raw[u][k] = pg[u] >= 0 ? ldg_stream(base + (k * kTpl + sub) * D) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int ii = i + u * kTsWarps;
#pragma unroll
      for (int k = 0; k < kLoads; ++k) {
        float f[8];
        Elem<__nv_bfloat16>::unpack(raw[u][k], f);
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) part = fmaf(qv[e], f[e], part);
#pragma unroll
        for (int o = 1; o < kCpt; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        const int t = (j0 + ii) * kBlock + k * kTpl + sub;
        if (c == 0 && ii < np && t < L) srow[t] = pg[u] >= 0 ? part : -INFINITY;
      }
    }
  }
}

// ----------------------------------------------------------------------------- select
// One CTA of NTHR threads per row.  Thread x owns the contiguous positions
// [x KPT, (x + 1) KPT) of the row (KPT keys per thread, a multiple of 4) and holds their
// keys in registers, loaded once with 16-byte reads: four radix passes of 8 bits find the
// B-th largest key (counts per digit aggregated per warp before the shared-memory
// atomics), then two block scans place every kept position in ascending order.  Rows
// longer than 1024 x 32 positions go through token_select_long; rows of 8K-25.6K positions
// go through token_select_smem, which fits more of them on an SM.
template <int KPT, int NTHR>
__global__ void __launch_bounds__(NTHR) token_select_kernel(TokenParams p) {
  static_assert(KPT % kBlock == 0 || kBlock % KPT == 0, "a thread's run stays within whole pages");
  __shared__ int hist[256];
  __shared__ int scan_tmp[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int row = blockIdx.x;
  const int H = p.num_kv_heads;
  const int b = row / H, h = row % H;
  const int B = p.top_k;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  int32_t *gat = p.gather + static_cast<int64_t>(row) * B;
  int32_t *usr = p.sel_out == nullptr ? nullptr : p.sel_out + static_cast<int64_t>(row) * B;
  const int L = p.seq_lens[b];
  const int32_t *trow = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
  // kept position t at place pos: its row in the [P*H*16, d] view of the pages
  auto emit = [&](int pos, int t) {
    const int pg = trow[t / kBlock];
    const bool ok = pg >= 0 && pg < p.num_pages;
    gat[pos] = ok ? (pg * H + h) * kBlock + t % kBlock : -1;
    if (usr != nullptr) usr[pos] = t;
  };
  auto pad = [&](int from) {
    for (int i = from + tid; i < B; i += nt) {
      gat[i] = -1;
      if (usr != nullptr) usr[i] = -1;
    }
  };
  if (L < 1 || L > kBlock * p.max_blocks) {   // flagged by the score kernel
    pad(0);
    return;
  }
  if (L <= B) {
    for (int i = tid; i < L; i += nt) emit(i, i);
    pad(L);
    return;
  }
  const float *srow = p.scores + static_cast<int64_t>(row) * p.score_stride;
  const int t0 = tid * KPT;
  // the pages of this thread's run (KPT is a multiple of 16 or divides it, so the run
  // covers at most kRunPages pages), read now so that the emission waits on no load
  constexpr int kRunPages = KPT >= kBlock ? KPT / kBlock : 1;
  int run_pg[kRunPages];
#pragma unroll
  for (int u = 0; u < kRunPages; ++u) {
    const int t = t0 + u * kBlock;
    run_pg[u] = t < L ? trow[t / kBlock] : -1;
  }
  uint32_t key[KPT];   // 0: no position (past L)
#pragma unroll
  for (int i = 0; i < KPT; i += 4) {
    const int t = t0 + i;
    if (t + 3 < L) {   // rows start 16-byte aligned (the stride is a multiple of 64 floats)
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(srow + t));
      key[i] = token_key(v.x);
      key[i + 1] = token_key(v.y);
      key[i + 2] = token_key(v.z);
      key[i + 3] = token_key(v.w);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) key[i + u] = t + u < L ? token_key(__ldcg(srow + t + u)) : 0u;
    }
  }
  // keys of real positions are >= 1 except NaN scores (key 0), which rank last: count a
  // position by t < L, not by its key
  if (tid == 0) {
    s_prefix = 0u;
    s_remaining = B;
  }
  uint32_t mask = 0u;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += nt) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const bool in = t0 + i < L && (key[i] & mask) == prefix;
      const unsigned active = __ballot_sync(0xffffffffu, in);
      if (in) {
        const uint32_t dig = (key[i] >> shift) & 255u;
        const unsigned same = __match_any_sync(active, dig);
        if (lane == __ffs(same) - 1) atomicAdd(&hist[dig], __popc(same));
      }
    }
    __syncthreads();
    // thread x looks at digit 255 - x: count of keys whose digit is above it
    const int cnt = tid < 256 ? hist[255 - tid] : 0;
    int total;
    const int above = block_exclusive_scan(cnt, scan_tmp, &total);
    const int remaining = s_remaining;
    __syncthreads();
    if (tid < 256 && above < remaining && above + cnt >= remaining) {
      s_prefix = prefix | (static_cast<uint32_t>(255 - tid) << shift);
      s_remaining = remaining - above;
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t thr = s_prefix;     // key of the B-th largest score
  const int take_eq = s_remaining;   // keys equal to thr that are kept (>= 1), lowest first
  int gt = 0, eq = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const bool real = t0 + i < L;
    gt += real && key[i] > thr ? 1 : 0;
    eq += real && key[i] == thr ? 1 : 0;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, scan_tmp, &tot);
  const int my_eq = max(0, min(eq, take_eq - eq_before));
  int w = block_exclusive_scan(gt + my_eq, scan_tmp, &tot);
  int used_eq = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    if (t0 + i >= L) continue;
    bool keep = key[i] > thr;
    if (key[i] == thr && used_eq < my_eq) {
      keep = true;
      ++used_eq;
    }
    if (keep) {
      const int t = t0 + i;
      const int pg = run_pg[i / kBlock < kRunPages ? i / kBlock : kRunPages - 1];
      const bool ok = pg >= 0 && pg < p.num_pages;
      gat[w] = ok ? (pg * H + h) * kBlock + t % kBlock : -1;
      if (usr != nullptr) usr[w] = t;
      ++w;
    }
  }
}

// The same selection with the row's keys and page ids in shared memory instead of
// registers (512 threads, few registers): for rows whose keys take at most ~100 KB, two or
// more rows then run on one SM (the register-resident version above fits one 1024-thread
// CTA per SM once a row exceeds 512 x 32 positions).  Radix passes walk the keys in a
// strided order (conflict-free); the compaction walks contiguous runs.
constexpr int kSelSmemThreads = 512;
constexpr int kSelSmemMaxKeys = 25600;   // 100 KB of keys

__global__ void __launch_bounds__(kSelSmemThreads) token_select_smem(TokenParams p) {
  extern __shared__ uint32_t skeys[];   // [16 max_blocks] keys, then [max_blocks] pages
  __shared__ int hist[256];
  __shared__ int scan_tmp[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int row = blockIdx.x;
  const int H = p.num_kv_heads;
  const int b = row / H, h = row % H;
  const int B = p.top_k;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  int32_t *gat = p.gather + static_cast<int64_t>(row) * B;
  int32_t *usr = p.sel_out == nullptr ? nullptr : p.sel_out + static_cast<int64_t>(row) * B;
  const int L = p.seq_lens[b];
  const int32_t *trow = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
  auto pad = [&](int from) {
    for (int i = from + tid; i < B; i += nt) {
      gat[i] = -1;
      if (usr != nullptr) usr[i] = -1;
    }
  };
  if (L < 1 || L > kBlock * p.max_blocks) {
    pad(0);
    return;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  int *spages = reinterpret_cast<int *>(skeys + kBlock * p.max_blocks);
  for (int j = tid; j < nb; j += nt) spages[j] = trow[j];
  auto emit = [&](int pos, int t) {
    const int pg = spages[t / kBlock];
    const bool ok = pg >= 0 && pg < p.num_pages;
    gat[pos] = ok ? (pg * H + h) * kBlock + t % kBlock : -1;
    if (usr != nullptr) usr[pos] = t;
  };
  if (L <= B) {
    __syncthreads();
    for (int i = tid; i < L; i += nt) emit(i, i);
    pad(L);
    return;
  }
  const float *srow = p.scores + static_cast<int64_t>(row) * p.score_stride;
  for (int i = 4 * tid; i < L; i += 4 * nt) {   // rows start 16-byte aligned
    if (i + 3 < L) {
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(srow + i));
      skeys[i] = token_key(v.x);
      skeys[i + 1] = token_key(v.y);
      skeys[i + 2] = token_key(v.z);
      skeys[i + 3] = token_key(v.w);
    } else {
      for (int u = 0; u < 4 && i + u < L; ++u) skeys[i + u] = token_key(__ldcg(srow + i + u));
    }
  }
  if (tid == 0) {
    s_prefix = 0u;
    s_remaining = B;
  }
  uint32_t mask = 0u;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += nt) hist[i] = 0;
    __syncthreads();   // (first pass: also the keys and pages in shared memory)
    const uint32_t prefix = s_prefix;
#pragma unroll 4
    for (int t0 = 0; t0 < L; t0 += nt) {
      const int t = t0 + tid;
      const uint32_t key = t < L ? skeys[t] : 0u;
      const bool in = t < L && (key & mask) == prefix;
      const unsigned active = __ballot_sync(0xffffffffu, in);
      if (in) {
        const uint32_t dig = (key >> shift) & 255u;
        const unsigned same = __match_any_sync(active, dig);
        if (lane == __ffs(same) - 1) atomicAdd(&hist[dig], __popc(same));
      }
    }
    __syncthreads();
    const int cnt = tid < 256 ? hist[255 - tid] : 0;
    int total;
    const int above = block_exclusive_scan(cnt, scan_tmp, &total);
    const int remaining = s_remaining;
    __syncthreads();
    if (tid < 256 && above < remaining && above + cnt >= remaining) {
      s_prefix = prefix | (static_cast<uint32_t>(255 - tid) << shift);
      s_remaining = remaining - above;
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t thr = s_prefix;
  const int take_eq = s_remaining;
  const int per = (L + nt - 1) / nt;
  const int lo = min(L, tid * per), hi = min(L, lo + per);
  int gt = 0, eq = 0;
  for (int t = lo; t < hi; ++t) {
    const uint32_t key = skeys[t];
    gt += key > thr ? 1 : 0;
    eq += key == thr ? 1 : 0;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, scan_tmp, &tot);
  const int my_eq = max(0, min(eq, take_eq - eq_before));
  int w = block_exclusive_scan(gt + my_eq, scan_tmp, &tot);
  int used_eq = 0;
  for (int t = lo; t < hi; ++t) {
    const uint32_t key = skeys[t];
    bool keep = key > thr;
    if (key == thr && used_eq < my_eq) {
      keep = true;
      ++used_eq;
    }
    if (keep) emit(w++, t);
  }
}

// Rows longer than 1024 x 32 positions: the same radix select with the keys
// re-read from L2 on every pass (eight loads in flight per thread), and a compaction over
// contiguous runs.
__global__ void __launch_bounds__(kTselThreads) token_select_long(TokenParams p) {
  __shared__ int hist[256];
  __shared__ int scan_tmp[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int row = blockIdx.x;
  const int H = p.num_kv_heads;
  const int b = row / H, h = row % H;
  const int B = p.top_k;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  int32_t *gat = p.gather + static_cast<int64_t>(row) * B;
  int32_t *usr = p.sel_out == nullptr ? nullptr : p.sel_out + static_cast<int64_t>(row) * B;
  const int L = p.seq_lens[b];
  const int32_t *trow = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
  auto emit = [&](int pos, int t) {
    const int pg = trow[t / kBlock];
    const bool ok = pg >= 0 && pg < p.num_pages;
    gat[pos] = ok ? (pg * H + h) * kBlock + t % kBlock : -1;
    if (usr != nullptr) usr[pos] = t;
  };
  auto pad = [&](int from) {
    for (int i = from + tid; i < B; i += nt) {
      gat[i] = -1;
      if (usr != nullptr) usr[i] = -1;
    }
  };
  if (L < 1 || L > kBlock * p.max_blocks) {
    pad(0);
    return;
  }
  if (L <= B) {
    for (int i = tid; i < L; i += nt) emit(i, i);
    pad(L);
    return;
  }
  const float *srow = p.scores + static_cast<int64_t>(row) * p.score_stride;
  if (tid == 0) {
    s_prefix = 0u;
    s_remaining = B;
  }
  constexpr int kBatch = 8;
  uint32_t mask = 0u;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += nt) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
#pragma unroll 1
    for (int base = 0; base < L; base += kBatch * nt) {
      uint32_t kb[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int t = base + u * nt + tid;
        kb[u] = t < L ? token_key(__ldcg(srow + t)) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int t = base + u * nt + tid;
        const bool in = t < L && (kb[u] & mask) == prefix;
        const unsigned active = __ballot_sync(0xffffffffu, in);
        if (in) {
          const uint32_t dig = (kb[u] >> shift) & 255u;
          const unsigned same = __match_any_sync(active, dig);
          if (lane == __ffs(same) - 1) atomicAdd(&hist[dig], __popc(same));
        }
      }
    }
    __syncthreads();
    const int cnt = tid < 256 ? hist[255 - tid] : 0;
    int total;
    const int above = block_exclusive_scan(cnt, scan_tmp, &total);
    const int remaining = s_remaining;
    __syncthreads();
    if (tid < 256 && above < remaining && above + cnt >= remaining) {
      s_prefix = prefix | (static_cast<uint32_t>(255 - tid) << shift);
      s_remaining = remaining - above;
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t thr = s_prefix;
  const int take_eq = s_remaining;
  const int per = (L + nt - 1) / nt;
  const int lo = min(L, tid * per), hi = min(L, lo + per);
  int gt = 0, eq = 0;
  for (int t = lo; t < hi; ++t) {
    const uint32_t key = token_key(__ldcg(srow + t));
    gt += key > thr ? 1 : 0;
    eq += key == thr ? 1 : 0;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, scan_tmp, &tot);
  const int my_eq = max(0, min(eq, take_eq - eq_before));
  int w = block_exclusive_scan(gt + my_eq, scan_tmp, &tot);
  int used_eq = 0;
  for (int t = lo; t < hi; ++t) {
    const uint32_t key = token_key(__ldcg(srow + t));
    bool keep = key > thr;
    if (key == thr && used_eq < my_eq) {
      keep = true;
      ++used_eq;
    }
    if (keep) emit(w++, t);
  }
}

// ----------------------------------------------------------------------------- attend
// Gather one 16-token tile of kept tokens [tb, tb + 16) ∩ [tb, te) into a stage: K rows
// then V rows in the swizzled page layout; entries past te or with no valid row are zero.
// offs: the rows of the kept tokens from position ob on (shared memory).
template <int D>
__device__ __forceinline__ int gather_tile(const TokenParams &p, const int *offs, int ob, int tb,
                                           int te, uint8_t *stage, int lane) {
  constexpr int kCpt = D / 8;
  const int n = min(kBlock, te - tb);
  int off = lane < n ? offs[tb - ob + lane] : -1;
  if (lane < n && off < 0) flag_error(p.err, KIN_DEVERR_PAGE_ID);
  const uint32_t sK = smem_u32(stage), sV = sK + BfTile<D>::kKBytes;
#pragma unroll
  for (int k = 0; k < kBlock * kCpt / 32; ++k) {
    const int idx = lane + 32 * k;
    const int slot = idx / kCpt, ch = idx % kCpt;
    const int o = __shfl_sync(0xffffffffu, off, slot);
    const uint32_t dk = sK + swz_chunk(slot, ch), dv = sV + swz_chunk(slot, ch);
    if (o >= 0) {
      cp_async16(dk, p.k_pages + static_cast<int64_t>(o) * D + ch * 8);
      cp_async16(dv, p.v_pages + static_cast<int64_t>(o) * D + ch * 8);
    } else {
      asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dk), "r"(0u) : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dv), "r"(0u) : "memory");
    }
  }
  return n;
}

template <int D, int NT>
__global__ void __launch_bounds__(kTaThreads) token_attn_kernel(TokenParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int QMAX = 8 * NT;
  __shared__ float wm[kTaWarps * QMAX], wl[kTaWarps * QMAX];
  __shared__ int offs[kTaOffChunk];
  __shared__ int s_flag;
  uint8_t *smem = align1024(smem_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  const int H = p.num_kv_heads, G = p.group;
  const int b = row / H, h = row % H;
  const int L = p.seq_lens[b];
  const EmitCtx e{p.out, p.lse, p.part_o, p.part_ml, p.counters, p.splits, G, H};
  if (L < 1 || L > kBlock * p.max_blocks) {
    if (split == 0) write_empty_row<__nv_bfloat16, D, kTaThreads>(e, b, h);
    return;
  }
  const int n_kept = min(L, p.top_k);
  const int t0 = split * p.tokens_per_split;
  if (t0 >= n_kept) return;
  const int t1 = min(n_kept, t0 + p.tokens_per_split);
  const int splits = (n_kept + p.tokens_per_split - 1) / p.tokens_per_split;
  const int32_t *gat = p.gather + static_cast<int64_t>(row) * p.top_k;
  uint32_t qb[D / 16][NT][2];
  load_qT_frags<D, NT>(qb, p.q + (static_cast<int64_t>(b) * H * G + h * G) * D, G, lane);
  WarpSoftmaxT<D, NT> st;
  st.init();
  const float scale_log2 = p.sm_scale * kLog2e;
  uint8_t *wst = smem + warp * kTaStages * BfTile<D>::kStageBytes;
  // Chunks of kTaOffChunk kept tokens: their rows staged in shared memory by one coalesced
  // read, then this warp's 16-token tiles of the chunk (tb = c0 + 16 (warp + kTaWarps i)),
  // kTaStages gathers in flight.
#pragma unroll 1
  for (int c0 = t0; c0 < t1; c0 += kTaOffChunk) {
    const int c1 = min(t1, c0 + kTaOffChunk);
    __syncthreads();   // the previous chunk's offsets are no longer read
    for (int i = threadIdx.x; i < c1 - c0; i += kTaThreads) offs[i] = __ldcg(gat + c0 + i);
    __syncthreads();
    const int n_tiles = (c1 - c0 + kBlock - 1) / kBlock;
    int ntok[kTaStages];
#pragma unroll
    for (int s = 0; s < kTaStages; ++s) {
      const int tile = warp + kTaWarps * s;
      ntok[s] = tile < n_tiles ? gather_tile<D>(p, offs, c0, c0 + kBlock * tile, c1,
                                                wst + s * BfTile<D>::kStageBytes, lane)
                               : 0;
      cp_async_commit();
    }
    for (int i = 0;; ++i) {
      const int tile = warp + kTaWarps * i;
      if (tile >= n_tiles) break;
      const int s = i % kTaStages;
      cp_async_wait<kTaStages - 1>();
      __syncwarp();
      const uint32_t sK = smem_u32(wst + s * BfTile<D>::kStageBytes);
      st.page(qb, sK, sK + BfTile<D>::kKBytes, ntok[s], scale_log2, lane);
      __syncwarp();
      const int nxt = tile + kTaWarps * kTaStages;
      ntok[s] = nxt < n_tiles ? gather_tile<D>(p, offs, c0, c0 + kBlock * nxt, c1,
                                               wst + s * BfTile<D>::kStageBytes, lane)
                              : 0;
      cp_async_commit();
    }
    cp_async_wait<0>();
  }
  __syncthreads();   // every warp is done with its stages: the combine reuses them
  float *wo = reinterpret_cast<float *>(smem);
  st.store(wm + warp * QMAX, wl + warp * QMAX, wo + warp * QMAX * D, lane, G);
  __syncthreads();
  combine_and_emit<__nv_bfloat16, D, kTaWarps, QMAX, kTaThreads, CtaBarrier>(
      e, row, b, h, split, splits, wm, wl, wo, &s_flag);
  // the merging CTA leaves the row's arrival counter zero for the next call
  if (splits > 1 && s_flag && threadIdx.x == 0) p.counters[row] = 0;
}

template <int D, int NT>
cudaError_t launch_attn_t(const TokenParams &p, cudaStream_t stream) {
  const size_t smem = token_attn_smem<D>();
  static int set_device = -1;   // the device whose attribute was raised (one per process)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (set_device != dev) {
    e = cudaFuncSetAttribute(token_attn_kernel<D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    set_device = dev;
  }
  const int rows = p.batch * p.num_kv_heads;
  token_attn_kernel<D, NT><<<rows * p.splits, kTaThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_token_score(int head_dim, const TokenParams &p, cudaStream_t stream) {
  const int rows = p.batch * p.num_kv_heads;
  dim3 grid((p.max_blocks + kTsPages - 1) / kTsPages, rows);
  if (head_dim == 128)
    token_score_kernel<128><<<grid, kTsThreads, 0, stream>>>(p);
  else
    token_score_kernel<64><<<grid, kTsThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_token_select(const TokenParams &p, cudaStream_t stream) {
  // keys per thread: the smallest register run that covers the longest possible row
  const int64_t longest = static_cast<int64_t>(kBlock) * p.max_blocks;
  const int rows = p.batch * p.num_kv_heads;
  if (longest > 512 * 16 && longest <= kSelSmemMaxKeys) {
    // keys in shared memory: two to three rows per SM instead of one 1024-thread CTA
    const size_t smem = sizeof(uint32_t) * static_cast<size_t>(longest + p.max_blocks);
    static int set_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (set_device != dev) {
      e = cudaFuncSetAttribute(token_select_smem, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sizeof(uint32_t) * (kSelSmemMaxKeys + kSelSmemMaxKeys / kBlock)));
      if (e != cudaSuccess) return e;
      set_device = dev;
    }
    token_select_smem<<<rows, kSelSmemThreads, smem, stream>>>(p);
    return cudaGetLastError();
  }
  if (longest <= 512 * 8)
    token_select_kernel<8, 512><<<rows, 512, 0, stream>>>(p);
  else if (longest <= 512 * 16)
    token_select_kernel<16, 512><<<rows, 512, 0, stream>>>(p);
  else if (longest <= 1024 * 32)
    token_select_kernel<32, 1024><<<rows, 1024, 0, stream>>>(p);
  else
    token_select_long<<<rows, kTselThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_token_attn(int head_dim, const TokenParams &p, cudaStream_t stream) {
  const bool wide = p.group > 8;
  if (head_dim == 128) return wide ? launch_attn_t<128, 2>(p, stream) : launch_attn_t<128, 1>(p, stream);
  return wide ? launch_attn_t<64, 2>(p, stream) : launch_attn_t<64, 1>(p, stream);
}

int token_tile_tokens() { return kTaWarps * kBlock; }

}  // namespace kin
