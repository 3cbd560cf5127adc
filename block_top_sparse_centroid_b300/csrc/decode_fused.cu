// One persistent kernel for a whole bf16 decode step: group scoring, top-k block
// selection and split-KV attention, plus the centroid append of complete final blocks.
//
// Block top-k ranks key blocks by their mean key vectors and keeps the k best blocks of
// each GQA query group (Pith review of "Kinetics: Rethinking Test-Time Scaling Laws",
// "What carries the argument"); blocks are 16-token pages and k counts pages (Kinetics
// README, "Benchmark Block TopK Attention throughput").
//
// Work queue.  A global counter hands out items in this order:
//   score items      (row, chunk of 256 candidate blocks), rows with nb > k only;
//   attention items  (row, split of the row's kept-block list).
// A score item writes s_j = (sum_g q_g) . c_j for its chunk; the last score item of a row
// to finish (an atomic arrival count) selects the row's kept blocks and then releases
// the row's ready flag.  An attention item of a row that needs selection waits on that
// flag (bounded; a timeout sets KIN_DEVERR_TIMEOUT).  The wait cannot deadlock: every
// score item is handed out before any attention item, and score items never wait, so
// the item that completes a row is always held by a running CTA.
//
// Selection: radix select of the (k-1)-th largest order-preserving score key, 4 bits per
// pass.  Each thread packs its digit counts into two 64-bit words (8 bits per digit),
// each warp sums them with redux.sync, the CTA combines the 4 warps' 16 counts through
// shared memory (one barrier per pass); then an index-ordered compaction emits the kept
// blocks ascending, equal scores going to the lower block index.
//
// Attention: as in the standalone kernels -- TMA tiled copies of each kept page (K and V,
// 64-column boxes, 128-byte swizzle) into per-warp shared-memory rings completed on
// mbarriers, mma.m16n8k16 bf16 for S = Q K^T and O += P V with an online softmax, the
// warps of a CTA combined in shared memory, and the row's splits merged by the last
// split to arrive.
#include "attn_common.cuh"
#include "kin_internal.h"

namespace kin {
namespace {

constexpr int kChunk = 256;          // candidate blocks per score item
constexpr int kScoreUnroll = 8;      // centroid loads in flight per thread
constexpr int kMaxKeys = 16384;      // selection keys (one per candidate) in shared memory

// Dynamic shared memory: the attention stages, which also hold the selection keys and
// the combine buffers (never at the same time).
template <int D>
constexpr size_t fused_smem_bytes() {
  return BfTile<D>::kSmemBytes > kMaxKeys * 4 ? BfTile<D>::kSmemBytes : kMaxKeys * 4;
}

__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 0u;             // NaN ranks below every number
  s = s + 0.0f;                      // -0 and +0 compare equal
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int ld_acquire(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Kept blocks of one row: {nb-1} plus the m = k-1 largest of the n = nb-1 scores (ties to
// the lower index), ascending, into out[0..k-1].  CTA-wide; keys: n words of shared memory.
__device__ void select_row(const float *srow, int n, int m, int nb, uint32_t *keys,
                           int (*s_cnt)[kWarps * 16], int *scan_tmp, int32_t *out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int j = tid; j < n; j += kThreads) keys[j] = score_key(__ldcg(srow + j));
  __syncthreads();
  uint32_t prefix = 0u, mask = 0u;
  int remaining = m;
#pragma unroll 1
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 28 - 4 * pass;
    unsigned long long lo = 0ull, hi = 0ull;   // 8-bit count per digit (<= 128 keys/thread)
    for (int j = tid; j < n; j += kThreads) {
      const uint32_t key = keys[j];
      if ((key & mask) == prefix) {
        const uint32_t dg = (key >> shift) & 15u;
        if (dg < 8) lo += 1ull << (8 * dg);
        else hi += 1ull << (8 * (dg - 8));
      }
    }
    int mine = 0;
#pragma unroll
    for (int d = 0; d < 16; ++d) {
      const unsigned c = d < 8 ? static_cast<unsigned>((lo >> (8 * d)) & 255ull)
                               : static_cast<unsigned>((hi >> (8 * (d - 8))) & 255ull);
      const unsigned s = __reduce_add_sync(0xffffffffu, c);
      if (lane == d) mine = static_cast<int>(s);
    }
    if (lane < 16) s_cnt[pass & 1][warp * 16 + lane] = mine;
    __syncthreads();
    int above = 0, digit = 0;
    for (int d = 15; d >= 0; --d) {
      int c = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) c += s_cnt[pass & 1][w * 16 + d];
      if (above + c >= remaining) {
        digit = d;
        break;
      }
      above += c;
    }
    remaining -= above;
    prefix |= static_cast<uint32_t>(digit) << shift;
    mask |= 15u << shift;
  }
  const uint32_t thr = prefix;     // key of the m-th largest score
  const int take_eq = remaining;   // keys equal to thr that are kept (>= 1)
  const int per = (n + kThreads - 1) / kThreads;
  const int lo_j = min(n, tid * per), hi_j = min(n, lo_j + per);
  int gt = 0, eq = 0;
  for (int j = lo_j; j < hi_j; ++j) {
    const uint32_t key = keys[j];
    gt += key > thr;
    eq += key == thr;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, scan_tmp, &tot);
  const int my_eq = max(0, min(eq, take_eq - eq_before));
  int w = block_exclusive_scan(gt + my_eq, scan_tmp, &tot);
  int used = 0;
  for (int j = lo_j; j < hi_j; ++j) {
    const uint32_t key = keys[j];
    bool keep = key > thr;
    if (key == thr && used < my_eq) {
      keep = true;
      ++used;
    }
    if (keep) out[w++] = j;
  }
  if (tid == 0) out[m] = nb - 1;
}

struct Shared {
  uint64_t bars[kWarps * kStages];
  int page[kMaxItems];
  int ntok[kMaxItems];
  int chunk_pages[kChunk];
  int cnt[2][kWarps * 16];
  int scan_tmp[32];
  int next;
  int flag;
};

template <int D>
__device__ void score_item(const FusedParams &p, int item, uint8_t *smem, Shared &sh) {
  constexpr int kVec = 8;                          // bf16 per 16-byte slice
  constexpr int kTpi = D / kVec;                   // lanes per centroid (8 or 16)
  constexpr int kGroups = kThreads / kTpi;         // centroids per CTA per load slot
  const int tid = threadIdx.x;
  const int row = item / p.chunks_per_row, chunk = item % p.chunks_per_row;
  const int H = p.num_kv_heads, G = p.group;
  const int b = row / H, h = row % H;
  const int L = __ldg(p.seq_lens + b);
  if (L < 1 || L > kBlock * p.max_blocks) {
    if (chunk == 0 && h == 0 && tid == 0) flag_error(p.err, KIN_DEVERR_SEQ_LEN);
    return;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  if (nb <= p.top_k) return;                       // every block kept: nothing to score
  const int n = nb - 1;
  const int j0 = chunk * kChunk;
  if (j0 >= n) return;
  const int j1 = min(n, j0 + kChunk);
  const int32_t *trow = p.block_table + static_cast<int64_t>(b) * p.max_blocks;
  for (int i = tid; i < j1 - j0; i += kThreads) sh.chunk_pages[i] = __ldg(trow + j0 + i);

  const int grp = tid / kTpi, slice = tid % kTpi;
  float qs[kVec], f[kVec];
  const __nv_bfloat16 *qrow = p.q + (static_cast<int64_t>(b) * H * G + h * G) * D + slice * kVec;
  Elem<__nv_bfloat16>::unpack(__ldg(reinterpret_cast<const uint4 *>(qrow)), qs);
  for (int g = 1; g < G; ++g) {
    Elem<__nv_bfloat16>::unpack(__ldg(reinterpret_cast<const uint4 *>(qrow + g * D)), f);
#pragma unroll
    for (int i = 0; i < kVec; ++i) qs[i] += f[i];
  }
  __syncthreads();
  float *srow = p.scores + static_cast<int64_t>(row) * p.max_blocks;
  for (int base = j0; base < j1; base += kGroups * kScoreUnroll) {
    uint4 v[kScoreUnroll];
    int jj[kScoreUnroll];
    bool valid[kScoreUnroll];
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      jj[u] = base + u * kGroups + grp;
      valid[u] = false;
      v[u] = make_uint4(0, 0, 0, 0);
      if (jj[u] < j1) {
        const int64_t page = sh.chunk_pages[jj[u] - j0];
        if (page >= 0 && page < p.num_pages) {
          valid[u] = true;
          v[u] = ldg_stream(p.centroids + (page * H + h) * D + slice * kVec);
        } else if (slice == 0) {
          flag_error(p.err, KIN_DEVERR_PAGE_ID);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      Elem<__nv_bfloat16>::unpack(v[u], f);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < kVec; ++i) s = fmaf(qs[i], f[i], s);
#pragma unroll
      for (int o = kTpi / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (slice == 0 && jj[u] < j1) __stcg(srow + jj[u], valid[u] ? s : -INFINITY);
    }
  }
  // Arrival; the last chunk of the row to finish selects.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(p.score_cnt + row, 1);
    sh.flag = (prev == (n + kChunk - 1) / kChunk - 1);
  }
  __syncthreads();
  if (!sh.flag) return;
  __threadfence();
  select_row(srow, n, p.top_k - 1, nb, reinterpret_cast<uint32_t *>(smem), sh.cnt,
             sh.scan_tmp, p.sel + static_cast<int64_t>(row) * p.top_k);
  fence_proxy_async_smem();                        // keys area is reused by TMA copies
  __threadfence();
  __syncthreads();
  if (tid == 0) atomicExch(p.ready + row, 1);
}

template <int D>
__device__ void attention_item(const FusedParams &p, const CUtensorMap *kmap,
                               const CUtensorMap *vmap, int a, uint8_t *smem, Shared &sh,
                               uint32_t &uses, uint64_t policy) {
  using Tile = BfTile<D>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.num_kv_heads, G = p.group;
  const int row = a / p.splits_per_row, split = a % p.splits_per_row;
  const int b = row / H, h = row % H;
  const EmitCtx ec{p.out, p.lse, p.part_o, p.part_ml, p.attn_cnt, p.splits_per_row, G, H};
  const int L = __ldg(p.seq_lens + b);
  int32_t *srow_w = p.sel + static_cast<int64_t>(row) * p.top_k;
  if (L < 1 || L > kBlock * p.max_blocks) {
    if (split == 0) {
      write_empty_row<__nv_bfloat16, D>(ec, b, h);
      if (tid == 0 && h == 0) flag_error(p.err, KIN_DEVERR_SEQ_LEN);
      for (int i = tid; i < p.top_k; i += kThreads) srow_w[i] = -1;
    }
    return;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  const bool every_block = p.top_k == 0 || nb <= p.top_k;
  if (p.top_k > 0 && nb <= p.top_k && split == 0) {
    // no selection ran for this row: its kept list is every block, -1 padded
    for (int i = tid; i < p.top_k; i += kThreads) srow_w[i] = i < nb ? i : -1;
  }
  const int n_items = p.top_k == 0 ? nb : min(nb, p.top_k);
  const int splits = (n_items + p.items_per_split - 1) / p.items_per_split;
  if (split >= splits) return;
  const int i0 = split * p.items_per_split;
  const int cnt = min(n_items, i0 + p.items_per_split) - i0;

  if (!every_block) {
    if (tid == 0) {
      bool ok = false;
      for (uint32_t i = 0; i < kMaxWaitTries; ++i) {
        if (ld_acquire(p.ready + row) != 0) {
          ok = true;
          break;
        }
        __nanosleep(128);
      }
      if (!ok) flag_error(p.err, KIN_DEVERR_TIMEOUT);
    }
    __syncthreads();
  }
  const int32_t *srow = p.sel + static_cast<int64_t>(row) * p.top_k;
  for (int i = tid; i < cnt; i += kThreads) {
    const int j = every_block ? i0 + i : __ldcg(srow + i0 + i);
    int page = -1, ntok = 0;
    if (j >= 0 && j < nb) {
      const int pg = __ldg(p.block_table + static_cast<int64_t>(b) * p.max_blocks + j);
      if (pg >= 0 && pg < p.num_pages) {
        page = pg;
        ntok = min(kBlock, L - kBlock * j);
      } else {
        flag_error(p.err, KIN_DEVERR_PAGE_ID);
      }
    }
    sh.page[i] = page;
    sh.ntok[i] = ntok;
  }
  __syncthreads();

  const int my_cnt = cnt > warp ? (cnt - warp + kWarps - 1) / kWarps : 0;
  uint8_t *wbase = smem + warp * kStages * Tile::kStageBytes;
  uint64_t *wbar = sh.bars + warp * kStages;
  const int32_t ybase = h * kBlock;
  auto issue = [&](int n) {   // lane 0: stage the warp's n-th block of this item
    const uint32_t u = uses + n;
    const int s = u % kStages;
    const int page = sh.page[warp + n * kWarps];
    if (page < 0) {
      mbar_arrive(&wbar[s]);
      return;
    }
    uint8_t *dst = wbase + s * Tile::kStageBytes;
    mbar_arrive_expect_tx(&wbar[s], Tile::kStageBytes);
    const int32_t y = page * H * kBlock + ybase;
#pragma unroll
    for (int x = 0; x < Tile::kBoxes; ++x)
      tma_load_2d(dst + x * Tile::kBoxBytes, kmap, x * Tile::kBoxCols, y, &wbar[s], policy);
#pragma unroll
    for (int x = 0; x < Tile::kBoxes; ++x)
      tma_load_2d(dst + Tile::kKBytes + x * Tile::kBoxBytes, vmap, x * Tile::kBoxCols, y,
                  &wbar[s], policy);
  };
  if (lane == 0) {
    fence_proxy_async_smem();
    for (int n = 0; n < kStages && n < my_cnt; ++n) issue(n);
  }
  uint32_t qa[D / 16][4];
  load_q_frags<D>(qa, p.q + (static_cast<int64_t>(b) * H * G + h * G) * D, G, lane);
  const float scale_log2 = p.sm_scale * kLog2e;
  const bool append = p.append_final != 0 && (L % kBlock) == 0 && split == splits - 1;
  WarpSoftmax<D> st;
  st.init();
  for (int n = 0; n < my_cnt; ++n) {
    const uint32_t u = uses + n;
    const int s = u % kStages;
    const int it = warp + n * kWarps;
    const int ntok = sh.ntok[it];
    if (!mbar_wait(&wbar[s], (u / kStages) & 1)) {
      if (lane == 0) flag_error(p.err, KIN_DEVERR_TIMEOUT);
    } else if (ntok > 0) {
      uint8_t *stage = wbase + s * Tile::kStageBytes;
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
        __syncwarp();
      } else if (append && it == cnt - 1) {
        // The final block just became complete: its centroid (fp32 sum over the 16
        // tokens in order, times 1/16, rounded to bf16) from the staged keys.
        constexpr int kPer = D / 32;
        float acc[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
#pragma unroll
        for (int t = 0; t < kBlock; ++t) {
          const uint8_t *src = stage + swz_offset(t, lane * kPer);
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const float x = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(src)[i]);
            acc[i] = t == 0 ? x : __fadd_rn(acc[i], x);
          }
        }
        __nv_bfloat16 *dst = p.cent_out + (static_cast<int64_t>(sh.page[it]) * H + h) * D + lane * kPer;
#pragma unroll
        for (int i = 0; i < kPer; ++i) dst[i] = __float2bfloat16_rn(__fmul_rn(acc[i], 1.0f / kBlock));
      }
      const uint32_t sK = smem_u32(stage);
      st.page(qa, sK, sK + Tile::kKBytes, ntok, scale_log2, lane);
    }
    __syncwarp();
    if (lane == 0 && n + kStages < my_cnt) {
      fence_proxy_async_smem();
      issue(n + kStages);
    }
  }
  uses += my_cnt;
  __syncthreads();   // every stage consumed: reuse the stage memory for the combine
  float *wm = reinterpret_cast<float *>(smem);
  float *wl = wm + kWarps * kMaxGroup;
  float *wo = wl + kWarps * kMaxGroup;
  st.store(wm, wl, wo, warp, lane);
  __syncthreads();
  combine_and_emit<__nv_bfloat16, D>(ec, row, b, h, split, splits, wm, wl, wo, &sh.flag);
  fence_proxy_async_smem();   // the combine buffers are overwritten by the next copies
  __syncthreads();
}

template <int D>
__global__ void __launch_bounds__(kThreads, 3)
    fused_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  uint8_t *smem = align1024(smem_raw);
  const int tid = threadIdx.x;
  if (tid < kWarps * kStages) mbar_init(&sh.bars[tid], 1);
  fence_mbar_init();
  if (tid == 0) sh.next = atomicAdd(p.work_next, 1);
  __syncthreads();
  const uint64_t policy = l2_policy_evict_first();
  uint32_t uses = 0;
  const int total = p.n_score_items + p.n_attn_items;
  while (true) {
    const int item = sh.next;
    __syncthreads();
    if (item >= total) break;
    int next = 0;
    if (tid == 0) next = atomicAdd(p.work_next, 1);   // consumed at the end of the item
    if (item < p.n_score_items)
      score_item<D>(p, item, smem, sh);
    else
      attention_item<D>(p, &kmap, &vmap, item - p.n_score_items, smem, sh, uses, policy);
    if (tid == 0) sh.next = next;
    __syncthreads();
  }
}

template <int D>
cudaError_t launch_d(const FusedParams &p, const CUtensorMap *kmap, const CUtensorMap *vmap,
                     cudaStream_t stream) {
  static_assert(fused_smem_bytes<D>() >= combine_smem_bytes(D), "combine must fit");
  const size_t smem = fused_smem_bytes<D>() + 1024;
  static int occupancy = 0, sms = 0;
  if (occupancy == 0) {
    cudaError_t e = cudaFuncSetAttribute(fused_decode_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occupancy, fused_decode_kernel<D>,
                                                      kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occupancy < 1) occupancy = 1;
  }
  const int total = p.n_score_items + p.n_attn_items;
  const int grid = min(total, sms * occupancy);
  if (grid <= 0) return cudaSuccess;
  fused_decode_kernel<D><<<grid, kThreads, smem, stream>>>(*kmap, *vmap, p);
  return cudaGetLastError();
}

}  // namespace

int fused_chunk() { return kChunk; }

cudaError_t launch_fused(int head_dim, const FusedParams &p, const CUtensorMap *kmap,
                         const CUtensorMap *vmap, cudaStream_t stream) {
  return head_dim == 128 ? launch_d<128>(p, kmap, vmap, stream)
                         : launch_d<64>(p, kmap, vmap, stream);
}

}  // namespace kin
