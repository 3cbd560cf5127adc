// Split-KV paged decode attention over a list of kept blocks (block top-k) or over every
// block (dense), with the split merge fused through a last-arriver counter.
//
// The paged decode of one layer over 16-token pages is the benchmark of the Kinetics
// README ("Benchmark Block TopK Attention throughput"); block top-k restricts it to the
// kept blocks (Pith review of "Kinetics: Rethinking Test-Time Scaling Laws", "What
// carries the argument").  Per (sequence b, KV head h) row and query head g of the group:
//   o = sum_t softmax_t(sm_scale * q_g . k_t) v_t,   lse = ln sum_t exp(sm_scale * q_g . k_t)
// over the valid tokens (position < seq_len) of the row's blocks.
//
// Work decomposition: grid = (splits, rows).  A CTA takes a contiguous run of the row's
// block list; its 4 warps take every 4th block of the run, each warp with its own
// online-softmax state and its own ring of shared-memory stages.  At the end the warps'
// states are combined in shared memory; with one split the CTA writes the output, with
// several it writes an unnormalised partial and the last CTA of the row to arrive (an
// atomic counter, no waiting) merges all partials.
//
// bf16 path: every page of K and V for one head is 16 x d contiguous bf16 (4 KB at
// d = 128).  A TMA tiled copy moves it in 64-column boxes with the 128-byte swizzle, so
// that ldmatrix reads of 8 tokens at one column offset hit 8 different bank groups.  The
// group's G <= 16 query heads form the M = 16 rows of mma.m16n8k16 (bf16 in, fp32
// accumulate): S = Q K^T (N = 16 tokens, K = d) then O += P V (N = d, K = 16 tokens),
// with P rounded to bf16 and the running sum built from those rounded weights.
// fp32 path: CUDA-core FMAs, one lane per d/32 dimensions (exact fp32 arithmetic).
#include "kin_common.cuh"
#include "kin_internal.h"

namespace kin {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;          // shared-memory stages per warp (bf16 path)
constexpr int kMaxItems = 256;      // blocks per CTA (host keeps items_per_split below)
constexpr int kMaxGroup = 16;

template <int D>
struct BfTile {
  static constexpr int kBoxCols = 64;                       // 128 bytes of bf16
  static constexpr int kBoxes = D / kBoxCols;               // per page, per tensor
  static constexpr int kBoxBytes = kBlock * kBoxCols * 2;   // 2048
  static constexpr int kKBytes = kBoxes * kBoxBytes;        // one page of K (or V)
  static constexpr int kStageBytes = 2 * kKBytes;           // K + V
  static constexpr int kSmemBytes = kWarps * kStages * kStageBytes;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Row bookkeeping shared by both paths.  Returns false when the CTA has nothing to do.
struct RowInfo {
  int row, b, h, L, nb, n_items, splits, i0, cnt;
};

__device__ __forceinline__ bool row_setup(const AttnParams &p, RowInfo &ri) {
  ri.row = blockIdx.y;
  ri.b = ri.row / p.num_kv_heads;
  ri.h = ri.row % p.num_kv_heads;
  ri.L = p.seq_lens[ri.b];
  const int split = blockIdx.x;
  if (ri.L < 1 || ri.L > kBlock * p.max_blocks) {
    ri.nb = 0;
    return split == 0;  // split 0 writes the empty result
  }
  ri.nb = (ri.L + kBlock - 1) / kBlock;
  ri.n_items = p.sel != nullptr ? min(ri.nb, p.sel_stride) : ri.nb;
  ri.splits = (ri.n_items + p.items_per_split - 1) / p.items_per_split;
  if (split >= ri.splits) return false;
  ri.i0 = split * p.items_per_split;
  ri.cnt = min(ri.n_items, ri.i0 + p.items_per_split) - ri.i0;
  return true;
}

// Empty result for a row whose seq_len is out of range.
template <typename T, int D>
__device__ void write_empty_row(const AttnParams &p, const RowInfo &ri) {
  const int G = p.group, Hq = p.num_kv_heads * G;
  T *out = static_cast<T *>(p.out);
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int r = e / D, i = e % D;
    Elem<T>::store(out + (static_cast<int64_t>(ri.b) * Hq + ri.h * G + r) * D + i, 0.f);
    if (i == 0 && p.lse != nullptr) p.lse[static_cast<int64_t>(ri.b) * Hq + ri.h * G + r] = -INFINITY;
  }
  if (threadIdx.x == 0 && ri.h == 0) flag_error(p.err, KIN_DEVERR_SEQ_LEN);
}

// Load the CTA's block list: physical page and number of valid tokens per item.
__device__ __forceinline__ void load_items(const AttnParams &p, const RowInfo &ri, int *s_page,
                                           int *s_ntok) {
  for (int i = threadIdx.x; i < ri.cnt; i += blockDim.x) {
    const int idx = ri.i0 + i;
    const int j = p.sel != nullptr ? p.sel[static_cast<int64_t>(ri.row) * p.sel_stride + idx] : idx;
    int page = -1, ntok = 0;
    if (j >= 0 && j < ri.nb) {
      const int pg = p.block_table[static_cast<int64_t>(ri.b) * p.max_blocks + j];
      if (pg >= 0 && pg < p.num_pages) {
        page = pg;
        ntok = min(kBlock, ri.L - kBlock * j);
      } else {
        flag_error(p.err, KIN_DEVERR_PAGE_ID);
      }
    }
    s_page[i] = page;
    s_ntok[i] = ntok;
  }
}

// Combine the per-warp states (wm: running max in log2 units, wl: sum of weights,
// wo: unnormalised output, each [kWarps][16(...)]) and emit the row's result, directly
// or through the split partials and the last-arriver merge.
template <typename T, int D>
__device__ void combine_and_emit(const AttnParams &p, const RowInfo &ri, const float *wm,
                                 const float *wl, const float *wo) {
  __shared__ int s_last;
  const int G = p.group, Hq = p.num_kv_heads * G;
  const int split = blockIdx.x;
  T *out = static_cast<T *>(p.out);
  const int64_t obase = static_cast<int64_t>(ri.b) * Hq + ri.h * G;
  if (ri.splits == 1) {
    for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
      const int r = e / D, i = e % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kMaxGroup + r]);
      float Ls = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float a = exp2f(wm[w * kMaxGroup + r] - M);
          Ls += wl[w * kMaxGroup + r] * a;
          O += wo[(w * kMaxGroup + r) * D + i] * a;
        }
      }
      Elem<T>::store(out + (obase + r) * D + i, Ls > 0.f ? O / Ls : 0.f);
      if (i == 0 && p.lse != nullptr) p.lse[obase + r] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    }
    return;
  }
  const int64_t slot = static_cast<int64_t>(ri.row) * p.max_splits;
  float *po = p.part_o + (slot + split) * G * D;
  float *pml = p.part_ml + (slot + split) * G * 2;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int r = e / D, i = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kMaxGroup + r]);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float a = exp2f(wm[w * kMaxGroup + r] - M);
        Ls += wl[w * kMaxGroup + r] * a;
        O += wo[(w * kMaxGroup + r) * D + i] * a;
      }
    }
    po[e] = O;
    if (i == 0) {
      pml[2 * r] = M;
      pml[2 * r + 1] = Ls;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&p.counters[ri.row], 1);
    s_last = (prev == ri.splits - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) p.counters[ri.row] = 0;  // leave the workspace zeroed
  const float *po_row = p.part_o + slot * G * D;
  const float *pml_row = p.part_ml + slot * G * 2;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int r = e / D, i = e % D;
    float M = -INFINITY;
    for (int s = 0; s < ri.splits; ++s) M = fmaxf(M, __ldcg(pml_row + (s * G + r) * 2));
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < ri.splits; ++s) {
        const float ms = __ldcg(pml_row + (s * G + r) * 2);
        const float a = exp2f(ms - M);
        Ls += __ldcg(pml_row + (s * G + r) * 2 + 1) * a;
        O += __ldcg(po_row + static_cast<int64_t>(s) * G * D + e) * a;
      }
    }
    Elem<T>::store(out + (obase + r) * D + i, Ls > 0.f ? O / Ls : 0.f);
    if (i == 0 && p.lse != nullptr) p.lse[obase + r] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
  }
}

// ------------------------------------------------------------------------------------
// bf16: TMA + mma.sync
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads, 3)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
  using Tile = BfTile<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kWarps * kStages];
  __shared__ int s_page[kMaxItems], s_ntok[kMaxItems];
  uint8_t *smem = align1024(smem_raw);

  RowInfo ri;
  if (!row_setup(p, ri)) return;
  if (ri.nb == 0) {
    write_empty_row<__nv_bfloat16, D>(p, ri);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.num_kv_heads, G = p.group;
  load_items(p, ri, s_page, s_ntok);
  if (tid < kWarps * kStages) mbar_init(&bars[tid], 1);
  fence_mbar_init();
  __syncthreads();

  const int my_cnt = ri.cnt > warp ? (ri.cnt - warp + kWarps - 1) / kWarps : 0;
  uint8_t *wbase = smem + warp * kStages * Tile::kStageBytes;
  uint64_t *wbar = bars + warp * kStages;
  const uint64_t policy = l2_policy_evict_first();
  const int32_t ybase = ri.h * kBlock;

  auto issue = [&](int n) {  // lane 0 only: stage the warp's n-th block
    const int it = warp + n * kWarps;
    const int s = n % kStages;
    const int page = s_page[it];
    if (page < 0) {
      mbar_arrive(&wbar[s]);
      return;
    }
    uint8_t *dst = wbase + s * Tile::kStageBytes;
    mbar_arrive_expect_tx(&wbar[s], Tile::kStageBytes);
    const int32_t y = page * H * kBlock + ybase;
#pragma unroll
    for (int x = 0; x < Tile::kBoxes; ++x)
      tma_load_2d(dst + x * Tile::kBoxBytes, &kmap, x * Tile::kBoxCols, y, &wbar[s], policy);
#pragma unroll
    for (int x = 0; x < Tile::kBoxes; ++x)
      tma_load_2d(dst + Tile::kKBytes + x * Tile::kBoxBytes, &vmap, x * Tile::kBoxCols, y,
                  &wbar[s], policy);
  };
  if (lane == 0) {
    for (int n = 0; n < kStages && n < my_cnt; ++n) issue(n);
  }

  // Q fragments (A operand, rows = query heads of the group, zero beyond G).
  const int gq = lane >> 2, tq = lane & 3;
  const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q) +
                            (static_cast<int64_t>(ri.b) * H * G + ri.h * G) * D;
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int qrow = gq + 8 * (r & 1);
      const int col = 16 * ks + 2 * tq + 8 * (r >> 1);
      qa[ks][r] = qrow < G ? *reinterpret_cast<const uint32_t *>(qg + qrow * D + col) : 0u;
    }
  }
  const float scale_log2 = p.sm_scale * kLog2e;

  float o[D / 8][4];
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  const int mi = lane >> 3, mr = lane & 7;
  for (int n = 0; n < my_cnt; ++n) {
    const int s = n % kStages;
    const int it = warp + n * kWarps;
    const int ntok = s_ntok[it];
    if (!mbar_wait(&wbar[s], (n / kStages) & 1)) {
      if (lane == 0) flag_error(p.err, KIN_DEVERR_TIMEOUT);
      break;
    }
    if (ntok > 0) {
      const uint32_t sK = smem_u32(wbase + s * Tile::kStageBytes);
      const uint32_t sV = sK + Tile::kKBytes;
      if (ntok < kBlock) {
        // Stale slots of a partial final page may hold anything (even NaN): zero their
        // V rows so that P = 0 times V stays 0.
        uint8_t *vrow = wbase + s * Tile::kStageBytes + Tile::kKBytes;
        for (int e = lane; e < (kBlock - ntok) * Tile::kBoxes * 8; e += 32) {
          const int t = ntok + e / (Tile::kBoxes * 8);
          const int rem = e % (Tile::kBoxes * 8);
          *reinterpret_cast<uint4 *>(vrow + (rem / 8) * Tile::kBoxBytes + t * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // S = Q K^T over 16 tokens (two n-tiles of 8).
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int chunk = 2 * ks + (mi & 1);
        const int tok = mr + 8 * (mi >> 1);
        const uint32_t addr = sK + (chunk >> 3) * Tile::kBoxBytes + tok * 128 +
                              (((chunk & 7) ^ (tok & 7)) << 4);
        uint32_t b00, b01, b10, b11;
        ldmatrix_x4(addr, b00, b01, b10, b11);
        mma_bf16_16816(sc[0], qa[ks], b00, b01);
        mma_bf16_16816(sc[1], qa[ks], b10, b11);
      }
      // Scale to log2 units, mask tokens past the length, running max per query head.
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int tok = nt * 8 + 2 * tq + (c & 1);
          sc[nt][c] = tok < ntok ? sc[nt][c] * scale_log2 : -INFINITY;
        }
      }
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float a0 = exp2f(m0 - mu0), a1 = exp2f(m1 - mu1);
      m0 = mn0;
      m1 = mn1;
      uint32_t pa[4];
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint32_t top = pack_bf16x2(exp2f(sc[nt][0] - mu0), exp2f(sc[nt][1] - mu0));
        const uint32_t bot = pack_bf16x2(exp2f(sc[nt][2] - mu1), exp2f(sc[nt][3] - mu1));
        ps0 += bf16_lo(top) + bf16_hi(top);
        ps1 += bf16_lo(bot) + bf16_hi(bot);
        pa[2 * nt] = top;       // a0 / a2: row gq, tokens 8nt + 2tq, +1
        pa[2 * nt + 1] = bot;   // a1 / a3: row gq + 8
      }
      l0 = l0 * a0 + ps0;
      l1 = l1 * a1 + ps1;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        o[nt][0] *= a0;
        o[nt][1] *= a0;
        o[nt][2] *= a1;
        o[nt][3] *= a1;
      }
      // O += P V: B operand from V via transposing ldmatrix, two n-tiles per load.
#pragma unroll
      for (int pp = 0; pp < D / 16; ++pp) {
        const int chunk = 2 * pp + (mi >> 1);
        const int tok = mr + 8 * (mi & 1);
        const uint32_t addr = sV + (chunk >> 3) * Tile::kBoxBytes + tok * 128 +
                              (((chunk & 7) ^ (tok & 7)) << 4);
        uint32_t v0, v1, v2, v3;
        ldmatrix_x4_trans(addr, v0, v1, v2, v3);
        mma_bf16_16816(o[2 * pp], pa, v0, v1);
        mma_bf16_16816(o[2 * pp + 1], pa, v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0 && n + kStages < my_cnt) {
      fence_proxy_async_smem();
      issue(n + kStages);
    }
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  __syncthreads();  // every stage consumed: reuse the stage memory for the combine
  float *wm = reinterpret_cast<float *>(smem);
  float *wl = wm + kWarps * kMaxGroup;
  float *wo = wl + kWarps * kMaxGroup;
  if (tq == 0) {
    wm[warp * kMaxGroup + gq] = m0;
    wm[warp * kMaxGroup + gq + 8] = m1;
    wl[warp * kMaxGroup + gq] = l0;
    wl[warp * kMaxGroup + gq + 8] = l1;
  }
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    const int col = nt * 8 + 2 * tq;
    wo[(warp * kMaxGroup + gq) * D + col] = o[nt][0];
    wo[(warp * kMaxGroup + gq) * D + col + 1] = o[nt][1];
    wo[(warp * kMaxGroup + gq + 8) * D + col] = o[nt][2];
    wo[(warp * kMaxGroup + gq + 8) * D + col + 1] = o[nt][3];
  }
  __syncthreads();
  combine_and_emit<__nv_bfloat16, D>(p, ri, wm, wl, wo);
}

// ------------------------------------------------------------------------------------
// fp32: CUDA cores, loads straight from global memory
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) attn_f32_kernel(const AttnParams p) {
  constexpr int kPer = D / 32;  // dimensions per lane (2 or 4)
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_page[kMaxItems], s_ntok[kMaxItems];
  RowInfo ri;
  if (!row_setup(p, ri)) return;
  if (ri.nb == 0) {
    write_empty_row<float, D>(p, ri);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.num_kv_heads, G = p.group;
  load_items(p, ri, s_page, s_ntok);
  __syncthreads();

  const float *qg = static_cast<const float *>(p.q) + (static_cast<int64_t>(ri.b) * H * G + ri.h * G) * D;
  const float *kp = static_cast<const float *>(p.k_pages);
  const float *vp = static_cast<const float *>(p.v_pages);
  float qr[kMaxGroup][kPer], acc[kMaxGroup][kPer], m[kMaxGroup], l[kMaxGroup];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      qr[g][i] = g < G ? qg[g * D + lane * kPer + i] : 0.f;
      acc[g][i] = 0.f;
    }
  }
  const float scale_log2 = p.sm_scale * kLog2e;
  for (int it = warp; it < ri.cnt; it += kWarps) {
    const int page = s_page[it], ntok = s_ntok[it];
    if (page < 0) continue;
    const int64_t base = (static_cast<int64_t>(page) * H + ri.h) * kBlock * D;
    for (int t = 0; t < ntok; ++t) {
      float kv[kPer], vv[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        kv[i] = kp[base + t * D + lane * kPer + i];
        vv[i] = vp[base + t * D + lane * kPer + i];
      }
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) {
        if (g < G) {
          float s = 0.f;
#pragma unroll
          for (int i = 0; i < kPer; ++i) s = fmaf(qr[g][i], kv[i], s);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          const float z = s * scale_log2;
          const float mn = fmaxf(m[g], z);
          const float a = exp2f(m[g] - mn);
          const float w = exp2f(z - mn);
          l[g] = l[g] * a + w;
#pragma unroll
          for (int i = 0; i < kPer; ++i) acc[g][i] = acc[g][i] * a + w * vv[i];
          m[g] = mn;
        }
      }
    }
  }
  float *wm = reinterpret_cast<float *>(smem_raw);
  float *wl = wm + kWarps * kMaxGroup;
  float *wo = wl + kWarps * kMaxGroup;
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    if (lane == 0) {
      wm[warp * kMaxGroup + g] = m[g];
      wl[warp * kMaxGroup + g] = l[g];
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) wo[(warp * kMaxGroup + g) * D + lane * kPer + i] = acc[g][i];
  }
  __syncthreads();
  combine_and_emit<float, D>(p, ri, wm, wl, wo);
}

constexpr size_t combine_smem_bytes(int D) {
  return static_cast<size_t>(kWarps) * kMaxGroup * (D + 2) * sizeof(float);
}

template <int D>
cudaError_t launch_bf16(const AttnParams &p, const CUtensorMap *kmap, const CUtensorMap *vmap,
                        cudaStream_t stream) {
  static_assert(BfTile<D>::kSmemBytes >= combine_smem_bytes(D), "combine must fit the stages");
  const size_t smem = BfTile<D>::kSmemBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_splits, p.batch * p.num_kv_heads);
  attn_bf16_kernel<D><<<grid, kThreads, smem, stream>>>(*kmap, *vmap, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_f32(const AttnParams &p, cudaStream_t stream) {
  const size_t smem = combine_smem_bytes(D);
  cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_splits, p.batch * p.num_kv_heads);
  attn_f32_kernel<D><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int attention_warps() { return kWarps; }
int attention_max_items() { return kMaxItems; }

cudaError_t launch_attention(kin_dtype dtype, int head_dim, const AttnParams &p,
                             const CUtensorMap *kmap, const CUtensorMap *vmap,
                             cudaStream_t stream) {
  if (dtype == KIN_BF16)
    return head_dim == 128 ? launch_bf16<128>(p, kmap, vmap, stream)
                           : launch_bf16<64>(p, kmap, vmap, stream);
  return head_dim == 128 ? launch_f32<128>(p, stream) : launch_f32<64>(p, stream);
}

}  // namespace kin
