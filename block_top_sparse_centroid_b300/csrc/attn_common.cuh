// Device pieces shared by the attention kernels: tiling constants, the tensor-core page
// step (online softmax over one 16-token page), and the combine / split-merge epilogue.
//
// Per (sequence b, KV head h) row and query head g of its group:
//   o = sum_t softmax_t(sm_scale * q_g . k_t) v_t,   lse = ln sum_t exp(sm_scale * q_g . k_t)
// over the valid tokens (position < seq_len) of the row's kept blocks -- the paged decode
// of one layer (Kinetics README, "Benchmark Block TopK Attention throughput") restricted
// to the blocks block top-k keeps (Pith review of "Kinetics: Rethinking Test-Time Scaling
// Laws", "What carries the argument").
#pragma once

#include "kin_common.cuh"

namespace kin {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;          // shared-memory stages per warp (bf16 path)
constexpr int kMaxItems = 256;      // blocks per attention work item
constexpr int kMaxGroup = 16;

// One page of K (or V) for one head is 16 x D contiguous bf16; a TMA tiled copy moves it
// as D/64 boxes of 16 rows x 64 columns (128 bytes) with the 128-byte swizzle, so that
// ldmatrix reads of 8 tokens at one column offset hit 8 different bank groups.
template <int D>
struct BfTile {
  static constexpr int kBoxCols = 64;
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kBoxBytes = kBlock * kBoxCols * 2;   // 2048
  static constexpr int kKBytes = kBoxes * kBoxBytes;        // one page of K (or V)
  static constexpr int kStageBytes = 2 * kKBytes;           // K + V
  static constexpr int kSmemBytes = kWarps * kStages * kStageBytes;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                     ~uintptr_t(1023));
}

// Byte offset of element (token t, column c) inside one swizzled K or V page.
__device__ __forceinline__ uint32_t swz_offset(int t, int c) {
  const int box = c >> 6, col = c & 63;
  return box * 2048 + t * 128 + ((((col >> 3) ^ (t & 7))) << 4) + (col & 7) * 2;
}

// Where a row's result goes.
struct EmitCtx {
  void *out;           // [B, H*G, D]
  float *lse;          // [B, H*G] or NULL
  float *part_o;       // [rows, max_splits, G, D]
  float *part_ml;      // [rows, max_splits, G, 2]
  int32_t *counters;   // [rows] split arrivals, cleared before the kernel starts
  int max_splits;
  int G, H;
};

template <typename T, int D>
__device__ void write_empty_row(const EmitCtx &e, int b, int h) {
  const int Hq = e.H * e.G;
  T *out = static_cast<T *>(e.out);
  for (int x = threadIdx.x; x < e.G * D; x += blockDim.x) {
    const int r = x / D, i = x % D;
    Elem<T>::store(out + (static_cast<int64_t>(b) * Hq + h * e.G + r) * D + i, 0.f);
    if (i == 0 && e.lse != nullptr) e.lse[static_cast<int64_t>(b) * Hq + h * e.G + r] = -INFINITY;
  }
}

// Combine the per-warp states (wm: running max in log2 units, wl: sum of weights, wo:
// unnormalised output; [kWarps][kMaxGroup(...)]) and emit the row's result: directly
// when the row has one split, otherwise as a partial, the last split to arrive (an
// atomic counter, nothing waits) merging all partials.  Ends with a __syncthreads().
template <typename T, int D>
__device__ void combine_and_emit(const EmitCtx &e, int row, int b, int h, int split,
                                 int splits, const float *wm, const float *wl,
                                 const float *wo, int *s_flag) {
  const int G = e.G, Hq = e.H * G;
  T *out = static_cast<T *>(e.out);
  const int64_t obase = static_cast<int64_t>(b) * Hq + h * G;
  if (splits == 1) {
    for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
      const int r = x / D, i = x % D;
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
      if (i == 0 && e.lse != nullptr) e.lse[obase + r] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    return;
  }
  const int64_t slot = static_cast<int64_t>(row) * e.max_splits;
  float *po = e.part_o + (slot + split) * G * D;
  float *pml = e.part_ml + (slot + split) * G * 2;
  for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
    const int r = x / D, i = x % D;
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
    po[x] = O;
    if (i == 0) {
      pml[2 * r] = M;
      pml[2 * r + 1] = Ls;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&e.counters[row], 1);
    *s_flag = (prev == splits - 1);
  }
  __syncthreads();
  if (*s_flag) {
    __threadfence();
    const float *po_row = e.part_o + slot * G * D;
    const float *pml_row = e.part_ml + slot * G * 2;
    for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
      const int r = x / D, i = x % D;
      float M = -INFINITY;
      for (int s = 0; s < splits; ++s) M = fmaxf(M, __ldcg(pml_row + (s * G + r) * 2));
      float Ls = 0.f, O = 0.f;
      if (M != -INFINITY) {
        for (int s = 0; s < splits; ++s) {
          const float a = exp2f(__ldcg(pml_row + (s * G + r) * 2) - M);
          Ls += __ldcg(pml_row + (s * G + r) * 2 + 1) * a;
          O += __ldcg(po_row + static_cast<int64_t>(s) * G * D + x) * a;
        }
      }
      Elem<T>::store(out + (obase + r) * D + i, Ls > 0.f ? O / Ls : 0.f);
      if (i == 0 && e.lse != nullptr) e.lse[obase + r] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    }
  }
  __syncthreads();
}

// Online-softmax state of one warp for the query heads of a group: rows gq and gq + 8
// of the mma fragments (gq = lane / 4); O is [D/8 n-tiles][4] in C-fragment layout.
template <int D>
struct WarpSoftmax {
  float o[D / 8][4];
  float m0, m1, l0, l1;

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  // One staged page: S = Q K^T over 16 tokens, mask tokens >= ntok, online softmax,
  // O += P V.  sK / sV: shared addresses of the swizzled K and V pages.
  __device__ __forceinline__ void page(const uint32_t (&qa)[D / 16][4], uint32_t sK, uint32_t sV,
                                       int ntok, float scale_log2, int lane) {
    using Tile = BfTile<D>;
    const int tq = lane & 3, mi = lane >> 3, mr = lane & 7;
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
    if (a0 != 1.f || a1 != 1.f) {
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        o[nt][0] *= a0;
        o[nt][1] *= a0;
        o[nt][2] *= a1;
        o[nt][3] *= a1;
      }
    }
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

  // Reduce the quad-partial sums and store the state into the combine buffers.
  __device__ __forceinline__ void store(float *wm, float *wl, float *wo, int warp, int lane) {
    const int gq = lane >> 2, tq = lane & 3;
    float s0 = l0, s1 = l1;
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    if (tq == 0) {
      wm[warp * kMaxGroup + gq] = m0;
      wm[warp * kMaxGroup + gq + 8] = m1;
      wl[warp * kMaxGroup + gq] = s0;
      wl[warp * kMaxGroup + gq + 8] = s1;
    }
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + 2 * tq;
      wo[(warp * kMaxGroup + gq) * D + col] = o[nt][0];
      wo[(warp * kMaxGroup + gq) * D + col + 1] = o[nt][1];
      wo[(warp * kMaxGroup + gq + 8) * D + col] = o[nt][2];
      wo[(warp * kMaxGroup + gq + 8) * D + col + 1] = o[nt][3];
    }
  }
};

// Q fragments (A operand of S = Q K^T): rows = query heads of the group (zero past G).
template <int D>
__device__ __forceinline__ void load_q_frags(uint32_t (&qa)[D / 16][4], const __nv_bfloat16 *qg,
                                             int G, int lane) {
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int qrow = gq + 8 * (r & 1);
      const int col = 16 * ks + 2 * tq + 8 * (r >> 1);
      qa[ks][r] = qrow < G ? __ldg(reinterpret_cast<const unsigned int *>(qg + qrow * D + col)) : 0u;
    }
  }
}

constexpr size_t combine_smem_bytes(int D) {
  return static_cast<size_t>(kWarps) * kMaxGroup * (D + 2) * sizeof(float);
}

}  // namespace kin
