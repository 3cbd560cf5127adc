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

constexpr int kWarps = 4;           // warps of the fp32 attention kernel
constexpr int kThreads = kWarps * 32;
constexpr int kMaxItems = 256;      // blocks per attention work item
constexpr int kMaxGroup = 16;       // query heads per KV head

// One page of K (or V) for one head is 16 x D contiguous bf16.  In shared memory it is
// laid out as D/64 column halves of [16 rows][64 columns] (128 bytes per row) with the
// 128-byte swizzle, as a TMA tiled copy with that swizzle writes it, so that ldmatrix
// reads of 8 tokens at one column offset hit 8 different bank groups.
template <int D>
struct BfTile {
  static constexpr int kBoxCols = 64;
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kBoxBytes = kBlock * kBoxCols * 2;   // 2048
  static constexpr int kKBytes = kBoxes * kBoxBytes;        // one page of K (or V)
  static constexpr int kStageBytes = 2 * kKBytes;           // K + V
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

// Byte offset of the 16-byte chunk `chunk` (8 columns) of token t in a swizzled page.
__device__ __forceinline__ uint32_t swz_chunk(int t, int chunk) {
  return (chunk >> 3) * 2048 + t * 128 + (((chunk & 7) ^ (t & 7)) << 4);
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

// Barriers over the NTHR threads (threadIdx.x < NTHR) that run an epilogue: the whole
// CTA, or the consumer warps of a warp-specialised CTA (named barrier 1).
struct CtaBarrier {
  __device__ static __forceinline__ void sync() { __syncthreads(); }
};
template <int NTHR>
struct GroupBarrier {
  __device__ static __forceinline__ void sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NTHR) : "memory");
  }
};

template <typename T, int D, int NTHR>
__device__ void write_empty_row(const EmitCtx &e, int b, int h) {
  const int Hq = e.H * e.G;
  T *out = static_cast<T *>(e.out);
  for (int x = threadIdx.x; x < e.G * D; x += NTHR) {
    const int r = x / D, i = x % D;
    Elem<T>::store(out + (static_cast<int64_t>(b) * Hq + h * e.G + r) * D + i, 0.f);
    if (i == 0 && e.lse != nullptr) e.lse[static_cast<int64_t>(b) * Hq + h * e.G + r] = -INFINITY;
  }
}

// Combine NSTATES warp states (wm: running max in log2 units, wl: sum of weights, wo:
// unnormalised output; state w, query r at wm[w * QMAX + r], wo[(w * QMAX + r) * D + i])
// and emit the row's result: directly when the row has one split, otherwise as a partial,
// the last split to arrive (an atomic counter, nothing waits) merging all partials.  Run
// by the NTHR threads of the barrier group Bar; ends with a Bar::sync().
template <typename T, int D, int NSTATES, int QMAX, int NTHR, typename Bar>
__device__ void combine_and_emit(const EmitCtx &e, int row, int b, int h, int split,
                                 int splits, const float *wm, const float *wl,
                                 const float *wo, int *s_flag) {
  const int G = e.G, Hq = e.H * G;
  T *out = static_cast<T *>(e.out);
  const int64_t obase = static_cast<int64_t>(b) * Hq + h * G;
  const int64_t slot = static_cast<int64_t>(row) * e.max_splits;
  float *po = e.part_o + (slot + split) * G * D;
  float *pml = e.part_ml + (slot + split) * G * 2;
  for (int x = threadIdx.x; x < G * D; x += NTHR) {
    const int r = x / D, i = x % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NSTATES; ++w) M = fmaxf(M, wm[w * QMAX + r]);
    float Ls = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NSTATES; ++w) {
        const float a = exp2f(wm[w * QMAX + r] - M);
        Ls += wl[w * QMAX + r] * a;
        O += wo[(w * QMAX + r) * D + i] * a;
      }
    }
    if (splits == 1) {
      Elem<T>::store(out + (obase + r) * D + i, Ls > 0.f ? O / Ls : 0.f);
      if (i == 0 && e.lse != nullptr) e.lse[obase + r] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    } else {
      po[x] = O;
      if (i == 0) {
        pml[2 * r] = M;
        pml[2 * r + 1] = Ls;
      }
    }
  }
  if (splits == 1) {
    Bar::sync();
    return;
  }
  // One thread publishes the group's partial: the barrier orders the other threads'
  // stores before its release, which is cumulative; its acquire (when it arrives last)
  // makes the other splits' partials visible to the group after the next barrier.
  Bar::sync();
  if (threadIdx.x == 0) *s_flag = atom_add_acq_rel_gpu(&e.counters[row], 1) == splits - 1;
  Bar::sync();
  if (*s_flag) {
    constexpr int kFast = 8;   // splits merged with every load issued up front
    const float *po_row = e.part_o + slot * G * D;
    const float *pml_row = e.part_ml + slot * G * 2;
    for (int x = threadIdx.x; x < G * D; x += NTHR) {
      const int r = x / D, i = x % D;
      float M = -INFINITY, Ls = 0.f, O = 0.f;
      if (splits <= kFast) {
        float ms[kFast], ls[kFast], os[kFast];
#pragma unroll
        for (int s = 0; s < kFast; ++s) {
          ms[s] = s < splits ? __ldcg(pml_row + (s * G + r) * 2) : -INFINITY;
          ls[s] = s < splits ? __ldcg(pml_row + (s * G + r) * 2 + 1) : 0.f;
          os[s] = s < splits ? __ldcg(po_row + static_cast<int64_t>(s) * G * D + x) : 0.f;
        }
#pragma unroll
        for (int s = 0; s < kFast; ++s) M = fmaxf(M, ms[s]);
        if (M != -INFINITY) {
#pragma unroll
          for (int s = 0; s < kFast; ++s) {
            const float a = exp2f(ms[s] - M);
            Ls += ls[s] * a;
            O += os[s] * a;
          }
        }
      } else {
        for (int s = 0; s < splits; ++s) M = fmaxf(M, __ldcg(pml_row + (s * G + r) * 2));
        if (M != -INFINITY) {
          for (int s = 0; s < splits; ++s) {
            const float a = exp2f(__ldcg(pml_row + (s * G + r) * 2) - M);
            Ls += __ldcg(pml_row + (s * G + r) * 2 + 1) * a;
            O += __ldcg(po_row + static_cast<int64_t>(s) * G * D + x) * a;
          }
        }
      }
      Elem<T>::store(out + (obase + r) * D + i, Ls > 0.f ? O / Ls : 0.f);
      if (i == 0 && e.lse != nullptr) e.lse[obase + r] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
    }
  }
  Bar::sync();
}

// Online-softmax state of one warp over pages, in transposed form: per page
//   S^T = K Q^T    (mma M = 16 tokens, N = 8 NT query heads, K = d)
//   O^T += V^T P^T (mma M = 16 dims,   N = 8 NT query heads, K = 16 tokens)
// so a group of up to 8 query heads costs d/16 + d/16 mma per page.  Lane (gq, tq) =
// (lane / 4, lane % 4) holds, per n-tile nt, query heads 8 nt + 2 tq and 8 nt + 2 tq + 1:
// their running max m (log2 units), a partial weight sum l over this lane's tokens, and
// O^T for dims 16 mt + gq and 16 mt + gq + 8.
template <int D, int NT>
struct WarpSoftmaxT {
  static constexpr int kSteps = D / 16;
  float o[kSteps][NT][4];
  float m[NT][2], l[NT][2];

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int mt = 0; mt < kSteps; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
    }
  }

  // One staged page (sK / sV: shared addresses of the swizzled K and V pages); tokens
  // >= ntok are masked.  qb: B fragments of Q^T (load_qT_frags).
  __device__ __forceinline__ void page(const uint32_t (&qb)[kSteps][NT][2], uint32_t sK,
                                       uint32_t sV, int ntok, float scale_log2, int lane) {
    const int gq = lane >> 2, mj = lane >> 3, mr = lane & 7;
    // K as the A operand: matrix j of ldmatrix.x4 = tokens 8 (j & 1) .. +7 and columns
    // 8 (j >> 1) .. +7 of the k-step.
    uint32_t fa[kSteps][4];
#pragma unroll
    for (int ks = 0; ks < kSteps; ++ks)
      ldmatrix_x4(sK + swz_chunk(mr + 8 * (mj & 1), 2 * ks + (mj >> 1)), fa[ks][0], fa[ks][1],
                  fa[ks][2], fa[ks][3]);
    float sc[NT][4], sd[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[nt][c] = sd[nt][c] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kSteps; ks += 2) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16_16816(sc[nt], fa[ks], qb[ks][nt][0], qb[ks][nt][1]);
        mma_bf16_16816(sd[nt], fa[ks + 1], qb[ks + 1][nt][0], qb[ks + 1][nt][1]);
      }
    }
    // V^T as the A operand (transposed loads): matrix j = tokens 8 (j >> 1) .. +7 and
    // dims 16 mt + 8 (j & 1) .. +7.  Independent of the softmax below.
#pragma unroll
    for (int mt = 0; mt < kSteps; ++mt)
      ldmatrix_x4_trans(sV + swz_chunk(mr + 8 * (mj >> 1), 2 * mt + (mj & 1)), fa[mt][0],
                        fa[mt][1], fa[mt][2], fa[mt][3]);
    const bool v0 = gq < ntok, v1 = gq + 8 < ntok;   // tokens gq and gq + 8
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // c0 / c1: token gq, query heads 2tq / 2tq+1; c2 / c3: token gq + 8
      const float s0 = v0 ? (sc[nt][0] + sd[nt][0]) * scale_log2 : -INFINITY;
      const float s1 = v0 ? (sc[nt][1] + sd[nt][1]) * scale_log2 : -INFINITY;
      const float s2 = v1 ? (sc[nt][2] + sd[nt][2]) * scale_log2 : -INFINITY;
      const float s3 = v1 ? (sc[nt][3] + sd[nt][3]) * scale_log2 : -INFINITY;
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);   // over this lane's two tokens
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {              // over the 8 lanes of a column
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
      }
      const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float a0 = exp2f(m[nt][0] - mu0), a1 = exp2f(m[nt][1] - mu1);
      m[nt][0] = mn0;
      m[nt][1] = mn1;
      const uint32_t top = pack_bf16x2(exp2f(s0 - mu0), exp2f(s1 - mu1));   // token gq
      const uint32_t bot = pack_bf16x2(exp2f(s2 - mu0), exp2f(s3 - mu1));   // token gq + 8
      l[nt][0] = l[nt][0] * a0 + (bf16_lo(top) + bf16_lo(bot));
      l[nt][1] = l[nt][1] * a1 + (bf16_hi(top) + bf16_hi(bot));
      if (a0 != 1.f || a1 != 1.f) {
#pragma unroll
        for (int mt = 0; mt < kSteps; ++mt) {
          o[mt][nt][0] *= a0;
          o[mt][nt][1] *= a1;
          o[mt][nt][2] *= a0;
          o[mt][nt][3] *= a1;
        }
      }
      // P (tokens x query heads) -> P^T as the B operand: transpose each 8 x 8 half
      pb[nt][0] = movmatrix_trans(top);   // tokens 2tq, 2tq+1 of query head 8nt + gq
      pb[nt][1] = movmatrix_trans(bot);   // tokens 8 + 2tq, 8 + 2tq + 1
    }
#pragma unroll
    for (int mt = 0; mt < kSteps; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[mt][nt], fa[mt], pb[nt][0], pb[nt][1]);
  }

  // Reduce the partial weight sums over each column's lanes and store the state of the
  // G live query heads: wm / wl [8 NT], wo [8 NT][D].
  __device__ __forceinline__ void store(float *wm, float *wl, float *wo, int lane, int G) {
    const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float s0 = l[nt][0], s1 = l[nt][1];
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, sh);
        s1 += __shfl_xor_sync(0xffffffffu, s1, sh);
      }
      const int q0 = 8 * nt + 2 * tq;
      if (gq == 0) {
        if (q0 < G) {
          wm[q0] = m[nt][0];
          wl[q0] = s0;
        }
        if (q0 + 1 < G) {
          wm[q0 + 1] = m[nt][1];
          wl[q0 + 1] = s1;
        }
      }
#pragma unroll
      for (int mt = 0; mt < kSteps; ++mt) {
        const int d0 = 16 * mt + gq;
        if (q0 < G) {
          wo[q0 * D + d0] = o[mt][nt][0];
          wo[q0 * D + d0 + 8] = o[mt][nt][2];
        }
        if (q0 + 1 < G) {
          wo[(q0 + 1) * D + d0] = o[mt][nt][1];
          wo[(q0 + 1) * D + d0 + 8] = o[mt][nt][3];
        }
      }
    }
  }
};

// B fragments of Q^T for the transposed page step: qb[ks][nt] = (Q[8nt + gq][16ks + 2tq],
// +1) and (Q[8nt + gq][16ks + 8 + 2tq], +1); zero for query heads >= G.
template <int D, int NT>
__device__ __forceinline__ void load_qT_frags(uint32_t (&qb)[D / 16][NT][2],
                                              const __nv_bfloat16 *qg, int G, int lane) {
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int qrow = 8 * nt + gq;
      const unsigned int *src =
          reinterpret_cast<const unsigned int *>(qg + qrow * D + 16 * ks + 2 * tq);
      qb[ks][nt][0] = qrow < G ? __ldg(src) : 0u;
      qb[ks][nt][1] = qrow < G ? __ldg(src + 4) : 0u;
    }
}

constexpr size_t combine_smem_bytes(int D) {
  return static_cast<size_t>(kWarps) * kMaxGroup * (D + 2) * sizeof(float);
}

}  // namespace kin
