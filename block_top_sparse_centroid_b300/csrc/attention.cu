// fp32 split-KV paged decode attention (CUDA cores) over a list of kept blocks (block
// top-k) or over every block (dense); the split merge goes through the last-arriver
// epilogue of attn_common.cuh.  bf16 caches use the fused tensor-core kernel instead.
//
// Grid = (splits, rows).  A CTA takes a contiguous run of the row's block list; its 4
// warps take every 4th block of the run.  One lane owns d/32 dimensions; per token each
// warp forms q_g . k_t for the group's query heads with a butterfly reduction and updates
// its online softmax (exact fp32 arithmetic, exp2 in log2 units).
#include "attn_common.cuh"
#include "kin_internal.h"

namespace kin {
namespace {

template <int D>
__global__ void __launch_bounds__(kThreads) attn_f32_kernel(const AttnParams p) {
  constexpr int kPer = D / 32;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_page[kMaxItems], s_ntok[kMaxItems];
  __shared__ int s_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.num_kv_heads, G = p.group;
  const int row = blockIdx.y, split = blockIdx.x;
  const int b = row / H, h = row % H;
  const EmitCtx ec{p.out, p.lse, p.part_o, p.part_ml, p.counters, p.max_splits, G, H};
  const int L = p.seq_lens[b];
  if (L < 1 || L > kBlock * p.max_blocks) {
    if (split == 0) {
      write_empty_row<float, D, kThreads>(ec, b, h);
      if (tid == 0 && h == 0) flag_error(p.err, KIN_DEVERR_SEQ_LEN);
    }
    return;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  const int n_items = p.sel != nullptr ? min(nb, p.sel_stride) : nb;
  const int splits = (n_items + p.items_per_split - 1) / p.items_per_split;
  if (split >= splits) return;
  const int i0 = split * p.items_per_split;
  const int cnt = min(n_items, i0 + p.items_per_split) - i0;
  for (int i = tid; i < cnt; i += kThreads) {
    const int j = p.sel != nullptr ? p.sel[static_cast<int64_t>(row) * p.sel_stride + i0 + i] : i0 + i;
    int page = -1, ntok = 0;
    if (j >= 0 && j < nb) {
      const int pg = p.block_table[static_cast<int64_t>(b) * p.max_blocks + j];
      if (pg >= 0 && pg < p.num_pages) {
        page = pg;
        ntok = min(kBlock, L - kBlock * j);
      } else {
        flag_error(p.err, KIN_DEVERR_PAGE_ID);
      }
    }
    s_page[i] = page;
    s_ntok[i] = ntok;
  }
  __syncthreads();

  const float *qg = static_cast<const float *>(p.q) + (static_cast<int64_t>(b) * H * G + h * G) * D;
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
  const bool append = p.append_final != 0 && (L % kBlock) == 0 && split == splits - 1;
  for (int it = warp; it < cnt; it += kWarps) {
    const int page = s_page[it], ntok = s_ntok[it];
    if (page < 0) continue;
    const int64_t base = (static_cast<int64_t>(page) * H + h) * kBlock * D;
    if (append && it == cnt - 1) {
      // The final block just became complete: its centroid (fp32 sum over the 16
      // tokens in order, times 1/16).
      float c[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) c[i] = kp[base + lane * kPer + i];
      for (int t = 1; t < kBlock; ++t) {
#pragma unroll
        for (int i = 0; i < kPer; ++i) c[i] = __fadd_rn(c[i], kp[base + t * D + lane * kPer + i]);
      }
      float *dst = static_cast<float *>(p.cent_out) + (static_cast<int64_t>(page) * H + h) * D + lane * kPer;
#pragma unroll
      for (int i = 0; i < kPer; ++i) dst[i] = __fmul_rn(c[i], 1.0f / kBlock);
    }
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
  combine_and_emit<float, D, kWarps, kMaxGroup, kThreads, CtaBarrier>(ec, row, b, h, split, splits, wm, wl, wo, &s_flag);
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

cudaError_t launch_attention_f32(int head_dim, const AttnParams &p, cudaStream_t stream) {
  return head_dim == 128 ? launch_f32<128>(p, stream) : launch_f32<64>(p, stream);
}

}  // namespace kin
