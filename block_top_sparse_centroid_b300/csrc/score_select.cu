// Group scoring of candidate blocks and top-k block selection as standalone kernels,
// used for fp32 caches (bf16 caches score and select inside the fused decode kernel).
//
// Block top-k ranks key blocks by their mean key vectors and keeps, for each GQA query
// group, only the k best blocks (Pith review of "Kinetics: Rethinking Test-Time Scaling
// Laws", section "What carries the argument"); k is counted in 16-token pages (Kinetics
// README, "Benchmark Block TopK Attention throughput", --topk_page).
//
// score:  s[b,h,j] = sum_g q[b,hG+g,:] . c[page(b,j),h,:]   for j < nb-1  (fp32)
//         computed as (sum_g q_g) . c_j: the group sum of the query is formed once per
//         row, so every candidate costs one d-long dot product.  HBM-bound on the
//         centroid reads (d * esize bytes per candidate); one 16-byte vector per lane,
//         a d-wide centroid spread over d/vec lanes and reduced with xor shuffles.
// select: per row keep {nb-1} plus the k-1 largest scores of blocks 0..nb-2, ties to
//         the lower block index, emitted ascending; rows with nb <= k keep every block.
//         One CTA per row: radix select over order-preserving 32-bit keys in shared
//         memory (4 passes of 8 bits), then an index-ordered compaction.
#include "kin_common.cuh"
#include "kin_internal.h"

namespace kin {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreUnroll = 4;
constexpr int kSelectThreads = 512;

template <typename T, int D>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(ScoreParams p) {
  constexpr int kVec = Elem<T>::kVec;
  constexpr int kTpi = D / kVec;                 // lanes per centroid (8, 16 or 32)
  constexpr int kGroups = kScoreThreads / kTpi;  // centroids per CTA per unrolled slot
  const int row = blockIdx.y;
  const int b = row / p.num_kv_heads, h = row % p.num_kv_heads;
  const int L = p.seq_lens[b];
  if (L < 1 || L > kBlock * p.max_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && h == 0) flag_error(p.err, KIN_DEVERR_SEQ_LEN);
    return;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  if (nb <= p.top_k) return;                     // every block is kept: nothing to score
  const int n = nb - 1;
  const int j0 = blockIdx.x * p.chunk;
  if (j0 >= n) return;
  const int j1 = min(n, j0 + p.chunk);
  const int grp = threadIdx.x / kTpi, slice = threadIdx.x % kTpi;
  const int G = p.group;
  const T *q = static_cast<const T *>(p.q);
  const T *cents = static_cast<const T *>(p.centroids);
  const int32_t *trow = p.block_table + static_cast<int64_t>(b) * p.max_blocks;

  // Group-summed query slice, fp32, ascending g.
  float qs[kVec], f[kVec];
  const T *qrow = q + (static_cast<int64_t>(b) * p.num_kv_heads * G + h * G) * D + slice * kVec;
  Elem<T>::unpack(*reinterpret_cast<const uint4 *>(qrow), qs);
  for (int g = 1; g < G; ++g) {
    Elem<T>::unpack(*reinterpret_cast<const uint4 *>(qrow + g * D), f);
#pragma unroll
    for (int i = 0; i < kVec; ++i) qs[i] += f[i];
  }

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
        const int64_t page = trow[jj[u]];
        if (page >= 0 && page < p.num_pages) {
          valid[u] = true;
          v[u] = ldg_stream(cents + (page * p.num_kv_heads + h) * D + slice * kVec);
        } else if (slice == 0) {
          flag_error(p.err, KIN_DEVERR_PAGE_ID);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kScoreUnroll; ++u) {
      Elem<T>::unpack(v[u], f);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < kVec; ++i) s = fmaf(qs[i], f[i], s);
#pragma unroll
      for (int o = kTpi / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (slice == 0 && jj[u] < j1) srow[jj[u]] = valid[u] ? s : -INFINITY;
    }
  }
}

// Order-preserving map of a float score to an unsigned key (larger score, larger key).
// -0 is folded onto +0 so that the two compare equal, as real numbers do; NaN maps
// below every number.
__device__ __forceinline__ uint32_t score_key(float s) {
  if (s != s) return 0u;
  s = s + 0.0f;
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kSelectThreads) select_kernel(ScoreParams p) {
  extern __shared__ uint32_t keys[];            // [max_blocks]
  __shared__ int hist[256];
  __shared__ int scan_tmp[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  const int row = blockIdx.x;
  const int b = row / p.num_kv_heads;
  const int k = p.top_k;
  int32_t *out = p.sel + static_cast<int64_t>(row) * k;
  const int L = p.seq_lens[b];
  const int tid = threadIdx.x, nt = blockDim.x;
  if (L < 1 || L > kBlock * p.max_blocks) {
    for (int i = tid; i < k; i += nt) out[i] = -1;
    return;
  }
  const int nb = (L + kBlock - 1) / kBlock;
  if (nb <= k) {
    for (int i = tid; i < k; i += nt) out[i] = i < nb ? i : -1;
    return;
  }
  const int n = nb - 1;          // scored candidates 0..n-1
  const int m = k - 1;           // how many of them to keep
  if (m == 0) {
    if (tid == 0) out[0] = nb - 1;
    return;
  }
  const float *srow = p.scores + static_cast<int64_t>(row) * p.max_blocks;
  for (int j = tid; j < n; j += nt) keys[j] = score_key(srow[j]);
  if (tid == 0) { s_prefix = 0u; s_remaining = m; }
  __syncthreads();

  // Radix select of the m-th largest key, 8 bits per pass from the top.
  uint32_t mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += nt) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int j = tid; j < n; j += nt) {
      const uint32_t key = keys[j];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    // Thread t looks at digit 255-t: inclusive count of digits >= 255-t.
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
  const uint32_t thr = s_prefix;        // key of the m-th largest score
  const int take_eq = s_remaining;      // how many keys equal to thr are kept (>= 1)

  // Index-ordered compaction: each thread owns a contiguous run of candidates.
  const int per = (n + nt - 1) / nt;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int gt = 0, eq = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = keys[j];
    gt += key > thr;
    eq += key == thr;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, scan_tmp, &tot);
  const int my_eq = max(0, min(eq, take_eq - eq_before));
  const int pos = block_exclusive_scan(gt + my_eq, scan_tmp, &tot);
  int w = pos, used_eq = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = keys[j];
    bool keep = key > thr;
    if (key == thr && used_eq < my_eq) { keep = true; ++used_eq; }
    if (keep) out[w++] = j;
  }
  if (tid == 0) out[m] = nb - 1;         // the final block, largest id, goes last
}

template <typename T, int D>
cudaError_t launch_score_t(const ScoreParams &p, cudaStream_t stream) {
  const int rows = p.batch * p.num_kv_heads;
  const int chunks = (p.max_blocks + p.chunk - 1) / p.chunk;
  dim3 grid(chunks, rows);
  score_kernel<T, D><<<grid, kScoreThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score(kin_dtype dtype, int head_dim, const ScoreParams &p,
                         cudaStream_t stream) {
  if (dtype != KIN_F32) return cudaErrorInvalidValue;  // bf16 scores in the fused kernel
  return head_dim == 128 ? launch_score_t<float, 128>(p, stream)
                         : launch_score_t<float, 64>(p, stream);
}

cudaError_t launch_select(const ScoreParams &p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(p.max_blocks) * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  select_kernel<<<p.batch * p.num_kv_heads, kSelectThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kin
