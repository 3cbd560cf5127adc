// Block centroid (mean key) kernel.
//
// Block top-k ranks each key block by the mean of its key vectors (Pith review of
// "Kinetics: Rethinking Test-Time Scaling Laws", section "What carries the argument").
// One block is one 16-token KV page (Kinetics README, "Benchmark Block TopK Attention
// throughput").
//
// c[p, h, :] = (sum_{t=0..15} K[p, h, t, :]) * (1/16), summed in fp32 in ascending t.
// fp32 caches store c.  bf16 caches store two bf16 codes per element in two planes of the
// table: plane 0 holds c rounded to bf16 (round-to-nearest-even), plane 1 the residual
// c - plane 0 (exact in fp32) rounded to bf16, so that plane 0 + plane 1 is c to about
// 2^-16 of its size.  HBM-bound: 16*d elements in, d (fp32) or 2d (bf16) out per
// (page, head).  Each thread owns one 16-byte column slice of the page and
// walks the 16 rows, so every element is accumulated by one thread in token order; the
// 16 row loads are issued back to back for memory-level parallelism.
#include "kin_common.cuh"
#include "kin_internal.h"

namespace kin {
namespace {

template <typename T, int D>
__global__ void __launch_bounds__(256) centroid_kernel(const T *__restrict__ k_pages,
                                                       const int32_t *__restrict__ page_ids,
                                                       int64_t n, int H, int64_t num_pages,
                                                       T *__restrict__ cents,
                                                       int32_t *__restrict__ err) {
  constexpr int kVec = Elem<T>::kVec;        // elements per 16-byte slice
  constexpr int kTpi = D / kVec;              // threads per (page, head) item
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t item = gtid / kTpi;
  const int slice = static_cast<int>(gtid % kTpi);
  if (item >= n * H) return;
  const int64_t idx = item / H;
  const int h = static_cast<int>(item % H);
  const int64_t page = page_ids != nullptr ? static_cast<int64_t>(page_ids[idx]) : idx;
  if (page < 0 || page >= num_pages) {
    if (slice == 0 && h == 0) flag_error(err, KIN_DEVERR_PAGE_ID);
    return;
  }
  const T *base = k_pages + ((page * H + h) * kBlock) * D + slice * kVec;
  uint4 rows[kBlock];
#pragma unroll
  for (int t = 0; t < kBlock; ++t) rows[t] = ldg_stream(base + t * D);
  float acc[kVec], f[kVec];
  Elem<T>::unpack(rows[0], acc);
#pragma unroll
  for (int t = 1; t < kBlock; ++t) {
    Elem<T>::unpack(rows[t], f);
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
  }
#pragma unroll
  for (int i = 0; i < kVec; ++i) acc[i] = __fmul_rn(acc[i], 1.0f / kBlock);
  T *dst = cents + (page * H + h) * D + slice * kVec;
  const uint4 code = Elem<T>::pack(acc);
  *reinterpret_cast<uint4 *>(dst) = code;
  if constexpr (sizeof(T) == 2) {
    // plane 1: the residual of the rounding, itself rounded to bf16
    float hi[kVec];
    Elem<T>::unpack(code, hi);
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = __fsub_rn(acc[i], hi[i]);
    *reinterpret_cast<uint4 *>(dst + num_pages * H * D) = Elem<T>::pack(acc);
  }
}

template <typename T, int D>
cudaError_t launch_t(int H, const void *k_pages, int64_t num_pages, const int32_t *page_ids,
                     int64_t n, void *cents, int32_t *err, cudaStream_t stream) {
  constexpr int kTpi = D / Elem<T>::kVec;
  const int64_t threads = n * H * kTpi;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  if (grid == 0) return cudaSuccess;
  centroid_kernel<T, D><<<static_cast<unsigned>(grid), block, 0, stream>>>(
      static_cast<const T *>(k_pages), page_ids, n, H, num_pages, static_cast<T *>(cents), err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_centroids(kin_dtype dtype, int head_dim, int num_kv_heads,
                             const void *k_pages, int64_t num_pages, const int32_t *page_ids,
                             int64_t n, void *centroids, int32_t *err, cudaStream_t stream) {
  if (dtype == KIN_BF16) {
    if (head_dim == 128)
      return launch_t<__nv_bfloat16, 128>(num_kv_heads, k_pages, num_pages, page_ids, n,
                                          centroids, err, stream);
    return launch_t<__nv_bfloat16, 64>(num_kv_heads, k_pages, num_pages, page_ids, n,
                                       centroids, err, stream);
  }
  if (head_dim == 128)
    return launch_t<float, 128>(num_kv_heads, k_pages, num_pages, page_ids, n, centroids, err,
                                stream);
  return launch_t<float, 64>(num_kv_heads, k_pages, num_pages, page_ids, n, centroids, err,
                             stream);
}

}  // namespace kin
