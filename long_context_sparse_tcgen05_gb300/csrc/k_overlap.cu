// Overlap of two index buffers, row by row: |A_r and B_r| / |A_r| over the valid (>= 0)
// entries.  Rows are ascending lists of valid positions followed by -1 padding (the form
// dsa_topk writes), so one warp per row binary-searches every entry of A_r in B_r.  A row
// that is not ascending raises DSA_FLAG_UNSORTED.  The mean over rows is a single-CTA
// reduction in double, in a fixed order (deterministic).
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kWarpsPerCta = 8;

// Length of the valid prefix of an index row (entries >= 0 come first).
__device__ __forceinline__ int valid_len(const int32_t* r, int k) {
  int lo = 0, hi = k;  // first index with r[i] < 0
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(r + mid) >= 0) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32) k_topk_overlap(const int32_t* a, const int32_t* b,
                                                                    int rows, int k, float* per_row,
                                                                    uint32_t* flags) {
  const int warp = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int32_t* ra = a + (int64_t)warp * k;
  const int32_t* rb = b + (int64_t)warp * k;
  const int na = valid_len(ra, k), nb = valid_len(rb, k);
  int common = 0;
  bool unsorted = false;
  for (int j = lane; j < na; j += 32) {
    const int32_t x = __ldg(ra + j);
    if (j + 1 < na && __ldg(ra + j + 1) <= x) unsorted = true;
    if (j + 1 < nb && __ldg(rb + j + 1) <= __ldg(rb + j)) unsorted = true;
    int lo = 0, hi = nb;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(rb + mid) < x) lo = mid + 1; else hi = mid;
    }
    common += (lo < nb && __ldg(rb + lo) == x);
  }
  for (int j = na + lane; j + 1 < nb; j += 32)
    if (__ldg(rb + j + 1) <= __ldg(rb + j)) unsorted = true;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) common += __shfl_xor_sync(0xffffffffu, common, o);
  if (__any_sync(0xffffffffu, unsorted) && lane == 0) atomicOr(flags, DSA_FLAG_UNSORTED);
  if (lane == 0) per_row[warp] = na == 0 ? 1.f : (float)((double)common / (double)na);
}

// Mean of per_row in double: each thread sums a strided slice, then a fixed-order tree.
__global__ void __launch_bounds__(1024) k_mean(const float* per_row, int rows, double* out) {
  __shared__ double part[1024];
  double s = 0.0;
  for (int i = threadIdx.x; i < rows; i += 1024) s += (double)per_row[i];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = rows > 0 ? part[0] / (double)rows : 1.0;
}

}  // namespace

cudaError_t launch_topk_overlap(const int32_t* a, const int32_t* b, int rows, int k,
                                float* per_row, double* mean_dev, uint32_t* flags,
                                cudaStream_t st) {
  TraceScope trace(kTraceOverlap, st);
  if (rows > 0) {
    const int ctas = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
    k_topk_overlap<<<ctas, kWarpsPerCta * 32, 0, st>>>(a, b, rows, k, per_row, flags);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  k_mean<<<1, 1024, 0, st>>>(per_row, rows, mean_dev);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
