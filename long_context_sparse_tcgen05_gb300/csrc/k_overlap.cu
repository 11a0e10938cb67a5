// Overlap of two index buffers, row by row: |A_r and B_r| / |A_r| over the valid (>= 0)
// entries.  Rows are ascending lists of valid positions followed by -1 padding (the form
// dsa_topk writes), so one warp per row binary-searches every entry of A_r in B_r.  A row
// that is not ascending raises DSA_FLAG_UNSORTED.  The mean over rows is a single-CTA
// reduction in double, in a fixed order (deterministic).
//
// The all-pairs form (the layer-overlap heatmap of an all-F pass, IndexCache notes,
// section 2) takes n buffers of the same query rows.  One CTA holds a row of every buffer in
// shared memory; each warp takes whole pairs (i < j) and each lane a contiguous run of the
// shorter list, found in the other list by one binary search and then a forward walk (both
// lists ascend).  A row of each buffer arrives by cp.async, word by word.  Lists are stored with one pad word per 64 entries, so the lanes' runs of 64
// start in different banks.  Per-row fractions |A_i and A_j| / |A_i| are summed in double by
// the thread that owns the ordered pair (i, j); per-CTA sums are reduced in a fixed order.
#include <algorithm>

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

// --- all pairs ---------------------------------------------------------------------

constexpr int kMatThreads = 1024;
constexpr int kMatWarps = kMatThreads / 32;

__device__ __forceinline__ int padded(int e) { return e + (e >> 6); }

__device__ __forceinline__ int lower_bound_padded(const int32_t* l, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (l[padded(mid)] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kMatThreads) k_overlap_matrix(OverlapMatrixLaunch p) {
  extern __shared__ __align__(16) int32_t lists[];  // n lists of padded(k) + 1 words
  __shared__ int vlen[kMaxOverlapLayers];
  __shared__ int cnt[kMaxOverlapLayers * kMaxOverlapLayers];  // |A_i and A_j| for i < j at i*16+j
  __shared__ uint8_t pair_i[kMaxOverlapLayers * (kMaxOverlapLayers - 1) / 2];
  __shared__ uint8_t pair_j[kMaxOverlapLayers * (kMaxOverlapLayers - 1) / 2];
  const int n = p.n, k = p.k, nn = n * n, npairs = n * (n - 1) / 2;
  const int stride = padded(k) + 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    int q = 0;
    for (int i = 0; i < n; ++i)
      for (int j = i + 1; j < n; ++j) {
        pair_i[q] = (uint8_t)i;
        pair_j[q] = (uint8_t)j;
        ++q;
      }
  }
  double acc = 0.0;  // sum over this CTA's rows of the fraction of ordered pair threadIdx.x
  bool unsorted = false;
  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
    // the row of every buffer, copied asynchronously word by word (rows need not be 16-byte
    // aligned), then one wait
    for (int i = 0; i < n; ++i) {
      const int32_t* src = p.bufs[i] + row * k;
      const uint32_t dst = (uint32_t)__cvta_generic_to_shared(lists + i * stride);
      for (int j = threadIdx.x; j < k; j += kMatThreads)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst + 4u * (uint32_t)padded(j)),
                     "l"(src + j)
                     : "memory");
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    __syncthreads();
    // the previous row's counts were read before the barrier above
    for (int t = threadIdx.x; t < kMaxOverlapLayers * kMaxOverlapLayers; t += kMatThreads) cnt[t] = 0;
    if (threadIdx.x < n) {
      const int32_t* l = lists + threadIdx.x * stride;
      int lo = 0, hi = k;  // first padding entry: valid entries come first
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (l[padded(mid)] >= 0) lo = mid + 1; else hi = mid;
      }
      vlen[threadIdx.x] = lo;
    }
    // form check: ascending valid entries, then only padding
    for (int i = 0; i < n; ++i) {
      const int32_t* l = lists + i * stride;
      for (int j = threadIdx.x; j + 1 < k; j += kMatThreads) {
        const int32_t a = l[padded(j)], b = l[padded(j + 1)];
        if (b >= 0 && (a < 0 || b <= a)) unsorted = true;
      }
    }
    __syncthreads();
    for (int q = warp; q < npairs; q += kMatWarps) {
      int i = pair_i[q], j = pair_j[q];
      // walk the shorter list through the longer one
      const int32_t* la = lists + i * stride;
      const int32_t* lb = lists + j * stride;
      int na = vlen[i], nb = vlen[j];
      if (nb < na) {
        const int32_t* t = la; la = lb; lb = t;
        const int u = na; na = nb; nb = u;
      }
      const int run = (na + 31) >> 5;
      const int e0 = lane * run, e1 = min(na, e0 + run);
      int c = 0;
      if (e0 < e1) {
        // merge walk without branches: advance the smaller side (both on a match)
        int b = lower_bound_padded(lb, nb, la[padded(e0)]), e = e0;
        while (e < e1 && b < nb) {
          const int32_t x = la[padded(e)], y = lb[padded(b)];
          c += x == y;
          e += x <= y;
          b += y <= x;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (lane == 0) cnt[i * kMaxOverlapLayers + j] = c;
    }
    __syncthreads();
    if ((int)threadIdx.x < nn) {
      const int i = threadIdx.x / n, j = threadIdx.x - i * n;
      const int c = i == j ? vlen[i] : cnt[min(i, j) * kMaxOverlapLayers + max(i, j)];
      acc += vlen[i] == 0 ? 1.0 : (double)c / (double)vlen[i];
      if (p.counts) p.counts[row * nn + threadIdx.x] = c;
    }
  }
  if (__syncthreads_or(unsorted) && threadIdx.x == 0) atomicOr(p.flags, DSA_FLAG_UNSORTED);
  if ((int)threadIdx.x < nn) p.part[(int64_t)blockIdx.x * nn + threadIdx.x] = acc;
}

// matrix[t] = (sum over CTAs, in CTA order, of part[c][t]) / rows; 1 everywhere for no rows
__global__ void __launch_bounds__(256) k_overlap_matrix_mean(const double* part, int ctas, int nn,
                                                             int64_t rows, double* matrix) {
  const int t = threadIdx.x;
  if (t >= nn) return;
  double s = 0.0;
  for (int c = 0; c < ctas; ++c) s += part[(int64_t)c * nn + t];
  matrix[t] = rows > 0 ? s / (double)rows : 1.0;
}

int device_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

size_t overlap_matrix_smem(int n, int k) {
  return (size_t)n * ((size_t)k + ((size_t)k >> 6) + 1) * sizeof(int32_t);
}

cudaError_t launch_overlap_matrix(const OverlapMatrixLaunch& p, double* matrix_dev, cudaStream_t st) {
  TraceScope trace(kTraceOverlap, st);
  const size_t smem = overlap_matrix_smem(p.n, p.k);
  int ctas = 0;
  if (p.rows > 0) {
    cudaError_t e = cudaFuncSetAttribute(k_overlap_matrix, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_overlap_matrix, kMatThreads, smem);
    if (e != cudaSuccess) return e;
    const int64_t want = (int64_t)device_sms() * (per_sm > 0 ? per_sm : 1);
    ctas = (int)std::min<int64_t>(std::min<int64_t>(p.rows, want), kMaxOverlapCtas);
    k_overlap_matrix<<<ctas, kMatThreads, smem, st>>>(p);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  k_overlap_matrix_mean<<<1, 256, 0, st>>>(p.part, ctas, p.n * p.n, p.rows, matrix_dev);
  count_launches(1);
  return cudaGetLastError();
}

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
