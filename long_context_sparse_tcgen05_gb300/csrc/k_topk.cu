// Per-row top-k over materialised fp32 score rows: an exact radix select on the
// order-preserving 32-bit keys of the scores (three histogram passes of 11, 11 and 10
// bits in shared memory), then one stable compaction pass that writes the selected
// positions in ascending order.  Ties at the k-th key go to the lowest positions.
//
// One 1024-thread CTA owns one row.  The row is re-read once per pass; between passes it
// stays in L2 (a resident CTA's row is at most 4 MB and usually far less), so DRAM sees
// roughly one read of the scores.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kPerThread = 4;  // consecutive scores per thread per sweep

struct TopkSmem {
  uint32_t hist[kBins];
  uint32_t warp_sums[kWarps];
  uint32_t sel_bin, sel_above;
};

// Exclusive block-wide prefix sum; *total receives the block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_sums,
                                                    uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const uint32_t base = wid > 0 ? warp_sums[wid - 1] : 0u;
  *total = warp_sums[kWarps - 1];
  __syncthreads();
  return base + x - v;
}

// Warp 0: find the bin b (scanning from the top) with above(b) < need <= above(b)+hist[b].
__device__ __forceinline__ void select_bin(TopkSmem& sm, uint32_t need) {
  const int lane = threadIdx.x;
  const int hi = kBins - 64 * lane, lo = hi - 64;
  uint32_t s = 0;
  for (int b = lo; b < hi; ++b) s += sm.hist[b];
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t above = incl - s;
  if (above < need && need <= incl) {
    uint32_t acc = above;
    for (int b = hi - 1; b >= lo; --b) {
      const uint32_t h = sm.hist[b];
      if (acc + h >= need) {
        sm.sel_bin = (uint32_t)b;
        sm.sel_above = acc;
        break;
      }
      acc += h;
    }
  }
}

__device__ __forceinline__ void load4(const float* x, int64_t p, int64_t n, bool vec, float v[4]) {
  if (vec && p + 3 < n) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(x + p));
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = (p + j < n) ? __ldg(x + p + j) : 0.f;
  }
}

__global__ void __launch_bounds__(kThreads, 1) k_topk_rows(TopkLaunch p) {
  __shared__ TopkSmem sm;
  const int row = blockIdx.x;
  const int b = row / p.Tc, tl = row % p.Tc, t = p.t0 + tl;
  const float* x = p.scores + (int64_t)b * p.bstride + (int64_t)tl * p.ld;
  int32_t* out = p.idx + ((int64_t)b * p.T + t) * p.k;
  int64_t n = p.q_pos0 + t + p.diag;
  n = n < 0 ? 0 : (n > p.S ? p.S : n);
  const int k = p.k;

  if (n <= k) {
    for (int j = threadIdx.x; j < k; j += kThreads) out[j] = j < n ? j : -1;
    return;
  }
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;

  uint32_t prefix = 0, pmask = 0, need = (uint32_t)k;
  bool saw_nan = false;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t wmask = pass == 2 ? 0x3ffu : 0x7ffu;
    for (int i = threadIdx.x; i < kBins; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    for (int64_t q = (int64_t)threadIdx.x * kPerThread; q < n; q += (int64_t)kThreads * kPerThread) {
      float v[4];
      load4(x, q, n, vec, v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (q + j >= n) break;
        const uint32_t key = score_key(v[j]);
        if (pass == 0 && isnan(v[j])) saw_nan = true;
        if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & wmask], 1u);
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) select_bin(sm, need);
    __syncthreads();
    prefix |= sm.sel_bin << shift;
    pmask |= wmask << shift;
    need -= sm.sel_above;
    __syncthreads();
  }
  if (saw_nan) atomicOr(p.flags, DSA_FLAG_NAN_SCORE);
  const uint32_t tau = prefix;  // key of the k-th largest score
  // `need` ties (key == tau) are taken, lowest positions first; all keys > tau are taken.

  uint32_t out_base = 0, eq_seen = 0;
#pragma unroll 1
  for (int64_t base = 0; base < n; base += (int64_t)kThreads * kPerThread) {
    const int64_t q = base + (int64_t)threadIdx.x * kPerThread;
    float v[4];
    load4(x, q, n, vec, v);
    uint32_t key[4];
    uint32_t cg = 0, ce = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool valid = q + j < n;
      key[j] = score_key(v[j]);
      cg += (valid && key[j] > tau);
      ce += (valid && key[j] == tau);
    }
    uint32_t tot;
    const uint32_t ex = block_excl_scan((cg << 16) | ce, sm.warp_sums, &tot);
    const uint32_t gt_before = ex >> 16, eq_before = ex & 0xffffu;
    const uint32_t gt_tot = tot >> 16, eq_tot = tot & 0xffffu;
    const uint32_t rem = need > eq_seen ? need - eq_seen : 0u;  // ties still to take
    uint32_t pos = out_base + gt_before + (eq_before < rem ? eq_before : rem);
    uint32_t eq_idx = eq_seen + eq_before;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (q + j >= n) break;
      if (key[j] > tau) {
        out[pos++] = (int32_t)(q + j);
      } else if (key[j] == tau) {
        if (eq_idx < need) out[pos++] = (int32_t)(q + j);
        ++eq_idx;
      }
    }
    out_base += gt_tot + (eq_tot < rem ? eq_tot : rem);
    eq_seen += eq_tot;
    if (out_base >= (uint32_t)k) break;
  }
}

}  // namespace

cudaError_t launch_topk_rows(const TopkLaunch& p, cudaStream_t st) {
  const int rows = p.B * p.Tc;
  if (rows <= 0) return cudaSuccess;
  k_topk_rows<<<rows, kThreads, 0, st>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
