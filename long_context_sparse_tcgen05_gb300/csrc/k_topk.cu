// Per-row top-k over materialised fp32 score rows, exact, ties to the lower position, output
// in ascending position order.
//
// One 512-thread CTA owns one row (two CTAs per SM).  Scores are compared through their
// order-preserving 32-bit keys.
//   * Rows with at most kCap visible scores are copied to shared memory whole.
//   * Longer rows: a sample of at most kSampleMax keys (whole 8-key groups, evenly strided)
//     gives, by an exact radix select
//     in shared memory, a threshold theta that about 1.25k of the row's keys exceed; one
//     streaming pass then appends every key >= theta, in position order (block-wide prefix
//     sums of warp ballots), to shared memory.  Every key below theta has at least k larger
//     keys, so the row's top-k lies among the candidates.
//   * An exact radix select (11/11/10-bit histograms) among the candidates finds the k-th key;
//     a stable compaction writes the selected positions in order.
// If the sample misjudges the threshold (fewer than k candidates, or more than fit), the CTA
// falls back to three histogram passes over the row in global memory and a final ordered
// compaction pass.  Either way DRAM sees about one read of the row.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kCap = 8192;         // candidates held in shared memory
constexpr int kSampleMax = 8192;   // sampled keys of a long row
constexpr int kPer = 8;            // consecutive scores per thread per streaming step

struct TopkSmem {
  uint32_t key[kCap];
  int32_t pos[kCap];
  uint32_t hist[kBins];
  uint32_t warp_sums[kWarps];
  uint32_t sel_bin, sel_above;
};

// Exclusive block-wide prefix sum; *total receives the block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = lane < kWarps ? warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kWarps) warp_sums[lane] = s;
  }
  __syncthreads();
  const uint32_t base = wid > 0 ? warp_sums[wid - 1] : 0u;
  *total = warp_sums[kWarps - 1];
  __syncthreads();
  return base + x - v;
}

// Warp 0: the bin b (scanning from the top) with above(b) < need <= above(b) + hist[b].
__device__ __forceinline__ void select_bin(TopkSmem& sm, uint32_t need) {
  const int lane = threadIdx.x;
  const int hi = kBins - 64 * lane, lo = hi - 64;
  uint32_t s = 0;
  for (int b = lo; b < hi; ++b) s += sm.hist[b];
  uint32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
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

// The need-th largest key (need >= 1) among keys delivered by get(i), i < n, by three
// histogram passes.  Returns the key; *ties receives how many keys equal to it are taken.
template <class Get>
__device__ uint32_t radix_select(TopkSmem& sm, int64_t n, uint32_t need, Get get, uint32_t* ties) {
  uint32_t prefix = 0, pmask = 0;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t wmask = pass == 2 ? 0x3ffu : 0x7ffu;
    for (int i = threadIdx.x; i < kBins; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = get(i);
      if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & wmask], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) select_bin(sm, need);
    __syncthreads();
    prefix |= sm.sel_bin << shift;
    pmask |= wmask << shift;
    need -= sm.sel_above;
    __syncthreads();
  }
  *ties = need;
  return prefix;
}

__device__ __forceinline__ void load8(const float* x, int64_t q, int64_t n, bool vec, float v[kPer]) {
  if (vec && q + kPer <= n) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(x + q));
    const float4 b = __ldg(reinterpret_cast<const float4*>(x + q + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < kPer; ++j) v[j] = (q + j < n) ? __ldg(x + q + j) : 0.f;
  }
}

// Stable ordered compaction: writes out[0..k) with the positions of the entries whose key is
// > tau, plus the first `ties` entries whose key == tau, in stream order.  get(i) gives
// (key, position) of entry i < n.
template <class Get>
__device__ void ordered_output(TopkSmem& sm, int64_t n, uint32_t tau, uint32_t ties, int k, int32_t* out, Get get) {
  uint32_t out_base = 0, eq_seen = 0;
#pragma unroll 1
  for (int64_t base = 0; base < n; base += (int64_t)kThreads * kPer) {
    const int64_t q = base + (int64_t)threadIdx.x * kPer;
    uint32_t key[kPer];
    int32_t ps[kPer];
    uint32_t cg = 0, ce = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const bool valid = q + j < n;
      get(valid ? q + j : 0, key[j], ps[j]);
      cg += (valid && key[j] > tau);
      ce += (valid && key[j] == tau);
      if (!valid) key[j] = 0, ps[j] = -1;
    }
    uint32_t tot;
    const uint32_t ex = block_excl_scan((cg << 16) | ce, sm.warp_sums, &tot);
    const uint32_t gt_before = ex >> 16, eq_before = ex & 0xffffu;
    const uint32_t gt_tot = tot >> 16, eq_tot = tot & 0xffffu;
    const uint32_t rem = ties > eq_seen ? ties - eq_seen : 0u;
    uint32_t o = out_base + gt_before + (eq_before < rem ? eq_before : rem);
    uint32_t eq_idx = eq_seen + eq_before;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (ps[j] < 0) continue;
      if (key[j] > tau) {
        out[o++] = ps[j];
      } else if (key[j] == tau) {
        if (eq_idx < ties) out[o++] = ps[j];
        ++eq_idx;
      }
    }
    out_base += gt_tot + (eq_tot < rem ? eq_tot : rem);
    eq_seen += eq_tot;
    if (out_base >= (uint32_t)k) break;
  }
}

__global__ void __launch_bounds__(kThreads, 2) k_topk_rows(TopkLaunch p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw);
  __shared__ uint32_t s_count;
  __shared__ int s_nan;
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
  if (threadIdx.x == 0) {
    s_count = 0;
    s_nan = 0;
  }
  __syncthreads();

  int64_t c = 0;  // candidates in shared memory
  bool ok = true;
  if (n <= kCap) {
    for (int64_t i = threadIdx.x; i < n; i += kThreads) {
      const float v = __ldg(x + i);
      if (isnan(v)) s_nan = 1;
      sm.key[i] = score_key(v);
      sm.pos[i] = (int32_t)i;
    }
    c = n;
  } else {
    // threshold from a sample of whole 8-score groups (one 32-byte sector each), evenly
    // strided over the row, so the sample touches only every g-th sector
    const int64_t groups = n / 8;
    const int64_t gstride = (groups * 8 + kSampleMax - 1) / kSampleMax;  // >= 1 since n > kCap
    const int64_t mg = (groups + gstride - 1) / gstride;
    const int64_t m = mg * 8;
    for (int64_t i = threadIdx.x; i < m; i += kThreads)
      sm.key[i] = score_key(__ldg(x + (i >> 3) * gstride * 8 + (i & 7)));
    __syncthreads();
    int64_t ks = (int64_t)ceil(1.25 * (double)k * (double)m / (double)n) + 16;
    if (ks > m) ks = m;
    uint32_t dummy;
    const uint32_t theta = radix_select(sm, m, (uint32_t)ks, [&](int64_t i) { return sm.key[i]; }, &dummy);
    // one streaming pass: append every key >= theta in position order
    uint32_t count = 0;
#pragma unroll 1
    for (int64_t base = 0; base < n; base += (int64_t)kThreads * kPer) {
      const int64_t q = base + (int64_t)threadIdx.x * kPer;
      float v[kPer];
      load8(x, q, n, vec, v);
      uint32_t key[kPer];
      uint32_t cnt = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const bool valid = q + j < n;
        if (valid && isnan(v[j])) s_nan = 1;
        key[j] = score_key(v[j]);
        cnt += (valid && key[j] >= theta);
      }
      uint32_t tot;
      uint32_t o = count + block_excl_scan(cnt, sm.warp_sums, &tot);
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        if (q + j < n && key[j] >= theta) {
          if (o < (uint32_t)kCap) {
            sm.key[o] = key[j];
            sm.pos[o] = (int32_t)(q + j);
          }
          ++o;
        }
      }
      count += tot;
    }
    __syncthreads();
    c = count;
    ok = count >= (uint32_t)k && count <= (uint32_t)kCap;
  }
  __syncthreads();
  if (s_nan && threadIdx.x == 0) atomicOr(p.flags, DSA_FLAG_NAN_SCORE);

  if (ok) {
    uint32_t ties;
    const uint32_t tau = radix_select(sm, c, (uint32_t)k, [&](int64_t i) { return sm.key[i]; }, &ties);
    ordered_output(sm, c, tau, ties, k, out, [&](int64_t i, uint32_t& key, int32_t& ps) {
      key = sm.key[i];
      ps = sm.pos[i];
    });
  } else {
    // the sample misjudged the threshold: three histogram passes over the row in global memory
    auto gkey = [&](int64_t i) { return score_key(__ldg(x + i)); };
    uint32_t ties;
    const uint32_t tau = radix_select(sm, n, (uint32_t)k, gkey, &ties);
    ordered_output(sm, n, tau, ties, k, out, [&](int64_t i, uint32_t& key, int32_t& ps) {
      key = gkey(i);
      ps = (int32_t)i;
    });
  }
}

}  // namespace

cudaError_t launch_topk_rows(const TopkLaunch& p, cudaStream_t st) {
  const int rows = p.B * p.Tc;
  if (rows <= 0) return cudaSuccess;
  const int smem = (int)sizeof(TopkSmem);
  cudaError_t e = cudaFuncSetAttribute(k_topk_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k_topk_rows<<<rows, kThreads, smem, st>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
