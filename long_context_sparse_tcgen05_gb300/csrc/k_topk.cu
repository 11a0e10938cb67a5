// Per-row top-k over materialised fp32 score rows, exact, ties to the lower position, output
// in ascending position order.
//
// One 512-thread CTA owns one row (two CTAs per SM).  Scores are compared through their
// order-preserving 32-bit keys.
//   * Rows with at most Cap visible scores are copied to shared memory whole.
//   * Longer rows: a sample of at most Cap keys (whole 8-key groups, evenly strided) gives, by
//     two 11-bit radix passes in shared memory, a threshold theta that about 1.5k of the row's
//     keys exceed; one streaming pass then appends every key >= theta, in position order
//     (block-wide prefix sums of per-thread counts), to shared memory.  Every key below theta
//     has at least k larger keys, so the row's top-k lies among the candidates.  The pass
//     reads the row through a ring of bulk copies (cp.async.bulk into shared memory,
//     completion on an mbarrier) of Per scores per thread each, and is bound by its per-score
//     instruction count: one block-wide scan per Per x 512 scores, 32-bit indices, no
//     per-score bounds checks on whole chunks, the NaN flag kept in a register.  A buffer
//     about to overflow is compacted in place to its exact top-k and theta raised to the k-th
//     key (a later equal key loses the tie).
//   * An exact radix select among the candidates, starting at the first bit where theta and
//     the largest candidate differ, finds the k-th key; a stable compaction writes the
//     selected positions in order.
//   * Fewer rows than SMs (decode): each row is split into segments of at least 32K scores,
//     one CTA each; a segment writes its exact top-k with the keys, sorted by position, and
//     k_topk_merge selects the row's top-k from the concatenated lists.
// If the sample overestimates the threshold (fewer than k candidates), or one chunk brings more
// candidates than the buffer holds, the CTA falls back to histogram passes over the row in
// global memory and a final ordered compaction pass.
//
// k_topk_cand is the top-k of the path that stores no scores: a row's candidates (score,
// position) from the selecting indexer are loaded into shared memory, a radix select (starting
// at the first bit where the smallest and largest candidate keys differ) finds the k-th key and
// the positions of its ties, and the selected positions are written in order by marking them
// in a bitmap of the row and compacting it (rows up to 262,144 keys; longer rows sort the k
// positions bitonically).
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kPer = 8;                     // consecutive entries per thread per compaction step

// Cap: candidates (and sampled keys) held in shared memory; Ring: bulk-copy slots;
// Per: consecutive scores per thread per streaming step (a slot holds Per x 512 scores).
template <int Cap, int Ring, int Per>
struct TopkSmem {
  float ring[Ring][kThreads * Per];
  uint32_t key[Cap];
  int32_t pos[Cap];
  uint32_t hist[kBins];
  uint32_t warp_sums[kWarps];
  uint32_t stream_sums[2][kWarps];  // per-warp totals of the streaming pass, by chunk parity
  uint32_t sel_bin, sel_above;
  uint64_t full[Ring];
  int abort;
  uint32_t kmax;  // largest candidate key
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

// The same prefix sum with a single barrier: after it every warp scans the kWarps warp totals
// itself. Consecutive calls must alternate between two sums arrays, so that a warp writing the
// next call's totals cannot overwrite ones that a slower warp has still to read.
__device__ __forceinline__ uint32_t block_excl_scan1(uint32_t v, uint32_t* sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sums[wid] = x;
  __syncthreads();
  uint32_t s = lane < kWarps ? sums[lane] : 0u;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
    if (lane >= o) s += y;
  }
  *total = __shfl_sync(0xffffffffu, s, kWarps - 1);
  const uint32_t before = __shfl_sync(0xffffffffu, s, wid > 0 ? wid - 1 : 0);
  return (wid > 0 ? before : 0u) + x - v;
}

// The bin b (counting from the top) with above(b) < need <= above(b) + hist[b], among the
// nbins <= 2048 bins: thread t sums the four bins nbins-1-4t .. nbins-4-4t, one block scan
// gives each thread the count above its bins, and the thread whose bins hold the need-th key
// writes sel_bin / sel_above.
template <class Sm>
__device__ __forceinline__ void select_bin(Sm& sm, uint32_t need, int nbins) {
  uint32_t h[4], s = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int b = nbins - 1 - 4 * (int)threadIdx.x - j;
    h[j] = b >= 0 ? sm.hist[b] : 0u;
    s += h[j];
  }
  uint32_t tot;
  const uint32_t above = block_excl_scan(s, sm.warp_sums, &tot);
  if (above < need && need <= above + s) {
    uint32_t acc = above;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (acc + h[j] >= need) {
        sm.sel_bin = (uint32_t)(nbins - 1 - 4 * (int)threadIdx.x - j);
        sm.sel_above = acc;
        break;
      }
      acc += h[j];
    }
  }
}

// Radix select over keys delivered by get(i), i < n, that all carry `prefix` in their bits at
// and above `top` (prefix has no bits below `top`): histograms of 11-bit digits from bit `top`
// down to bit `stop` locate the need-th largest key (need >= 1).  Returns its bits at and
// above `stop` (lower bits zero); with stop = 0 that is the key itself and *ties receives how
// many keys equal to it are taken.
template <class Sm, class Get>
__device__ uint32_t radix_select(Sm& sm, int64_t n, uint32_t need, Get get, uint32_t* ties, uint32_t prefix, int top,
                                 int stop) {
  uint32_t pmask = top >= 32 ? 0u : ~((1u << top) - 1u);
#pragma unroll 1
  while (top > stop) {
    const int width = top - stop < 11 ? top - stop : 11;
    const int shift = top - width;
    const uint32_t wmask = (1u << width) - 1u;
    for (int i = threadIdx.x; i < (1 << width); i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = get(i);
      if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & wmask], 1u);
    }
    __syncthreads();
    select_bin(sm, need, 1 << width);
    __syncthreads();
    prefix |= sm.sel_bin << shift;
    pmask |= wmask << shift;
    need -= sm.sel_above;
    __syncthreads();
    top = shift;
  }
  *ties = need;
  return prefix;
}

// Keeps, in place and in position order, the exact top-k of the first `count` candidates
// (count >= k; ties go to the lower position, i.e. the earlier entry) and returns the k-th key.
template <class Sm>
__device__ uint32_t compact_top(Sm& sm, uint32_t count, int k) {
  uint32_t ties;
  const uint32_t tau =
      radix_select(sm, (int64_t)count, (uint32_t)k, [&](int64_t i) { return sm.key[i]; }, &ties, 0u, 32, 0);
  uint32_t out_base = 0, eq_seen = 0;
#pragma unroll 1
  for (uint32_t base = 0; base < count; base += (uint32_t)kThreads * kPer) {
    const uint32_t q = base + threadIdx.x * kPer;
    uint32_t kk[kPer];
    int32_t ps[kPer];
    uint32_t cg = 0, ce = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const bool valid = q + j < count;
      kk[j] = valid ? sm.key[q + j] : 0u;
      ps[j] = valid ? sm.pos[q + j] : -1;
      cg += valid && kk[j] > tau;
      ce += valid && kk[j] == tau;
    }
    uint32_t tot;  // every entry of this pass is in registers once the scan returns
    const uint32_t ex = block_excl_scan((cg << 16) | ce, sm.warp_sums, &tot);
    const uint32_t rem = ties > eq_seen ? ties - eq_seen : 0u;
    uint32_t o = out_base + (ex >> 16) + ((ex & 0xffffu) < rem ? (ex & 0xffffu) : rem);
    uint32_t eq_idx = eq_seen + (ex & 0xffffu);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (ps[j] < 0) continue;
      if (kk[j] > tau || (kk[j] == tau && eq_idx++ < ties)) {
        sm.key[o] = kk[j];
        sm.pos[o] = ps[j];
        ++o;
      }
    }
    out_base += (tot >> 16) + ((tot & 0xffffu) < rem ? (tot & 0xffffu) : rem);
    eq_seen += tot & 0xffffu;
  }
  __syncthreads();
  return tau;
}

// Stable ordered compaction: writes out[0..k) with the positions of the entries whose key is
// > tau, plus the first `ties` entries whose key == tau, in stream order.  get(i) gives
// (key, position) of entry i < n.
template <class Sm, class Get>
__device__ void ordered_output(Sm& sm, int64_t n, uint32_t tau, uint32_t ties, int k, int32_t* out, Get get,
                               int32_t pos_off = 0, uint32_t* kout = nullptr) {
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
        if (kout) kout[o] = key[j];
        out[o++] = ps[j] + pos_off;
      } else if (key[j] == tau) {
        if (eq_idx < ties) {
          if (kout) kout[o] = key[j];
          out[o++] = ps[j] + pos_off;
        }
        ++eq_idx;
      }
    }
    out_base += gt_tot + (eq_tot < rem ? eq_tot : rem);
    eq_seen += eq_tot;
    if (out_base >= (uint32_t)k) break;
  }
}

__device__ __forceinline__ uint32_t sa(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
// Waits for a ring slot's copy; gives up after `limit` cycles (raising *abort) or when another
// thread has raised *abort.  kPoll (the instantiation for a bound shorter than the default,
// used to test the timeout path) polls with test_wait, which never suspends (try_wait may
// sleep until the copy lands and so hide a short bound).
template <bool kPoll>
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, volatile int* abort, long long limit) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    if constexpr (kPoll)
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(ok)
          : "r"(sa(bar)), "r"(parity)
          : "memory");
    else
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(ok)
          : "r"(sa(bar)), "r"(parity)
          : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      return false;
    }
  }
}

template <int Cap, int Ring, int Per, bool kPoll>
__global__ void __launch_bounds__(kThreads, 2) k_topk_rows(TopkLaunch p) {
  using Sm = TopkSmem<Cap, Ring, Per>;
  constexpr int kChunk = kThreads * Per;
  static_assert(kChunk < (1 << 16), "a chunk's candidate count must stay below the timeout flag");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
  __shared__ int s_nan;
  const int parts = p.parts > 1 ? p.parts : 1;
  const int row = (int)(blockIdx.x / parts), part = (int)(blockIdx.x % parts);
  // recomputing pass: only rows the selection left over
  if (p.gate && !p.gate[(int64_t)(row / p.Tc) * p.gate_bstride + row % p.Tc]) return;
  const int b = row / p.Tc, tl = row % p.Tc, t = p.t0 + tl;
  const float* x = p.scores + (int64_t)b * p.bstride + (int64_t)tl * p.ld;
  int32_t* out = p.idx + ((int64_t)b * p.T + t) * p.k;
  int64_t n = p.q_pos0 + t + p.diag;
  n = n < 0 ? 0 : (n > p.S ? p.S : n);
  const int k = p.k;
  // a split row: this CTA's segment [seg0, seg0 + n), whole 4,096-score pieces but the last
  int32_t seg0 = 0;
  uint32_t* kout = nullptr;
  if (parts > 1) {
    const int64_t seg_len = ((n + parts - 1) / parts + 4095) / 4096 * 4096;
    const int64_t s0 = (int64_t)part * seg_len, s1 = s0 + seg_len < n ? s0 + seg_len : n;
    seg0 = (int32_t)s0;
    n = s1 > s0 ? s1 - s0 : 0;
    x += s0;
    const int64_t slot = (int64_t)row * parts + part;
    out = p.part_pos + slot * k;
    kout = p.part_key + slot * k;
    if (threadIdx.x == 0) p.part_cnt[slot] = (int32_t)(n < k ? n : k);
  }

  if (n <= k) {
    for (int j = threadIdx.x; j < k; j += kThreads) {
      out[j] = j < n ? seg0 + j : -1;
      if (kout && j < n) {
        const float v = __ldg(x + j);
        if (isnan(v)) atomicOr(p.flags, DSA_FLAG_NAN_SCORE);
        kout[j] = score_key(v);
      }
    }
    return;
  }
  const bool vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
  if (threadIdx.x == 0) {
    s_nan = 0;
    sm.abort = 0;
    sm.kmax = 0;
    for (int i = 0; i < Ring; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(sa(&sm.full[i])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  int64_t c = 0;  // candidates in shared memory
  bool ok = true;
  uint32_t theta_s = 0;  // candidate threshold of a long row
  if (n <= Cap) {
#pragma unroll 4
    for (int64_t i = threadIdx.x; i < n; i += kThreads) {
      const float v = __ldg(x + i);
      if (isnan(v)) s_nan = 1;
      sm.key[i] = score_key(v);
      sm.pos[i] = (int32_t)i;
    }
    c = n;
  } else {
    const int64_t nchunks = (n + kChunk - 1) / kChunk;
    // ring slot s holds chunk ci; the bulk copy covers the chunk's whole 16-byte units, the
    // last 1-3 scores of a ragged row tail are read directly
    auto bulk_len = [&](int64_t ci) -> int64_t {
      const int64_t len = n - ci * kChunk < kChunk ? n - ci * kChunk : kChunk;
      return vec ? (len & ~(int64_t)3) : 0;
    };
    auto issue = [&](int64_t ci) {
      const int s = (int)(ci % Ring);
      const uint32_t bytes = (uint32_t)(bulk_len(ci) * 4);
      if (bytes) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(sa(&sm.full[s])), "r"(bytes)
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                sa(&sm.ring[s][0])),
            "l"(reinterpret_cast<uint64_t>(x + ci * kChunk)), "r"(bytes), "r"(sa(&sm.full[s]))
            : "memory");
      } else {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(sa(&sm.full[s])) : "memory");
      }
    };
    // the stream starts before the sample is taken, so its latency hides behind the select;
    // chunks [0, issued) have had their copies started (thread 0 keeps the count)
    int64_t issued = 0;
    if (threadIdx.x == 0)
      for (; issued < Ring && issued < nchunks; ++issued) issue(issued);
    // threshold from a sample of whole 8-score groups (one 32-byte sector each), evenly
    // strided over the row, so the sample touches only every g-th sector
    const int64_t groups = n / 8;
    const int64_t gstride = (groups * 8 + Cap - 1) / Cap;  // >= 1 since n > Cap
    const int64_t mg = (groups + gstride - 1) / gstride;
    const int64_t m = mg * 8;
#pragma unroll 4
    for (int64_t i = threadIdx.x; i < m; i += kThreads)
      sm.key[i] = score_key(__ldg(x + (i >> 3) * gstride * 8 + (i & 7)));
    __syncthreads();
    // aim at about 1.5k candidates: too few (< k) costs a fallback, too many only a compaction
    int64_t ks = (int64_t)ceil(1.5 * (double)k * (double)m / (double)n) + 8;
    if (ks > m) ks = m;
    // the ks-th largest sampled key rounded down to a multiple of 2^10: two digit passes; a
    // lower threshold only admits more candidates
    uint32_t dummy;
    uint32_t theta =
        radix_select(sm, m, (uint32_t)ks, [&](int64_t i) { return sm.key[i]; }, &dummy, 0u, 32, 10);
    theta_s = theta;  // lower bound of every candidate key
    // one streaming pass: append every key >= theta in position order (32-bit indices: n < 2^31)
    const int n32 = (int)n;
    uint32_t count = 0, kmax = 0;
    bool nan_seen = false;
    bool overflow = false;  // a chunk brought more candidates than the buffer can hold
#pragma unroll 1
    for (int64_t ci = 0; ci < nchunks; ++ci) {
      const int s = (int)(ci % Ring);
      // a thread whose copy wait timed out adds 2^16 to the block sum below (a chunk holds at
      // most 8,192 candidates), and the whole block leaves the pass after that sum
      const bool landed = ring_wait<kPoll>(&sm.full[s], (uint32_t)((ci / Ring) & 1), &sm.abort, p.wait);
      const int base = (int)ci * kChunk, blen = (int)bulk_len(ci);
      const int q = base + (int)threadIdx.x * Per;
      const float* slot = &sm.ring[s][threadIdx.x * Per];
      uint32_t key[Per];
      uint32_t cnt = 0;
      if (blen == kChunk) {  // whole chunk in the slot
#pragma unroll
        for (int j = 0; j < Per; j += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(slot + j);
          const float v4[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            nan_seen |= v4[u] != v4[u];
            key[j + u] = score_key(v4[u]);
            cnt += key[j + u] >= theta;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < Per; ++j) {
          const int i = q + j;
          const float v = i < base + blen ? slot[j] : (i < n32 ? __ldg(x + i) : 0.f);
          nan_seen |= i < n32 && v != v;
          key[j] = i < n32 ? score_key(v) : 0u;
          cnt += i < n32 && key[j] >= theta;
        }
      }
      uint32_t tot;
      uint32_t o = count + block_excl_scan1(cnt + (landed ? 0u : 1u << 16), sm.stream_sums[ci & 1], &tot);
      if (tot >> 16) break;
      // every thread has read slot s (the scan synchronised the block): refill it
      if (threadIdx.x == 0 && ci + Ring < nchunks) issue(issued++);
      if (count + tot > (uint32_t)Cap && count >= (uint32_t)k) {
        // the buffer would overflow: keep only its exact top-k and raise the threshold to the
        // k-th key -- a later key equal to it loses the tie to every kept one -- then recount
        const uint32_t tau = compact_top(sm, count, k);
        count = (uint32_t)k;
        theta_s = tau;
        theta = tau == 0xffffffffu ? tau : tau + 1u;
        cnt = 0;
#pragma unroll
        for (int j = 0; j < Per; ++j) cnt += q + j < n32 && key[j] >= theta;
        o = count + block_excl_scan(cnt, sm.warp_sums, &tot);
      }
      if (count + tot > (uint32_t)Cap) {
        // even compacted the buffer cannot hold this chunk's candidates (a threshold far below
        // the k-th key, e.g. a row of equal scores): leave the row to the exact passes below
        overflow = true;
        break;
      }
      if (cnt) {
#pragma unroll
        for (int j = 0; j < Per; ++j) {
          if (key[j] >= theta && q + j < n32) {
            kmax = key[j] > kmax ? key[j] : kmax;
            if (o < (uint32_t)Cap) {
              sm.key[o] = key[j];
              sm.pos[o] = q + j;
            }
            ++o;
          }
        }
      }
      count += tot;
    }
    if (nan_seen) s_nan = 1;
    if (kmax) atomicMax(&sm.kmax, kmax);
    __syncthreads();
    if (sm.abort || overflow) {
      // the pass ended early (a wait ran out, or the buffer overflowed): let the copies still in
      // flight -- the last Ring chunks issued, one per ring slot -- land before the CTA goes on
      // or exits (with the default bound)
      if (threadIdx.x == 0) {
        for (int64_t ci = issued - Ring > 0 ? issued - Ring : 0; ci < issued; ++ci) {
          const long long t0 = clock64();
          uint32_t okw = 0;
          while (!okw && clock64() - t0 < kDefaultWaitCycles)
            asm volatile(
                "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, "
                "p;\n}\n"
                : "=r"(okw)
                : "r"(sa(&sm.full[ci % Ring])), "r"((uint32_t)((ci / Ring) & 1))
                : "memory");
        }
        if (sm.abort) atomicOr(p.flags, DSA_FLAG_TIMEOUT);
      }
      if (sm.abort) return;
      __syncthreads();
    }
    c = count;
    ok = !overflow && count >= (uint32_t)k && count <= (uint32_t)Cap;
  }
  __syncthreads();
  if (s_nan && threadIdx.x == 0) atomicOr(p.flags, DSA_FLAG_NAN_SCORE);

  if (ok) {
    // every candidate key lies in [theta, kmax] (short rows: the whole key range), so the
    // bits above the highest one where theta and kmax differ are common to all of them
    uint32_t ties, prefix = 0;
    int top = 32;
    if (n > Cap) {
      const uint32_t diff = theta_s ^ sm.kmax;
      top = diff ? 32 - __clz(diff) : 0;
      prefix = top >= 32 ? 0u : (sm.kmax & ~((1u << top) - 1u));
    }
    const uint32_t tau =
        radix_select(sm, c, (uint32_t)k, [&](int64_t i) { return sm.key[i]; }, &ties, prefix, top, 0);
    ordered_output(sm, c, tau, ties, k, out, [&](int64_t i, uint32_t& key, int32_t& ps) {
      key = sm.key[i];
      ps = sm.pos[i];
    }, seg0, kout);
  } else {
    // the sample misjudged the threshold: three histogram passes over the row in global memory
    auto gkey = [&](int64_t i) { return score_key(__ldg(x + i)); };
    uint32_t ties;
    const uint32_t tau = radix_select(sm, n, (uint32_t)k, gkey, &ties, 0u, 32, 0);
    ordered_output(sm, n, tau, ties, k, out, [&](int64_t i, uint32_t& key, int32_t& ps) {
      key = gkey(i);
      ps = (int32_t)i;
    }, seg0, kout);
  }
}

struct MergeSmem {
  uint32_t hist[kBins];
  uint32_t warp_sums[kWarps];
  uint32_t sel_bin, sel_above;
  int32_t pre[kMaxTopkParts + 1];  // start of each segment's list in the concatenation
};

// One split row: the exact top-k of its segments' lists, concatenated in segment order (so in
// position order).  kSmemKeys: the row's keys are first gathered densely into shared memory
// (at most kMergeSmemKeys), the radix passes start at the first bit where the smallest and
// largest key differ, and only entries at or above the k-th key fetch their position; otherwise
// every pass reads the lists in global memory.
constexpr int kMergeSmemKeys = 40960;  // 160 KB
template <bool kSmemKeys>
__global__ void __launch_bounds__(kThreads) k_topk_merge(TopkLaunch p) {
  __shared__ MergeSmem sm;
  extern __shared__ uint32_t mkeys[];
  const int row = blockIdx.x, parts = p.parts, k = p.k;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int s = 0; s < parts; ++s) {
      sm.pre[s] = acc;
      acc += p.part_cnt[(int64_t)row * parts + s];
    }
    sm.pre[parts] = acc;
  }
  __syncthreads();
  const int64_t n = sm.pre[parts];
  const int b = row / p.Tc, tl = row % p.Tc;
  int32_t* out = p.idx + ((int64_t)b * p.T + p.t0 + tl) * k;
  const int64_t base = (int64_t)row * parts * k;
  auto locate = [&](int64_t i) -> int64_t {  // entry i of the concatenation -> list offset
    int lo = 0, hi = parts;                  // largest s with pre[s] <= i
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sm.pre[mid] <= i) lo = mid; else hi = mid;
    }
    return base + (int64_t)lo * k + (i - sm.pre[lo]);
  };
  if (n <= k) {
    for (int j = threadIdx.x; j < k; j += kThreads) out[j] = j < n ? p.part_pos[locate(j)] : -1;
    return;
  }
  uint32_t ties;
  if constexpr (kSmemKeys) {
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int s = 0; s < parts; ++s) {
      const int c = sm.pre[s + 1] - sm.pre[s];
      const uint32_t* src = p.part_key + base + (int64_t)s * k;
      for (int j = threadIdx.x; j < c; j += kThreads) {
        const uint32_t kk = __ldg(src + j);
        mkeys[sm.pre[s] + j] = kk;
        lo = kk < lo ? kk : lo;
        hi = kk > hi ? kk : hi;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if ((threadIdx.x & 31) == 0) sm.warp_sums[threadIdx.x >> 5] = lo;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t m = 0xffffffffu;
      for (int w = 0; w < kWarps; ++w) m = sm.warp_sums[w] < m ? sm.warp_sums[w] : m;
      sm.sel_bin = m;
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sm.warp_sums[threadIdx.x >> 5] = hi;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t m = 0u;
      for (int w = 0; w < kWarps; ++w) m = sm.warp_sums[w] > m ? sm.warp_sums[w] : m;
      sm.sel_above = m;
    }
    __syncthreads();
    // every key shares the bits of the smallest and largest above their highest differing bit
    const uint32_t kmin = sm.sel_bin, kmax = sm.sel_above, d = kmin ^ kmax;
    const int top = d ? 32 - __clz(d) : 0;
    const uint32_t prefix = top >= 32 ? 0u : (kmax & ~((1u << top) - 1u));
    __syncthreads();
    const uint32_t tau =
        radix_select(sm, n, (uint32_t)k, [&](int64_t i) { return mkeys[i]; }, &ties, prefix, top, 0);
    ordered_output(sm, n, tau, ties, k, out, [&](int64_t i, uint32_t& key, int32_t& ps) {
      key = mkeys[i];
      ps = key >= tau ? p.part_pos[locate(i)] : 0;  // only taken entries need their position
    });
  } else {
    const uint32_t tau =
        radix_select(sm, n, (uint32_t)k, [&](int64_t i) { return p.part_key[locate(i)]; }, &ties, 0u, 32, 0);
    ordered_output(sm, n, tau, ties, k, out, [&](int64_t i, uint32_t& key, int32_t& ps) {
      const int64_t o = locate(i);
      key = p.part_key[o];
      ps = p.part_pos[o];
    });
  }
}

constexpr int kBitmapKeys = 262144;  // rows this long or shorter are ordered through a bitmap
struct CandSmem {
  uint32_t key[kCandMaxCap];
  int32_t pos[kCandMaxCap];
  union {
    int32_t sel[2 * kCandMaxK];           // longer rows: the k positions, bitonic-sorted
    uint32_t bits[kBitmapKeys / 32];      // shorter rows: one bit per position
  };
  uint32_t hist[kBins];
  uint32_t warp_sums[kWarps];
  uint32_t sel_bin, sel_above;
  uint32_t eq;                  // candidates whose key equals the k-th key
  uint32_t kmin, kmax;          // smallest and largest candidate key
  uint32_t pmin, pmax;          // smallest and largest inverted position among those equal to tau
};

// One row's exact top-k from its candidates (see CandLaunch): the k-th key tau by radix
// select; when more candidates equal tau than the row can take, the lowest positions among them
// (a radix select on inverted positions); the k selected positions are then sorted ascending
// (bitonic) and written.
__global__ void __launch_bounds__(kThreads, 2) k_topk_cand(CandLaunch p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  CandSmem& sm = *reinterpret_cast<CandSmem*>(smem_raw);
  const int row = blockIdx.x;
  const int b = row / p.Tc, tl = row % p.Tc, t = p.t0 + tl;
  int32_t* out = p.idx + ((int64_t)b * p.T + t) * p.k;
  int64_t n = p.q_pos0 + t + p.diag;
  n = n < 0 ? 0 : (n > p.S ? p.S : n);
  const int k = p.k;
  if (n <= k) {  // every visible key
    for (int j = threadIdx.x; j < k; j += kThreads) out[j] = j < n ? j : -1;
    if (threadIdx.x == 0) p.fail[row] = 0;
    return;
  }
  // the row's list is four segments of cap/4 (one per epilogue warp of the indexer)
  const int cap4 = p.cap / 4;
  int cs[4], pre[4], cnt = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    cs[q] = __ldg(p.cand_cnt + (int64_t)row * 4 + q);
    pre[q] = cnt;
    cnt += cs[q];
  }
  if (cnt < k || cs[0] > cap4 || cs[1] > cap4 || cs[2] > cap4 || cs[3] > cap4) {
    if (threadIdx.x == 0) p.fail[row] = 1;
    return;
  }
  const uint2* cd = p.cand + (int64_t)row * p.cap;
  if (threadIdx.x == 0) {
    sm.eq = 0;
    sm.kmin = 0xffffffffu;
    sm.kmax = 0u;
    sm.pmin = 0xffffffffu;
    sm.pmax = 0u;
  }
  __syncthreads();
  uint32_t lo = 0xffffffffu, hi = 0u;
  {
    // every load of the four segments in flight at once, then into shared memory contiguously
    constexpr int kU = kCandMaxCap / 4 / kThreads;  // entries per thread and segment
    uint2 cv[4][kU];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = u * kThreads + (int)threadIdx.x;
        cv[q][u] = i < cs[q] ? __ldg(cd + q * cap4 + i) : make_uint2(0u, 0u);
      }
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = u * kThreads + (int)threadIdx.x;
        if (i < cs[q]) {
          const uint32_t kk = score_key(__uint_as_float(cv[q][u].x));
          sm.key[pre[q] + i] = kk;
          sm.pos[pre[q] + i] = (int32_t)cv[q][u].y;
          lo = kk < lo ? kk : lo;
          hi = kk > hi ? kk : hi;
        }
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&sm.kmin, lo);
    atomicMax(&sm.kmax, hi);
  }
  __syncthreads();
  // every candidate shares the bits of kmin and kmax above their highest differing bit: the
  // radix passes start there (a row's candidates sit in a narrow range of scores, so the
  // leading digits would put them all in one histogram bin)
  auto common = [](uint32_t a, uint32_t b, uint32_t* prefix) {
    const uint32_t d = a ^ b;
    const int top = d ? 32 - __clz(d) : 0;
    *prefix = top >= 32 ? 0u : (b & ~((1u << top) - 1u));
    return top;
  };
  uint32_t ties, prefix;
  int top = common(sm.kmin, sm.kmax, &prefix);
  const uint32_t tau =
      radix_select(sm, (int64_t)cnt, (uint32_t)k, [&](int64_t i) { return sm.key[i]; }, &ties, prefix, top, 0);
  uint32_t eq_local = 0, plo = 0xffffffffu, phi = 0u;
  for (int i = threadIdx.x; i < cnt; i += kThreads)
    if (sm.key[i] == tau) {
      ++eq_local;
      const uint32_t ip = ~(uint32_t)sm.pos[i];
      plo = ip < plo ? ip : plo;
      phi = ip > phi ? ip : phi;
    }
  if (eq_local) {
    atomicAdd(&sm.eq, eq_local);
    atomicMin(&sm.pmin, plo);
    atomicMax(&sm.pmax, phi);
  }
  __syncthreads();
  // the ties lowest positions among the keys equal to tau: those up to pi (a radix select of
  // the ties-th largest inverted position; entries of other keys map to 0, below every one)
  int32_t pi = INT32_MAX;
  if (sm.eq > ties) {
    uint32_t t2, pprefix;
    const int ptop = common(sm.pmin, sm.pmax, &pprefix);
    const uint32_t inv = radix_select(sm, (int64_t)cnt, ties,
                                      [&](int64_t i) { return sm.key[i] == tau ? ~(uint32_t)sm.pos[i] : 0u; }, &t2,
                                      pprefix, ptop, 0);
    pi = (int32_t)~inv;
  }
  auto selected = [&](int i) { return sm.key[i] > tau || (sm.key[i] == tau && sm.pos[i] <= pi); };
  if (n <= kBitmapKeys) {
    // mark the selected positions in a bitmap of the row, then one ordered compaction of its
    // words (each thread a contiguous run of words; a block scan places the runs)
    const int words = (int)((n + 31) / 32);
    for (int w = threadIdx.x; w < words; w += kThreads) sm.bits[w] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < cnt; i += kThreads)
      if (selected(i) && (uint32_t)sm.pos[i] < (uint32_t)n) atomicOr(&sm.bits[sm.pos[i] >> 5], 1u << (sm.pos[i] & 31));
    __syncthreads();
    const int per = (words + kThreads - 1) / kThreads;
    const int w0 = (int)threadIdx.x * per, w1 = min(words, w0 + per);
    uint32_t c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(sm.bits[w]);
    uint32_t tot;
    uint32_t o = block_excl_scan(c, sm.warp_sums, &tot);
    for (int w = w0; w < w1 && o < (uint32_t)k; ++w) {
      uint32_t m = sm.bits[w];
      while (m && o < (uint32_t)k) {
        out[o++] = w * 32 + (__ffs(m) - 1);
        m &= m - 1;
      }
    }
    for (int j = (int)tot + threadIdx.x; j < k; j += kThreads) out[j] = -1;  // (tot == k)
    if (threadIdx.x == 0) p.fail[row] = 0;
    return;
  }
  // compact the k selected positions (any order), then sort them
  int P = 1;
  while (P < k) P <<= 1;
  uint32_t out_base = 0;
  for (int base = 0; base < cnt; base += kThreads * kPer) {
    const int q = base + (int)threadIdx.x * kPer;
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = q + j;
      c += i < cnt && (sm.key[i] > tau || (sm.key[i] == tau && sm.pos[i] <= pi));
    }
    uint32_t tot;
    uint32_t o = out_base + block_excl_scan(c, sm.warp_sums, &tot);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = q + j;
      if (i < cnt && (sm.key[i] > tau || (sm.key[i] == tau && sm.pos[i] <= pi)) && o < (uint32_t)k) sm.sel[o++] = sm.pos[i];
    }
    out_base += tot;
  }
  for (int i = k + threadIdx.x; i < P; i += kThreads) sm.sel[i] = INT32_MAX;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int tt = threadIdx.x; tt < P / 2; tt += kThreads) {
        const int lo = 2 * tt - (tt & (stride - 1));
        const int hi = lo + stride;
        const bool asc = (lo & size) == 0;
        const int32_t a = sm.sel[lo], c = sm.sel[hi];
        if ((a > c) == asc) {
          sm.sel[lo] = c;
          sm.sel[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int j = threadIdx.x; j < k; j += kThreads) out[j] = sm.sel[j];
  if (threadIdx.x == 0) p.fail[row] = 0;
}

// ---- few long rows of stored scores: a sampled threshold, one filtering pass, candidate top-k ----
// (decode: 32 rows of 200,000 scores.)  k_row_threshold estimates, from an evenly spread sample
// of each row, the key that about `target` of its scores reach; k_row_filter streams every
// score once over many CTAs and appends those at or above it, as (score, position) pairs, to
// the row's candidate list (the format of the selecting indexer, one quarter per warp of four);
// k_topk_cand then selects the exact top-k.  A row whose candidates are fewer than k or overflow
// a quarter is recomputed by the one-CTA-per-row pass, gated on its flag.
constexpr int kFiltSamples = 8192;  // sampled scores per row
constexpr int kFiltChunk = 8192;    // scores per filtering CTA
constexpr int kFiltThreads = 256;
struct ThreshSmem {
  uint32_t key[kFiltSamples];
  uint32_t hist[kBins];
  uint32_t warp_sums[kWarps];
  uint32_t key_hi[kWarps];
  uint32_t sel_bin, sel_above;
};

__device__ __forceinline__ int64_t launch_row_visible(const TopkLaunch& p, int tl) {
  const int64_t n = p.q_pos0 + p.t0 + tl + p.diag;
  return n < 0 ? 0 : (n > p.S ? (int64_t)p.S : n);
}

// One row per CTA: the sample's need-th largest key, need = ceil(target' m / n) for m sampled of
// n visible scores, where target' (at most `target`) stays 4.5 standard deviations of the
// estimate above k; 0 (keep every visible score) when the sample cannot tell.  The sample is 64
// runs of 128 consecutive scores spread evenly over the row (coalesced loads), and the radix
// passes start at the first bit where its smallest and largest keys differ.  Also clears the
// row's four counts.
__global__ void __launch_bounds__(kThreads) k_row_threshold(TopkLaunch p, int target, uint32_t* tau, int32_t* cnt) {
  __shared__ ThreshSmem sm;
  const int row = blockIdx.x, b = row / p.Tc, tl = row % p.Tc;
  if (threadIdx.x < 4) cnt[row * 4 + threadIdx.x] = 0;
  const int64_t n = launch_row_visible(p, tl);
  const int m = n < kFiltSamples ? (int)n : kFiltSamples;
  int64_t need = 0;
  if (n > p.k && m > 0) {
    const float ratio = (float)n / (float)m;
    const float a = 4.5f * sqrtf(ratio);
    const float r = 0.5f * (a + sqrtf(a * a + 4.0f * (float)p.k));
    need = (int64_t)ceilf(fminf(r * r, (float)target) / ratio);
  }
  // (the same decision in every thread; a row of at most kFiltSamples scores keeps them all)
  if (need < 1 || need >= m || n <= kFiltSamples) {
    if (threadIdx.x == 0) tau[row] = 0u;
    return;
  }
  const float* sr = p.scores + (int64_t)b * p.bstride + (int64_t)tl * p.ld;
  // sample i: element i % 128 of run i / 128, the runs starting evenly over the row (n > m =
  // 8,192 here, so they do not overlap); all of a thread's loads in flight at once
  constexpr int kRun = 128, kRuns = kFiltSamples / kRun, kPerT = kFiltSamples / kThreads;
  float v[kPerT];
#pragma unroll
  for (int u = 0; u < kPerT; ++u) {
    const int i = u * kThreads + (int)threadIdx.x, r = i / kRun;
    const int64_t start = (int64_t)r * (n - kRun) / (kRuns - 1);
    v[u] = __ldg(sr + start + (i % kRun));
  }
  uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
  for (int u = 0; u < kPerT; ++u) {
    const uint32_t key = score_key(v[u]);
    sm.key[u * kThreads + (int)threadIdx.x] = key;
    lo = key < lo ? key : lo;
    hi = key > hi ? key : hi;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if ((threadIdx.x & 31) == 0) {
    sm.warp_sums[threadIdx.x >> 5] = lo;
    sm.key_hi[threadIdx.x >> 5] = hi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = 0xffffffffu, z = 0u;
    for (int w = 0; w < kWarps; ++w) {
      a = sm.warp_sums[w] < a ? sm.warp_sums[w] : a;
      z = sm.key_hi[w] > z ? sm.key_hi[w] : z;
    }
    sm.sel_bin = a;
    sm.sel_above = z;
  }
  __syncthreads();
  const uint32_t d = sm.sel_bin ^ sm.sel_above;
  const int top = d ? 32 - __clz(d) : 0;
  const uint32_t prefix = top >= 32 ? 0u : (sm.sel_above & ~((1u << top) - 1u));
  __syncthreads();
  uint32_t ties;
  const uint32_t t =
      radix_select(sm, (int64_t)kFiltSamples, (uint32_t)need, [&](int64_t i) { return sm.key[i]; }, &ties, prefix, top, 0);
  if (threadIdx.x == 0) tau[row] = t;
}

// Grid (chunks, rows): chunk c streams scores [c kFiltChunk, (c + 1) kFiltChunk) of the row's
// visible range and gathers those at or above the row's threshold in shared memory (a
// block-local count: one atomic per warp and pass on the same global counter serialised the
// whole pass); then entry i of the CTA's gathered list goes to quarter i % 4 of the row's list,
// after one global atomic per quarter reserves the room.  NaN scores raise DSA_FLAG_NAN_SCORE.
constexpr int kFiltBuf = 2048;  // gathered entries per CTA (8,192 scores: about 2% qualify)
constexpr int kFiltUnroll = 8;  // scores per thread per pass, loaded together
__global__ void __launch_bounds__(kFiltThreads) k_row_filter(TopkLaunch p, const uint32_t* tau, int cap, uint2* cand,
                                                             int32_t* cnt) {
  __shared__ uint2 buf[kFiltBuf];
  __shared__ int nbuf, over;
  __shared__ int qbase[4];
  const int row = blockIdx.y, b = row / p.Tc, tl = row % p.Tc;
  const int64_t n = launch_row_visible(p, tl);
  const int64_t c0 = (int64_t)blockIdx.x * kFiltChunk;
  if (c0 >= n) return;
  const int64_t c1 = n < c0 + kFiltChunk ? n : c0 + kFiltChunk;
  const float* sr = p.scores + (int64_t)b * p.bstride + (int64_t)tl * p.ld;
  const uint32_t th = tau[row];
  const int lane = threadIdx.x & 31, cap4 = cap / 4;
  const uint32_t below = (1u << lane) - 1u;
  if (threadIdx.x == 0) nbuf = 0, over = 0;
  __syncthreads();
  bool nan = false;
  auto consider = [&](float v, int64_t i, bool valid) {  // warp-uniform call
    nan |= valid && v != v;
    const bool take = valid && score_key(v) >= th;
    const uint32_t bal = __ballot_sync(0xffffffffu, take);
    if (bal) {
      int slot0 = 0;
      if (lane == 0) slot0 = atomicAdd(&nbuf, __popc(bal));
      slot0 = __shfl_sync(0xffffffffu, slot0, 0);
      if (take) {
        const int slot = slot0 + __popc(bal & below);
        if (slot < kFiltBuf) buf[slot] = make_uint2(__float_as_uint(v), (uint32_t)i);
        else over = 1;
      }
    }
  };
  if (c1 - c0 == kFiltChunk && (reinterpret_cast<uintptr_t>(sr + c0) & 15u) == 0) {
    // a whole 16-byte-aligned chunk: 16-byte loads, two per thread and pass in flight
    const float4* s4 = reinterpret_cast<const float4*>(sr + c0);
    for (int base = 0; base < kFiltChunk / 4; base += 2 * kFiltThreads) {
      float4 w[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) w[u] = __ldg(s4 + base + u * kFiltThreads + threadIdx.x);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int64_t i = c0 + 4 * (int64_t)(base + u * kFiltThreads + threadIdx.x);
        consider(w[u].x, i, true);
        consider(w[u].y, i + 1, true);
        consider(w[u].z, i + 2, true);
        consider(w[u].w, i + 3, true);
      }
    }
  } else {
    for (int64_t base = c0; base < c1; base += (int64_t)kFiltThreads * kFiltUnroll) {
      float v[kFiltUnroll];
#pragma unroll
      for (int u = 0; u < kFiltUnroll; ++u) {
        const int64_t i = base + u * kFiltThreads + threadIdx.x;
        v[u] = i < c1 ? __ldg(sr + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kFiltUnroll; ++u) {
        const int64_t i = base + u * kFiltThreads + threadIdx.x;
        consider(v[u], i, i < c1);
      }
    }
  }
  __syncthreads();
  const int m = nbuf < kFiltBuf ? nbuf : kFiltBuf;
  if (threadIdx.x < 4) {
    // an overflowing CTA claims more than a quarter holds, so the row is recomputed exactly
    const int add = over ? cap4 + 1 : (m - (int)threadIdx.x + 3) / 4;
    qbase[threadIdx.x] = atomicAdd(cnt + row * 4 + threadIdx.x, add);
  }
  __syncthreads();
  if (!over)
    for (int i = threadIdx.x; i < m; i += kFiltThreads) {
      const int q = i & 3, slot = qbase[q] + (i >> 2);
      if (slot < cap4) cand[(int64_t)row * cap + q * cap4 + slot] = buf[i];
    }
  if (nan) atomicOr(p.flags, DSA_FLAG_NAN_SCORE);
}

template <int Cap, int Ring, int Per>
cudaError_t launch_rows(const TopkLaunch& p, int rows, cudaStream_t st) {
  TraceScope trace(kTraceTopk, st);
  const int smem = (int)sizeof(TopkSmem<Cap, Ring, Per>);
  TopkLaunch q = p;
  if (q.wait <= 0) q.wait = wait_limit();
  auto kern = q.wait < kDefaultWaitCycles ? k_topk_rows<Cap, Ring, Per, true> : k_topk_rows<Cap, Ring, Per, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<rows * (p.parts > 1 ? p.parts : 1), kThreads, smem, st>>>(q);
  return cudaGetLastError();
}

}  // namespace

int topk_parts(int64_t rows, int64_t n) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (rows <= 0 || rows >= sms) return 1;
  int64_t parts = (2LL * sms) / rows;        // about two CTAs per SM
  const int64_t by_len = n / 32768;           // segments of at least 32K scores
  if (parts > by_len) parts = by_len;
  if (parts > kMaxTopkParts) parts = kMaxTopkParts;
  return parts < 2 ? 1 : (int)parts;
}

cudaError_t launch_topk_cand(const CandLaunch& p, cudaStream_t st) {
  const int rows = p.B * p.Tc;
  if (rows <= 0) return cudaSuccess;
  if (p.k < 1 || p.k > kCandMaxK || p.cap > kCandMaxCap || p.cap < p.k) return cudaErrorInvalidValue;
  TraceScope trace(kTraceTopk, st);
  const int smem = (int)sizeof(CandSmem);
  cudaError_t e = cudaFuncSetAttribute(k_topk_cand, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k_topk_cand<<<rows, kThreads, smem, st>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_topk_rows(const TopkLaunch& p, cudaStream_t st) {
  const int rows = p.B * p.Tc;
  if (rows <= 0) return cudaSuccess;
  if (p.parts > kMaxTopkParts || (p.parts > 1 && !(p.part_pos && p.part_key && p.part_cnt)))
    return cudaErrorInvalidValue;
  if (p.parts > 1 && !p.gate && p.k <= kCandMaxK) {
    // few long rows: threshold, filter and candidate top-k in the room planned for the segment
    // lists, when it holds the candidate lists (decode: 67 -> about 30 us for 32 rows of 200K)
    const int cap = ((p.k * 4 < 2048 ? 2048 : p.k * 4) + 127) / 128 * 128;
    // (the room starts wherever the caller's score chunk ends: 4-byte aligned; the pairs want 8)
    const uintptr_t at = reinterpret_cast<uintptr_t>(p.part_pos), at16 = (at + 15) & ~(uintptr_t)15;
    const size_t room = (size_t)rows * p.parts * ((size_t)p.k * 8 + 4) - (size_t)(at16 - at);
    const size_t cand_b = (size_t)rows * cap * 8, cnt_b = (size_t)rows * 16, tau_b = (size_t)rows * 4;
    if (cap <= kCandMaxCap && cand_b + cnt_b + tau_b + rows <= room) {
      uint8_t* w = reinterpret_cast<uint8_t*>(at16);
      uint2* cand = reinterpret_cast<uint2*>(w);
      int32_t* cnt = reinterpret_cast<int32_t*>(w + cand_b);
      uint32_t* tau = reinterpret_cast<uint32_t*>(w + cand_b + cnt_b);
      uint8_t* fail = w + cand_b + cnt_b + tau_b;
      int64_t n_max = p.q_pos0 + p.t0 + p.Tc - 1 + p.diag;
      n_max = n_max < 0 ? 0 : (n_max > p.S ? p.S : n_max);
      {
        TraceScope trace(kTraceTopk, st);
        k_row_threshold<<<rows, kThreads, 0, st>>>(p, cap / 2, tau, cnt);
        count_launches(1);
        const unsigned chunks = (unsigned)((n_max + kFiltChunk - 1) / kFiltChunk);
        if (chunks > 0) {
          k_row_filter<<<dim3(chunks, (unsigned)rows), kFiltThreads, 0, st>>>(p, tau, cap, cand, cnt);
          count_launches(1);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
      }
      CandLaunch C{};
      C.B = p.B; C.T = p.T; C.S = p.S; C.t0 = p.t0; C.Tc = p.Tc;
      C.q_pos0 = p.q_pos0; C.diag = p.diag; C.k = p.k; C.cap = cap;
      C.cand = cand; C.cand_cnt = cnt; C.fail = fail; C.idx = p.idx;
      cudaError_t e = launch_topk_cand(C, st);
      if (e != cudaSuccess) return e;
      // rows the candidates could not finish: the one-CTA-per-row pass over their scores
      TopkLaunch g = p;
      g.parts = 1;
      g.gate = fail;
      g.gate_bstride = p.Tc;
      e = p.k <= 2560 ? launch_rows<4096, 2, 16>(g, rows, st) : launch_rows<8192, 2, 8>(g, rows, st);
      count_launches(1);
      return e;
    }
  }
  // about 1.25k + 16 n / Cap candidates are expected: 4096 slots hold them for k <= 2560
  cudaError_t e =
      p.k <= 2560 ? launch_rows<4096, 2, 16>(p, rows, st) : launch_rows<8192, 2, 8>(p, rows, st);
  count_launches(1);
  if (e != cudaSuccess || p.parts <= 1) return e;
  TraceScope trace(kTraceTopk, st);
  if ((int64_t)p.parts * p.k <= kMergeSmemKeys) {
    const int smem = (int)((size_t)p.parts * p.k * sizeof(uint32_t));
    if ((e = cudaFuncSetAttribute(k_topk_merge<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
      return e;
    k_topk_merge<true><<<rows, kThreads, smem, st>>>(p);
  } else {
    k_topk_merge<false><<<rows, kThreads, 0, st>>>(p);
  }
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
