// Lightning-indexer scores on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
//   I[t,s] = sq[t] * sk[s] * sum_h w[t,h] * ReLU(q[t,h] . k[s])
//
// One CTA owns a block of query tokens and walks the key tiles they can see (all of them, or
// one of `ksplit` equal key ranges when there are too few token blocks to fill the GPU, as in
// decode):
//   * MMA shape M = 128 keys (A: the key tile, K-major), N = 256 columns = tokens x heads
//     (B: the stationary query tile, K-major), K = d_I; fp32 accumulators in TMEM, two
//     256-column buffers so the epilogue of tile i overlaps the MMAs of tile i+1 (N = 256
//     reads each key tile from shared memory once; two N = 128 halves were measured slower);
//   * warp 0 streams key tiles with TMA (128-byte swizzle) through a ring of smem stages;
//   * warp 1 allocates TMEM and issues the MMAs from one thread (tcgen05.commit frees the
//     stage and publishes the accumulator);
//   * warps 2..17 read the accumulator (TMEM lane = key) with tcgen05.ld, apply ReLU and the
//     head weights with packed fp32x2 FMAs, apply the per-token scales and write the fp32 score
//     row with coalesced stores.  With 64 heads per token a warp owns one token's 64 columns
//     of its 32 TMEM lanes and reads them with the 16x256b shape, so a thread holds 4 keys x
//     16 heads: its 16 head weights stay in registers for the whole CTA (re-reading them from
//     shared memory every tile saturated the LSU pipe), and a 3-shuffle reduce-scatter over
//     the 4 threads that share the keys leaves each thread one key's sum.
// Selecting mode (the top-k path that stores no scores): a CTA whose rows are longer than the
// candidate room first scores an evenly spread sample of its key tiles and records each
// sampled score's top 16 order-key bits; each token's eight warps then set its threshold (the
// sample's quantile that about `target` of the row's keys should exceed); every tile is then
// scored in order and each score at or above the threshold is kept as a (score, position) pair
// in the row's candidate list quarter of the warp's TMEM lane quarter: where over half a score
// per warp and step qualifies, a lane parks each step's score in shared memory and sets a bit,
// and once per 16 steps (4 for bf16) the warp scans its lanes' counts, claims slots from the
// quarter's count in shared memory and each lane appends its own; sparser rows append under a
// per-step ballot.  The sampled tiles are scored twice (1/64 of the tiles, at least 16), which
// keeps the main pass in plain tile order.  Here the sixteen epilogue warps form two groups of
// eight that take the steps in turn (group g reads accumulator buffer g), each warp reading
// two tokens' columns in four 16-lane loads: a warp's fixed work per step (waits, loads,
// fences, release, key scale, loop) is paid once per two tokens, and every scheduler keeps
// four warps, two working on each buffer (4,096 rows x 128K keys: 4.19 against 4.33 ms with
// one token per warp and step; eight warps of two tokens each, with only two warps per
// scheduler to hide the load latency, took 4.75).
// One-token mode (one query token per block, as in decode): each step's four products cover
// four key tiles (N = 64: the token's heads), one per 64-column group, so all sixteen epilogue
// warps work.
// Every wait is bounded; a timeout raises DSA_FLAG_TIMEOUT, drains the copies in flight,
// frees TMEM and returns.
#include <cuda_bf16.h>

#include <cstdlib>
#include <mutex>

#include "dsa_internal.cuh"
#include "sm100.cuh"

namespace dsa {
namespace {
using namespace sm100;

constexpr int kM = 128;        // keys per tile
constexpr int kN = 256;        // token x head columns per tile and per MMA
constexpr int kBufs = 2;       // TMEM accumulator buffers of kN columns (512 columns)
constexpr int kEpiWarps = 16;  // four per TMEM lane quarter, one per 64-column quarter of N
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr uint32_t kTmemCols = kBufs * kN;
// Selecting mode: at most kSampMax sampled key tiles per CTA, their scores' top 16 key bits
// kept per token in shared memory, two 8-bit histogram passes per token for the threshold.
constexpr int kSampMax = 64;
constexpr int kThBins = 512;  // bins of the threshold histogram (a window of sampled key prefixes)
template <int SAMP>
struct SelSmem {
  uint16_t samp[4][SAMP * kM];
  uint32_t hist[4][kThBins];
  uint32_t part[4][8]; // per token: each warp's bin total
  uint32_t claim[4][4];   // per token and TMEM lane quarter: candidate slots claimed
  int mvis[4];         // visible sampled keys per token
  uint32_t lo[4], hi[4];  // smallest and largest sampled key prefix per token
  uint32_t theta[4];   // per-token threshold key
  int tile[SAMP];      // key tile of each sample step
};

// Sampled tiles of a CTA whose rows are longer than the candidate capacity: 1/64 of its tiles,
// between 16 and `most` (at most all of them).
__host__ __device__ inline int sample_tiles(int ktiles, int most) {
  int ns = ktiles / 64;
  ns = ns < 16 ? 16 : (ns > most ? most : ns);
  return ns < ktiles ? ns : ktiles;
}
// Tile processed at step i of a CTA that first scores nsamp evenly spread sample tiles (their
// tiles listed in `tiles`), then every tile in order.
__device__ __forceinline__ int tile_at(int i, int nsamp, const int* tiles) { return i < nsamp ? tiles[i] : i - nsamp; }
// the kTokThreads epilogue threads of token tok (both groups' warps of its column quarter)
constexpr int kTokThreads = 256;
__device__ __forceinline__ void token_sync(int tok) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(1 + tok), "r"(kTokThreads) : "memory");
}

// The threshold key of token `tok` from its recorded sample, computed by the token's eight
// epilogue warps (thread tt of kTokThreads; every one must call it): the sample's need-th largest
// score, need = ceil(target * sampled / visible), so that about `target` of the row's keys reach
// it, rounded down to a bin of a histogram of the sampled 16-bit key prefixes over the window
// [smallest, largest] (one pass; a row's scores span a narrow range of prefixes).  A threshold
// of 1 keeps every visible non-NaN key (the sample suggests about all of them).
// The target is the least number of keys whose estimate from need sampled ones stays 4.5
// standard deviations (relative error about 1/sqrt(need)) above k: sqrt(target) = (a +
// sqrt(a^2 + 4k)) / 2 with a = 4.5 sqrt(visible / sampled), capped at `most` (the candidate
// room the row has, with margin).
template <class SelSmem>
__device__ __noinline__ uint32_t token_threshold(SelSmem* ss, int tok, int tt, int nsamp, int mv, int64_t n_vis,
                                                 int k, int most) {
  uint32_t* hist = ss->hist[tok];
  const uint16_t* sp = ss->samp[tok];
  const int total = nsamp * kM;
  const int lane = tt & 31, w = tt >> 5;
  token_sync(tok);  // every warp of the token has recorded its sample entries
  uint32_t lo = 0xffffu, hi = 0u;
  for (int i = tt; i < total; i += kTokThreads) {
    const uint32_t k = sp[i];
    if (k) {
      lo = k < lo ? k : lo;
      hi = k > hi ? k : hi;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    atomicMin(&ss->lo[tok], lo);
    atomicMax(&ss->hi[tok], hi);
  }
  atomicAdd(&ss->mvis[tok], mv);
  for (int i = tt; i < kThBins; i += kTokThreads) hist[i] = 0;
  token_sync(tok);
  const int m = ss->mvis[tok];
  // (single precision: the threshold is an estimate, any value keeps the result exact, and
  // double-precision arithmetic is slow on this part)
  int64_t need = 0;
  if (n_vis > 0 && m > 0) {
    const float ratio = (float)n_vis / (float)m;
    const float a = 4.5f * sqrtf(ratio);
    const float r = 0.5f * (a + sqrtf(a * a + 4.0f * (float)k));
    const float target = fminf(r * r, (float)most);
    need = (int64_t)ceilf(target / ratio);
  }
  if (need < 1 || need >= m) return 1u;  // (the same decision in every thread)
  const uint32_t wlo = ss->lo[tok], span = ss->hi[tok] - wlo;
  int sh = 0;
  while ((span >> sh) >= (uint32_t)kThBins) ++sh;
  for (int i = tt; i < total; i += kTokThreads) {
    const uint32_t k = sp[i];
    const uint32_t bin = (k - wlo) >> sh;  // every recorded non-zero prefix lies in the window
    if (k && bin < (uint32_t)kThBins) atomicAdd(&hist[bin], 1u);
  }
  token_sync(tok);
  // thread tt owns the kPer bins kPer*tt .. counted from the top; a scan over the token's
  // threads gives the count above them
  constexpr int kPer = kThBins / kTokThreads;
  uint32_t c[kPer], sum = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    c[j] = hist[kThBins - 1 - (kPer * tt + j)];
    sum += c[j];
  }
  uint32_t inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) ss->part[tok][w] = inc;
  token_sync(tok);
  uint32_t above = inc - sum;
  for (int q = 0; q < w; ++q) above += ss->part[tok][q];
  if (above < (uint32_t)need && (uint32_t)need <= above + sum) {
    uint32_t acc = above;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (acc + c[j] >= (uint32_t)need) {
        const uint32_t bin = (uint32_t)(kThBins - 1 - (kPer * tt + j));
        ss->theta[tok] = (wlo + (bin << sh)) << 16;
        break;
      }
      acc += c[j];
    }
  }
  token_sync(tok);
  return ss->theta[tok];
}

template <int HI, int DI, bool FP8>
struct Cfg {
  static constexpr int kEsz = FP8 ? 1 : 2;
  static constexpr int kRowBytes = DI * kEsz;
  static constexpr int kKBlocks = kRowBytes / 128;  // 128-byte swizzle atoms along d_I
  static constexpr int kAtomElems = 128 / kEsz;
  static constexpr int kTB = kN / HI;               // tokens per CTA
  static constexpr uint32_t kQBlock = kN * 128;
  static constexpr uint32_t kKBlock = kM * 128;
  static constexpr uint32_t kQBytes = kN * kRowBytes;
  static constexpr uint32_t kKTile = kM * kRowBytes;
  static constexpr int kStages = FP8 ? 6 : 4;
  static constexpr int kCols = kN / 4;              // columns read by one epilogue warp
  static constexpr int kBarOff = kQBytes + kStages * kKTile;
  static constexpr size_t kSmem = 1024 + kBarOff + 256 + (size_t)kTB * HI * 4;
  static constexpr uint32_t kIdesc = idesc_mn(FP8 ? 0u : 1u, FP8 ? 0u : 1u, kM, kN);
  static constexpr uint32_t kIdescTok = idesc_mn(FP8 ? 0u : 1u, FP8 ? 0u : 1u, kM, HI);  // one token's heads
  // selecting mode: sampled tiles whose score prefixes fit beside the stages (FP8: 64; the
  // bf16 stages are twice as large, so 16)
  static constexpr int kSamp = FP8 ? kSampMax : 16;
  static_assert(kRowBytes % 128 == 0, "d_I must fill whole 128-byte rows");
  static_assert(kN % HI == 0, "heads must tile the N columns");
};

// Thread t of a warp receives, for each of the x8 repetitions j, TMEM lanes base + t/4 and
// base + t/4 + 8 at columns 8j + 2(t%4) and 8j + 2(t%4) + 1, in that order (r[4j .. 4j+3]).
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ int64_t visible_keys(const IndexerLaunch& p, int t_local) {
  int64_t n = p.q_pos0 + p.t0 + t_local + p.diag;
  return n < 0 ? 0 : (n > p.S ? (int64_t)p.S : n);
}

// Out-of-line append of one batch (see the selecting main loop): the lanes' qualifying scores
// (bit t of a lane's mask: its score of the batch's entry t, parked at vbuf[t * 32 + lane], key
// key0 + t * kstep) go to slots the warp claims from the count it shares with the other group's
// warp of its list quarter.
__device__ __noinline__ void sel_flush(uint32_t mask, const float* vbuf, int lane, uint32_t* claim, int cap4,
                                       uint2* cand, int key0, int kstep) {
  const uint32_t c = __popc(mask);
  uint32_t inc = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, inc, 31);
  if (total == 0) return;
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(claim, total);
  uint32_t slot = __shfl_sync(0xffffffffu, base, 0) + inc - c;
  for (uint32_t mm = mask; mm; mm &= mm - 1, ++slot) {
    const int tb = __ffs(mm) - 1;
    if (slot < (uint32_t)cap4) cand[slot] = make_uint2(__float_as_uint(vbuf[tb * 32 + lane]), (uint32_t)(key0 + tb * kstep));
  }
}

template <int HI, int DI, bool FP8, bool kPoll, bool SEL, bool DEC>
__global__ void __launch_bounds__(kThreads, 1)
    k_indexer_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 IndexerLaunch p) {
  using C = Cfg<HI, DI, FP8>;
  static_assert(!SEL || HI == 64, "the selecting epilogue is written for 64 heads (one token per warp)");
  // DEC (one query token per block, as in decode): each step's four products cover four key
  // tiles (N = 64, the token's heads) in the four 64-column groups of the accumulator, so all
  // sixteen epilogue warps work, one key tile per column group, where one token alone would
  // leave twelve of them idle
  static_assert(!DEC || (HI == 64 && !SEL), "the one-token layout is written for 64 heads, scores stored");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* k_s = smem + C::kQBytes;
  uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* k_empty = k_full + C::kStages;
  uint64_t* q_full = k_empty + C::kStages;
  uint64_t* tm_full = q_full + 1;
  uint64_t* tm_empty = tm_full + kBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tm_empty + kBufs);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* w_s = reinterpret_cast<float*>(smem + C::kBarOff + 256);
  using Sel = SelSmem<C::kSamp>;
  Sel* ss = reinterpret_cast<Sel*>(smem + C::kBarOff + 256 + (size_t)C::kTB * HI * 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = (p.Tc + C::kTB - 1) / C::kTB;
  const int tb = nblk - 1 - (int)(blockIdx.x / p.ksplit);  // latest (longest) token blocks first
  const int split = (int)(blockIdx.x % p.ksplit);
  const int b = blockIdx.y;
  const int tl0 = tb * C::kTB;
  const int ntok = min(C::kTB, p.Tc - tl0);
  if (p.gate) {
    // recomputing only the rows a selecting pass could not finish: leave unless one of this
    // block's rows is marked (before any barrier, copy or tensor memory is touched)
    bool any = false;
    for (int i = 0; i < ntok; ++i) any |= p.gate[(int64_t)b * p.gate_bstride + tl0 + i] != 0;
    if (!any) return;
  }
  // epilogue warps own one column quarter each; quarters that hold none of this block's
  // tokens (decode: one token per block) have no work, so they sit the tiles out and the
  // accumulator buffers wait only for the others
  constexpr int kTokWarp = C::kCols / HI > 0 ? C::kCols / HI : 1;
  const int active_ch = DEC ? kEpiWarps / 4 : min(kEpiWarps / 4, (ntok + kTokWarp - 1) / kTokWarp);
  // selecting mode: the epilogue warps form two groups of eight, group g reading accumulator
  // buffer g (the steps of its parity); a warp reads the column quarters of a token pair
  const int active_pairs = (active_ch + 1) / 2;
  const int64_t nmax = visible_keys(p, tl0 + ntok - 1);
  // this CTA's key tiles: [kt_lo, kt_lo + ktiles) of the ceil(S / kM) tiles of the row
  const int tiles_all = (p.S + kM - 1) / kM;
  const int tps = (tiles_all + p.ksplit - 1) / p.ksplit;
  const int kt_lo = split * tps;
  const int kt_vis = (int)((nmax + kM - 1) / kM);
  const int ktiles = max(0, min(kt_vis, kt_lo + tps) - kt_lo);
  const int key_hi = min(p.S, (kt_lo + tps) * kM);  // end of this CTA's key range
  const int64_t row0 = (int64_t)b * p.T + p.t0 + tl0;  // flat (b, t) of the block's first token
  // selecting mode: rows longer than the candidate capacity first score a sample of tiles
  const int nsamp = (SEL && nmax > p.cap) ? sample_tiles(ktiles, C::kSamp) : 0;
  const int nproc = DEC ? (ktiles + 3) / 4 : nsamp + ktiles;  // steps of the MMA and the epilogue
  const int nload = DEC ? ktiles : nproc;                      // tiles the producer streams

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
    }
    mbar_init(q_full, 1);
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(tm_full + i, 1);
      mbar_init(tm_empty + i, SEL ? 4 * active_pairs : 4 * active_ch);  // the warps that read buffer i
    }
    *abort_flag = 0;
    if constexpr (SEL)
      for (int i = 0; i < 4; ++i) {
        ss->mvis[i] = 0;
        ss->lo[i] = 0xffffu;
        ss->hi[i] = 0u;
        ss->theta[i] = 1u;
        for (int q = 0; q < 4; ++q) ss->claim[i][q] = 0u;
      }
    fence_barrier_init();
  }
  if constexpr (SEL)  // the sample tiles, evenly spread over the CTA's tiles
    for (int s2 = threadIdx.x; s2 < nsamp; s2 += kThreads) ss->tile[s2] = ((2 * s2 + 1) * ktiles) / (2 * nsamp);
  for (int i = threadIdx.x; i < C::kTB * HI; i += kThreads)
    w_s[i] = (i / HI < ntok) ? __ldg(p.w + row0 * HI + i) : 0.f;
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && ktiles > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      mbar_arrive_expect_tx(q_full, C::kQBytes);
      for (int kb = 0; kb < C::kKBlocks; ++kb)
        tma_load_4d(q_s + kb * C::kQBlock, &tm_q, q_full, kb * C::kAtomElems, 0, p.t0 + tl0, b);
      int issued = 0;
      for (int i = 0; i < nload; ++i) {
        const int kt = SEL ? tile_at(i, nsamp, ss->tile) : i;
        const int st = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        if (!mbar_wait<kPoll, true>(k_empty + st, ph ^ 1, abort_flag, p.wait)) break;
        mbar_arrive_expect_tx(k_full + st, C::kKTile);
        for (int kb = 0; kb < C::kKBlocks; ++kb)
          tma_load_3d(k_s + st * C::kKTile + kb * C::kKBlock, &tm_k, k_full + st, kb * C::kAtomElems,
                      (kt_lo + kt) * kM, b);
        issued = i + 1;
      }
      // every copy issued lands before the CTA can exit: a wait elsewhere in the CTA may run
      // out after this loop has ended (in a normal run these phases are long complete)
      mbar_wait_drain(q_full, 0);
      for (int kt = issued > C::kStages ? issued - C::kStages : 0; kt < issued; ++kt)
        mbar_wait_drain(k_full + kt % C::kStages, (kt / C::kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && ktiles > 0) {
      bool ok = mbar_wait<kPoll>(q_full, 0, abort_flag, p.wait);
      int done = 0;
      const uint64_t q_desc0 = desc_sw128(smem_addr(q_s));
      const uint64_t k_desc0 = desc_sw128(smem_addr(k_s));
      for (int kt = 0; ok && kt < nproc; ++kt) {  // kt: processing step (the tile itself is the producer's)
        const int buf = kt & (kBufs - 1);
        if (!(ok = mbar_wait<kPoll, true>(tm_empty + buf, ((kt / kBufs) & 1) ^ 1, abort_flag, p.wait))) break;
        // one tile (N = 256: the block's tokens x heads), or DEC: up to four tiles, one per
        // 64-column group (N = 64: the token's heads)
        const int ntile = DEC ? min(4, ktiles - 4 * kt) : 1;
        int issued_c = 0;
        for (int c = 0; ok && c < ntile; ++c) {
          const int ti = DEC ? 4 * kt + c : kt;  // the tile's place in the producer's stream
          const int st = ti % C::kStages;
          if (!(ok = mbar_wait<kPoll, true>(k_full + st, (ti / C::kStages) & 1, abort_flag, p.wait))) break;
          tc_fence_after();
          const uint32_t d = tmem + buf * kN + (DEC ? c * 64 : 0);
          const uint64_t kd = k_desc0 + (uint64_t)((st * C::kKTile) >> 4);
#pragma unroll
          for (int kb = 0; kb < C::kKBlocks; ++kb)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              // base descriptors + compile-time offsets in the 16-byte start-address field
              const uint64_t ad = kd + (uint64_t)((kb * C::kKBlock + j * 32) >> 4);
              const uint64_t bd = q_desc0 + (uint64_t)((kb * C::kQBlock + j * 32) >> 4);
              constexpr uint32_t id = DEC ? C::kIdescTok : C::kIdesc;
              if constexpr (FP8)
                mma_fp8(d, ad, bd, id, (kb | j) != 0);
              else
                mma_bf16(d, ad, bd, id, (kb | j) != 0);
            }
          mma_commit(k_empty + st);
          ++issued_c;
        }
        // the accumulator's commit also covers a step cut short by a wait that ran out, so the
        // drain below waits for every product issued
        if (issued_c > 0) {
          mma_commit(tm_full + buf);
          done = kt + 1;
        }
        if (!ok) break;
      }
      // the products issued are complete before TMEM can be freed, whichever wait ran out
      if (done > 0) mbar_wait_drain(tm_full + ((done - 1) & (kBufs - 1)), ((done - 1) / kBufs) & 1);
    }
  } else if (SEL ? (((warp - 2) >> 2) & 1) < active_pairs : ((warp - 2) >> 2) < active_ch) {
    // ---------------- epilogue ----------------
    const int e = warp - 2;
    const int lq = warp & 3;                 // TMEM lane quarter this warp may read
    const int ch = e >> 2;                   // column quarter (one 64-column slice of N)
    const int wtok = DEC ? 0 : ch;           // HI = 64: the token of this warp's columns
    const int key_in_tile = lq * 32 + lane;  // TMEM lane = key
    const uint32_t t_lane = tmem + ((uint32_t)(lq * 32) << 16);
    float* out_b = p.out + (int64_t)b * p.out_bstride;
    const float* skg = FP8 ? p.k_scale + (int64_t)b * p.S : nullptr;

    constexpr int kTokW = C::kCols / HI > 0 ? C::kCols / HI : 1;  // tokens per epilogue warp
    const float* w_warp = w_s + (DEC ? 0 : ch * C::kCols);          // this warp's columns' weights

    // per-token constants of this warp's tokens, held in registers
    int64_t nvis[kTokW];
    float sq[kTokW];
#pragma unroll
    for (int tk = 0; tk < kTokW; ++tk) {
      const int tok = DEC ? 0 : ch * kTokW + tk;
      nvis[tk] = tok < ntok ? visible_keys(p, tl0 + tok) : 0;
      sq[tk] = (FP8 && tok < ntok) ? __ldg(p.q_scale + row0 + tok) : 1.f;
    }
    // key scales are fetched one tile ahead so their latency hides behind the tile's work
    auto key_scale = [&](int kt) -> float {
      const int key = (kt_lo + kt) * kM + key_in_tile;
      return (FP8 && kt < ktiles && key < p.S) ? __ldg(skg + key) : 1.f;
    };
    float sk_next = key_scale(0);

    if constexpr (HI == 64) {
      // one token per warp; thread t: keys kq + t/4 + {0, 8, 16, 24}, heads 8j + 2(t%4) + {0, 1}
      const int m = lane & 3, rq = lane >> 2;
      const int my_key = lq * 32 + (m >> 1) * 16 + (m & 1) * 8 + rq;  // the key this thread stores
      // halved weights: w * ReLU(x) = (w / 2) * (x + |x|), both factors exact, so the product
      // rounds exactly as w * max(x, 0) does (finite x); the add runs on the FMA pipe with a
      // free |.| operand, where a max would take an ALU-pipe slot
      unsigned long long wp[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        wp[j] = pack2(0.5f * w_warp[8 * j + 2 * m], 0.5f * w_warp[8 * j + 2 * m + 1]);
      auto key_scale16 = [&](int kt) -> float {  // key scale of this thread's key in tile kt
        const int key = (kt_lo + kt) * kM + my_key;
        return (FP8 && kt < ktiles && key < p.S) ? __ldg(skg + key) : 1.f;
      };
      // the same by key, clamped to the last key (a key past the row's end is never kept)
      auto key_scale_at = [&](int key) -> float { return FP8 ? __ldg(skg + min(key, p.S - 1)) : 1.f; };
      // Head-weighted ReLU sums over this thread's 16 heads of one token for the two keys of
      // a 16-lane half a (keys a*16 + {0, 8} + rq), from that half's 32 registers of a 16x256b
      // load (ra[4j + 2e + {0,1}]: key a*16 + e*8 + rq, heads 8j + 2m + {0,1}), into acc_e0 and
      // acc_e1 as two partial sums each (even / odd head of each pair).
      auto accum_half = [&](const uint32_t (&ra)[32], const unsigned long long (&w)[8], unsigned long long& acc_e0,
                            unsigned long long& acc_e1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float y0 = __uint_as_float(ra[4 * j]), y1 = __uint_as_float(ra[4 * j + 1]);
          const float y2 = __uint_as_float(ra[4 * j + 2]), y3 = __uint_as_float(ra[4 * j + 3]);
          acc_e0 = fma2(pack2(y0 + fabsf(y0), y1 + fabsf(y1)), w[j], acc_e0);
          acc_e1 = fma2(pack2(y2 + fabsf(y2), y3 + fabsf(y3)), w[j], acc_e1);
        }
      };
      // reduce-scatter of the four keys' sums over the 4 threads of a key group: thread m ends
      // with key index m's total
      auto xlane = [&](const unsigned long long (&acc)[4]) -> float {
        float v4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v4[q] = lo2(acc[q]) + hi2(acc[q]);
        const bool hi1 = (m & 2) != 0, hi0 = (m & 1) != 0;
        const float s0 = hi1 ? v4[0] : v4[2], s1 = hi1 ? v4[1] : v4[3];
        const float k0 = hi1 ? v4[2] : v4[0], k1 = hi1 ? v4[3] : v4[1];
        const float u0 = k0 + __shfl_xor_sync(0xffffffffu, s0, 2);
        const float u1 = k1 + __shfl_xor_sync(0xffffffffu, s1, 2);
        return (hi0 ? u1 : u0) + __shfl_xor_sync(0xffffffffu, hi0 ? u0 : u1, 1);
      };
      // The head-weighted ReLU sum of this thread's key for the accumulator of step i (false:
      // a wait ran out).  The buffer goes back to the MMA right after the TMEM loads.
      auto score_step = [&](int i, float& v) -> bool {
        const int buf = i & (kBufs - 1);
        if (!mbar_wait<kPoll, true>(tm_full + buf, (i / kBufs) & 1, abort_flag, p.wait)) return false;
        tc_fence_after();
        const uint32_t col0 = tmem + ((uint32_t)(lq * 32) << 16) + buf * kN + ch * C::kCols;
        uint32_t r[2][32];
        tmem_ld_16x256b_x8(col0, r[0]);
        tmem_ld_16x256b_x8(col0 + (16u << 16), r[1]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tm_empty + buf);
        unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
        accum_half(r[0], wp, acc[0], acc[1]);
        accum_half(r[1], wp, acc[2], acc[3]);
        v = xlane(acc);
        return true;
      };
      if constexpr (SEL) {
        // Selecting mode.  Two groups of eight warps take the steps in turn (group g: the steps
        // of parity g, whose accumulator is buffer g), each warp reading the column quarters of
        // a token pair, so a warp's fixed work per step (waits, loads, fences, release, key
        // scale, loop) is paid once per two tokens while each scheduler still holds four
        // working warps.  Sample steps record the top 16 key bits of each sampled score; each
        // token's eight warps then set its threshold (every visible non-NaN key when the row is
        // short enough to keep whole); the main steps keep (key, position) of every score that
        // reaches it, in the row's list quarter of the warp's TMEM lane quarter (the two groups'
        // warps of a quarter claim its slots from a count in shared memory).
        const int grp = e >> 3;              // this warp's group, and the buffer it reads
        const int pr = (e >> 2) & 1;         // its token pair
        const int c0 = 2 * pr;               // the pair's first token (column quarter)
        const bool has1 = c0 + 1 < ntok;     // the pair's second token exists
        unsigned long long wq0[8], wq1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          wq0[j] = pack2(0.5f * w_s[c0 * HI + 8 * j + 2 * m], 0.5f * w_s[c0 * HI + 8 * j + 2 * m + 1]);
          wq1[j] = pack2(0.5f * w_s[(c0 + 1) * HI + 8 * j + 2 * m], 0.5f * w_s[(c0 + 1) * HI + 8 * j + 2 * m + 1]);
        }
        const int nv0 = (int)visible_keys(p, tl0 + c0);
        const int nv1 = has1 ? (int)visible_keys(p, tl0 + c0 + 1) : 0;
        const float sq0 = FP8 ? __ldg(p.q_scale + row0 + c0) : 1.f;
        const float sq1 = (FP8 && has1) ? __ldg(p.q_scale + row0 + c0 + 1) : 1.f;
        const uint32_t t_pair = tmem + ((uint32_t)(lq * 32) << 16) + grp * kN + c0 * C::kCols;  // in buffer grp
        // Both tokens' sums for step i (of this group's parity; false: a wait ran out): four
        // loads of 16 lanes x 64 columns into one set of registers, each summed before the next;
        // the buffer goes back to the MMA once the last is loaded.
        auto step2 = [&](int i, float& v0, float& v1) -> bool {
          if (!mbar_wait<kPoll, true>(tm_full + grp, (i / kBufs) & 1, abort_flag, p.wait)) return false;
          tc_fence_after();
          uint32_t r[32];
          unsigned long long x0[4] = {0ull, 0ull, 0ull, 0ull}, x1[4] = {0ull, 0ull, 0ull, 0ull};
          tmem_ld_16x256b_x8(t_pair, r);
          tmem_wait_ld();
          accum_half(r, wq0, x0[0], x0[1]);
          tmem_ld_16x256b_x8(t_pair + (16u << 16), r);
          tmem_wait_ld();
          accum_half(r, wq0, x0[2], x0[3]);
          tmem_ld_16x256b_x8(t_pair + C::kCols, r);
          tmem_wait_ld();
          accum_half(r, wq1, x1[0], x1[1]);
          tmem_ld_16x256b_x8(t_pair + C::kCols + (16u << 16), r);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tm_empty + grp);
          accum_half(r, wq1, x1[2], x1[3]);
          v0 = xlane(x0);
          v1 = xlane(x1);
          return true;
        };
        bool dead = false;
        int mv0 = 0, mv1 = 0;  // visible sampled keys seen by this thread, per token
        for (int i = grp; i < nsamp; i += kBufs) {
          if (dead) continue;  // still meet the threshold barriers below
          const int key = (kt_lo + ss->tile[i]) * kM + my_key;
          const float sk = key_scale_at(key);
          float v0, v1;
          if (!step2(i, v0, v1)) {
            dead = true;
            continue;
          }
          if constexpr (FP8) {
            v0 *= sq0 * sk;
            v1 *= sq1 * sk;
          }
          const bool vis0 = key < nv0, vis1 = key < nv1;
          ss->samp[c0][i * kM + my_key] = vis0 ? (uint16_t)(score_key(v0) >> 16) : (uint16_t)0;
          ss->samp[c0 + 1][i * kM + my_key] = vis1 ? (uint16_t)(score_key(v1) >> 16) : (uint16_t)0;
          mv0 += vis0;
          mv1 += vis1;
        }
        const int tt = (grp * 4 + (e & 3)) * 32 + lane;  // this thread among its tokens' kTokThreads
        const uint32_t theta0 = nsamp > 0 ? token_threshold(ss, c0, tt, nsamp, mv0, nv0, p.topk, p.target) : 1u;
        const uint32_t theta1 =
            (nsamp > 0 && has1) ? token_threshold(ss, c0 + 1, tt, nsamp, mv1, nv1, p.topk, p.target) : 1u;
        const int64_t crow0 = (int64_t)b * p.Tc + tl0 + c0;  // chunk-local row of the first token
        const int cap4 = p.cap / 4;
        uint2* cand0 = p.cand + crow0 * p.cap + lq * cap4;
        uint2* cand1 = cand0 + p.cap;  // the second token's row (written only when it exists)
        uint32_t* claim0 = &ss->claim[c0][lq];
        uint32_t* claim1 = &ss->claim[c0 + 1][lq];
        // the thresholds as floats: scores v >= thf are exactly those whose order key reaches
        // theta (-inf keeps every non-NaN score)
        auto th_float = [](uint32_t th) {
          return th == 1u ? -INFINITY : __uint_as_float((th & 0x80000000u) ? (th & 0x7fffffffu) : ~th);
        };
        const float thf0 = th_float(theta0), thf1 = th_float(theta1);
        // this group's first main step (parity grp) and its tile's key; a warp steps two tiles on
        const int i0 = nsamp + ((grp - nsamp) & 1);
        int key = (kt_lo + i0 - nsamp) * kM + my_key;
        float sk_next = key_scale_at(key);
        // Batched append: every step only records each lane's two scores in shared memory (the
        // tokens' sample areas, no longer read once the thresholds are set) and one bit per step
        // in a lane mask per token; once per batch of kBatch steps the warp scans the lanes'
        // counts and each lane appends its own qualifying scores.  The lists are unordered; the
        // top-k orders its selection by position.
        constexpr int kBatch = FP8 ? 16 : 4;
        static_assert(sizeof(ss->samp[0]) >= 8 * kBatch * 32 * sizeof(float), "batch exceeds the token's sample area");
        const int slice = (grp * 4 + (e & 3)) * kBatch * 32;  // this warp's part of a sample area
        float* vbuf0 = reinterpret_cast<float*>(ss->samp[c0]) + slice;
        float* vbuf1 = reinterpret_cast<float*>(ss->samp[c0 + 1]) + slice;
        const uint32_t vb0 = smem_addr(vbuf0 + lane), vb1 = smem_addr(vbuf1 + lane);  // slots of entry 0
        // Rows whose threshold keeps under half a score per warp and step (long rows: 0.15 at
        // 1M keys, 1.2 at 128K) append at once under a ballot instead, which skips most steps
        // entirely.
        const bool batched = (float)p.target * 32.f >= 0.5f * (float)(nv0 > 0 ? nv0 : 1);
        if (batched) {
          uint32_t mask0 = 0, mask1 = 0;  // bit t: this lane's score of the batch's entry t qualifies
          int tb = 0, kbase = key;        // entries parked; the key of entry 0
          auto flush = [&]() {
            sel_flush(mask0, vbuf0, lane, claim0, cap4, cand0, kbase, kBufs * kM);
            if (has1) sel_flush(mask1, vbuf1, lane, claim1, cap4, cand1, kbase, kBufs * kM);
            mask0 = mask1 = 0;
          };
          for (int i = i0; !dead && i < nproc; i += kBufs, key += kBufs * kM) {
            const float sk = sk_next;
            sk_next = key_scale_at(key + kBufs * kM);
            float v0, v1;
            if (!step2(i, v0, v1)) break;
            if constexpr (FP8) {
              v0 *= sq0 * sk;
              v1 *= sq1 * sk;
            }
            asm volatile("st.shared.f32 [%0], %1;\n" ::"r"(vb0 + (uint32_t)tb * 128u), "f"(v0) : "memory");
            asm volatile("st.shared.f32 [%0], %1;\n" ::"r"(vb1 + (uint32_t)tb * 128u), "f"(v1) : "memory");
            mask0 |= (key < nv0 && v0 >= thf0 ? 1u : 0u) << tb;
            mask1 |= (key < nv1 && v1 >= thf1 ? 1u : 0u) << tb;
            if (++tb == kBatch) {
              flush();
              tb = 0;
              kbase = key + kBufs * kM;
            }
          }
          if (tb) flush();  // the last, partial batch
        } else {
          const uint32_t below = (1u << lane) - 1u;
          auto append = [&](bool take, float v, uint32_t* claim, uint2* cand) {
            const uint32_t bal = __ballot_sync(0xffffffffu, take);
            if (bal) {
              uint32_t base = 0;
              if (lane == 0) base = atomicAdd(claim, (uint32_t)__popc(bal));
              base = __shfl_sync(0xffffffffu, base, 0);
              if (take) {
                const uint32_t slot = base + __popc(bal & below);
                if (slot < (uint32_t)cap4) cand[slot] = make_uint2(__float_as_uint(v), (uint32_t)key);
              }
            }
          };
          for (int i = i0; !dead && i < nproc; i += kBufs, key += kBufs * kM) {
            const float sk = sk_next;
            sk_next = key_scale_at(key + kBufs * kM);
            float v0, v1;
            if (!step2(i, v0, v1)) break;
            if constexpr (FP8) {
              v0 *= sq0 * sk;
              v1 *= sq1 * sk;
            }
            append(key < nv0 && v0 >= thf0, v0, claim0, cand0);
            append(key < nv1 && v1 >= thf1, v1, claim1, cand1);
          }
        }
        // both groups' warps of the pair have claimed their slots; group 0 publishes the counts
        asm volatile("bar.sync %0, %1;\n" ::"r"(5 + pr), "r"(kTokThreads) : "memory");
        if (grp == 0 && lane == 0) {
          p.cand_cnt[crow0 * 4 + lq] = (int32_t)*claim0;
          if (has1) p.cand_cnt[(crow0 + 1) * 4 + lq] = (int32_t)*claim1;
        }
      } else {
        // step i holds tile i (the block's tokens in the column groups), or DEC: tiles 4i .. 4i+3,
        // tile 4i + ch in this warp's column group
        auto tile_of = [&](int i) { return DEC ? 4 * i + ch : i; };
        float sk16_next = key_scale16(tile_of(0));
        for (int kt = 0; kt < nproc; ++kt) {
          const float sk = sk16_next;
          sk16_next = key_scale16(tile_of(kt + 1));
          float v;
          if (!score_step(kt, v)) break;
          const int ti = tile_of(kt);
          const int key = (kt_lo + ti) * kM + my_key;
          if ((DEC ? ti < ktiles : ntok > ch) && key < p.S) {
            float* dst = out_b + (int64_t)(tl0 + wtok) * p.ld + key;
            if (key < nvis[0]) {
              if constexpr (FP8) v *= sq[0] * sk;
              *dst = v;
            } else if (p.write_masked) {
              *dst = -INFINITY;
            }
          }
        }
      }
    } else {
    for (int kt = 0; kt < ktiles; ++kt) {
        const int buf = kt & (kBufs - 1);
        const float sk = sk_next;
        sk_next = key_scale(kt + 1);
        if (!mbar_wait<kPoll, true>(tm_full + buf, (kt / kBufs) & 1, abort_flag, p.wait)) break;
        tc_fence_after();
        const uint32_t col0 = t_lane + buf * kN + ch * C::kCols;
        // all of this warp's accumulator columns in one go, then the buffer goes back to the MMA
        uint32_t r[C::kCols / 32][32];
#pragma unroll
        for (int cb = 0; cb < C::kCols / 32; ++cb) tmem_ld32(col0 + cb * 32, r[cb]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tm_empty + buf);
        const int key = (kt_lo + kt) * kM + key_in_tile;
#pragma unroll
        for (int tk = 0; tk < kTokW; ++tk) {
          // four independent partial sums per token keep the FMA pipe fed
          unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
          float acc1 = 0.f;
#pragma unroll
          for (int c4 = 0; c4 < HI / 4; ++c4) {
            const int c = tk * HI + c4 * 4;  // column within the warp
            const float4 wv = *reinterpret_cast<const float4*>(w_warp + c);
            const float x0 = fmaxf(__uint_as_float(r[c >> 5][c & 31]), 0.f);
            const float x1 = fmaxf(__uint_as_float(r[(c + 1) >> 5][(c + 1) & 31]), 0.f);
            const float x2 = fmaxf(__uint_as_float(r[(c + 2) >> 5][(c + 2) & 31]), 0.f);
            const float x3 = fmaxf(__uint_as_float(r[(c + 3) >> 5][(c + 3) & 31]), 0.f);
            if constexpr (HI >= 8) {
              acc[(2 * c4) & 3] = fma2(pack2(wv.x, wv.y), pack2(x0, x1), acc[(2 * c4) & 3]);
              acc[(2 * c4 + 1) & 3] = fma2(pack2(wv.z, wv.w), pack2(x2, x3), acc[(2 * c4 + 1) & 3]);
            } else {
              acc1 += wv.x * x0 + wv.y * x1 + wv.z * x2 + wv.w * x3;
            }
          }
          float v;
          if constexpr (HI >= 8)
            v = ((lo2(acc[0]) + hi2(acc[0])) + (lo2(acc[1]) + hi2(acc[1]))) +
                ((lo2(acc[2]) + hi2(acc[2])) + (lo2(acc[3]) + hi2(acc[3])));
          else
            v = acc1;
          const int tok = ch * kTokW + tk;
          if (tok < ntok && key < p.S) {
            float* dst = out_b + (int64_t)(tl0 + tok) * p.ld + key;
            if (key < nvis[tk]) {
              if constexpr (FP8) v *= sq[tk] * sk;
              *dst = v;
            } else if (p.write_masked) {
              *dst = -INFINITY;
            }
          }
        }
      }
    }
    if (p.write_masked && !*abort_flag) {  // keys beyond every visible tile
      for (int tk = 0; tk < kTokW; ++tk) {
        const int tok = ch * kTokW + tk;
        if (tok >= ntok) break;
        for (int key = (kt_lo + ktiles) * kM + key_in_tile; key < key_hi; key += kM)
          out_b[(int64_t)(tl0 + tok) * p.ld + key] = -INFINITY;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }

  if (threadIdx.x == 0 && *abort_flag && p.flags) atomicOr(p.flags, DSA_FLAG_TIMEOUT);
}

// ---- host side -------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// Map over a `rank`-dimensional tensor whose innermost dimension holds row_elems contiguous
// codes: dims[0] = row_elems, dims[1..rank-1] with byte strides strides[0..rank-2]; box
// (atom_elems x box[1] x ...), 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, bool fp8, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int HI, int DI, bool FP8, bool SEL, bool DEC = false>
cudaError_t launch_cfg(const IndexerLaunch& p, cudaStream_t st) {
  TraceScope trace(kTraceIndexer, st);
  using C = Cfg<HI, DI, FP8>;
  CUtensorMap tq, tk;
  const cuuint64_t esz = FP8 ? 1 : 2;
  // queries [B][T][H_I][d_I] with token strides q_st / q_sb: a box is the block's kTB tokens
  // x H_I heads x one swizzle atom of d_I, i.e. the [kTB * H_I = kN][atom] tile the MMA reads
  const cuuint64_t qdims[4] = {(cuuint64_t)DI, (cuuint64_t)HI, (cuuint64_t)p.T, (cuuint64_t)p.B};
  const cuuint64_t qstr[3] = {(cuuint64_t)DI * esz, (cuuint64_t)p.q_st * esz, (cuuint64_t)p.q_sb * esz};
  const cuuint32_t qbox[4] = {(cuuint32_t)C::kAtomElems, (cuuint32_t)HI, (cuuint32_t)C::kTB, 1};
  cudaError_t e = make_map(&tq, p.q, FP8, 4, qdims, qstr, qbox);
  if (e != cudaSuccess) return e;
  const cuuint64_t kdims[3] = {(cuuint64_t)DI, (cuuint64_t)p.S, (cuuint64_t)p.B};
  const cuuint64_t kstr[2] = {(cuuint64_t)DI * esz, (cuuint64_t)p.k_sb * esz};
  const cuuint32_t kbox[3] = {(cuuint32_t)C::kAtomElems, (cuuint32_t)kM, 1};
  if ((e = make_map(&tk, p.k, FP8, 3, kdims, kstr, kbox)) != cudaSuccess) return e;
  IndexerLaunch q = p;
  if (q.wait <= 0) q.wait = wait_limit();
  auto kern = q.wait < kDefaultWaitCycles ? k_indexer_tc<HI, DI, FP8, true, SEL, DEC>
                                          : k_indexer_tc<HI, DI, FP8, false, SEL, DEC>;
  const size_t smem = C::kSmem + (SEL ? sizeof(SelSmem<C::kSamp>) : 0);
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return e;
  const int nblk = (p.Tc + C::kTB - 1) / C::kTB;
  if (SEL) q.ksplit = 1;  // a row's candidates come from one CTA
  if (q.ksplit <= 0) {
    // split the key range when the token blocks alone would not give about four waves of
    // CTAs (or ctas_min), keeping at least 16 key tiles per split
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long ctas = (long long)nblk * p.B;
    const int tiles_all = (p.S + kM - 1) / kM;
    const long long goal = p.ctas_min > 4LL * sms ? (long long)p.ctas_min : 4LL * sms;
    long long want = ctas >= goal ? 1 : (goal + ctas - 1) / ctas;
    const long long most = tiles_all / 16 > 0 ? tiles_all / 16 : 1;
    q.ksplit = (int)(want < most ? want : most);
  }
  dim3 grid((unsigned)(nblk * q.ksplit), p.B);
  kern<<<grid, kThreads, smem, st>>>(tq, tk, q);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_scores(const IndexerLaunch& p, cudaStream_t st) {
  if (p.B <= 0 || p.Tc <= 0 || p.S <= 0) return cudaSuccess;
  if (p.HI == 64 && p.DI == 128) {
    if (p.select)
      return p.fp8 ? launch_cfg<64, 128, true, true>(p, st) : launch_cfg<64, 128, false, true>(p, st);
    if (p.Tc == 1)  // one query token per block (decode): four key tiles per step
      return p.fp8 ? launch_cfg<64, 128, true, false, true>(p, st) : launch_cfg<64, 128, false, false, true>(p, st);
    return p.fp8 ? launch_cfg<64, 128, true, false>(p, st) : launch_cfg<64, 128, false, false>(p, st);
  }
  if (p.HI == 4 && p.DI == 64 && !p.fp8 && !p.select) return launch_cfg<4, 64, false, false>(p, st);
  return cudaErrorInvalidValue;
}

}  // namespace dsa
