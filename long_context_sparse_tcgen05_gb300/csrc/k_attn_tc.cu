// Sparse MLA attention over index-selected latent-KV rows on tcgen05 tensor cores.
//
// Shapes: H = 64 query heads of width 576 (512 latent + 64 rope) attend, multi-query,
// over k selected rows of a shared 576-wide latent KV; the value is the first 512 columns
// of the same row, so each gathered row feeds both products.
//
// Persistent CTAs (one per SM) walk query rows.  For each row:
//   * warps 0..3 gather the selected KV rows, 64 per block,
//     with 16-byte cp.async copies into two 128-byte-swizzled stages, prefetching the rows of
//     the block two ahead into L2 (the stage's fill latency, mostly DRAM misses, paces the
//     ring).  A stage lands in three groups of three atoms (an atom: 64 columns of all 64
//     rows), each group with its own barrier, so the score product starts on the first columns
//     while the rest are still in flight.  Every copying thread arrives on a group's barrier,
//     and those arrivals pace the gather: one barrier per atom moved about 17% fewer bytes per
//     second than one per stage (and 32-row stages, with twice the arrivals per byte, half as
//     many);
//   * warp 4 loads each row's query tile with TMA, once its own last score product of the
//     previous row is done with the buffer (so the gathers never wait for it), and issues
//     S = Q K^T  (M = 64 heads, N = 64 keys, K = 576) into TMEM, group by group;
//   * warp 5 issues  O^T += V^T P^T  (M = 128 value dims x 4, N = 64 heads, K = 64 keys) -- the
//     transposed value product keeps the 64 x 512 fp32 accumulator in 256 TMEM columns.  Two
//     issuing threads let the tensor pipe interleave the two products (a single issuer stalls
//     in the 36-instruction score chain while a value product is ready).  It runs dimension
//     chunk by chunk, each chunk releasing its two atoms of the stage (the last also the rope
//     atom), so the gather of the block two ahead refills the stage while the rest of the value
//     product still runs (8,192 rows x 2,048 keys: 3.47 -> 3.24 ms against one release per
//     stage);
//   * warps 6..13 run the softmax, two warps per TMEM lane quarter, each on 32 of the block's
//     64 keys (base-2 exponent, fp32 row sums; the two halves of a head exchange partial sums
//     through shared memory; bf16 P is written into the block's rope columns, free once S is
//     done).  The fixed-reference pass takes a reference maximum of 0 (below); the
//     running-maximum form raises its maximum only when a block exceeds it by more than 2^8
//     (the two halves exchange block maxima) and then rescales O^T in TMEM.  At the end they
//     normalise O and write bf16 O -- each warp's four 32-head slices of O^T loaded in turn, a
//     slice landing while the one before it is stored, lane pairs storing two neighbouring
//     dimensions of a head as one 4-byte word (the epilogue took about 7,450 cycles a row with
//     one 2-byte store per element, 4,650 this way) -- and the natural-log LSE.
// One launch may cover several layers that read the same index rows (each with its own
// queries, latent KV, output and LSE): work items run over layers x rows.  With fewer rows
// than SMs (decode) a row's blocks are split over several CTAs: each writes its part
// normalised by its own row sums, in fp32, with its LSE, and k_attn_combine merges the parts
// (weights exp(LSE_part - LSE_row)).
// Entries of -1 are skipped (masked), out-of-range entries raise DSA_FLAG_BAD_INDEX and are
// skipped.  Every wait is bounded (DSA_FLAG_TIMEOUT); TMEM is freed on every exit path.
#include <cuda_bf16.h>

#include <cstdlib>
#include <mutex>

#include "dsa_internal.cuh"
#include "sm100.cuh"

namespace dsa {
namespace {
using namespace sm100;

constexpr int kH = 64, kDQK = 576, kDV = 512;
// Keys per block (N of the S product, K of the PV product) and blocks in flight.  64 x 2 fills
// shared memory beside the query tile; 32 x 4 (the same bytes, shorter per-block steps) was
// measured 1.55x slower (5.98 against 3.87 ms over 8,192 rows of 2,048 keys).
constexpr int kNB = 64;
constexpr int kStages = 2;
static_assert(kNB == 64 || kNB == 32, "P rows are 128- or 64-byte swizzled");
constexpr int kHalf = kNB / 2;             // keys of a block per softmax warp
constexpr int kAtoms = kDQK / 64;          // 9 swizzle atoms of 64 bf16 per row
constexpr uint32_t kAtomQ = kH * 128;      // 8 KB
constexpr uint32_t kAtomKV = kNB * 128;    // kNB rows of 128 bytes
constexpr uint32_t kQBytes = kAtoms * kAtomQ;
constexpr uint32_t kKVBytes = kAtoms * kAtomKV;
constexpr int kPAtom = kAtoms - 1;         // P(g) overwrites block g's rope atom once S(g) is done
constexpr int kBarAtoms = 3;               // atoms per landing barrier (a group of atoms lands together)
constexpr int kGroups = kAtoms / kBarAtoms;
static_assert(kAtoms % kBarAtoms == 0, "landing groups must tile the atoms");
constexpr int kProdWarps = 4;              // cp.async gather warps
constexpr int kMmaWarp = kProdWarps;       // warp 4: score product issuer (and TMEM owner)
constexpr int kPvWarp = kProdWarps + 1;    // warp 5: value product issuer
constexpr int kSmWarp0 = kProdWarps + 2;   // warps 6..13: softmax + epilogue
constexpr int kSmWarps = 8;
constexpr int kSmThreads = kSmWarps * 32;
constexpr int kThreads = (kProdWarps + 2 + kSmWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;              // O^T: 4 chunks x 64 columns
constexpr uint32_t kColS = 256;            // S: 2 buffers x kNB columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;

struct Bars {
  uint64_t q_full, q_empty;
  // kv_empty[st][c]: the value product's dimension chunk c (atoms 2c, 2c + 1; chunk 3 also
  // the rope atom, which holds P) is done with stage st, so its atoms can be refilled
  uint64_t kv_full[kStages][kGroups], kv_empty[kStages][kDV / 128];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2];
  uint64_t o_full, o_empty;
  uint64_t info_full[2], info_empty[2];
  uint64_t drain[2];  // end of kernel: each issuer waits for its own products
};

struct Small {
  Bars bar;
  uint32_t tmem;
  int abort;
  int nb[2];                       // blocks of the work item in flight (by item parity)
  int j0[2];                       // its first block within the row
  float alpha[kH];
  alignas(16) float lsum[kH];
  float bmax[2][2][kH];           // [block parity][key half][head]: block maxima of the two halves
  float lpart[2][kH];             // [key half][head]: partial row sums at the end of a row
  int any_rescale[2][kSmWarps];   // by block parity, so a fast warp never overwrites an unread flag
  int bad;                        // fixed reference: a row sum of this row left the exact range
};

constexpr size_t kSmem = 1024 + kQBytes + kStages * kKVBytes + sizeof(Small);

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Thread t of the warp receives, for each of the x2 / x4 repetitions j, TMEM lanes base + t/4
// and base + t/4 + 8 at columns 8j + 2(t%4) and 8j + 2(t%4) + 1, in that order (r[4j .. 4j+3]).
// (x2: the 32-key block width, which the kernel keeps buildable.)
[[maybe_unused]] __device__ __forceinline__ void tmem_ld_16x256b(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_16x256b(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory"); }
// Named barrier that also ORs a predicate over the n participating threads: every thread gets
// the same answer, so a decision taken on it (leaving the loop after a wait ran out in some
// warp) is uniform and no warp is left waiting at a later barrier.
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// MN-major 128-byte-swizzled operand descriptor: 64-element MN atoms `lbo` bytes apart, 8-row
// K groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = desc_sw128(saddr);
  d &= ~((uint64_t)0x3FFF << 16);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  return d;
}

// One query tensor map per layer of the launch.
struct QMaps {
  CUtensorMap m[kMaxAttnLayers];
};
// Entry l of a per-layer array of the launch parameters, selected with constant indices (a
// runtime index into a parameter array makes the compiler copy the array to local memory).
template <class T>
__device__ __forceinline__ T layer_pick(const T (&a)[kMaxAttnLayers], int l) {
  T r = a[0];
#pragma unroll
  for (int i = 1; i < kMaxAttnLayers; ++i) r = l == i ? a[i] : r;
  return r;
}

// kFixed: the softmax uses a fixed reference maximum of 0 (base-2 units) instead of a running
// one, so a block needs no exchange of maxima between the warps that share a head and O^T is
// never rescaled; exact while every row sum stays within [2^-64, 2^64] (P <= 2^64 in bf16, O^T
// and the sums in fp32).  A row outside that range is marked in p.redo and recomputed by the
// running-maximum kernel, which then runs only the marked rows (p.gate).
template <bool kPoll, bool kFixed>
__global__ void __launch_bounds__(kThreads, 1)
    k_sparse_mla_tc(const __grid_constant__ QMaps qm, AttnLaunch p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = base;
  uint8_t* kv_s = base + kQBytes;               // kStages stages
  Small* sm = reinterpret_cast<Small*>(kv_s + kStages * kKVBytes);
  Bars& bar = sm->bar;
  volatile int* abort_flag = &sm->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows1 = p.B * p.T;                     // query rows of one layer
  const int rows = rows1 * (p.layers > 1 ? p.layers : 1);
  const int splits = p.splits > 1 ? p.splits : 1;  // work item = (layer x row, part of its blocks)
  const int items = rows * splits;
  // items in order, skipping rows that a recomputing pass (p.gate) does not run; every role walks
  // the same sequence, so the barriers they share stay in step (a warp-uniform call)
  auto next_item = [&](int i) -> int {
    if (!p.gate) return i;
    const int G = (int)gridDim.x, ln = (int)(threadIdx.x & 31);
    for (int base = i; base < items; base += 32 * G) {
      const int cand = base + ln * G;
      const bool f = cand < items && p.gate[cand / splits] != 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, f);
      if (bal) return base + (__ffs(bal) - 1) * G;
    }
    return items;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      for (int gr = 0; gr < kGroups; ++gr) mbar_init(&bar.kv_full[i][gr], kProdWarps * 32);
      for (int c = 0; c < kDV / 128; ++c) mbar_init(&bar.kv_empty[i][c], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.s_empty[i], kSmWarps);
      mbar_init(&bar.p_full[i], kSmWarps);
      mbar_init(&bar.info_full[i], 1);
      mbar_init(&bar.info_empty[i], 3);
      mbar_init(&bar.drain[i], 1);
    }
    mbar_init(&bar.o_full, 1);
    mbar_init(&bar.o_empty, kSmWarps);
    sm->abort = 0;
    sm->bad = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sm->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem;

  if (warp < kProdWarps) {
    // ================= producers: row info, Q tile, KV gathers (cp.async), L2 prefetch ==========
    // Each of the four warps copies 16 of a block's 64 rows, atom by atom (8 lanes per row,
    // one 16-byte chunk each), into the 128-byte-swizzled K-major layout the MMAs read.  After
    // each atom every copying thread arms an asynchronous arrive on that atom's kv_full
    // barrier, which fires once its own copies have landed, so the producer never waits for
    // its copies and all stages stay in flight.
    const int64_t row_bytes = p.k_ld * 2;
    int it = 0;
    long long g = 0;  // global block counter
    bool ok = true;
    const bool vec = ((p.kk | p.idx_st | p.idx_sb) & 3) == 0 && (reinterpret_cast<uintptr_t>(p.idx) & 15u) == 0;
    for (int item = next_item(blockIdx.x); ok && item < items; item = next_item(item + (int)gridDim.x), ++it) {
      const int lrow = item / splits, layer = lrow / rows1, row = lrow % rows1;  // row within its layer
      const int32_t* irow = attn_idx_row(p, row);
      const int b = row / p.T;
      const uint8_t* kvb = static_cast<const uint8_t*>(layer_pick(p.lk, layer)) + (int64_t)b * p.k_sb * 2;  // its latent rows
      // blocks = 1 + (last entry other than -1) / kNB: the last 32 entries first (a full row
      // ends in a valid one), else a scan of the row with all its loads issued together
      int last = -1;
      {
        const int e = p.kk - 1 - lane;
        const int v = e >= 0 ? __ldg(irow + e) : -1;
        const uint32_t bal = __ballot_sync(0xffffffffu, v != -1);
        if (bal) last = p.kk - __ffs(bal);  // the lowest such lane holds the highest entry
      }
      if (last >= 0) {
      } else if (vec) {
        const int n4 = p.kk >> 2;
        for (int c0 = 0; c0 < n4; c0 += 32 * 8) {
          int4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * 32 + lane;
            v[u] = c < n4 ? __ldg(reinterpret_cast<const int4*>(irow) + c) : make_int4(-1, -1, -1, -1);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = 4 * (c0 + u * 32 + lane);
            if (v[u].x != -1) last = max(last, c);
            if (v[u].y != -1) last = max(last, c + 1);
            if (v[u].z != -1) last = max(last, c + 2);
            if (v[u].w != -1) last = max(last, c + 3);
          }
        }
      } else {
        for (int j = lane; j < p.kk; j += 32)
          if (__ldg(irow + j) != -1) last = j;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      const int nbr = (last + kNB) / kNB;  // blocks of the row
      const int split = item % splits;
      const int j0 = split * nbr / splits, nb = (split + 1) * nbr / splits - j0;  // this item's blocks
      if (warp == 0) {
        if (lane == 0) ok = mbar_wait<kPoll>(&bar.info_empty[it & 1], ((it >> 1) & 1) ^ 1, abort_flag, p.wait);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && lane == 0) {
          sm->nb[it & 1] = nb;
          sm->j0[it & 1] = j0;
          mbar_arrive(&bar.info_full[it & 1]);
        }
      }
      if (!ok || *abort_flag) break;
      if (nb == 0) continue;
      if (warp == 0) {
        const int next = (item + (int)gridDim.x) / splits;
        if (lane == 0 && next < rows && next != lrow) {
          const int nr = next % rows1;
          prefetch_l2(static_cast<const __nv_bfloat16*>(layer_pick(p.lq, next / rows1)) + (int64_t)(nr / p.T) * p.q_sb +
                          (int64_t)(nr % p.T) * p.q_st,
                      kQBytes);
        }
      }
      for (int j = 0; ok && j < nb; ++j, ++g) {
        const int st = (int)(g % kStages);
        // ids of this warp's 16 rows
        constexpr int kRowsW = kNB / kProdWarps;
        const int rl = warp * kRowsW + (lane & (kRowsW - 1));
        const int e = (j0 + j) * kNB + rl;
        int id = e < p.kk ? __ldg(irow + e) : -1;
        const bool valid = id >= 0 && id < p.S;
        if (lane < kRowsW && !valid && id != -1) atomicOr(p.flags, DSA_FLAG_BAD_INDEX);
        if (!valid) id = 0;
        const uint32_t epar = (uint32_t)((g / kStages) & 1) ^ 1;  // the stage's release phase
        uint8_t* stage = kv_s + st * kKVBytes;
        // atom by atom: 8 lanes per row (one 16-byte chunk each), 4 rows per pass, 4 passes
        // cover the warp's 16 rows; the row of each pass is fixed, so its id is fetched once
        int rid[kRowsW / 4];
        bool rv[kRowsW / 4];
#pragma unroll
        for (int pass = 0; pass < kRowsW / 4; ++pass) {
          rid[pass] = __shfl_sync(0xffffffffu, id, pass * 4 + (lane >> 3));
          rv[pass] = __shfl_sync(0xffffffffu, valid, pass * 4 + (lane >> 3));
        }
        const int cc = lane & 7;
        // atom by atom, each pair of atoms once the value product has released it (the
        // block two back in this stage), so refilling overlaps the rest of that product
#pragma unroll
        for (int a = 0; a < kAtoms; ++a) {
          if (a % 2 == 0 && a / 2 < kDV / 128 &&
              !(ok = mbar_wait<kPoll>(&bar.kv_empty[st][a / 2], epar, abort_flag, p.wait)))
            break;
#pragma unroll
          for (int pass = 0; pass < kRowsW / 4; ++pass) {
            const int r = warp * kRowsW + pass * 4 + (lane >> 3);
            const uint32_t dst = smem_addr(stage + a * kAtomKV + r * 128 + ((cc ^ (r & 7)) << 4));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
                         "l"(kvb + rid[pass] * row_bytes + (a * 8 + cc) * 16), "r"(rv[pass] ? 16 : 0)
                         : "memory");
          }
          if (a % kBarAtoms == kBarAtoms - 1)
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(
                             smem_addr(&bar.kv_full[st][a / kBarAtoms]))
                         : "memory");
        }
        if (!ok) break;
        // L2 prefetch of the rows of the block two ahead (two stages: the next block this
        // stage will hold), so that its gathers hit L2: the fill latency of a stage, mostly
        // DRAM misses, sets the pace of the two-stage ring (8,192 rows x 2,048 keys: 3.83 ->
        // 3.65 ms; three ahead 3.66; also the next row's first blocks 3.66).
        if (j + 2 < nb && lane < kRowsW) {
          const int ep = (j0 + j + 2) * kNB + warp * kRowsW + lane;
          const int idp = ep < p.kk ? __ldg(irow + ep) : -1;
          if (idp >= 0 && idp < p.S) prefetch_l2(kvb + (int64_t)idp * row_bytes, (uint32_t)row_bytes);
        }
      }
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ================= score product issuer (one thread) =================
    const uint32_t id_s = idesc_mn(1, 1, kH, kNB);  // S: M=64 heads, N=32 keys
    const uint64_t q_desc0 = desc_sw128(smem_addr(q_s));
    const uint64_t kv_desc0 = desc_sw128(smem_addr(kv_s));
    int it = 0, qc = 0, qi = 0;  // rows begun; query tiles loaded
    long long g = 0;
    bool ok = true;
    for (int item = next_item(blockIdx.x); ok && item < items; item = next_item(item + (int)gridDim.x), ++it) {
      int nb = 0;
      if (lane == 0) {
        ok = mbar_wait<kPoll>(&bar.info_full[it & 1], (it >> 1) & 1, abort_flag, p.wait);
        nb = sm->nb[it & 1];
        mbar_arrive(&bar.info_empty[it & 1]);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      nb = __shfl_sync(0xffffffffu, nb, 0);
      if (!ok) break;
      if (nb == 0) continue;
      if (lane == 0) {
        // this row's query tile, once the previous row's last score product (issued by this
        // thread) is done with the buffer: the gathers never wait for it
        ok = mbar_wait<kPoll>(&bar.q_empty, (qc & 1) ^ 1, abort_flag, p.wait);
        if (ok) {
          const int lrow = item / splits, layer = lrow / rows1, row = lrow % rows1;
          mbar_arrive_expect_tx(&bar.q_full, kQBytes);
          for (int a = 0; a < kAtoms; ++a)
            tma_load_4d(q_s + a * kAtomQ, &qm.m[layer], &bar.q_full, a * 64, 0, row % p.T, row / p.T);
          ++qi;
          ok = mbar_wait<kPoll>(&bar.q_full, qc & 1, abort_flag, p.wait);
        }
        for (int j = 0; ok && j < nb; ++j) {
          const long long gs = g + j;
          const int st = (int)(gs % kStages), sb = (int)(gs & 1);
          const uint32_t kvpar = (uint32_t)((gs / kStages) & 1);
          if (!(ok = mbar_wait<kPoll>(&bar.s_empty[sb], (uint32_t)((gs >> 1) & 1) ^ 1, abort_flag, p.wait))) break;
          // descriptors: base + compile-time offsets in the 16-byte start-address field
          const uint64_t qd = q_desc0, kd = kv_desc0 + (uint64_t)((st * kKVBytes) >> 4);
          const uint32_t d = tmem + kColS + sb * kNB;
#pragma unroll
          for (int a = 0; a < kAtoms; ++a) {
            if (a % kBarAtoms == 0 && !(ok = mbar_wait<kPoll>(&bar.kv_full[st][a / kBarAtoms], kvpar, abort_flag, p.wait)))
              break;
            fence_async_smem();  // the stage was written by cp.async (generic proxy)
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16(d, qd + (uint64_t)((a * kAtomQ + k * 32) >> 4), kd + (uint64_t)((a * kAtomKV + k * 32) >> 4),
                       id_s, (a | k) != 0 ? 1u : 0u);
          }
          if (!ok) break;
          mma_commit(&bar.s_full[sb]);
          if (j == nb - 1) mma_commit(&bar.q_empty);  // last use of this row's Q
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      g += nb;
      ++qc;
    }
    if (lane == 0) {  // wait for this thread's own products before TMEM can be freed
      mma_commit(&bar.drain[0]);
      mbar_wait_drain(&bar.drain[0], 0);
      // and for the last query tile it loaded (whichever wait ran out)
      if (qi > 0) mbar_wait_drain(&bar.q_full, (uint32_t)((qi - 1) & 1));
    }
  } else if (warp == kPvWarp) {
    // ================= value product issuer (one thread) =================
    const uint32_t id_o = idesc_mn(1, 1, 128, kH) | (1u << 15);  // O^T: M=128 dims (MN-major A), N=64 heads
    // P: 64 rows (heads) of kNB keys, 128- or 64-byte swizzled rows
    const uint64_t p_desc0 = kNB == 64 ? desc_sw128(smem_addr(kv_s)) : desc_sw64(smem_addr(kv_s));
    const uint64_t v_desc0 = desc_sw128_mn(smem_addr(kv_s), kAtomKV);
    int it = 0, oc = 0;
    long long g = 0;
    bool ok = true;
    for (int item = next_item(blockIdx.x); ok && item < items; item = next_item(item + (int)gridDim.x), ++it) {
      int nb = 0;
      if (lane == 0) {
        ok = mbar_wait<kPoll>(&bar.info_full[it & 1], (it >> 1) & 1, abort_flag, p.wait);
        nb = sm->nb[it & 1];
        mbar_arrive(&bar.info_empty[it & 1]);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      nb = __shfl_sync(0xffffffffu, nb, 0);
      if (!ok) break;
      if (nb == 0) continue;
      if (lane == 0) {
        ok = mbar_wait<kPoll>(&bar.o_empty, (oc & 1) ^ 1, abort_flag, p.wait);
        for (int j = 0; ok && j < nb; ++j) {
          const long long gp = g + j;
          const int st = (int)(gp % kStages), pb = (int)(gp & 1);
          if (!(ok = mbar_wait<kPoll>(&bar.p_full[pb], (uint32_t)((gp >> 1) & 1), abort_flag, p.wait))) break;
          fence_async_smem();
          tc_fence_after();
          const uint64_t vd = v_desc0 + (uint64_t)((st * kKVBytes) >> 4);
          const uint64_t pd = p_desc0 + (uint64_t)((st * kKVBytes + kPAtom * kAtomKV) >> 4);
          // chunk by chunk, each releasing its atoms of the stage when done
#pragma unroll
          for (int c = 0; c < kDV / 128; ++c) {
#pragma unroll
            for (int k = 0; k < kNB / 16; ++k)
              mma_bf16(tmem + kColO + c * kH, vd + (uint64_t)((2 * c * kAtomKV + k * 2048) >> 4),
                       pd + (uint64_t)((k * 32) >> 4), id_o, (j | k) != 0 ? 1u : 0u);
            mma_commit(&bar.kv_empty[st][c]);
          }
          if (j == nb - 1) mma_commit(&bar.o_full);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      g += nb;
      ++oc;
    }
    if (lane == 0) {
      mma_commit(&bar.drain[1]);
      mbar_wait_drain(&bar.drain[1], 0);
    }
  } else {
    // ================= softmax + epilogue (warps 6..13) =================
    const int q4 = warp & 3;                    // TMEM lane quarter
    const int sw = warp - kSmWarp0;             // softmax warp index 0..7
    const int kh = sw >> 2;                     // key half: columns kHalf * kh .. + kHalf - 1 of each block
    // The M = 64 score rows sit in lanes 0..15 of each lane quarter; the 16x256b TMEM shape
    // spreads them over all 32 threads: thread t holds heads hd[0] = 16 q4 + t/4 and hd[1] =
    // hd[0] + 8, each at the keys 8j + 2m + {0, 1} (m = t % 4, j < kHalf / 8) of the warp's key
    // half; a head's four threads (one quad) combine their maxima and sums with two shuffles.
    const int m = lane & 3;
    const int hd[2] = {q4 * 16 + (lane >> 2), q4 * 16 + (lane >> 2) + 8};
    const bool quad_lead = m == 0;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const float sl2 = p.scale * kLog2e;
    const int t = threadIdx.x - kSmWarp0 * 32;  // 0..255
    int it = 0, oc = 0;
    long long g = 0;
    bool ok = true;
    for (int item = next_item(blockIdx.x); ok && item < items; item = next_item(item + (int)gridDim.x), ++it) {
      const int lrow = item / splits, layer = lrow / rows1, row = lrow % rows1;
      float* const lse_out = layer_pick(p.llse, layer);
      // every wait of these eight warps is followed by a barrier that ORs "it ran out" over
      // them, so they leave together
      const bool got_info = mbar_wait<kPoll>(&bar.info_full[it & 1], (it >> 1) & 1, abort_flag, p.wait);
      if (named_sync_or(1, kSmThreads, !got_info)) {
        ok = false;
        break;
      }
      const int nb = sm->nb[it & 1], j0 = sm->j0[it & 1];
      if (t == 0) mbar_arrive(&bar.info_empty[it & 1]);
      __nv_bfloat16* og = static_cast<__nv_bfloat16*>(layer_pick(p.lout, layer)) + (int64_t)row * kH * kDV;
      float* po = splits > 1 ? p.part_o + (int64_t)item * kH * kDV : nullptr;  // this part's output
      const int32_t* irow = attn_idx_row(p, row);
      if (nb == 0) {  // nothing visible: O = 0, LSE = -inf
        if (po) {
          for (int i = t; i < kH * kDV / 4; i += kSmThreads) reinterpret_cast<float4*>(po)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (t < kH) p.part_lse[(int64_t)item * kH + t] = -INFINITY;
        } else {
          for (int i = t; i < kH * kDV / 8; i += kSmThreads) reinterpret_cast<uint4*>(og)[i] = make_uint4(0, 0, 0, 0);
          if (lse_out && t < kH) lse_out[(int64_t)row * kH + t] = -INFINITY;
        }
        if (kFixed && t == 0 && p.redo) p.redo[lrow] = 0;
        continue;
      }
      float m_used[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
      const uint32_t kv_base_s = smem_addr(kv_s);  // the stages' shared-space address
      bool failed = false;  // kFixed: a wait ran out; the warp goes to the row's end barrier
      for (int j = 0; ok && j < nb; ++j, ++g) {
        const int sb = (int)(g & 1);
        // this lane's key slot (lanes 16..31 repeat 0..15), loaded before the wait so that its
        // latency hides behind it
        const int e = (j0 + j) * kNB + kh * kHalf + (lane & (kHalf - 1));
        const int id = e < p.kk ? __ldg(irow + e) : -1;
        const bool got_s = mbar_wait<kPoll>(&bar.s_full[sb], (uint32_t)((g >> 1) & 1), abort_flag, p.wait);
        uint32_t sr[kHalf / 2];
        if (got_s) {
          tc_fence_after();
          tmem_ld_16x256b(tmem + lane_base + kColS + sb * kNB + kh * kHalf, sr);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar.s_empty[sb]);
        } else {
#pragma unroll
          for (int c = 0; c < kHalf / 2; ++c) sr[c] = 0u;  // leaving at the barrier below
        }
        // scores in base-2 units, masked by the validity of each key slot (lane c checks key c)
        const uint32_t vm = __ballot_sync(0xffffffffu, id >= 0 && id < p.S);
        float s[2][kHalf / 4];
        float bmax[2] = {-INFINITY, -INFINITY};
        if (vm == 0xffffffffu) {  // every key of the half valid (warp-uniform): no mask
#pragma unroll
          for (int jj = 0; jj < kHalf / 8; ++jj)
#pragma unroll
            for (int hs = 0; hs < 2; ++hs)
#pragma unroll
              for (int e2 = 0; e2 < 2; ++e2) {
                const float x = __uint_as_float(sr[4 * jj + 2 * hs + e2]) * sl2;
                s[hs][2 * jj + e2] = x;
                bmax[hs] = fmaxf(bmax[hs], x);
              }
        } else {
#pragma unroll
          for (int jj = 0; jj < kHalf / 8; ++jj)
#pragma unroll
            for (int hs = 0; hs < 2; ++hs)
#pragma unroll
              for (int e2 = 0; e2 < 2; ++e2) {
                const float x = __uint_as_float(sr[4 * jj + 2 * hs + e2]) * sl2;
                const float y = ((vm >> (8 * jj + 2 * m + e2)) & 1u) ? x : -INFINITY;
                s[hs][2 * jj + e2] = y;
                bmax[hs] = fmaxf(bmax[hs], y);
              }
        }
        float m_new[2];
        if constexpr (kFixed) {
          if (!got_s) {
            failed = true;
            break;
          }
          m_new[0] = m_new[1] = 0.f;
        } else {
  #pragma unroll
          for (int hs = 0; hs < 2; ++hs) {
            bmax[hs] = fmaxf(bmax[hs], __shfl_xor_sync(0xffffffffu, bmax[hs], 1));
            bmax[hs] = fmaxf(bmax[hs], __shfl_xor_sync(0xffffffffu, bmax[hs], 2));
          }
          const bool need_h = bmax[0] > m_used[0] + kRescaleLog2 || bmax[1] > m_used[1] + kRescaleLog2;
          const int any = __any_sync(0xffffffffu, need_h);
          if (quad_lead) {
            sm->bmax[sb][kh][hd[0]] = bmax[0];
            sm->bmax[sb][kh][hd[1]] = bmax[1];
          }
          if (lane == 0) sm->any_rescale[sb][sw] = any;
          if (named_sync_or(1, kSmThreads, !got_s)) {
            ok = false;
            break;
          }
          int anyr = 0;
  #pragma unroll
          for (int w = 0; w < kSmWarps; ++w) anyr |= sm->any_rescale[sb][w];
          bool need[2];
  #pragma unroll
          for (int hs = 0; hs < 2; ++hs) {
            const float bm = fmaxf(sm->bmax[sb][0][hd[hs]], sm->bmax[sb][1][hd[hs]]);
            need[hs] = bm > m_used[hs] + kRescaleLog2;  // the same decision in both key halves
            m_new[hs] = need[hs] ? bm : m_used[hs];
          }
          if (j > 0 && anyr) {
            // O^T must be complete for the previous block before it is rescaled: the last
            // chunk of the value product of block g-1 releases its stage's last atoms, and its
            // commit covers the earlier chunks
            const long long gp = g - 1;
            const bool got_o = mbar_wait<kPoll>(&bar.kv_empty[gp % kStages][kDV / 128 - 1], (uint32_t)((gp / kStages) & 1), abort_flag, p.wait);
  #pragma unroll
            for (int hs = 0; hs < 2; ++hs) {
              const float alpha = need[hs] ? ex2(m_used[hs] - m_new[hs]) : 1.f;
              if (quad_lead && kh == 0) sm->alpha[hd[hs]] = alpha;
              l[hs] *= alpha;
            }
            if (named_sync_or(1, kSmThreads, !got_o)) {
              ok = false;
              break;
            }
            tc_fence_after();
  #pragma unroll 1
            for (int c = 2 * kh; c < 2 * kh + 2; ++c)  // each key half rescales two of the four chunks
  #pragma unroll 1
              for (int half = 0; half < 2; ++half) {
                uint32_t r[32];
                const uint32_t ta = tmem + lane_base + kColO + c * kH + half * 32;
                tmem_ld32(ta, r);
                tmem_wait_ld();
  #pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * sm->alpha[half * 32 + i]);
                tmem_st32(ta, r);
              }
            tmem_wait_st();
            tc_fence_before();
          }
        }
        // P rows (bf16) of this thread's two heads, in the block's rope atom, which S(g) -- now
        // complete -- was the last to read: key 8j + 2m + {0, 1} of the key half is the 4-byte
        // word m of 16-byte chunk (kHalf / 8) kh + j of the head's 2 kNB-byte row, whose chunks
        // the swizzle permutes (128-byte rows: by head mod 8; 64-byte rows: by (head / 2) mod 4)
        const uint32_t patom = kv_base_s + (uint32_t)(g % kStages) * kKVBytes + kPAtom * kAtomKV;
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          m_used[hs] = m_new[hs];
          const float mu = m_used[hs] == -INFINITY ? 0.f : m_used[hs];
          const uint32_t prow = patom + hd[hs] * (2 * kNB) + m * 4;
          const int perm = kNB == 64 ? (hd[hs] & 7) : ((hd[hs] >> 1) & 3);
#pragma unroll
          for (int jj = 0; jj < kHalf / 8; ++jj) {
            const float a = ex2(s[hs][2 * jj] - mu), bq = ex2(s[hs][2 * jj + 1] - mu);
            l[hs] += a + bq;
            __nv_bfloat162 v2 = __floats2bfloat162_rn(a, bq);
            asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(prow + ((uint32_t)((kh * (kHalf / 8) + jj) ^ perm) << 4)),
                         "r"(*reinterpret_cast<uint32_t*>(&v2))
                         : "memory");
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.p_full[sb]);
      }
      if (!ok) break;
      // ---- epilogue: O = O^T / l, LSE ----
#pragma unroll
      for (int hs = 0; hs < 2; ++hs) {
        l[hs] += __shfl_xor_sync(0xffffffffu, l[hs], 1);
        l[hs] += __shfl_xor_sync(0xffffffffu, l[hs], 2);
        if (quad_lead) sm->lpart[kh][hd[hs]] = l[hs];
      }
      if (named_sync_or(1, kSmThreads, failed)) {
        ok = false;
        break;
      }
      if (quad_lead && kh == 0) {
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          const int hh = hd[hs];
          const float lt = sm->lpart[0][hh] + sm->lpart[1][hh];
          if (kFixed && !(lt >= 0x1p-64f && lt <= 0x1p64f)) sm->bad = 1;  // (also inf, NaN)
          sm->lsum[hh] = lt > 0.f ? 1.f / lt : 0.f;  // reciprocal row sums
          const float lse_v = lt > 0.f ? (m_used[hs] + log2f(lt)) * kLn2 : -INFINITY;
          if (po) p.part_lse[(int64_t)item * kH + hh] = lse_v;
          else if (lse_out) lse_out[(int64_t)row * kH + hh] = lse_v;
        }
      }
      const bool got_o = mbar_wait<kPoll>(&bar.o_full, oc & 1, abort_flag, p.wait);
      if (named_sync_or(1, kSmThreads, !got_o)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this warp's four slices of O^T (dimension chunks 2kh, 2kh + 1; heads 0-31, 32-63), each
      // loaded while the previous one is stored; the reciprocal row sums are read four at a time
      {
        uint32_t ra[32], rb[32];
        auto slice = [&](int n) {  // TMEM address of slice n
          return tmem + lane_base + kColO + (uint32_t)((2 * kh + (n >> 1)) * kH + (n & 1) * 32);
        };
        auto store = [&](const uint32_t (&r)[32], int n) {
          const int d = (2 * kh + (n >> 1)) * 128 + q4 * 32 + lane, h0 = (n & 1) * 32;
          const float4* ls4 = reinterpret_cast<const float4*>(sm->lsum + h0);
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 L = ls4[i4];
            const float lv[4] = {L.x, L.y, L.z, L.w};
            if (po) {
#pragma unroll
              for (int u = 0; u < 4; ++u)
                po[(int64_t)(h0 + 4 * i4 + u) * kDV + d] = __uint_as_float(r[4 * i4 + u]) * lv[u];
            } else {
              // lane pairs write two neighbouring dimensions of one head as one 4-byte word:
              // of heads (i, i + 1) the even lane keeps i and takes its partner's value of i,
              // the odd lane keeps i + 1 and takes its partner's value of i + 1
              const bool odd = (lane & 1) != 0;
#pragma unroll
              for (int u = 0; u < 4; u += 2) {
                const int i = 4 * i4 + u;
                const float a = __uint_as_float(r[i]) * lv[u], bq = __uint_as_float(r[i + 1]) * lv[u + 1];
                const float other = __shfl_xor_sync(0xffffffffu, odd ? a : bq, 1);
                const __nv_bfloat162 w = odd ? __floats2bfloat162_rn(other, bq) : __floats2bfloat162_rn(a, other);
                *reinterpret_cast<__nv_bfloat162*>(og + (int64_t)(h0 + i + (odd ? 1 : 0)) * kDV + (d & ~1)) = w;
              }
            }
          }
        };
        tmem_ld32(slice(0), ra);
        tmem_wait_ld();
        tmem_ld32(slice(1), rb);
        store(ra, 0);
        tmem_wait_ld();
        tmem_ld32(slice(2), ra);
        store(rb, 1);
        tmem_wait_ld();
        tmem_ld32(slice(3), rb);
        store(ra, 2);
        tmem_wait_ld();
        store(rb, 3);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.o_empty);
      named_sync(1, kSmThreads);  // lsum and lpart are reused by the next row
      if (kFixed && t == 0) {
        if (p.redo) p.redo[lrow] = (uint8_t)sm->bad;
        sm->bad = 0;
      }
      ++oc;
    }
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.flags, DSA_FLAG_TIMEOUT);
}

// Merge of a split row's parts: O = sum_s w_s O_s, w_s = exp(LSE_s - LSE), LSE = log sum_s exp(LSE_s).
// One CTA per (row, group of kCombHeads heads): a decode call has few rows, and one CTA per row
// left most of the GPU idle (26 us for 32 rows of 4 parts).
constexpr int kCombHeads = 4;
__global__ void __launch_bounds__(128) k_attn_combine(AttnLaunch p) {
  __shared__ float wgt[kMaxAttnSplits][kCombHeads];
  // blockIdx.x: flat (layer, row); parts of flat row r are items r*S .. r*S + S - 1
  const int lrow = blockIdx.x, h0 = blockIdx.y * kCombHeads, S = p.splits;
  const int rows1 = p.B * p.T, layer = lrow / rows1, row = lrow % rows1;
  float* const lse_out = layer_pick(p.llse, layer);
  const float* pl = p.part_lse + (int64_t)lrow * S * kH;
  if (threadIdx.x < kCombHeads) {
    const int h = h0 + threadIdx.x;
    float mx = -INFINITY;
    for (int s = 0; s < S; ++s) mx = fmaxf(mx, pl[s * kH + h]);
    float sum = 0.f;
    for (int s = 0; s < S; ++s) {
      const float w = mx == -INFINITY ? 0.f : expf(pl[s * kH + h] - mx);
      wgt[s][threadIdx.x] = w;
      sum += w;
    }
    for (int s = 0; s < S; ++s) wgt[s][threadIdx.x] = sum > 0.f ? wgt[s][threadIdx.x] / sum : 0.f;
    if (lse_out) lse_out[(int64_t)row * kH + h] = sum > 0.f ? mx + logf(sum) : -INFINITY;
  }
  __syncthreads();
  const int64_t first = (int64_t)h0 * kDV / 4;  // this CTA's first float4 within a part
  const float4* po = reinterpret_cast<const float4*>(p.part_o + (int64_t)lrow * S * kH * kDV) + first;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(layer_pick(p.lout, layer)) + (int64_t)row * kH * kDV;
  for (int i = threadIdx.x; i < kCombHeads * kDV / 4; i += 128) {
    const int hl = (i * 4) / kDV;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float4 v = po[(int64_t)s * kH * kDV / 4 + i];
      const float w = wgt[s][hl];
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(og)[first + i] = u;
  }
}

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

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace

bool sparse_mla_tc_supported(const AttnLaunch& p) {
  return p.H == kH && p.DQK == kDQK && p.DV == kDV && p.v == p.k && p.v_ld == p.k_ld && p.k_ld == kDQK &&
         p.v_sb == p.k_sb && p.S < (1 << 30);
}

cudaError_t launch_sparse_mla_tc(const AttnLaunch& p, cudaStream_t st) {
  if (p.splits > kMaxAttnSplits || (p.splits > 1 && !(p.part_o && p.part_lse))) return cudaErrorInvalidValue;
  if (p.layers > kMaxAttnLayers) return cudaErrorInvalidValue;
  TraceScope trace(kTraceAttention, st);
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  // a single-layer call describes its layer in q / k / out / lse
  AttnLaunch q = p;
  if (q.layers <= 1) {
    q.layers = 1;
    q.lq[0] = p.q;
    q.lk[0] = p.k;
    q.lout[0] = p.out;
    q.llse[0] = p.lse;
  }
  QMaps qm;
  for (int l = 0; l < q.layers; ++l) {
    // queries [B][T][H][576] with token strides q_st / q_sb; a box is one swizzle atom (64
    // columns) of one query's 64 heads
    cuuint64_t dims[4] = {(cuuint64_t)kDQK, (cuuint64_t)kH, (cuuint64_t)p.T, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {(cuuint64_t)kDQK * 2, (cuuint64_t)p.q_st * 2, (cuuint64_t)p.q_sb * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)kH, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&qm.m[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q.lq[l]), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (q.wait <= 0) q.wait = wait_limit();
  const bool poll = q.wait < kDefaultWaitCycles;
  // with room for the row marks and no split: the fixed-reference pass, then the running-maximum
  // pass over the rows it marked (its CTAs skip every other row)
  const bool fixed = q.redo != nullptr && q.splits <= 1;
  if (!fixed) q.redo = nullptr;
  auto kern_exact = poll ? k_sparse_mla_tc<true, false> : k_sparse_mla_tc<false, false>;
  auto kern = fixed ? (poll ? k_sparse_mla_tc<true, true> : k_sparse_mla_tc<false, true>) : kern_exact;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  const int rows = p.B * p.T * q.layers;
  const int items = rows * (p.splits > 1 ? p.splits : 1);
  const int grid = items < num_sms() ? items : num_sms();
  kern<<<grid, kThreads, kSmem, st>>>(qm, q);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (fixed) {
    AttnLaunch r = q;
    r.redo = nullptr;
    r.gate = q.redo;
    if ((e = cudaFuncSetAttribute(kern_exact, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem)) != cudaSuccess)
      return e;
    kern_exact<<<grid, kThreads, kSmem, st>>>(qm, r);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (p.splits <= 1) return e;
  k_attn_combine<<<dim3((unsigned)rows, kH / kCombHeads), 128, 0, st>>>(q);
  count_launches(1);
  return cudaGetLastError();
}


int attn_splits(const AttnLaunch& p) {
  if (!sparse_mla_tc_supported(p)) return 1;
  const int rows = p.B * p.T * (p.layers > 1 ? p.layers : 1), sms = num_sms();
  if (rows <= 0 || rows * 2 > sms) return 1;
  int s = sms / rows;                                       // about one CTA per SM
  const int by_len = (p.kk + 255) / 256;                    // parts of at least 256 keys
  if (s > by_len) s = by_len;
  if (s > kMaxAttnSplits) s = kMaxAttnSplits;
  return s < 2 ? 1 : s;
}

}  // namespace dsa
