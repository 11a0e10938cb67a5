// Lightning-indexer scores on warp-level mma.sync tensor-core instructions, materialised
// to an fp32 score buffer.  I[t,s] = sq[t] * sk[s] * sum_h w[t,h] * ReLU(q[t,h] . k[s]):
// the per-token fp32 scales of e4m3 operands are positive, so they leave the ReLU and
// multiply the head sum once.
//
// Tile: 128 keys (M, 16 per warp) x TB tokens; the tokens' query heads form the N columns
// (column j = token * H_I + head), d_I is the contraction.  The key fragments stay in
// registers for the whole CTA; the query tile sits in shared memory with a 16-byte row pad
// so that fragment loads are bank-conflict free.  The head-weighted ReLU sum runs in the
// fragment registers, then across the 4 lanes of a quad; scores are staged in shared memory
// and written with coalesced stores.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kKeysPerCta = 128;
constexpr int kThreads = 256;

template <bool FP8>
__device__ __forceinline__ void mma_tile(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (FP8) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <int HI, int DI, bool FP8, int TB>
struct IxTile {
  static constexpr int kEsz = FP8 ? 1 : 2;
  static constexpr int kRowBytes = DI * kEsz;       // one head vector
  static constexpr int kRowPad = kRowBytes + 16;    // shared-memory row stride
  static constexpr int kKSteps = kRowBytes / 32;    // 32 bytes of K per mma
  static constexpr int kCols = TB * HI;
  static constexpr int kNTiles = kCols / 8;
  static constexpr size_t kSmemQ = (size_t)kCols * kRowPad;
  static constexpr size_t kSmemW = (size_t)TB * HI * 4;
  static constexpr size_t kSmemOut = (size_t)TB * kKeysPerCta * 4;
  static constexpr size_t kSmem = kSmemQ + kSmemW + TB * 4 + kSmemOut;
  static_assert(kCols % 8 == 0, "columns come in n8 tiles");
};

template <int HI, int DI, bool FP8, int TB>
__global__ void __launch_bounds__(kThreads) k_indexer_mma(IndexerLaunch p) {
  using C = IxTile<HI, DI, FP8, TB>;
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* q_s = smem;
  float* w_s = reinterpret_cast<float*>(smem + C::kSmemQ);
  float* sq_s = w_s + TB * HI;
  float* o_s = sq_s + TB;

  const int key0 = blockIdx.x * kKeysPerCta;
  const int tl0 = blockIdx.y * TB;
  const int b = blockIdx.z;
  if (tl0 >= p.Tc || key0 >= p.S) return;
  const int ntok = min(TB, p.Tc - tl0);
  const int t_first = p.t0 + tl0;
  auto visible = [&](int t) -> int64_t {
    int64_t n = p.q_pos0 + t + p.diag;
    return n < 0 ? 0 : (n > p.S ? (int64_t)p.S : n);
  };
  const int64_t nmax = visible(t_first + ntok - 1);
  float* out_b = p.out + (int64_t)b * p.out_bstride;
  const int kend = min(kKeysPerCta, p.S - key0);

  if (key0 >= nmax) {  // the whole tile is masked
    if (p.write_masked)
      for (int i = threadIdx.x; i < ntok * kKeysPerCta; i += kThreads) {
        const int tok = i / kKeysPerCta, kk = i % kKeysPerCta;
        if (kk < kend) out_b[(int64_t)(tl0 + tok) * p.ld + key0 + kk] = -INFINITY;
      }
    return;
  }

  // ---- stage the query tile, head weights and query scales -------------------------
  {
    constexpr int kChunks = C::kRowBytes / 16;
    const uint8_t* qg = static_cast<const uint8_t*>(p.q) +
                        (((int64_t)b * p.T + t_first) * HI) * C::kRowBytes;
    for (int i = threadIdx.x; i < C::kCols * kChunks; i += kThreads) {
      const int j = i / kChunks, c16 = i % kChunks;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (j / HI < ntok) v = __ldg(reinterpret_cast<const uint4*>(qg + (int64_t)j * C::kRowBytes) + c16);
      *reinterpret_cast<uint4*>(q_s + j * C::kRowPad + c16 * 16) = v;
    }
    const float* wg = p.w + ((int64_t)b * p.T + t_first) * HI;
    for (int i = threadIdx.x; i < TB * HI; i += kThreads) w_s[i] = (i / HI < ntok) ? __ldg(wg + i) : 0.f;
    if (threadIdx.x < TB) {
      const int tok = threadIdx.x;
      sq_s[tok] = (FP8 && tok < ntok) ? __ldg(p.q_scale + (int64_t)b * p.T + t_first + tok) : 1.f;
    }
  }

  // ---- key fragments of this warp's 16 keys, straight from global ------------------
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int kr0 = key0 + warp * 16 + g, kr1 = kr0 + 8;
  uint32_t afr[C::kKSteps][4];
  {
    const uint8_t* kg = static_cast<const uint8_t*>(p.k) + (int64_t)b * p.S * C::kRowBytes;
    const bool v0 = kr0 < p.S, v1 = kr1 < p.S;
#pragma unroll
    for (int ks = 0; ks < C::kKSteps; ++ks) {
      const int off = ks * 32 + 4 * c;
      afr[ks][0] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(kg + (int64_t)kr0 * C::kRowBytes + off)) : 0u;
      afr[ks][1] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(kg + (int64_t)kr1 * C::kRowBytes + off)) : 0u;
      afr[ks][2] = v0 ? __ldg(reinterpret_cast<const uint32_t*>(kg + (int64_t)kr0 * C::kRowBytes + off + 16)) : 0u;
      afr[ks][3] = v1 ? __ldg(reinterpret_cast<const uint32_t*>(kg + (int64_t)kr1 * C::kRowBytes + off + 16)) : 0u;
    }
  }
  __syncthreads();

  // ---- MMA + fused ReLU / head-weighted sum ----------------------------------------
  float part0 = 0.f, part1 = 0.f;  // running head sums for keys kr0, kr1
#pragma unroll 1
  for (int nt = 0; nt < C::kNTiles; ++nt) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const uint8_t* brow = q_s + (nt * 8 + g) * C::kRowPad + 4 * c;
#pragma unroll
    for (int ks = 0; ks < C::kKSteps; ++ks) {
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(brow + ks * 32);
      const uint32_t b1 = *reinterpret_cast<const uint32_t*>(brow + ks * 32 + 16);
      mma_tile<FP8>(d, afr[ks], b0, b1);
    }
    const int j0 = nt * 8 + 2 * c;  // this thread's two columns: j0, j0 + 1
    const float w0 = w_s[j0], w1 = w_s[j0 + 1];
    part0 += w0 * fmaxf(d[0], 0.f) + w1 * fmaxf(d[1], 0.f);
    part1 += w0 * fmaxf(d[2], 0.f) + w1 * fmaxf(d[3], 0.f);

    bool token_done;
    int tok;
    if constexpr (HI >= 8) {
      token_done = ((nt + 1) % (HI / 8)) == 0;
      tok = nt / (HI / 8);
    } else {
      token_done = true;
      tok = j0 / HI;
    }
    if (token_done) {
      part0 += __shfl_xor_sync(0xffffffffu, part0, 1);
      part1 += __shfl_xor_sync(0xffffffffu, part1, 1);
      if constexpr (HI >= 8) {
        part0 += __shfl_xor_sync(0xffffffffu, part0, 2);
        part1 += __shfl_xor_sync(0xffffffffu, part1, 2);
      }
      const bool writer = (HI >= 8) ? (c == 0) : ((c & 1) == 0);
      if (writer) {
        o_s[tok * kKeysPerCta + warp * 16 + g] = part0;
        o_s[tok * kKeysPerCta + warp * 16 + g + 8] = part1;
      }
      part0 = part1 = 0.f;
    }
  }
  __syncthreads();

  // ---- scale, mask and write the tile rows -----------------------------------------
  const float* skg = FP8 ? p.k_scale + (int64_t)b * p.S : nullptr;
  for (int i = threadIdx.x; i < ntok * kKeysPerCta; i += kThreads) {
    const int tok = i / kKeysPerCta, kk = i % kKeysPerCta;
    if (kk >= kend) continue;
    const int s = key0 + kk;
    const int64_t n = visible(t_first + tok);
    float v;
    if (s < n) {
      v = o_s[i];
      if (FP8) v *= sq_s[tok] * __ldg(skg + s);
    } else {
      if (!p.write_masked) continue;
      v = -INFINITY;
    }
    out_b[(int64_t)(tl0 + tok) * p.ld + s] = v;
  }
}

template <int HI, int DI, bool FP8, int TB>
cudaError_t launch_tb(const IndexerLaunch& p, cudaStream_t st) {
  using C = IxTile<HI, DI, FP8, TB>;
  auto kern = k_indexer_mma<HI, DI, FP8, TB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.S + kKeysPerCta - 1) / kKeysPerCta, (p.Tc + TB - 1) / TB, p.B);
  kern<<<grid, kThreads, C::kSmem, st>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_scores_mma(const IndexerLaunch& p, cudaStream_t st) {
  if (p.B <= 0 || p.Tc <= 0 || p.S <= 0) return cudaSuccess;
  if (p.HI == 64 && p.DI == 128) return p.fp8 ? launch_tb<64, 128, true, 4>(p, st) : launch_tb<64, 128, false, 4>(p, st);
  if (p.HI == 4 && p.DI == 64 && !p.fp8) return launch_tb<4, 64, false, 32>(p, st);
  return cudaErrorInvalidValue;
}

}  // namespace dsa
