// Sparse multi-query attention over index-selected KV rows, warp-level mma.sync version.
//
// One CTA owns one query row (all H heads).  It walks the row's index list in blocks of
// NB entries: the selected KV rows are gathered with 16-byte cp.async copies into a
// double-buffered shared-memory stage (an entry of -1 is zero-filled and masked), then
//   S = Q K^T (heads x NB) on tensor cores, online softmax in fp32 with base-2 exponents,
//   P (bf16) to shared memory, O += P V on tensor cores (V read transposed from the same
//   stage; with a latent KV, V is the first d_v columns of the gathered rows).
// Warps are arranged WM x 2: WM groups of 16 heads; the two warps of a group split the
// keys of S and the value columns of O.  Rows are padded by 16 bytes in shared memory so
// that every ldmatrix is bank-conflict free.
#include <cuda_bf16.h>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int HP, int DQK, int DV, bool SEPV, int NB>
struct AtCfg {
  static constexpr int kWM = HP / 16, kWN = 2, kThreads = 32 * kWM * kWN;
  static constexpr int kQPad = DQK + 8, kKPad = DQK + 8, kVPad = DV + 8, kPPad = NB + 8;
  static constexpr int kKChunks = DQK * 2 / 16, kVChunks = DV * 2 / 16;
  static constexpr int kOTiles = DV / kWN / 8;  // n8 tiles of O per warp
  static constexpr size_t kQBytes = (size_t)HP * kQPad * 2;
  static constexpr size_t kKBytes = (size_t)NB * kKPad * 2;
  static constexpr size_t kVBytes = SEPV ? (size_t)NB * kVPad * 2 : 0;
  static constexpr size_t kPBytes = (size_t)HP * kPPad * 2;
  static constexpr size_t kSmem = kQBytes + 2 * kKBytes + 2 * kVBytes + kPBytes +
                                  (size_t)kWN * HP * 4 * 2 + 2 * NB * 4 + 16;
  static_assert(HP % 16 == 0 && NB == 16 * kWN && kOTiles % 2 == 0, "tile shape");
};

template <int HP, int DQK, int DV, bool SEPV, int NB>
__global__ void __launch_bounds__(AtCfg<HP, DQK, DV, SEPV, NB>::kThreads, 1)
    k_sparse_attn_mma(AttnLaunch p) {
  using C = AtCfg<HP, DQK, DV, SEPV, NB>;
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16* q_s = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* k_s = reinterpret_cast<__nv_bfloat16*>(smem + C::kQBytes);  // [2][NB][kKPad]
  __nv_bfloat16* v_s = reinterpret_cast<__nv_bfloat16*>(smem + C::kQBytes + 2 * C::kKBytes);
  __nv_bfloat16* p_s = reinterpret_cast<__nv_bfloat16*>(smem + C::kQBytes + 2 * C::kKBytes + 2 * C::kVBytes);
  float* red_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(p_s) + C::kPBytes);  // [kWN][HP]
  float* lsum_s = red_s + C::kWN * HP;                                                    // [kWN][HP]
  int* valid_s = reinterpret_cast<int*>(lsum_s + C::kWN * HP);                             // [2][NB]
  int* last_s = valid_s + 2 * NB;

  const int row = blockIdx.x;  // flat b*T + t
  const int b = row / p.T;
  const int32_t* irow = attn_idx_row(p, row);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp / C::kWN, wn = warp % C::kWN;
  const int g = lane >> 2, c = lane & 3;

  // Number of index blocks that hold any entry other than -1.
  if (threadIdx.x == 0) *last_s = -1;
  __syncthreads();
  {
    int last = -1;
    for (int j = threadIdx.x; j < p.kk; j += C::kThreads)
      if (irow[j] != -1) last = j;
    if (last >= 0) atomicMax(last_s, last);
  }
  // Query tile (heads beyond H are zero).
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) + (int64_t)b * p.q_sb + (int64_t)(row % p.T) * p.q_st;
  for (int i = threadIdx.x; i < HP * C::kKChunks; i += C::kThreads) {
    const int h = i / C::kKChunks, c16 = i % C::kKChunks;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (h < p.H) v = __ldg(reinterpret_cast<const uint4*>(qg + (int64_t)h * DQK) + c16);
    *reinterpret_cast<uint4*>(q_s + h * C::kQPad + c16 * 8) = v;
  }
  __syncthreads();
  const int nblocks = (*last_s + NB) / NB;

  const __nv_bfloat16* kbase = static_cast<const __nv_bfloat16*>(p.k) + (int64_t)b * p.k_sb;
  const __nv_bfloat16* vbase = static_cast<const __nv_bfloat16*>(p.v) + (int64_t)b * p.v_sb;
  auto gather = [&](int jb, int stage) {
    for (int i = threadIdx.x; i < NB * C::kKChunks; i += C::kThreads) {
      const int r = i / C::kKChunks, c16 = i % C::kKChunks;
      const int j = jb * NB + r;
      const int id = j < p.kk ? __ldg(irow + j) : -1;
      const bool ok = id >= 0 && id < p.S;
      if (c16 == 0) {
        valid_s[stage * NB + r] = ok;
        if (!ok && id != -1) atomicOr(p.flags, DSA_FLAG_BAD_INDEX);
      }
      const __nv_bfloat16* src = ok ? kbase + (int64_t)id * p.k_ld + c16 * 8 : kbase;
      cp_async16(smem_u32(k_s + (stage * NB + r) * C::kKPad + c16 * 8), src, ok);
    }
    if constexpr (SEPV) {
      for (int i = threadIdx.x; i < NB * C::kVChunks; i += C::kThreads) {
        const int r = i / C::kVChunks, c16 = i % C::kVChunks;
        const int j = jb * NB + r;
        const int id = j < p.kk ? __ldg(irow + j) : -1;
        const bool ok = id >= 0 && id < p.S;
        const __nv_bfloat16* src = ok ? vbase + (int64_t)id * p.v_ld + c16 * 8 : vbase;
        cp_async16(smem_u32(v_s + (stage * NB + r) * C::kVPad + c16 * 8), src, ok);
      }
    }
    cp_async_commit();
  };

  float o[C::kOTiles][4];
#pragma unroll
  for (int i = 0; i < C::kOTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows g, g+8 of the warp's group
  const float sl2 = p.scale * kLog2e;
  const int hr0 = wm * 16 + g, hr1 = hr0 + 8;

  if (nblocks > 0) gather(0, 0);
#pragma unroll 1
  for (int jb = 0; jb < nblocks; ++jb) {
    const int st = jb & 1;
    if (jb + 1 < nblocks) {
      gather(jb + 1, st ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    // ---- S = Q K^T for 16 heads x 16 keys per warp --------------------------------
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const __nv_bfloat16* ks_ = k_s + st * NB * C::kKPad;
    const uint32_t qa = smem_u32(q_s + (wm * 16 + (lane & 15)) * C::kQPad + (lane >> 4) * 8);
    const uint32_t kb = smem_u32(ks_ + (wn * 16 + (lane & 7) + (lane >> 4) * 8) * C::kKPad + ((lane >> 3) & 1) * 8);
#pragma unroll 4
    for (int kstep = 0; kstep < DQK / 16; ++kstep) {
      uint32_t a[4], bb[4];
      ldsm_x4(qa + kstep * 32, a);
      ldsm_x4(kb + kstep * 32, bb);
      mma_bf16(s[0], a, bb[0], bb[1]);
      mma_bf16(s[1], a, bb[2], bb[3]);
    }
    // ---- online softmax ------------------------------------------------------------
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int key = wn * 16 + nt * 8 + 2 * c;
      const bool v0 = valid_s[st * NB + key], v1 = valid_s[st * NB + key + 1];
      s[nt][0] = v0 ? s[nt][0] * sl2 : -INFINITY;
      s[nt][1] = v1 ? s[nt][1] * sl2 : -INFINITY;
      s[nt][2] = v0 ? s[nt][2] * sl2 : -INFINITY;
      s[nt][3] = v1 ? s[nt][3] * sl2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (c == 0) {
      red_s[wn * HP + hr0] = mx0;
      red_s[wn * HP + hr1] = mx1;
    }
    __syncthreads();
    mx0 = fmaxf(red_s[hr0], red_s[HP + hr0]);
    mx1 = fmaxf(red_s[hr1], red_s[HP + hr1]);
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = ex2(m0 - mu0), al1 = ex2(m1 - mu1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int key = wn * 16 + nt * 8 + 2 * c;
      // the row sums use the fp32 weights; P enters the PV product rounded to bf16
      const float p0 = ex2(s[nt][0] - mu0), p1 = ex2(s[nt][1] - mu0);
      const float p2 = ex2(s[nt][2] - mu1), p3 = ex2(s[nt][3] - mu1);
      const uint32_t u01 = pack_bf16(p0, p1);
      const uint32_t u23 = pack_bf16(p2, p3);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      *reinterpret_cast<uint32_t*>(p_s + hr0 * C::kPPad + key) = u01;
      *reinterpret_cast<uint32_t*>(p_s + hr1 * C::kPPad + key) = u23;
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int i = 0; i < C::kOTiles; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al0;
      o[i][2] *= al1;
      o[i][3] *= al1;
    }
    __syncthreads();

    // ---- O += P V --------------------------------------------------------------------
    const __nv_bfloat16* vs_ = SEPV ? v_s + st * NB * C::kVPad : ks_;
    constexpr int kVP = SEPV ? C::kVPad : C::kKPad;
    const int dbase = wn * (DV / C::kWN);
#pragma unroll
    for (int kstep = 0; kstep < NB / 16; ++kstep) {
      uint32_t a[4];
      ldsm_x4(smem_u32(p_s + (wm * 16 + (lane & 15)) * C::kPPad + kstep * 16 + (lane >> 4) * 8), a);
      const uint32_t vb = smem_u32(vs_ + (kstep * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kVP + dbase + (lane >> 4) * 8);
#pragma unroll
      for (int np = 0; np < C::kOTiles / 2; ++np) {
        uint32_t bb[4];
        ldsm_x4_t(vb + np * 32, bb);
        mma_bf16(o[2 * np], a, bb[0], bb[1]);
        mma_bf16(o[2 * np + 1], a, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }

  // ---- normalise and store --------------------------------------------------------
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (c == 0) {
    lsum_s[wn * HP + hr0] = l0;
    lsum_s[wn * HP + hr1] = l1;
  }
  __syncthreads();
  const float L0 = lsum_s[hr0] + lsum_s[HP + hr0];
  const float L1 = lsum_s[hr1] + lsum_s[HP + hr1];
  const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(p.out) + (int64_t)row * p.H * DV;
  const int dbase = wn * (DV / C::kWN);
#pragma unroll
  for (int i = 0; i < C::kOTiles; ++i) {
    const int d = dbase + i * 8 + 2 * c;
    if (hr0 < p.H)
      *reinterpret_cast<__nv_bfloat162*>(og + (int64_t)hr0 * DV + d) = __floats2bfloat162_rn(o[i][0] * inv0, o[i][1] * inv0);
    if (hr1 < p.H)
      *reinterpret_cast<__nv_bfloat162*>(og + (int64_t)hr1 * DV + d) = __floats2bfloat162_rn(o[i][2] * inv1, o[i][3] * inv1);
  }
  if (p.lse && wn == 0 && c == 0) {
    float* lg = p.lse + (int64_t)row * p.H;
    if (hr0 < p.H) lg[hr0] = L0 > 0.f ? (m0 + log2f(L0)) * kLn2 : -INFINITY;
    if (hr1 < p.H) lg[hr1] = L1 > 0.f ? (m1 + log2f(L1)) * kLn2 : -INFINITY;
  }
}

template <int HP, int DQK, int DV, bool SEPV>
cudaError_t launch_cfg(const AttnLaunch& p, cudaStream_t st) {
  TraceScope trace(kTraceAttention, st);
  constexpr int NB = 32;
  using C = AtCfg<HP, DQK, DV, SEPV, NB>;
  auto kern = k_sparse_attn_mma<HP, DQK, DV, SEPV, NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<p.B * p.T, C::kThreads, C::kSmem, st>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_attn(const AttnLaunch& p, cudaStream_t st) {
  if (p.B * p.T <= 0) return cudaSuccess;
  if (sparse_mla_tc_supported(p)) return launch_sparse_mla_tc(p, st);
  if (p.layers > 1) return cudaErrorInvalidValue;  // several layers per launch: the tcgen05 kernel only
  const bool latent = p.v == p.k && p.v_ld == p.k_ld && p.v_sb == p.k_sb;
  if (p.H == 64 && p.DQK == 576 && p.DV == 512)
    return latent ? launch_cfg<64, 576, 512, false>(p, st) : launch_cfg<64, 576, 512, true>(p, st);
  if (p.H <= 16 && p.DQK == 64 && p.DV == 64)
    return latent ? launch_cfg<16, 64, 64, false>(p, st) : launch_cfg<16, 64, 64, true>(p, st);
  return cudaErrorInvalidValue;
}

}  // namespace dsa
