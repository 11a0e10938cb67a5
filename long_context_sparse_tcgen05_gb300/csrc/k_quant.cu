// FP8 e4m3 quantisation of indexer rows, one fp32 scale per row, written into a cache (the
// step before the FP8 indexer, which reads e4m3 codes with per-token scales: IndexCache
// notes, section 1, "few heads, low-rank, FP8").  For a row x of `width` bf16 values:
// scale = amax / 448 (1 for an all-zero row) and code = e4m3(x / scale), rounded to nearest
// even and saturated to +-448, in fp32 (IEEE division, no reciprocal).
//
// One warp per row: pass 1 takes the row maximum of |x| (8-byte loads, a warp max), pass 2
// reads the row again (from L1/L2), divides and packs four codes into one 32-bit store.
// HBM-bound: 2*width bytes read, width + 4 written per row.
#include <algorithm>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kQuantWarps = 8;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// two fp32 -> two e4m3 codes (lo in the low byte), round to nearest even, saturate finite
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

__global__ void __launch_bounds__(kQuantWarps * 32) k_quant_e4m3_rows(QuantLaunch p) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)p.B * p.n;
  for (int64_t r = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5); r < rows;
       r += (int64_t)gridDim.x * kQuantWarps) {
    const int b = (int)(r / p.n), i = (int)(r - (int64_t)b * p.n);
    const int64_t pos = p.positions ? p.positions[b] : p.pos0;
    if (pos < 0 || pos > (int64_t)p.S_cap - p.n) {
      if (lane == 0) atomicOr(p.flags, DSA_FLAG_BAD_INDEX);
      continue;
    }
    const uint16_t* x = p.x + (int64_t)b * p.x_stride_b + (int64_t)i * p.width;
    const int64_t dst = (int64_t)b * p.S_cap + pos + i;
    float amax = 0.f;
    for (int j = lane * 4; j < p.width; j += 128) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(x + j));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                               fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? amax / 448.f : 1.f;
    uint8_t* codes = p.codes + dst * p.width;
    for (int j = lane * 4; j < p.width; j += 128) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(x + j));
      const uint32_t c01 = e4m3x2(bf16_lo(v.x) / scale, bf16_hi(v.x) / scale);
      const uint32_t c23 = e4m3x2(bf16_lo(v.y) / scale, bf16_hi(v.y) / scale);
      *reinterpret_cast<uint32_t*>(codes + j) = c01 | (c23 << 16);
    }
    if (lane == 0) p.scales[dst] = scale;
  }
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_quant_e4m3_rows(const QuantLaunch& p, cudaStream_t st) {
  const int64_t rows = (int64_t)p.B * p.n;
  if (rows == 0) return cudaSuccess;
  const int64_t want = (rows + kQuantWarps - 1) / kQuantWarps;
  const int grid = (int)std::min<int64_t>(want, (int64_t)sm_count() * 8);
  k_quant_e4m3_rows<<<grid, kQuantWarps * 32, 0, st>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
