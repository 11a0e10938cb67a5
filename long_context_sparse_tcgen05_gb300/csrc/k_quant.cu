// FP8 e4m3 quantisation of indexer rows, one fp32 scale per row, written into a cache (the
// step before the FP8 indexer, which reads e4m3 codes with per-token scales: IndexCache
// notes, section 1, "few heads, low-rank, FP8").  For a row x of `width` bf16 values:
// scale = amax / 448 (1 for an all-zero row) and code = e4m3(x / scale), rounded to nearest
// even and saturated to +-448, in fp32 (IEEE division, no reciprocal).
//
// Rows of up to 8,192 values are read once: a team of threads (a warp for rows of up to
// 1,024 values, a 256-thread CTA above) holds the row in registers, four values per 8-byte
// load, takes the team maximum of |x|, then divides and packs four codes into each 32-bit
// store.  Wider rows take a warp each and read the row twice (maximum, then codes).
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

// destination row of row r (sequence b, new row i), or -1 for a position outside the cache
__device__ __forceinline__ int64_t quant_dst(const QuantLaunch& p, int64_t r) {
  const int b = (int)(r / p.n), i = (int)(r - (int64_t)b * p.n);
  const int64_t pos = p.positions ? p.positions[b] : p.pos0;
  if (pos < 0 || pos > (int64_t)p.S_cap - p.n) return -1;
  return (int64_t)b * p.S_cap + pos + i;
}

// Team of kTeam threads per row (32: a warp, else the whole CTA), kUnits 4-value units per
// thread; a row is at most kTeam * kUnits * 4 values.
template <int kTeam, int kUnits>
__global__ void __launch_bounds__(256) k_quant_e4m3_rows_reg(QuantLaunch p) {
  __shared__ float team_max[256 / 32];
  const int lane = threadIdx.x & 31;
  const int t = kTeam == 32 ? lane : threadIdx.x;
  const int teams = kTeam == 32 ? 8 : 1;
  const int team = kTeam == 32 ? (threadIdx.x >> 5) : 0;
  const int64_t rows = (int64_t)p.B * p.n;
  for (int64_t r = (int64_t)blockIdx.x * teams + team; r < rows; r += (int64_t)gridDim.x * teams) {
    const int64_t dst = quant_dst(p, r);  // uniform over the team
    if (dst < 0) {
      if (t == 0) atomicOr(p.flags, DSA_FLAG_BAD_INDEX);
      continue;
    }
    const int b = (int)(r / p.n), i = (int)(r - (int64_t)b * p.n);
    const uint16_t* x = p.x + (int64_t)b * p.x_stride_b + (int64_t)i * p.width;
    uint2 v[kUnits];
    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
      const int j = (t + u * kTeam) * 4;
      v[u] = j < p.width ? __ldg(reinterpret_cast<const uint2*>(x + j)) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUnits; ++u)
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(v[u].x)), fabsf(bf16_hi(v[u].x))),
                               fmaxf(fabsf(bf16_lo(v[u].y)), fabsf(bf16_hi(v[u].y)))));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (kTeam > 32) {
      if (lane == 0) team_max[threadIdx.x >> 5] = amax;
      __syncthreads();
#pragma unroll
      for (int w = 0; w < kTeam / 32; ++w) amax = fmaxf(amax, team_max[w]);
      __syncthreads();  // team_max is rewritten for the next row
    }
    const float scale = amax > 0.f ? amax / 448.f : 1.f;
    uint8_t* codes = p.codes + dst * p.width;
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
      const int j = (t + u * kTeam) * 4;
      if (j < p.width) {
        const uint32_t c01 = e4m3x2(bf16_lo(v[u].x) / scale, bf16_hi(v[u].x) / scale);
        const uint32_t c23 = e4m3x2(bf16_lo(v[u].y) / scale, bf16_hi(v[u].y) / scale);
        *reinterpret_cast<uint32_t*>(codes + j) = c01 | (c23 << 16);
      }
    }
    if (t == 0) p.scales[dst] = scale;
  }
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
  const int64_t cap = (int64_t)sm_count() * 8;  // 8 resident 256-thread CTAs per SM
  const int64_t warp_grid = std::min<int64_t>((rows + 7) / 8, cap);
  const int64_t cta_grid = std::min<int64_t>(rows, cap);
  const int w = p.width;
  if (w <= 32 * 4 * 1) k_quant_e4m3_rows_reg<32, 1><<<(int)warp_grid, 256, 0, st>>>(p);
  else if (w <= 32 * 4 * 2) k_quant_e4m3_rows_reg<32, 2><<<(int)warp_grid, 256, 0, st>>>(p);
  else if (w <= 32 * 4 * 8) k_quant_e4m3_rows_reg<32, 8><<<(int)warp_grid, 256, 0, st>>>(p);
  else if (w <= 256 * 4 * 2) k_quant_e4m3_rows_reg<256, 2><<<(int)cta_grid, 256, 0, st>>>(p);
  else if (w <= 256 * 4 * 8) k_quant_e4m3_rows_reg<256, 8><<<(int)cta_grid, 256, 0, st>>>(p);
  else k_quant_e4m3_rows<<<(int)warp_grid, kQuantWarps * 32, 0, st>>>(p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace dsa
