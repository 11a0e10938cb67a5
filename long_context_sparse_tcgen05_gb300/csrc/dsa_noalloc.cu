// dsa_topk_indexer_noalloc: the indexer -> top-k path with its scratch space in a
// library-owned, statically sized device array instead of a caller workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where they call
// us -- code running inside a custom allocator or memory-pool callback, plugins of
// runtimes that own and pre-partition all device memory, or code that must not grow its
// footprint after start-up.  They still own and pass the inputs and the output buffer;
// the score chunks that dsa_topk(FROM_INDEXER) keeps in the caller's workspace live here
// in a fixed 64 MiB array that every GPU which loads this library holds until exit.
#include <cstdio>
#include <mutex>

#include "dsa_internal.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;
constexpr size_t kFlagBytes = 256;  // flag word at the front, scores after it
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.  In host
// code `g_static_scratch` names a host-side stand-in, so the address has to come from
// cudaGetSymbolAddress with that device current.
dsa_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dsa::record_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return dsa::record_error(DSA_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch failed: %s", cudaGetErrorString(e));
      return dsa::record_error(DSA_ERR_CUDA, msg);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" dsa_status dsa_topk_indexer_noalloc(const dsa_indexer_args* ix, int32_t k, int32_t* idx,
                                               uint32_t* flags, void* stream) {
  dsa_status s = dsa::validate_indexer(ix);
  if (s != DSA_OK) return s;
  if (!idx) return dsa::record_error(DSA_ERR_INVALID_ARG, "idx is NULL");
  if (k < 1 || k > 4096) return dsa::record_error(DSA_ERR_UNSUPPORTED, "k outside [1, 4096]");
  const size_t row_bytes = (size_t)ix->B * (size_t)ix->S * sizeof(float);
  if (row_bytes > kStaticScratchBytes - kFlagBytes)
    return dsa::record_error(DSA_ERR_UNSUPPORTED,
                             "B*S too large for the 64 MiB static scratch (needs B*S*4 <= 64 MiB - 256 B)");
  void* base = nullptr;
  if ((s = scratch_address(&base)) != DSA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* flag_word = flags ? flags : static_cast<uint32_t*>(base);
  if (!flags) {  // the array keeps the previous call's contents: the flag word starts at 0
    cudaError_t e = cudaMemsetAsync(base, 0, sizeof(uint32_t), st);
    if (e != cudaSuccess) return dsa::record_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  }
  float* sc = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kFlagBytes);
  const int64_t chunk_max = (int64_t)((kStaticScratchBytes - kFlagBytes) / row_bytes);
  for (int64_t t0 = 0; t0 < ix->T; t0 += chunk_max) {
    const int Tc = (int)((ix->T - t0) < chunk_max ? (ix->T - t0) : chunk_max);
    dsa::IndexerLaunch L = dsa::make_indexer_launch(ix, t0, Tc);
    L.out = sc; L.ld = ix->S; L.out_bstride = (int64_t)Tc * ix->S; L.write_masked = 0;
    L.flags = flag_word;
    cudaError_t e = dsa::launch_indexer_scores(L, st);
    if (e != cudaSuccess) return dsa::record_error(DSA_ERR_CUDA, cudaGetErrorString(e));
    dsa::TopkLaunch P{};
    P.scores = sc; P.ld = ix->S; P.bstride = (int64_t)Tc * ix->S;
    P.B = ix->B; P.T = ix->T; P.S = ix->S; P.t0 = (int)t0; P.Tc = Tc;
    P.q_pos0 = ix->q_pos0; P.diag = ix->diag; P.k = k; P.idx = idx; P.flags = flag_word;
    // few long rows (decode): split each over CTAs when the array's tail, after this chunk's
    // scores, holds the segments' lists (B = 32 rows of 200,000 keys: 25.6 MB of scores and
    // 8.4 MB of lists)
    const size_t lists_off = (kFlagBytes + (size_t)Tc * row_bytes + 255) & ~(size_t)255;
    dsa::plan_topk_split(P, (int64_t)ix->B * Tc, dsa::max_visible_keys(ix->q_pos0, ix->T, ix->diag, ix->S), base,
                         lists_off, kStaticScratchBytes);
    e = dsa::launch_topk_rows(P, st);
    if (e != cudaSuccess) return dsa::record_error(DSA_ERR_CUDA, cudaGetErrorString(e));
  }
  return DSA_OK;
}
