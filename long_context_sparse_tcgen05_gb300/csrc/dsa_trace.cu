// Launch tracing: when enabled, each launcher's kernels are bracketed by a pair of CUDA events
// recorded on the launch stream, so a host program can read per-kernel device durations of
// work it timed as a whole (a benchmark's timed region) without synchronising inside it.
// Events come from a pool created by dsa_trace_enable; when the pool runs out, further
// launches go unrecorded (dsa_trace_read reports how many were dropped).
#include <mutex>
#include <vector>

#include "dsa.h"
#include "dsa_internal.cuh"

namespace dsa {
namespace {

struct Rec {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_mu;
bool g_on = false;
std::vector<cudaEvent_t> g_free;  // pooled events
std::vector<Rec> g_recs;          // open and closed records, in launch order
int g_dropped = 0;

}  // namespace

int trace_open(int kind, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return -1;
  if (g_free.size() < 2) {
    ++g_dropped;
    return -1;
  }
  Rec r{kind, g_free.back(), nullptr};
  g_free.pop_back();
  r.b = g_free.back();
  g_free.pop_back();
  if (cudaEventRecord(r.a, st) != cudaSuccess) {
    g_free.push_back(r.b);
    g_free.push_back(r.a);
    return -1;
  }
  g_recs.push_back(r);
  return (int)g_recs.size() - 1;
}

void trace_close(int slot, cudaStream_t st) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (slot < (int)g_recs.size()) cudaEventRecord(g_recs[slot].b, st);
}

}  // namespace dsa

extern "C" {

dsa_status dsa_trace_enable(int max_launches) {
  if (max_launches <= 0 || max_launches > (1 << 20)) return DSA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(dsa::g_mu);
  for (int i = (int)dsa::g_free.size(); i < 2 * max_launches; ++i) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return DSA_ERR_CUDA;
    dsa::g_free.push_back(e);
  }
  dsa::g_recs.clear();
  dsa::g_dropped = 0;
  dsa::g_on = true;
  return DSA_OK;
}

int dsa_trace_read(int* kinds, float* ms, int max_records, int* dropped) {
  std::lock_guard<std::mutex> lk(dsa::g_mu);
  int n = 0;
  for (const dsa::Rec& r : dsa::g_recs) {
    float t = -1.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) t = -1.f;
    if (n < max_records) {
      if (kinds) kinds[n] = r.kind;
      if (ms) ms[n] = t;
    }
    ++n;
    dsa::g_free.push_back(r.a);
    dsa::g_free.push_back(r.b);
  }
  dsa::g_recs.clear();
  if (dropped) *dropped = dsa::g_dropped;
  dsa::g_dropped = 0;
  return n < max_records ? n : max_records;
}

void dsa_trace_disable(void) {
  std::lock_guard<std::mutex> lk(dsa::g_mu);
  dsa::g_on = false;
  for (const dsa::Rec& r : dsa::g_recs) {
    cudaEventSynchronize(r.b);
    dsa::g_free.push_back(r.a);
    dsa::g_free.push_back(r.b);
  }
  dsa::g_recs.clear();
  for (cudaEvent_t e : dsa::g_free) cudaEventDestroy(e);
  dsa::g_free.clear();
}

}  // extern "C"
