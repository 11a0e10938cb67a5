// Internal launch interface between the host API (dsa_api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "dsa.h"

namespace dsa {

// Workspace layout: the flag word and a double for reductions live in the first
// DSA_WS_MIN bytes; scratch buffers start at kWsScratch.
constexpr size_t kWsFlags = 0;
constexpr size_t kWsMean = 8;
constexpr size_t kWsScratch = DSA_WS_MIN;

// Kernel launches issued by this library since load (diagnostics; see dsa_launch_count).
void count_launches(uint64_t n);

// Bound, in SM clock cycles, on the waits of kernels launched now (dsa_set_wait_limit).
constexpr long long kDefaultWaitCycles = 2000000000LL;  // ~1 s at 2 GHz
long long wait_limit();

// Launch tracing (dsa_trace_enable): when on, a scope brackets one launcher's kernels with
// CUDA events on its stream; durations are read back by dsa_trace_read.
enum TraceKind { kTraceIndexer = 1, kTraceTopk = 2, kTraceAttention = 3, kTraceOverlap = 4 };
int trace_open(int kind, cudaStream_t st);
void trace_close(int slot, cudaStream_t st);
struct TraceScope {
  int slot;
  cudaStream_t st;
  TraceScope(int kind, cudaStream_t s) : slot(trace_open(kind, s)), st(s) {}
  ~TraceScope() { trace_close(slot, st); }
  TraceScope(const TraceScope&) = delete;
  TraceScope& operator=(const TraceScope&) = delete;
};

// Host-side helpers shared by the entry points: argument checks of an indexer operand set
// (sets the thread's last-error message on failure) and recording a failure message.
dsa_status validate_indexer(const dsa_indexer_args* ix);
dsa_status record_error(dsa_status s, const char* msg);

// Key transform of the selection order: a larger float gives a larger unsigned key.
// -0 and +0 share one key; NaN maps below -inf.
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 + 0 = +0; every other value is unchanged
  const uint32_t key = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);  // negatives: ~u, else u | sign
  return f != f ? 0u : key;                      // NaN ranks below every number
}

// Rows [t0, t0 + Tc) of every sequence of one layer's indexer.
struct IndexerLaunch;
IndexerLaunch make_indexer_launch(const dsa_indexer_args* ix, int64_t t0, int Tc);  // strides resolved

struct IndexerLaunch {
  int B, T, S, HI, DI;
  int fp8;
  const void* q;
  int64_t q_sb, q_st;   // token strides of q in elements (resolved: never 0)
  int64_t k_sb;         // sequence stride of k in elements
  const float* q_scale;
  const float* w;
  const void* k;
  const float* k_scale;
  int64_t q_pos0;
  int diag;
  int t0, Tc;
  float* out;           // out[b*out_bstride + (t - t0)*ld + s]
  int64_t ld;
  int64_t out_bstride;
  int write_masked;     // 1: write -inf over [n_t, S) as well
  uint32_t* flags;      // device flag word (DSA_FLAG_TIMEOUT)
  int ksplit;           // key-range splits per token block (0: chosen by the launcher)
  int ctas_min;         // launcher's split: at least this many CTAs (0: four waves)
  long long wait;       // wait bound in cycles (0: wait_limit() at launch)
  // selecting mode (select != 0; H_I = 64, one CTA per token block): instead of writing scores,
  // row r = b*Tc + (t - t0) keeps every key whose score reaches a threshold set from a sample of
  // its tiles (enough keys to hold the top k of them with high probability, at most `target`):
  // (score bits, position) pairs go to one of four segments of
  // cand[r*cap ..] (one per lane quarter of the key tiles, cap/4 each), the segment's count to
  // cand_cnt[r*4 + q]
  int select;
  int cap, target, topk;
  uint2* cand;
  int32_t* cand_cnt;
  // recomputing mode: when gate is set, only token blocks holding a row (b, t) whose flag
  // gate[b*gate_bstride + t - t0] is non-zero run
  const uint8_t* gate;
  int64_t gate_bstride;
};
cudaError_t launch_indexer_scores(const IndexerLaunch& p, cudaStream_t st);     // tcgen05 path

// Top-k over materialised score rows: rows [t0, t0 + Tc) of every sequence,
// scores[b*bstride + (t - t0)*ld + s], output idx[(b*T + t)*k + j].
struct TopkLaunch {
  const float* scores;
  int64_t ld, bstride;
  int B, T, S, t0, Tc;
  int64_t q_pos0;
  int diag, k;
  int32_t* idx;
  uint32_t* flags;
  long long wait;       // wait bound in cycles (0: wait_limit() at launch)
  // recomputing mode: when gate is set, only rows (b, t) whose flag gate[b*gate_bstride + t - t0]
  // is non-zero run
  const uint8_t* gate;
  int64_t gate_bstride;
  // few long rows: each row split into `parts` segments (> 1), one CTA each; segment s of row
  // r = b*Tc + tl writes its exact top-k, sorted by position, with the keys, to
  // part_pos / part_key[(r*parts + s)*k ..] and its length to part_cnt[r*parts + s]; a merge
  // kernel then writes idx
  int parts;
  int32_t* part_pos;
  uint32_t* part_key;
  int32_t* part_cnt;
};
// Few long rows: split each row of a top-k launch across CTAs when ws + off .. ws + ws_bytes
// holds the segments' lists (P.parts stays 1 otherwise); n_max: the longest row's keys.
void plan_topk_split(TopkLaunch& P, int64_t rows, int64_t n_max, void* ws, size_t off, size_t ws_bytes);
int64_t max_visible_keys(int64_t q_pos0, int T, int diag, int S);  // of the call's last row
cudaError_t launch_topk_rows(const TopkLaunch& p, cudaStream_t st);
constexpr int kMaxTopkParts = 16;

// Top-k of rows [t0, t0 + Tc) of every sequence from the candidates of a selecting indexer pass
// (IndexerLaunch::select): row r = b*Tc + (t - t0) holds four segments of candidates (fp32 score
// bits, position), segment q at cand[r*cap + q*cap/4 ..] with cand_cnt[r*4 + q] entries (more
// than cap/4 means it overflowed).  A row whose candidates cannot hold its top-k (fewer than
// min(k, visible) of them, or more than cap) gets fail[r] = 1 and is left for the recomputing
// pass; every other row gets fail[r] = 0 and its idx row.
struct CandLaunch {
  int B, T, S, t0, Tc;
  int64_t q_pos0;
  int diag, k, cap;
  const uint2* cand;
  const int32_t* cand_cnt;
  uint8_t* fail;
  int32_t* idx;
};
constexpr int kCandMaxK = 2048;     // selecting path: k up to this
constexpr int kCandMaxCap = 8192;   // candidates per row held in shared memory
cudaError_t launch_topk_cand(const CandLaunch& p, cudaStream_t st);
// Segments per row for `rows` rows of up to `n` visible scores (1: no split).
int topk_parts(int64_t rows, int64_t n);

constexpr int kMaxAttnLayers = 8;
struct AttnLaunch {
  int B, T, S, H, DQK, DV;
  float scale;
  const void* q;
  const void* k;
  int64_t k_ld;
  const void* v;
  int64_t v_ld;
  int64_t q_sb, q_st;   // query strides in elements (resolved: never 0)
  int64_t k_sb, v_sb;   // sequence strides of k and v in elements
  const int32_t* idx;
  int kk;
  // index-row strides in elements: row (b, t) reads idx + b*idx_sb + t*idx_st (dense rows:
  // kk and T*kk; the draft steps of a sequence sharing its one row: 0 and kk)
  int64_t idx_st, idx_sb;
  void* out;
  float* lse;
  uint32_t* flags;
  long long wait;       // wait bound in cycles (0: wait_limit() at launch)
  // few rows (decode): each row's selected blocks split into `splits` (> 1) parts, one CTA
  // each; part s of row r writes its output normalised by its own row sums, fp32,
  // part_o[((r*splits + s)*H + h)*DV ..], and its LSE part_lse[(r*splits + s)*H + h]; a
  // combine kernel merges them into out / lse
  int splits;
  float* part_o;
  float* part_lse;
  // several layers of one group in one launch (0 or 1: the one layer above): layer l has its
  // own queries, latent KV, output and LSE (same shapes and strides) and reads the same index
  // rows; work items run over layers x rows x parts, part_o / part_lse by that flat item
  int layers;
  // fixed-reference pass (redo set, no split): redo[r] = 1 for flat row r (layer x row) whose
  // row sums left the range the fixed reference keeps exact; a recomputing pass (gate set)
  // then runs only the marked rows
  uint8_t* redo;
  const uint8_t* gate;
  const void* lq[kMaxAttnLayers];
  const void* lk[kMaxAttnLayers];
  void* lout[kMaxAttnLayers];
  float* llse[kMaxAttnLayers];
};
// The index row of flat query row `row` = b*T + t.
__host__ __device__ inline const int32_t* attn_idx_row(const AttnLaunch& p, int row) {
  return p.idx + (int64_t)(row / p.T) * p.idx_sb + (int64_t)(row % p.T) * p.idx_st;
}
cudaError_t launch_sparse_attn(const AttnLaunch& p, cudaStream_t st);
constexpr int kMaxAttnSplits = 8;
int attn_splits(const AttnLaunch& p);  // parts per row the 64-head MLA kernel would use (1: none)
// tcgen05 sparse MLA kernel for the latent shape (H = 64, d_qk = 576, d_v = 512, v = k)
bool sparse_mla_tc_supported(const AttnLaunch& p);
cudaError_t launch_sparse_mla_tc(const AttnLaunch& p, cudaStream_t st);

cudaError_t launch_topk_overlap(const int32_t* a, const int32_t* b, int rows, int k,
                                float* per_row, double* mean_dev, uint32_t* flags,
                                cudaStream_t st);

// All-pairs overlap of n index buffers over the same rows.  part: kMaxOverlapCtas * n * n
// doubles of per-CTA sums; counts: [rows, n, n] int32 or nullptr.
constexpr int kMaxOverlapLayers = 16;
constexpr int kMaxOverlapCtas = 1024;
struct OverlapMatrixLaunch {
  const int32_t* bufs[kMaxOverlapLayers];
  int n, k;
  int64_t rows;
  int32_t* counts;
  double* part;
  uint32_t* flags;
};
size_t overlap_matrix_smem(int n, int k);  // dynamic shared memory of one CTA
cudaError_t launch_overlap_matrix(const OverlapMatrixLaunch& p, double* matrix_dev, cudaStream_t st);

// Per-row e4m3 quantisation into a cache: rows (b, i) of x [B, n, width] bf16 (sequence stride
// x_stride_b elements) go to row (b, pos_b + i) of codes [B, S_cap, width] and scales [B, S_cap],
// pos_b = positions[b] (device) or pos0.
struct QuantLaunch {
  const uint16_t* x;
  int B, n, width;
  int64_t x_stride_b;
  uint8_t* codes;
  float* scales;
  int S_cap;
  int64_t pos0;
  const int64_t* positions;
  uint32_t* flags;
};
cudaError_t launch_quant_e4m3_rows(const QuantLaunch& p, cudaStream_t st);

}  // namespace dsa
