// Host side of libdsa: argument validation, workspace planning, launch sequencing and the
// IndexShare schedule walk.  No device memory is allocated here; every buffer belongs to
// the caller.
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstring>
#include <string>
#include <vector>

#include "dsa_internal.cuh"

namespace dsa {
static std::atomic<uint64_t> g_launches{0};
void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
static std::atomic<long long> g_wait_limit{kDefaultWaitCycles};
long long wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }
}  // namespace dsa

namespace {

thread_local std::string g_last_error;

dsa_status fail(dsa_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
dsa_status fail(dsa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

dsa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

uint32_t* ws_flags(void* ws) { return reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + dsa::kWsFlags); }

dsa_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(DSA_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned16(ws)) return fail(DSA_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  if (ws_bytes < need) return fail(DSA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return DSA_OK;
}

dsa_status check_indexer(const dsa_indexer_args* ix) {
  if (!ix) return fail(DSA_ERR_INVALID_ARG, "indexer args are NULL");
  if (ix->B <= 0 || ix->T <= 0 || ix->S <= 0 || ix->H_I <= 0 || ix->d_I <= 0)
    return fail(DSA_ERR_INVALID_ARG, "indexer sizes must be positive (B=%d T=%d S=%d H_I=%d d_I=%d)",
                ix->B, ix->T, ix->S, ix->H_I, ix->d_I);
  if (ix->dtype != DSA_BF16 && ix->dtype != DSA_E4M3) return fail(DSA_ERR_INVALID_ARG, "unknown indexer dtype %d", (int)ix->dtype);
  const bool ok_shape = (ix->H_I == 64 && ix->d_I == 128) || (ix->dtype == DSA_BF16 && ix->H_I == 4 && ix->d_I == 64);
  if (!ok_shape) return fail(DSA_ERR_UNSUPPORTED, "indexer shape H_I=%d d_I=%d (%s) is not supported", ix->H_I, ix->d_I,
                             ix->dtype == DSA_E4M3 ? "e4m3" : "bf16");
  if (!ix->q || !ix->w || !ix->k) return fail(DSA_ERR_INVALID_ARG, "indexer q, w and k must be non-NULL");
  if (ix->dtype == DSA_E4M3 && (!ix->q_scale || !ix->k_scale))
    return fail(DSA_ERR_INVALID_ARG, "e4m3 indexer operands need q_scale and k_scale");
  if (!aligned16(ix->q) || !aligned16(ix->k)) return fail(DSA_ERR_MISALIGNED, "indexer q and k must be 16-byte aligned");
  if (!aligned16(ix->w)) return fail(DSA_ERR_MISALIGNED, "indexer w must be 16-byte aligned");
  if (ix->diag < 0 || ix->diag > 1) return fail(DSA_ERR_INVALID_ARG, "diag must be 0 or 1");
  if (ix->q_pos0 < 0) return fail(DSA_ERR_INVALID_ARG, "q_pos0 must be >= 0");
  if (ix->q_stride_b < 0 || ix->q_stride_t < 0 || ix->k_stride_b < 0)
    return fail(DSA_ERR_INVALID_ARG, "indexer strides must be >= 0 (0: dense)");
  if (ix->q_stride_t && ix->q_stride_t < (int64_t)ix->H_I * ix->d_I)
    return fail(DSA_ERR_INVALID_ARG, "q_stride_t = %lld is smaller than H_I * d_I", (long long)ix->q_stride_t);
  const int64_t esz = ix->dtype == DSA_E4M3 ? 1 : 2;
  if ((ix->q_stride_b * esz) % 16 || (ix->q_stride_t * esz) % 16 || (ix->k_stride_b * esz) % 16)
    return fail(DSA_ERR_MISALIGNED, "indexer strides must be multiples of 16 bytes");
  return DSA_OK;
}

// Indexer strides with the dense defaults filled in.
void indexer_strides(const dsa_indexer_args* ix, int64_t* q_sb, int64_t* q_st, int64_t* k_sb) {
  *q_st = ix->q_stride_t ? ix->q_stride_t : (int64_t)ix->H_I * ix->d_I;
  *q_sb = ix->q_stride_b ? ix->q_stride_b : (int64_t)ix->T * *q_st;
  *k_sb = ix->k_stride_b ? ix->k_stride_b : (int64_t)ix->S * ix->d_I;
}

// The launch description of an indexer call over query rows [t0, t0 + Tc).
dsa::IndexerLaunch indexer_launch(const dsa_indexer_args* ix, int64_t t0, int Tc) {
  dsa::IndexerLaunch L{};
  L.B = ix->B; L.T = ix->T; L.S = ix->S; L.HI = ix->H_I; L.DI = ix->d_I;
  L.fp8 = ix->dtype == DSA_E4M3;
  L.q = ix->q; L.q_scale = ix->q_scale; L.w = ix->w; L.k = ix->k; L.k_scale = ix->k_scale;
  indexer_strides(ix, &L.q_sb, &L.q_st, &L.k_sb);
  L.q_pos0 = ix->q_pos0; L.diag = ix->diag;
  L.t0 = (int)t0; L.Tc = Tc;
  return L;
}

dsa_status check_attn(const dsa_attn_args* at) {
  if (!at) return fail(DSA_ERR_INVALID_ARG, "attention args are NULL");
  if (at->B <= 0 || at->T <= 0 || at->S <= 0 || at->H <= 0 || at->d_qk <= 0 || at->d_v <= 0)
    return fail(DSA_ERR_INVALID_ARG, "attention sizes must be positive");
  const bool ok = (at->H == 64 && at->d_qk == 576 && at->d_v == 512) ||
                  (at->H <= 16 && at->d_qk == 64 && at->d_v == 64);
  if (!ok) return fail(DSA_ERR_UNSUPPORTED, "attention shape H=%d d_qk=%d d_v=%d is not supported", at->H, at->d_qk, at->d_v);
  if (!at->q || !at->k || !at->v) return fail(DSA_ERR_INVALID_ARG, "attention q, k and v must be non-NULL");
  if (!aligned16(at->q) || !aligned16(at->k) || !aligned16(at->v)) return fail(DSA_ERR_MISALIGNED, "attention q, k, v must be 16-byte aligned");
  if (at->k_ld < at->d_qk || at->v_ld < at->d_v || at->k_ld % 8 || at->v_ld % 8)
    return fail(DSA_ERR_MISALIGNED, "k_ld/v_ld must cover d_qk/d_v and be multiples of 8 elements");
  if (!(at->scale > 0.f)) return fail(DSA_ERR_INVALID_ARG, "scale must be positive");
  if (at->q_stride_b < 0 || at->q_stride_t < 0 || at->k_stride_b < 0 || at->v_stride_b < 0)
    return fail(DSA_ERR_INVALID_ARG, "attention strides must be >= 0 (0: dense)");
  if (at->q_stride_t && at->q_stride_t < (int64_t)at->H * at->d_qk)
    return fail(DSA_ERR_INVALID_ARG, "q_stride_t = %lld is smaller than H * d_qk", (long long)at->q_stride_t);
  if (at->q_stride_b % 8 || at->q_stride_t % 8 || at->k_stride_b % 8 || at->v_stride_b % 8)
    return fail(DSA_ERR_MISALIGNED, "attention strides must be multiples of 8 elements");
  return DSA_OK;
}

// The launch description of an attention call (strides resolved, no split planned).
dsa::AttnLaunch attn_launch(const dsa_attn_args* at, const int32_t* idx, int32_t k, void* out, float* lse) {
  dsa::AttnLaunch L{};
  L.B = at->B; L.T = at->T; L.S = at->S; L.H = at->H; L.DQK = at->d_qk; L.DV = at->d_v; L.scale = at->scale;
  L.q = at->q; L.k = at->k; L.k_ld = at->k_ld; L.v = at->v; L.v_ld = at->v_ld;
  L.q_st = at->q_stride_t ? at->q_stride_t : (int64_t)at->H * at->d_qk;
  L.q_sb = at->q_stride_b ? at->q_stride_b : (int64_t)at->T * L.q_st;
  L.k_sb = at->k_stride_b ? at->k_stride_b : (int64_t)at->S * at->k_ld;
  L.v_sb = at->v_stride_b ? at->v_stride_b : (int64_t)at->S * at->v_ld;
  L.idx = idx; L.kk = k; L.out = out; L.lse = lse;
  L.idx_st = k; L.idx_sb = (int64_t)at->T * k;
  return L;
}

// Workspace bytes beyond DSA_WS_MIN for the parts of a split attention call (0: no split).
size_t attn_split_bytes(const dsa::AttnLaunch& L) {
  const int splits = dsa::attn_splits(L);
  if (splits <= 1) return 0;
  return (size_t)L.B * L.T * (L.layers > 1 ? L.layers : 1) * splits * (size_t)L.H * ((size_t)L.DV + 1) * 4;
}

// Bytes of the fixed-reference pass's row marks (one per flat row; 0 where the call splits rows
// or takes the other kernel).
size_t attn_mark_bytes(const dsa::AttnLaunch& L) {
  if (!dsa::sparse_mla_tc_supported(L) || dsa::attn_splits(L) > 1) return 0;
  const size_t rows = (size_t)L.B * L.T * (L.layers > 1 ? L.layers : 1);
  return (rows + 255) & ~(size_t)255;
}

// All the workspace an attention call uses beyond DSA_WS_MIN.
size_t attn_extra_bytes(const dsa::AttnLaunch& L) { return attn_split_bytes(L) + attn_mark_bytes(L); }

constexpr int kMaxK = 4096;

// Bytes of the segment lists when `rows` rows of up to n_max scores are split across CTAs
// (0: no split).
size_t topk_split_bytes(int64_t rows, int64_t n_max, int k) {
  const int parts = dsa::topk_parts(rows, n_max);
  if (parts <= 1) return 0;
  return (size_t)rows * parts * ((size_t)k * 8 + 4);
}

// Few long rows: split each across CTAs (dsa::topk_parts) when the workspace from byte `off` on
// holds the segments' lists; otherwise one CTA per row.
void plan_topk_parts(dsa::TopkLaunch& P, int64_t rows, int64_t n_max, void* ws, size_t off, size_t ws_bytes) {
  P.parts = 1;
  const int parts = dsa::topk_parts(rows, n_max);
  if (parts <= 1) return;
  const size_t per = (size_t)rows * parts;
  const size_t need = topk_split_bytes(rows, n_max, P.k);
  if (off > ws_bytes || ws_bytes - off < need) return;
  uint8_t* w = static_cast<uint8_t*>(ws) + off;
  P.parts = parts;
  P.part_pos = reinterpret_cast<int32_t*>(w);
  P.part_key = reinterpret_cast<uint32_t*>(w + per * P.k * 4);
  P.part_cnt = reinterpret_cast<int32_t*>(w + per * P.k * 8);
}

int64_t max_visible(int64_t q_pos0, int T, int diag, int S) {
  const int64_t n = q_pos0 + T - 1 + diag;
  return n < 0 ? 0 : (n > S ? S : n);
}

// Query rows per chunk of the materialised score buffer that `bytes` of scratch (after the
// 256-byte header) can hold.
int64_t score_chunk_rows(const dsa_indexer_args* ix, size_t ws_bytes) {
  if (ws_bytes <= dsa::kWsScratch) return 0;
  const int64_t per_row = (int64_t)ix->B * ix->S * 4;
  int64_t rows = (int64_t)(ws_bytes - dsa::kWsScratch) / per_row;
  return rows > ix->T ? ix->T : rows;
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    sms = 148;
  return sms;
}

// The selecting path (scores never stored): a pass of the indexer keeps, per query row, the keys
// whose score reaches a threshold set from a sample of the row (about `target` of them, at most
// `cap` stored), an exact top-k runs over those candidates, and only rows whose candidates could
// not hold their top-k are recomputed through the score buffer.  It needs 64 indexer heads,
// k <= kCandMaxK, and enough 4-token blocks in a chunk to fill the GPU from one CTA per block.
constexpr size_t kCandBytes = (size_t)1 << 30;  // candidate lists of one chunk of rows
int cand_cap(int k) {
  int c = 4 * k < 2048 ? 2048 : 4 * k;
  return (c + 127) / 128 * 128;
}
// the largest number of candidates a row's threshold aims at: half the room, so that a
// segment (a quarter of the room, a quarter of the keys) rarely overflows (at 60%, 5 of 4,096
// rows of a 1M-key chunk overflowed a segment, each then recomputed over its million keys)
int cand_target(int k) { return cand_cap(k) / 2; }
size_t cand_area(int64_t rows, int cap) {  // key + position lists, four counts, fail flags
  const size_t b = (size_t)rows * ((size_t)cap * 8 + 16 + 1);
  return (b + 255) & ~(size_t)255;
}
bool select_blocks_ok(int64_t B, int64_t Tc) { return B * ((Tc + 3) / 4) >= 4LL * device_sms(); }
// Query rows per chunk of the selecting path (0: the path does not apply).
// The rows are split into equal chunks, each a whole number of waves of 4-token blocks (one
// CTA per block on every SM) where that still fits the candidate room: a chunk's last wave
// then runs full (128K rows: nine chunks of 14,592 rows, 24 waves each, where chunks of the
// most rows that fit left a last chunk of 2,048 of the longest rows, 3.4 waves).
int64_t select_chunk_rows(const dsa_indexer_args* ix, int k) {
  if (ix->H_I != 64 || k < 1 || k > dsa::kCandMaxK) return 0;
  const int64_t most = (int64_t)(kCandBytes / ((size_t)ix->B * ((size_t)cand_cap(k) * 8 + 17)));
  int64_t rows = ix->T;
  if (most < ix->T) {
    const int64_t n = (ix->T + most - 1) / most;  // chunks
    const int64_t sms = device_sms();
    const int64_t unit = 4 * (sms / ix->B > 1 ? sms / ix->B : 1);  // rows of one wave of blocks
    rows = (ix->T + n - 1) / n;
    rows = (rows + unit - 1) / unit * unit;
    if (rows > most) rows = most / unit * unit > 0 ? most / unit * unit : most;
  }
  if (rows < 1 || !select_blocks_ok(ix->B, rows)) return 0;
  return rows;
}

dsa_status run_materialised(const dsa_indexer_args* ix, int32_t k, int32_t* idx, void* ws, float* sc, size_t sc_bytes,
                            size_t split_off, size_t ws_bytes, int64_t t_begin, int64_t t_end, const uint8_t* gate,
                            int64_t gate_bstride, cudaStream_t st) {
  const int64_t per_row = (int64_t)ix->B * ix->S * 4;
  int64_t chunk = (int64_t)(sc_bytes / per_row);
  if (chunk > t_end - t_begin) chunk = t_end - t_begin;
  if (chunk < 1) return fail(DSA_ERR_WORKSPACE, "workspace too small for one row of indexer scores");
  for (int64_t t0 = t_begin; t0 < t_end; t0 += chunk) {
    const int Tc = (int)((t_end - t0) < chunk ? (t_end - t0) : chunk);
    dsa::IndexerLaunch L = indexer_launch(ix, t0, Tc);
    L.out = sc; L.ld = ix->S; L.out_bstride = (int64_t)Tc * ix->S; L.write_masked = 0;
    L.flags = ws_flags(ws);
    // a recomputing pass runs only the few flagged token blocks: with long rows, split their
    // key ranges over at least 4,096 CTAs (the others leave at once) -- a flagged 1M-key row
    // took 1.6 ms on three CTAs, 0.33 this way
    if (gate) {
      L.gate = gate + (t0 - t_begin);
      L.gate_bstride = gate_bstride;
      if (ix->S >= (1 << 18)) L.ctas_min = 4096;
    }
    cudaError_t e = dsa::launch_indexer_scores(L, st);
    if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
    dsa::TopkLaunch P{};
    P.scores = sc; P.ld = ix->S; P.bstride = (int64_t)Tc * ix->S;
    P.B = ix->B; P.T = ix->T; P.S = ix->S; P.t0 = (int)t0; P.Tc = Tc;
    P.q_pos0 = ix->q_pos0; P.diag = ix->diag; P.k = k; P.idx = idx; P.flags = ws_flags(ws);
    if (gate) { P.gate = gate + (t0 - t_begin); P.gate_bstride = gate_bstride; }
    else plan_topk_parts(P, (int64_t)ix->B * Tc, max_visible(ix->q_pos0, ix->T, ix->diag, ix->S), ws, split_off, ws_bytes);
    e = dsa::launch_topk_rows(P, st);
    if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  }
  return DSA_OK;
}

dsa_status run_indexer_topk(const dsa_indexer_args* ix, int32_t k, int32_t* idx, void* ws, size_t ws_bytes,
                            cudaStream_t st) {
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  const int64_t per_row = (int64_t)ix->B * ix->S * 4;
  const int64_t fchunk = select_chunk_rows(ix, k);
  const int cap = cand_cap(k);
  const size_t farea = fchunk > 0 ? cand_area((int64_t)ix->B * fchunk, cap) : 0;
  if (fchunk > 0 && ws_bytes >= dsa::kWsScratch + farea + (size_t)per_row) {
    // candidate lists first, the score buffer of the recomputing pass after them
    uint8_t* a = w8 + dsa::kWsScratch;
    const int64_t rows_max = (int64_t)ix->B * fchunk;
    uint2* cand = reinterpret_cast<uint2*>(a);
    int32_t* ccnt = reinterpret_cast<int32_t*>(a + (size_t)rows_max * cap * 8);
    uint8_t* fl = a + (size_t)rows_max * (cap * 8 + 16);
    float* sc = reinterpret_cast<float*>(a + farea);
    const size_t sc_bytes = ws_bytes - dsa::kWsScratch - farea;
    for (int64_t t0 = 0; t0 < ix->T; t0 += fchunk) {
      const int Tc = (int)((ix->T - t0) < fchunk ? (ix->T - t0) : fchunk);
      if (!select_blocks_ok(ix->B, Tc)) {  // a short tail chunk: the scores of its few rows
        dsa_status s = run_materialised(ix, k, idx, ws, sc, sc_bytes, ws_bytes, ws_bytes, t0, t0 + Tc, nullptr, 0, st);
        if (s != DSA_OK) return s;
        continue;
      }
      dsa::IndexerLaunch L = indexer_launch(ix, t0, Tc);
      L.flags = ws_flags(ws);
      L.select = 1; L.cap = cap; L.target = cand_target(k); L.topk = k;
      L.cand = cand; L.cand_cnt = ccnt;
      cudaError_t e = dsa::launch_indexer_scores(L, st);
      if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
      dsa::CandLaunch C{};
      C.B = ix->B; C.T = ix->T; C.S = ix->S; C.t0 = (int)t0; C.Tc = Tc;
      C.q_pos0 = ix->q_pos0; C.diag = ix->diag; C.k = k; C.cap = cap;
      C.cand = cand; C.cand_cnt = ccnt; C.fail = fl; C.idx = idx;
      if ((e = dsa::launch_topk_cand(C, st)) != cudaSuccess) return cuda_fail(e, "top-k launch");
      // rows whose candidates could not hold their top-k: scores and top-k again, through
      // the score buffer (each launch leaves at once unless one of its rows is marked)
      dsa_status s = run_materialised(ix, k, idx, ws, sc, sc_bytes, ws_bytes, ws_bytes, t0, t0 + Tc, fl, Tc, st);
      if (s != DSA_OK) return s;
    }
    return DSA_OK;
  }
  const int64_t chunk = score_chunk_rows(ix, ws_bytes);
  if (chunk < 1) return fail(DSA_ERR_WORKSPACE, "workspace too small for one row of indexer scores (%zu bytes)", ws_bytes);
  float* sc = reinterpret_cast<float*>(w8 + dsa::kWsScratch);
  return run_materialised(ix, k, idx, ws, sc, (size_t)(chunk * per_row), dsa::kWsScratch + (size_t)(chunk * per_row),
                          ws_bytes, 0, ix->T, nullptr, 0, st);
}

}  // namespace

namespace dsa {
dsa_status validate_indexer(const dsa_indexer_args* ix) { return check_indexer(ix); }
dsa_status record_error(dsa_status s, const char* msg) { return fail(s, "%s", msg); }
IndexerLaunch make_indexer_launch(const dsa_indexer_args* ix, int64_t t0, int Tc) { return indexer_launch(ix, t0, Tc); }
void plan_topk_split(TopkLaunch& P, int64_t rows, int64_t n_max, void* ws, size_t off, size_t ws_bytes) {
  plan_topk_parts(P, rows, n_max, ws, off, ws_bytes);
}
int64_t max_visible_keys(int64_t q_pos0, int T, int diag, int S) { return max_visible(q_pos0, T, diag, S); }
}  // namespace dsa

extern "C" {

size_t dsa_workspace_size(const dsa_indexer_args* ix, int32_t k) {
  if (!ix || ix->B <= 0 || ix->T <= 0 || ix->S <= 0) return DSA_WS_MIN;
  // Preferred score chunk: up to 4 GiB of fp32 scores, at least one row.
  const int64_t per_row = (int64_t)ix->B * ix->S * 4;
  int64_t rows = ((int64_t)4 << 30) / per_row;
  if (rows < 1) rows = 1;
  if (rows > ix->T) rows = ix->T;
  size_t bytes = dsa::kWsScratch + (size_t)(rows * per_row);
  // the selecting path's candidate lists (rows of the chunk x (cap keys + cap positions + count
  // + fail flag)) come first when it applies
  const int64_t fchunk = select_chunk_rows(ix, k);
  if (fchunk > 0) bytes += cand_area((int64_t)ix->B * fchunk, cand_cap(k));
  // a chunk of few rows may have them split across CTAs: room for the segments' lists (the
  // first chunk's rows are the most; the same room serves every later chunk)
  if (k >= 1 && k <= kMaxK) bytes += topk_split_bytes(rows * ix->B, max_visible(ix->q_pos0, ix->T, ix->diag, ix->S), k);
  return bytes;
}

size_t dsa_topk_workspace_size(int32_t B, int32_t T, int32_t S, int64_t q_pos0, int32_t diag, int32_t k) {
  if (B <= 0 || T <= 0 || S <= 0 || q_pos0 < 0 || diag < 0 || diag > 1 || k < 1 || k > kMaxK) return DSA_WS_MIN;
  return dsa::kWsScratch + topk_split_bytes((int64_t)B * T, max_visible(q_pos0, T, diag, S), k);
}

size_t dsa_attn_workspace_size(const dsa_attn_args* at, int32_t k) {
  if (!at || at->B <= 0 || at->T <= 0 || at->S <= 0 || k < 1 || k > kMaxK) return DSA_WS_MIN;
  return dsa::kWsScratch + attn_extra_bytes(attn_launch(at, nullptr, k, nullptr, nullptr));
}

dsa_status dsa_indexer_scores(const dsa_indexer_args* ix, float* scores, int64_t ld, void* ws, size_t ws_bytes,
                              void* stream) {
  dsa_status s = check_indexer(ix);
  if (s != DSA_OK) return s;
  if (!scores) return fail(DSA_ERR_INVALID_ARG, "scores is NULL");
  if (ld < ix->S) return fail(DSA_ERR_INVALID_ARG, "ld (%lld) < S (%d)", (long long)ld, ix->S);
  if ((s = check_ws(ws, ws_bytes, DSA_WS_MIN)) != DSA_OK) return s;
  dsa::IndexerLaunch L = indexer_launch(ix, 0, ix->T);
  L.out = scores; L.ld = ld; L.out_bstride = (int64_t)ix->T * ld; L.write_masked = 1;
  L.flags = ws_flags(ws);
  cudaError_t e = dsa::launch_indexer_scores(L, as_stream(stream));
  return e == cudaSuccess ? DSA_OK : cuda_fail(e, "indexer launch");
}

dsa_status dsa_topk(const dsa_topk_src* src, int32_t B, int32_t T, int32_t S, int64_t q_pos0, int32_t diag,
                    int32_t k, int32_t* idx, void* ws, size_t ws_bytes, void* stream) {
  if (!src) return fail(DSA_ERR_INVALID_ARG, "top-k source is NULL");
  if (!idx) return fail(DSA_ERR_INVALID_ARG, "idx is NULL");
  if (B <= 0 || T <= 0 || S <= 0) return fail(DSA_ERR_INVALID_ARG, "B, T, S must be positive");
  if (k < 1 || k > kMaxK) return fail(DSA_ERR_UNSUPPORTED, "k=%d outside [1, %d]", k, kMaxK);
  if (diag < 0 || diag > 1) return fail(DSA_ERR_INVALID_ARG, "diag must be 0 or 1");
  if (q_pos0 < 0) return fail(DSA_ERR_INVALID_ARG, "q_pos0 must be >= 0");
  dsa_status s = check_ws(ws, ws_bytes, DSA_WS_MIN);
  if (s != DSA_OK) return s;
  cudaStream_t st = as_stream(stream);
  if (src->kind == DSA_TOPK_FROM_SCORES) {
    if (!src->scores) return fail(DSA_ERR_INVALID_ARG, "scores is NULL");
    if (src->ld < S) return fail(DSA_ERR_INVALID_ARG, "ld < S");
    dsa::TopkLaunch P{};
    P.scores = src->scores; P.ld = src->ld; P.bstride = (int64_t)T * src->ld;
    P.B = B; P.T = T; P.S = S; P.t0 = 0; P.Tc = T;
    P.q_pos0 = q_pos0; P.diag = diag; P.k = k; P.idx = idx; P.flags = ws_flags(ws);
    plan_topk_parts(P, (int64_t)B * T, max_visible(q_pos0, T, diag, S), ws, dsa::kWsScratch, ws_bytes);
    cudaError_t e = dsa::launch_topk_rows(P, st);
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "top-k launch");
  }
  if (src->kind != DSA_TOPK_FROM_INDEXER) return fail(DSA_ERR_INVALID_ARG, "unknown top-k source kind");
  if ((s = check_indexer(src->ix)) != DSA_OK) return s;
  const dsa_indexer_args* ix = src->ix;
  if (ix->B != B || ix->T != T || ix->S != S || ix->q_pos0 != q_pos0 || ix->diag != diag)
    return fail(DSA_ERR_INVALID_ARG, "B/T/S/q_pos0/diag disagree with the indexer args");
  return run_indexer_topk(ix, k, idx, ws, ws_bytes, st);
}

namespace {

// Checks shared by the attention entry points (the attention args themselves checked before).
dsa_status check_attn_call(const int32_t* idx, int32_t k, const void* out, void* ws, size_t ws_bytes) {
  if (!idx || !out) return fail(DSA_ERR_INVALID_ARG, "idx and out must be non-NULL");
  if (k < 1 || k > kMaxK) return fail(DSA_ERR_UNSUPPORTED, "k=%d outside [1, %d]", k, kMaxK);
  if (!aligned16(out)) return fail(DSA_ERR_MISALIGNED, "out must be 16-byte aligned");
  return check_ws(ws, ws_bytes, DSA_WS_MIN);
}

// Launch of a described attention call: with few rows each row's blocks are split over CTAs
// when the workspace holds the parts.
dsa_status run_attn(dsa::AttnLaunch L, void* ws, size_t ws_bytes, void* stream) {
  L.flags = ws_flags(ws);
  const int splits = dsa::attn_splits(L);
  if (splits > 1) {
    const size_t parts = (size_t)L.B * L.T * (L.layers > 1 ? L.layers : 1) * splits;
    const size_t need = attn_split_bytes(L);
    if (ws_bytes > dsa::kWsScratch && ws_bytes - dsa::kWsScratch >= need) {
      uint8_t* w = static_cast<uint8_t*>(ws) + dsa::kWsScratch;
      L.splits = splits;
      L.part_o = reinterpret_cast<float*>(w);
      L.part_lse = reinterpret_cast<float*>(w + parts * (size_t)L.H * L.DV * 4);
    }
  } else {
    // the fixed-reference softmax when the workspace holds its row marks (else the running one)
    const size_t marks = attn_mark_bytes(L);
    if (marks > 0 && ws_bytes > dsa::kWsScratch && ws_bytes - dsa::kWsScratch >= marks)
      L.redo = static_cast<uint8_t*>(ws) + dsa::kWsScratch;
  }
  cudaError_t e = dsa::launch_sparse_attn(L, as_stream(stream));
  return e == cudaSuccess ? DSA_OK : cuda_fail(e, "attention launch");
}

// The draft steps of a sequence read its one index row: T query positions, row stride 0.
dsa::AttnLaunch draft_launch(const dsa_attn_args* at, const int32_t* idx, int32_t k, void* out, float* lse) {
  dsa::AttnLaunch L = attn_launch(at, idx, k, out, lse);
  L.idx_st = 0;
  L.idx_sb = k;
  return L;
}

dsa_status check_draft(const dsa_indexer_args* ix, const dsa_attn_args* at) {
  dsa_status s = check_indexer(ix);
  if (s != DSA_OK) return s;
  if ((s = check_attn(at)) != DSA_OK) return s;
  if (ix->T != 1)
    return fail(DSA_ERR_INVALID_ARG, "the first draft step's indexer has T=%d queries per sequence (1 expected)", ix->T);
  if (ix->B != at->B || ix->S != at->S)
    return fail(DSA_ERR_INVALID_ARG, "indexer B/S (%d/%d) differ from the attention's (%d/%d)", ix->B, ix->S, at->B, at->S);
  return DSA_OK;
}

}  // namespace

dsa_status dsa_sparse_attn(const dsa_attn_args* at, const int32_t* idx, int32_t k, void* out, float* lse, void* ws,
                           size_t ws_bytes, void* stream) {
  dsa_status s = check_attn(at);
  if (s != DSA_OK) return s;
  if ((s = check_attn_call(idx, k, out, ws, ws_bytes)) != DSA_OK) return s;
  return run_attn(attn_launch(at, idx, k, out, lse), ws, ws_bytes, stream);
}

dsa_status indexshare_draft_forward(const dsa_indexer_args* ix, const dsa_attn_args* at, int32_t k, int32_t* idx,
                                    void* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s = check_draft(ix, at);
  if (s != DSA_OK) return s;
  if ((s = check_attn_call(idx, k, out, ws, ws_bytes)) != DSA_OK) return s;
  // the first step's indexer + top-k, then every step over that one index row
  if ((s = run_indexer_topk(ix, k, idx, ws, ws_bytes, as_stream(stream))) != DSA_OK) return s;
  return run_attn(draft_launch(at, idx, k, out, lse), ws, ws_bytes, stream);
}

size_t indexshare_draft_workspace_size(const dsa_indexer_args* ix, const dsa_attn_args* at, int32_t k) {
  if (!ix || !at || at->B <= 0 || at->T <= 0 || at->S <= 0 || k < 1 || k > kMaxK) return DSA_WS_MIN;
  const size_t a = dsa::kWsScratch + attn_extra_bytes(draft_launch(at, nullptr, k, nullptr, nullptr));
  const size_t t = dsa_workspace_size(ix, k);
  return a > t ? a : t;
}

namespace {

// Validation of one group call: every layer, the schedule and the buffers; nothing launches.
dsa_status group_check(const dsa_layer* layers, int32_t n_layers, const char* schedule, int32_t k,
                       int32_t* const* idx_bufs, void* ws, size_t ws_bytes) {
  if (!layers || n_layers <= 0) return fail(DSA_ERR_INVALID_ARG, "no layers");
  if (!schedule) return fail(DSA_ERR_SCHEDULE, "schedule is NULL");
  if ((int32_t)strlen(schedule) != n_layers)
    return fail(DSA_ERR_SCHEDULE, "schedule has %zu roles for %d layers", strlen(schedule), n_layers);
  if (schedule[0] != 'F') return fail(DSA_ERR_SCHEDULE, "the first layer must be full ('F')");
  int n_full = 0;
  for (int i = 0; i < n_layers; ++i) {
    if (schedule[i] != 'F' && schedule[i] != 'S') return fail(DSA_ERR_SCHEDULE, "role '%c' at layer %d is not F or S", schedule[i], i);
    n_full += schedule[i] == 'F';
  }
  if (!idx_bufs) return fail(DSA_ERR_INVALID_ARG, "idx_bufs is NULL");
  if (k < 1 || k > kMaxK) return fail(DSA_ERR_UNSUPPORTED, "k=%d outside [1, %d]", k, kMaxK);
  dsa_status s;
  const dsa_attn_args& a0 = layers[0].at;
  for (int i = 0; i < n_layers; ++i) {
    const dsa_layer& L = layers[i];
    if ((s = check_attn(&L.at)) != DSA_OK) return fail(s, "layer %d: %s", i, g_last_error.c_str());
    if (L.at.B != a0.B || L.at.T != a0.T || L.at.S != a0.S) return fail(DSA_ERR_INVALID_ARG, "layer %d: B/T/S differ from layer 0", i);
    if (!L.out || !aligned16(L.out)) return fail(DSA_ERR_INVALID_ARG, "layer %d: out is NULL or misaligned", i);
    if (schedule[i] == 'F') {
      if ((s = check_indexer(&L.ix)) != DSA_OK) return fail(s, "layer %d: %s", i, g_last_error.c_str());
      if (L.ix.B != a0.B || L.ix.T != a0.T || L.ix.S != a0.S)
        return fail(DSA_ERR_INVALID_ARG, "layer %d: indexer B/T/S differ from the attention's", i);
      if (score_chunk_rows(&L.ix, ws_bytes) < 1) return fail(DSA_ERR_WORKSPACE, "layer %d: workspace too small for the indexer", i);
    }
  }
  for (int f = 0; f < n_full; ++f)
    if (!idx_bufs[f]) return fail(DSA_ERR_INVALID_ARG, "idx_bufs[%d] is NULL", f);
  return check_ws(ws, ws_bytes, DSA_WS_MIN);
}

// Layers a .. end-1 of a run of layers that read one index buffer (a full layer and the shared
// layers after it), attended in one launch: consecutive layers of the tcgen05 shape with equal
// scale and strides, when a single layer has too few query rows to fill the GPU (decode: a
// layer's 32 rows would be split over CTAs and merged; four layers' 128 rows fill it without
// splitting), at most kMaxAttnLayers.  Layer a alone otherwise.
int attn_batch_end(const dsa_layer* ls, int a, int run_end, int32_t k) {
  const dsa::AttnLaunch A = attn_launch(&ls[a].at, nullptr, k, nullptr, nullptr);
  if (!dsa::sparse_mla_tc_supported(A) || dsa::attn_splits(A) <= 1) return a + 1;
  int c = a + 1;
  while (c < run_end && c - a < dsa::kMaxAttnLayers) {
    const dsa::AttnLaunch C = attn_launch(&ls[c].at, nullptr, k, nullptr, nullptr);
    if (!dsa::sparse_mla_tc_supported(C) || C.scale != A.scale || C.q_st != A.q_st || C.q_sb != A.q_sb ||
        C.k_sb != A.k_sb || C.v_sb != A.v_sb || C.k_ld != A.k_ld)
      break;
    ++c;
  }
  return c;
}

// The attention launch of layers a .. c-1 over idx.
dsa::AttnLaunch batch_launch(const dsa_layer* ls, int a, int c, const int32_t* idx, int32_t k) {
  dsa::AttnLaunch L = attn_launch(&ls[a].at, idx, k, ls[a].out, ls[a].lse);
  if (c - a > 1) {
    L.layers = c - a;
    for (int l = 0; l < L.layers; ++l) {
      L.lq[l] = ls[a + l].at.q;
      L.lk[l] = ls[a + l].at.k;
      L.lout[l] = ls[a + l].out;
      L.llse[l] = ls[a + l].lse;
    }
  }
  return L;
}

// The schedule walk of a checked group.
dsa_status group_run(const dsa_layer* layers, int32_t n_layers, const char* schedule, int32_t k,
                     int32_t* const* idx_bufs, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s;
  cudaStream_t st = as_stream(stream);
  const int32_t* cur = nullptr;
  int f = 0;
  for (int i = 0; i < n_layers;) {
    if (schedule[i] == 'F') {
      // Full layer: indexer + top-k, positions kept in this F layer's buffer.
      if ((s = run_indexer_topk(&layers[i].ix, k, idx_bufs[f], ws, ws_bytes, st)) != DSA_OK) return s;
      cur = idx_bufs[f++];
    }
    // Every layer (full or shared) up to the next full one attends with its own operands over
    // `cur`, several layers per launch where that fills the GPU better.
    int run_end = i + 1;
    while (run_end < n_layers && schedule[run_end] != 'F') ++run_end;
    for (int a = i; a < run_end;) {
      const int c = attn_batch_end(layers, a, run_end, k);
      if ((s = run_attn(batch_launch(layers, a, c, cur, k), ws, ws_bytes, stream)) != DSA_OK) return s;
      a = c;
    }
    i = run_end;
  }
  return DSA_OK;
}

// Sequence b of a packed group as a one-sequence group: every pointer advanced to its first
// query row / key row, T and S its own, its indexer queries at q_pos0[b].
void varlen_view(const dsa_layer* layers, int32_t n_layers, const char* schedule, int32_t k, const dsa_varlen* v,
                 int b, int32_t* const* idx_bufs, std::vector<dsa_layer>& out, std::vector<int32_t*>& bufs) {
  const int64_t q0 = v->cu_q[b], k0 = v->cu_k[b];
  const int32_t T = (int32_t)(v->cu_q[b + 1] - q0), S = (int32_t)(v->cu_k[b + 1] - k0);
  out.assign(layers, layers + n_layers);
  int f = 0;
  bufs.clear();
  for (int i = 0; i < n_layers; ++i) {
    dsa_layer& L = out[i];
    dsa_attn_args& a = L.at;
    const int64_t aq_st = a.q_stride_t ? a.q_stride_t : (int64_t)a.H * a.d_qk;
    a.q_stride_t = aq_st;  // the view's rows keep the packed tensor's row stride
    a.T = T;
    a.S = S;
    a.q = static_cast<const uint16_t*>(a.q) + q0 * aq_st;
    a.k = static_cast<const uint16_t*>(a.k) + k0 * a.k_ld;
    a.v = a.v ? static_cast<const uint16_t*>(a.v) + k0 * a.v_ld : a.v;
    L.out = static_cast<uint16_t*>(L.out) + q0 * a.H * a.d_v;
    if (L.lse) L.lse += q0 * a.H;
    if (schedule[i] == 'F') {
      dsa_indexer_args& x = L.ix;
      const int64_t elt = x.dtype == DSA_E4M3 ? 1 : 2;
      const int64_t xq_st = x.q_stride_t ? x.q_stride_t : (int64_t)x.H_I * x.d_I;
      x.q_stride_t = xq_st;
      x.T = T;
      x.S = S;
      x.q = static_cast<const uint8_t*>(x.q) + q0 * xq_st * elt;
      if (x.q_scale) x.q_scale += q0;
      x.w += q0 * x.H_I;
      x.k = static_cast<const uint8_t*>(x.k) + k0 * x.d_I * elt;
      if (x.k_scale) x.k_scale += k0;
      x.q_pos0 = v->q_pos0[b];
      bufs.push_back(idx_bufs ? idx_bufs[f] + q0 * k : nullptr);
      ++f;
    }
  }
}

dsa_status check_varlen(const dsa_layer* layers, const dsa_varlen* v) {
  if (!v || v->n_seqs < 1 || !v->cu_q || !v->cu_k || !v->q_pos0)
    return fail(DSA_ERR_INVALID_ARG, "seqs needs n_seqs >= 1 and the cu_q, cu_k and q_pos0 arrays");
  if (v->cu_q[0] != 0 || v->cu_k[0] != 0) return fail(DSA_ERR_INVALID_ARG, "cu_q[0] and cu_k[0] must be 0");
  for (int b = 0; b < v->n_seqs; ++b) {
    const int64_t T = v->cu_q[b + 1] - v->cu_q[b], S = v->cu_k[b + 1] - v->cu_k[b];
    if (T < 0 || S < 1 || T > INT32_MAX || S > INT32_MAX)
      return fail(DSA_ERR_INVALID_ARG, "sequence %d: %lld query rows and %lld keys", b, (long long)T, (long long)S);
  }
  if (layers && (layers[0].at.B != 1 || v->cu_q[v->n_seqs] != layers[0].at.T || v->cu_k[v->n_seqs] != layers[0].at.S))
    return fail(DSA_ERR_INVALID_ARG, "packed layers must describe B = 1, T = cu_q[n_seqs], S = cu_k[n_seqs]");
  return DSA_OK;
}

}  // namespace

dsa_status indexshare_group_forward(const dsa_layer* layers, int32_t n_layers, const char* schedule, int32_t k,
                                    int32_t* const* idx_bufs, void* ws, size_t ws_bytes, void* stream) {
  dsa_status s = group_check(layers, n_layers, schedule, k, idx_bufs, ws, ws_bytes);
  if (s != DSA_OK) return s;
  return group_run(layers, n_layers, schedule, k, idx_bufs, ws, ws_bytes, stream);
}

dsa_status indexshare_group_forward_varlen(const dsa_layer* layers, int32_t n_layers, const char* schedule,
                                           int32_t k, const dsa_varlen* seqs, int32_t* const* idx_bufs, void* ws,
                                           size_t ws_bytes, void* stream) {
  // the packed layers are only read through the per-sequence views, which are fully checked
  if (!layers || n_layers <= 0) return fail(DSA_ERR_INVALID_ARG, "no layers");
  if (!schedule || (int32_t)strlen(schedule) != n_layers)
    return fail(DSA_ERR_SCHEDULE, "schedule must have one role per layer");
  if (!idx_bufs) return fail(DSA_ERR_INVALID_ARG, "idx_bufs is NULL");
  dsa_status s = check_varlen(layers, seqs);
  if (s != DSA_OK) return s;
  std::vector<dsa_layer> view;
  std::vector<int32_t*> bufs;
  // every sequence is checked before the first one launches
  for (int b = 0; b < seqs->n_seqs; ++b) {
    if (seqs->cu_q[b + 1] == seqs->cu_q[b]) continue;
    varlen_view(layers, n_layers, schedule, k, seqs, b, idx_bufs, view, bufs);
    if ((s = group_check(view.data(), n_layers, schedule, k, bufs.data(), ws, ws_bytes)) != DSA_OK)
      return fail(s, "sequence %d: %s", b, g_last_error.c_str());
  }
  for (int b = 0; b < seqs->n_seqs; ++b) {
    if (seqs->cu_q[b + 1] == seqs->cu_q[b]) continue;
    varlen_view(layers, n_layers, schedule, k, seqs, b, idx_bufs, view, bufs);
    if ((s = group_run(view.data(), n_layers, schedule, k, bufs.data(), ws, ws_bytes, stream)) != DSA_OK) return s;
  }
  return DSA_OK;
}

size_t indexshare_group_workspace_size(const dsa_layer* layers, int32_t n_layers, const char* schedule, int32_t k,
                                       const dsa_varlen* seqs) {
  if (!layers || n_layers <= 0 || !schedule || (int32_t)strnlen(schedule, (size_t)n_layers + 1) != n_layers)
    return DSA_WS_MIN;
  size_t best = DSA_WS_MIN;
  auto one_group = [&](const dsa_layer* ls) {
    for (int i = 0; i < n_layers; ++i) {
      if (schedule[i] == 'F') best = std::max(best, dsa_workspace_size(&ls[i].ix, k));
      best = std::max(best, dsa_attn_workspace_size(&ls[i].at, k));
    }
    if (k < 1 || k > kMaxK) return;
    for (int i = 0; i < n_layers;) {  // the split parts of the launches group_run makes
      int run_end = i + 1;
      while (run_end < n_layers && schedule[run_end] != 'F') ++run_end;
      for (int a = i; a < run_end;) {
        const int c = attn_batch_end(ls, a, run_end, k);
        best = std::max(best, dsa::kWsScratch + attn_extra_bytes(batch_launch(ls, a, c, nullptr, k)));
        a = c;
      }
      i = run_end;
    }
  };
  if (!seqs) {
    one_group(layers);
    return best;
  }
  if (check_varlen(layers, seqs) != DSA_OK) return DSA_WS_MIN;
  std::vector<dsa_layer> view;
  std::vector<int32_t*> bufs;
  for (int b = 0; b < seqs->n_seqs; ++b) {
    if (seqs->cu_q[b + 1] == seqs->cu_q[b]) continue;
    varlen_view(layers, n_layers, schedule, k, seqs, b, nullptr, view, bufs);
    one_group(view.data());
  }
  return best;
}

void dsa_set_wait_limit(uint64_t cycles) {
  const long long c = cycles == 0 || cycles > (uint64_t)dsa::kDefaultWaitCycles ? dsa::kDefaultWaitCycles : (long long)cycles;
  dsa::g_wait_limit.store(c, std::memory_order_relaxed);
}

size_t dsa_workspace_size_varlen(const dsa_indexer_args* ix, const dsa_varlen* seqs, int32_t k) {
  if (!ix || check_varlen(nullptr, seqs) != DSA_OK) return DSA_WS_MIN;
  size_t best = DSA_WS_MIN;
  for (int b = 0; b < seqs->n_seqs; ++b) {
    dsa_indexer_args x = *ix;
    x.B = 1;
    x.T = (int32_t)(seqs->cu_q[b + 1] - seqs->cu_q[b]);
    x.S = (int32_t)(seqs->cu_k[b + 1] - seqs->cu_k[b]);
    if (x.T < 1) continue;
    best = std::max(best, dsa_workspace_size(&x, k));
  }
  return best;
}

dsa_status topk_overlap(const int32_t* a, const int32_t* b, int32_t rows, int32_t k, float* per_row,
                        double* mean_out, void* ws, size_t ws_bytes, void* stream) {
  if (!a || !b || !mean_out) return fail(DSA_ERR_INVALID_ARG, "a, b and mean_out must be non-NULL");
  if (rows < 0 || k < 1) return fail(DSA_ERR_INVALID_ARG, "rows must be >= 0 and k >= 1");
  const size_t need = per_row ? DSA_WS_MIN : dsa::kWsScratch + (size_t)rows * 4;
  dsa_status s = check_ws(ws, ws_bytes, need);
  if (s != DSA_OK) return s;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  float* pr = per_row ? per_row : reinterpret_cast<float*>(w8 + dsa::kWsScratch);
  double* mean_dev = reinterpret_cast<double*>(w8 + dsa::kWsMean);
  cudaStream_t st = as_stream(stream);
  cudaError_t e = dsa::launch_topk_overlap(a, b, rows, k, pr, mean_dev, ws_flags(ws), st);
  if (e != cudaSuccess) return cuda_fail(e, "overlap launch");
  if ((e = cudaMemcpyAsync(mean_out, mean_dev, sizeof(double), cudaMemcpyDeviceToHost, st)) != cudaSuccess)
    return cuda_fail(e, "overlap mean copy");
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "overlap sync");
  return DSA_OK;
}

dsa_status topk_overlap_matrix(const int32_t* const* bufs, int32_t n, int32_t rows, int32_t k,
                               int32_t* counts, double* matrix_out, void* ws, size_t ws_bytes, void* stream) {
  if (!bufs || !matrix_out) return fail(DSA_ERR_INVALID_ARG, "bufs and matrix_out must be non-NULL");
  if (n < 1 || n > dsa::kMaxOverlapLayers)
    return fail(DSA_ERR_INVALID_ARG, "n = %d buffers; 1 <= n <= %d", n, dsa::kMaxOverlapLayers);
  if (rows < 0 || k < 1) return fail(DSA_ERR_INVALID_ARG, "rows must be >= 0 and k >= 1");
  for (int i = 0; i < n; ++i)
    if (!bufs[i]) return fail(DSA_ERR_INVALID_ARG, "bufs[%d] is NULL", i);
  if (dsa::overlap_matrix_smem(n, k) > DSA_OVERLAP_MATRIX_MAX_SMEM)
    return fail(DSA_ERR_UNSUPPORTED, "n = %d rows of k = %d do not fit in one CTA's shared memory", n, k);
  dsa_status s = check_ws(ws, ws_bytes, topk_overlap_matrix_workspace_size(n));
  if (s != DSA_OK) return s;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  double* matrix_dev = reinterpret_cast<double*>(w8 + dsa::kWsScratch);
  dsa::OverlapMatrixLaunch P{};
  for (int i = 0; i < n; ++i) P.bufs[i] = bufs[i];
  P.n = n;
  P.k = k;
  P.rows = rows;
  P.counts = counts;
  P.part = matrix_dev + dsa::kMaxOverlapLayers * dsa::kMaxOverlapLayers;
  P.flags = ws_flags(ws);
  cudaStream_t st = as_stream(stream);
  cudaError_t e = dsa::launch_overlap_matrix(P, matrix_dev, st);
  if (e != cudaSuccess) return cuda_fail(e, "overlap matrix launch");
  if ((e = cudaMemcpyAsync(matrix_out, matrix_dev, sizeof(double) * n * n, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
    return cuda_fail(e, "overlap matrix copy");
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "overlap matrix sync");
  return DSA_OK;
}

dsa_status dsa_quantize_e4m3_append(const void* x, int32_t B, int32_t n, int32_t width, int64_t x_stride_b,
                                    uint8_t* codes, float* scales, int32_t S_cap, int64_t pos0,
                                    const int64_t* positions, void* ws, size_t ws_bytes, void* stream) {
  if (!x || !codes || !scales) return fail(DSA_ERR_INVALID_ARG, "x, codes and scales must be non-NULL");
  if (B < 1 || n < 0 || S_cap < 1) return fail(DSA_ERR_INVALID_ARG, "B >= 1, n >= 0 and S_cap >= 1 are required");
  if (width < 4 || width > 65536 || width % 4)
    return fail(DSA_ERR_UNSUPPORTED, "width = %d; a multiple of 4 in [4, 65536] is required", width);
  if (x_stride_b < (int64_t)n * width)
    return fail(DSA_ERR_INVALID_ARG, "x_stride_b = %lld is smaller than n * width", (long long)x_stride_b);
  if ((reinterpret_cast<uintptr_t>(x) & 7u) || (x_stride_b & 3) || (reinterpret_cast<uintptr_t>(codes) & 3u) ||
      (reinterpret_cast<uintptr_t>(scales) & 3u))
    return fail(DSA_ERR_MISALIGNED, "x needs 8-byte alignment (and x_stride_b a multiple of 4), codes and "
                                    "scales 4-byte alignment");
  if (!positions && (pos0 < 0 || pos0 > (int64_t)S_cap - n))
    return fail(DSA_ERR_INVALID_ARG, "rows [%lld, %lld) fall outside the cache of %d rows", (long long)pos0,
                (long long)pos0 + n, S_cap);
  dsa_status s = check_ws(ws, ws_bytes, DSA_WS_MIN);
  if (s != DSA_OK) return s;
  dsa::QuantLaunch P{};
  P.x = static_cast<const uint16_t*>(x);
  P.B = B;
  P.n = n;
  P.width = width;
  P.x_stride_b = x_stride_b;
  P.codes = codes;
  P.scales = scales;
  P.S_cap = S_cap;
  P.pos0 = pos0;
  P.positions = positions;
  P.flags = ws_flags(ws);
  cudaError_t e = dsa::launch_quant_e4m3_rows(P, as_stream(stream));
  return e == cudaSuccess ? DSA_OK : cuda_fail(e, "quantisation launch");
}

size_t topk_overlap_matrix_workspace_size(int32_t n) {
  const size_t nn = n > 0 ? (size_t)n * (size_t)n : 0;
  return dsa::kWsScratch + sizeof(double) * (dsa::kMaxOverlapLayers * dsa::kMaxOverlapLayers + dsa::kMaxOverlapCtas * nn);
}

// --- F/S schedules scored by a measured overlap matrix (host only) ---------------------

namespace {

bool valid_schedule(const char* sched, int n) {
  if (!sched || (int)strnlen(sched, (size_t)n + 1) != n || sched[0] != 'F') return false;
  for (int i = 0; i < n; ++i)
    if (sched[i] != 'F' && sched[i] != 'S') return false;
  return true;
}

}  // namespace

dsa_status indexshare_schedule_score(const double* overlap, int32_t n, const char* schedule, double* score_out) {
  if (!overlap || !score_out) return fail(DSA_ERR_INVALID_ARG, "overlap and score_out must be non-NULL");
  if (n < 1) return fail(DSA_ERR_INVALID_ARG, "n must be >= 1");
  if (!valid_schedule(schedule, n))
    return fail(DSA_ERR_SCHEDULE, "schedule must be %d characters of 'F'/'S' starting with 'F'", n);
  double sum = 0.0;
  int f = 0;
  for (int l = 0; l < n; ++l) {
    if (schedule[l] == 'F') f = l;
    sum += overlap[(size_t)l * n + f];
  }
  *score_out = sum / n;
  return DSA_OK;
}

dsa_status indexshare_schedule_search(const double* overlap, int32_t n, int32_t n_full, char* schedule_out,
                                      double* score_out) {
  if (!overlap || !schedule_out || !score_out) return fail(DSA_ERR_INVALID_ARG, "pointers must be non-NULL");
  if (n < 1 || n > DSA_SCHEDULE_MAX_LAYERS)
    return fail(DSA_ERR_INVALID_ARG, "n = %d layers; 1 <= n <= %d", n, DSA_SCHEDULE_MAX_LAYERS);
  if (n_full < 1 || n_full > n) return fail(DSA_ERR_INVALID_ARG, "n_full = %d; 1 <= n_full <= n = %d", n_full, n);
  // seg(a, b): layers a .. b-1 served by an F layer at a = sum of overlap[l][a]
  // best[m][b]: the largest sum over layers 0 .. b-1 split into m such runs, the first at 0
  const int N = n + 1;
  std::vector<double> best((size_t)(n_full + 1) * N, -1.0), seg((size_t)n * N, 0.0);
  std::vector<int> from((size_t)(n_full + 1) * N, -1);
  for (int a = 0; a < n; ++a)
    for (int b = a + 1; b <= n; ++b) seg[(size_t)a * N + b] = seg[(size_t)a * N + b - 1] + overlap[(size_t)(b - 1) * n + a];
  for (int b = 1; b <= n; ++b) best[(size_t)1 * N + b] = seg[b];
  for (int m = 2; m <= n_full; ++m)
    for (int b = m; b <= n; ++b)
      for (int a = m - 1; a < b; ++a) {  // the m-th run starts at layer a; earlier a wins ties
        const double v = best[(size_t)(m - 1) * N + a] + seg[(size_t)a * N + b];
        if (from[(size_t)m * N + b] < 0 || v > best[(size_t)m * N + b]) {
          best[(size_t)m * N + b] = v;
          from[(size_t)m * N + b] = a;
        }
      }
  for (int l = 0; l < n; ++l) schedule_out[l] = 'S';
  schedule_out[n] = '\0';
  for (int m = n_full, b = n; m >= 1; --m) {
    const int a = m == 1 ? 0 : from[(size_t)m * N + b];
    schedule_out[a] = 'F';
    b = a;
  }
  *score_out = best[(size_t)n_full * N + n] / n;
  return DSA_OK;
}

dsa_status dsa_read_device_flags(void* ws, uint32_t* flags_out, void* stream) {
  if (!ws || !flags_out) return fail(DSA_ERR_INVALID_ARG, "ws and flags_out must be non-NULL");
  cudaStream_t st = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(flags_out, ws_flags(ws), sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws_flags(ws), 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? DSA_OK : cuda_fail(e, "reading device flags");
}

const char* dsa_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_MISALIGNED: return "DSA_ERR_MISALIGNED";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_SCHEDULE: return "DSA_ERR_SCHEDULE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_FLAG: return "DSA_ERR_DEVICE_FLAG";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
  }
  return "DSA_ERR_UNKNOWN";
}

const char* dsa_last_error(void) { return g_last_error.c_str(); }

uint64_t dsa_launch_count(void) { return dsa::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
