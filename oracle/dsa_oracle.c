/*
 * dsa_oracle.c -- plain, slow, fp64 CPU oracle for the DeepSeek Sparse Attention
 * hot path with IndexShare reuse.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark call this file.  It shares no code, header, table or helper with the
 * CUDA library; nothing in the product path may call it.
 *
 * What it computes (sources are the IndexShare explainer, "Why The Indexer Becomes
 * Expensive" and "How IndexShare Works", and the GLM-5.2 IndexShare article, "Where the
 * DSA indexer becomes expensive" / "What IndexShare reuses"):
 *   1. a lightweight indexer scores every preceding key of a query,
 *        I[t,s] = sum_h w[t,h] * max(0, q_I[t,h] . k_I[s])
 *      (the score formula itself is fixed by the project statement; the pages only
 *      say that the indexer scores the preceding tokens);
 *   2. the top-k positions of each query row are kept (ties: lower position wins);
 *   3. main attention runs over the selected rows only.
 * Everything is evaluated in double precision, one loop per term of the definition,
 * with no blocking, fusion or reordering.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_E4M3 = 1 };

/* Threads the OpenMP loops below use (reported beside CPU timings). */
int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* bfloat16 -> double.  A bfloat16 value is the upper 16 bits of an IEEE-754 binary32. */
double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits.  Exponent field 0 encodes subnormals m/8 * 2^-6; the pattern
 * S.1111.111 is NaN; there are no infinities, so the largest finite magnitude is
 * 1.75 * 2^8 = 448. */
double orc_e4m3_to_double(uint8_t b) {
  int sign = b >> 7;
  int e = (b >> 3) & 0xF;
  int m = b & 0x7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* The E4M3 code of the representable value nearest to v, ties to the even mantissa,
 * magnitudes beyond the largest finite value (448) saturated to it; NaN gives the NaN code.
 * Representable magnitudes are m * 2^(e-3) for m in [8, 16) and exponent e in [-6, 8], and
 * m * 2^-9 for m in [0, 8) (subnormals). */
uint8_t orc_encode_e4m3(float v) {
  if (v != v) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0;
  const double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  int e;
  frexp(a, &e); /* a in [2^(e-1), 2^e) */
  int ex = e - 1;
  if (ex < -6) ex = -6;
  const double quantum = ldexp(1.0, ex - 3);
  const double r = nearbyint(a / quantum) * quantum; /* default rounding: ties to even */
  if (r == 0.0) return sign;
  if (r < ldexp(1.0, -6)) return sign | (uint8_t)(r / ldexp(1.0, -9));
  int e2;
  frexp(r, &e2);
  const int E = e2 - 1; /* r in [2^E, 2^(E+1)) */
  const int mant = (int)((r / ldexp(1.0, E) - 1.0) * 8.0);
  return sign | (uint8_t)(((E + 7) << 3) | mant);
}

void orc_encode_e4m3_array(const float* src, uint8_t* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = orc_encode_e4m3(src[i]);
}

/* Per-row FP8 quantisation as the FP8 indexer consumes it (one scale per token row):
 * scale = amax / 448 (1 for an all-zero row), code = e4m3(x / scale); the scale and the
 * quotient are fp32 roundings (C float arithmetic). */
void orc_quantize_e4m3_rows(const uint16_t* x, int64_t rows, int width, uint8_t* codes, float* scales) {
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * (int64_t)width;
    float amax = 0.0f;
    for (int j = 0; j < width; ++j) {
      const float v = (float)orc_bf16_to_double(xr[j]);
      if (fabsf(v) > amax) amax = fabsf(v);
    }
    const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int j = 0; j < width; ++j) {
      const float v = (float)orc_bf16_to_double(xr[j]);
      const float y = v / scale;
      codes[r * (int64_t)width + j] = orc_encode_e4m3(y);
    }
    scales[r] = scale;
  }
}

void orc_decode_bf16(const uint16_t* src, double* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = orc_bf16_to_double(src[i]);
}

void orc_decode_e4m3(const uint8_t* src, double* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = orc_e4m3_to_double(src[i]);
}

static double load_elem(int dtype, const void* base, int64_t i) {
  if (dtype == ORC_BF16) return orc_bf16_to_double(((const uint16_t*)base)[i]);
  return orc_e4m3_to_double(((const uint8_t*)base)[i]);
}

/* Number of keys visible to a query at absolute position q_pos: the keys strictly
 * before it ("the preceding tokens"), s < q_pos + diag, clipped to [0, S].  diag = 0 is
 * the strictly-preceding reading; diag = 1 also lets a query see its own key. */
int64_t orc_visible(int64_t S, int64_t q_pos, int64_t diag) {
  int64_t n = q_pos + diag;
  if (n < 0) n = 0;
  if (n > S) n = S;
  return n;
}

/* Indexer scores of a set of query rows.
 *   q_rows   [n_rows,HI,DI]  bf16 or e4m3 codes of the rows' query vectors
 *   q_scale  [n_rows]        fp32 per-token dequantisation scale (NULL: 1)
 *   w_rows   [n_rows,HI]     fp32 head weights
 *   row_b    [n_rows]        batch of each row; row_pos [n_rows] its absolute position
 *   k        [B,S,DI]        bf16 or e4m3 codes of the indexer keys
 *   k_scale  [B,S]           fp32 (NULL: 1)
 *   out      [n_rows,S]      doubles; -inf where s is not visible
 * The dequantised operand is scale * decode(code); the score is the plain definition. */
void orc_indexer_scores(int dtype, int64_t S, int HI, int DI, int64_t n_rows, const void* q_rows,
                        const float* q_scale, const float* w_rows, const int64_t* row_b,
                        const int64_t* row_pos, const void* k, const float* k_scale,
                        int64_t diag, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t b = row_b[r];
    int64_t n = orc_visible(S, row_pos[r], diag);
    double* qd = (double*)malloc(sizeof(double) * (size_t)HI * DI);
    double* kd = (double*)malloc(sizeof(double) * (size_t)DI);
    double sq = q_scale ? (double)q_scale[r] : 1.0;
    for (int h = 0; h < HI; ++h)
      for (int d = 0; d < DI; ++d)
        qd[h * DI + d] = sq * load_elem(dtype, q_rows, (r * HI + h) * (int64_t)DI + d);
    for (int64_t s = 0; s < S; ++s) {
      if (s >= n) {
        out[r * S + s] = -INFINITY;
        continue;
      }
      double sk = k_scale ? (double)k_scale[b * S + s] : 1.0;
      for (int d = 0; d < DI; ++d) kd[d] = sk * load_elem(dtype, k, (b * S + s) * (int64_t)DI + d);
      double acc = 0.0;
      for (int h = 0; h < HI; ++h) {
        double dot = 0.0;
        for (int d = 0; d < DI; ++d) dot += qd[h * DI + d] * kd[d];
        double relu = dot > 0.0 ? dot : 0.0;
        acc += (double)w_rows[r * HI + h] * relu;
      }
      out[r * S + s] = acc;
    }
    free(qd);
    free(kd);
  }
}

typedef struct {
  double v;
  int64_t s;
} orc_pair;

/* Total order of the selection: larger score first; equal scores -> lower position
 * first.  -0.0 equals +0.0 under double comparison.  NaN ranks below every number. */
static int cmp_rank(const void* pa, const void* pb) {
  const orc_pair* a = (const orc_pair*)pa;
  const orc_pair* b = (const orc_pair*)pb;
  int an = isnan(a->v), bn = isnan(b->v);
  if (an != bn) return an ? 1 : -1;
  if (!an) {
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
  }
  return (a->s < b->s) ? -1 : (a->s > b->s);
}

static int cmp_i32(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a < b) ? -1 : (a > b);
}

/* Top-k of each row by the plain definition: sort all visible (score, position) pairs
 * by the order above, keep the first min(k, n), list those positions in ascending order,
 * and pad the row with -1 up to length k.
 *   scores  [n_rows, ld] doubles, only the first n_valid[r] entries of a row are read
 *   idx     [n_rows, k]  int32 output */
void orc_topk_rows(int64_t n_rows, const double* scores, int64_t ld, const int64_t* n_valid,
                   int k, int32_t* idx) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t n = n_valid[r];
    orc_pair* p = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)(n > 0 ? n : 1));
    for (int64_t s = 0; s < n; ++s) {
      p[s].v = scores[r * ld + s];
      p[s].s = s;
    }
    qsort(p, (size_t)n, sizeof(orc_pair), cmp_rank);
    int64_t m = n < k ? n : k;
    int32_t* out = idx + r * (int64_t)k;
    for (int64_t j = 0; j < m; ++j) out[j] = (int32_t)p[j].s;
    qsort(out, (size_t)m, sizeof(int32_t), cmp_i32);
    for (int64_t j = m; j < k; ++j) out[j] = -1;
    free(p);
  }
}

/* Sparse attention of a set of query rows over their own index rows (multi-query
 * form: every head h of a query reads the same gathered key/value rows).
 *   q_rows [n_rows,H,DQK] bf16;  row_b [n_rows] batch of each row
 *   k      [B,S,*] bf16, key row j of batch b starts at (b*S + j)*k_ld
 *   v      [B,S,*] bf16, row stride v_ld; may be the same buffer as k (latent KV)
 *   idx    [n_rows,kk] positions; -1 entries are skipped
 *   out    [n_rows,H,DV], lse [n_rows,H] (natural log)
 * For each head: z_j = scale * q . K[idx_j]; m = max z; p_j = exp(z_j - m);
 * O = sum p_j V[idx_j] / sum p_j; LSE = m + log(sum p_j).  No valid entry: O = 0,
 * LSE = -inf.  Returns the number of index entries outside [-1, S) (they are skipped). */
int64_t orc_sparse_attn(int64_t S, int H, int DQK, int DV, double scale, int64_t n_rows,
                        const uint16_t* q_rows, const int64_t* row_b, const uint16_t* k,
                        int64_t k_ld, const uint16_t* v, int64_t v_ld, const int32_t* idx, int kk,
                        double* out, double* lse) {
  int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t b = row_b[r];
    const int32_t* ir = idx + r * (int64_t)kk;
    double* z = (double*)malloc(sizeof(double) * (size_t)(kk > 0 ? kk : 1));
    for (int j = 0; j < kk; ++j)
      if (ir[j] < -1 || ir[j] >= S) ++bad;
    for (int h = 0; h < H; ++h) {
      const uint16_t* qh = q_rows + (r * H + h) * (int64_t)DQK;
      double m = -INFINITY;
      int any = 0;
      for (int j = 0; j < kk; ++j) {
        if (ir[j] < 0 || ir[j] >= S) continue;
        const uint16_t* kr = k + (b * S + ir[j]) * k_ld;
        double dot = 0.0;
        for (int d = 0; d < DQK; ++d) dot += orc_bf16_to_double(qh[d]) * orc_bf16_to_double(kr[d]);
        z[j] = scale * dot;
        if (!any || z[j] > m) m = z[j];
        any = 1;
      }
      double* o = out + (r * H + h) * (int64_t)DV;
      for (int d = 0; d < DV; ++d) o[d] = 0.0;
      if (!any) {
        lse[r * H + h] = -INFINITY;
        continue;
      }
      double l = 0.0;
      for (int j = 0; j < kk; ++j) {
        if (ir[j] < 0 || ir[j] >= S) continue;
        double p = exp(z[j] - m);
        l += p;
        const uint16_t* vr = v + (b * S + ir[j]) * v_ld;
        for (int d = 0; d < DV; ++d) o[d] += p * orc_bf16_to_double(vr[d]);
      }
      for (int d = 0; d < DV; ++d) o[d] /= l;
      lse[r * H + h] = m + log(l);
    }
    free(z);
  }
  return bad;
}

/* Overlap of two index rows: |A and B| / |A| over their valid (>= 0) entries, computed
 * as a set intersection (sort both, then walk them together).  A row whose A side is
 * empty counts as 1.  Returns the mean over rows. */
double orc_topk_overlap(const int32_t* a, const int32_t* b, int64_t rows, int k, double* per_row) {
  double sum = 0.0;
#pragma omp parallel for schedule(static) reduction(+ : sum)
  for (int64_t r = 0; r < rows; ++r) {
    int32_t* x = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    int32_t* y = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    int nx = 0, ny = 0;
    for (int j = 0; j < k; ++j) {
      if (a[r * (int64_t)k + j] >= 0) x[nx++] = a[r * (int64_t)k + j];
      if (b[r * (int64_t)k + j] >= 0) y[ny++] = b[r * (int64_t)k + j];
    }
    qsort(x, (size_t)nx, sizeof(int32_t), cmp_i32);
    qsort(y, (size_t)ny, sizeof(int32_t), cmp_i32);
    int i = 0, j = 0, common = 0;
    while (i < nx && j < ny) {
      if (x[i] == y[j]) {
        ++common;
        ++i;
        ++j;
      } else if (x[i] < y[j]) {
        ++i;
      } else {
        ++j;
      }
    }
    double f = nx == 0 ? 1.0 : (double)common / (double)nx;
    if (per_row) per_row[r] = f;
    sum += f;
    free(x);
    free(y);
  }
  return rows > 0 ? sum / (double)rows : 1.0;
}
