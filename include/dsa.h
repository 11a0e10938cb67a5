/*
 * dsa.h -- C ABI of libdsa: DeepSeek Sparse Attention with IndexShare reuse on one GPU.
 *
 * The library computes the three stages of a DSA layer and the IndexShare schedule that
 * ties layers together:
 *   - the lightning indexer scores every preceding key of a query
 *     (IndexShare explainer, "Why The Indexer Becomes Expensive"; the score formula
 *      I[t,s] = sum_h w[t,h] * ReLU(q_I[t,h] . k_I[s]) is the project's statement of it);
 *   - a per-query top-k keeps the k best positions, ties going to the lower position
 *     (same section; k = 2048 in the GLM-5.2 article, "Where the DSA indexer becomes
 *      expensive");
 *   - main attention runs over the selected rows only (same sections);
 *   - a full (F) layer runs indexer + top-k and keeps the positions; a shared (S) layer
 *     reuses the most recent F layer's positions with its own Q/KV and outputs
 *     (explainer, "How IndexShare Works"; article, "What IndexShare reuses"; IndexCache
 *      notes, section 2: the first layer is always F);
 *   - the overlap of two layers' selections (explainer, "Why Reusing Indices Can Work").
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller, unless a parameter says
 *     "host".  The library allocates no device memory; scratch space is the caller's
 *     workspace `ws` of `ws_bytes` bytes (see dsa_workspace_size).  The workspace must be
 *     zero-filled once before first use (its first bytes hold the device flag word).
 *   - `stream` is a cudaStream_t (NULL: the legacy default stream).  Every call only
 *     enqueues work on it, except topk_overlap (returns a host mean) and
 *     dsa_read_device_flags, which synchronise that stream.
 *   - Arguments are validated on the host before anything is launched; a rejected call
 *     launches nothing and returns a status other than DSA_OK.  dsa_last_error() gives
 *     a message for the last failure of the calling thread.
 *   - Faults found in the data on the device (an index outside [-1, S), a NaN score)
 *     never trap: the element is skipped (attention) or ranked lowest (top-k), and a bit
 *     is OR-ed into the device flag word, read by dsa_read_device_flags.
 *   - Tensors are row-major in the shapes given ("[B,T,H,d]": the last index varies
 *     fastest) and dense, except where a struct gives strides for its operands.  Query row i of every sequence sits at absolute position
 *     q_pos0 + i and sees the keys s < q_pos0 + i + diag (clipped to [0, S)).  diag = 0 is
 *     the strictly-preceding rule of the pages; diag = 1 also admits the query's own key.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, inconsistent shapes      */
  DSA_ERR_UNSUPPORTED = 2,  /* a shape the kernels are not built for                     */
  DSA_ERR_MISALIGNED = 3,   /* a pointer or row stride breaks the 16-byte rule            */
  DSA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than needed                  */
  DSA_ERR_SCHEDULE = 5,     /* schedule not 'F'/'S' per layer, or not starting with 'F'  */
  DSA_ERR_CUDA = 6,         /* a CUDA runtime call or kernel launch failed               */
  DSA_ERR_DEVICE_FLAG = 7,  /* reserved: returned by callers that treat flags as errors  */
  DSA_ERR_TIMEOUT = 8       /* a bounded device wait gave up                             */
} dsa_status;

typedef enum { DSA_BF16 = 0, DSA_E4M3 = 1 } dsa_dtype;

/* Bits of the device flag word. */
#define DSA_FLAG_BAD_INDEX 0x1u /* attention met an index outside [-1, S): entry skipped  */
#define DSA_FLAG_NAN_SCORE 0x2u /* top-k met a NaN score: ranked below every number       */
#define DSA_FLAG_UNSORTED 0x4u  /* topk_overlap met a row that is not ascending           */
#define DSA_FLAG_TIMEOUT 0x8u   /* a bounded device wait gave up                          */

/* Indexer operands of one layer (lightning indexer, "Why The Indexer Becomes Expensive").
 *   q       [B,T,H_I,d_I]  bf16 or e4m3 codes                      (16-byte aligned)
 *           token (b, t) starts at q + b*q_stride_b + t*q_stride_t (elements); its H_I*d_I
 *           codes are contiguous, heads of d_I codes each
 *   q_scale [B,T]  fp32 per-token dequantisation scale; required for E4M3, NULL for BF16
 *   w       [B,T,H_I] fp32 head weights (any sign), dense
 *   k       [B,S,d_I]  same dtype as q                              (16-byte aligned)
 *           key (b, s) starts at k + b*k_stride_b + s*d_I (elements)
 *   k_scale [B,S]  fp32, dense; required for E4M3, NULL for BF16
 * A dequantised operand is scale * code.  Supported: (H_I, d_I) in {(4,64), (64,128)}
 * for BF16 and {(64,128)} for E4M3.
 * Strides are in elements; 0 selects the dense value (q_stride_t = H_I*d_I, q_stride_b =
 * T*q_stride_t, k_stride_b = S*d_I).  Non-zero strides must be multiples of 16 bytes
 * (the operands are read by TMA) and q_stride_t >= H_I*d_I, else DSA_ERR_MISALIGNED /
 * DSA_ERR_INVALID_ARG.  A row chunk of a larger batch is a strided view: pass the chunk's
 * first token as q and the full tensor's strides. */
typedef struct {
  int32_t B, T, S, H_I, d_I;
  dsa_dtype dtype;
  const void* q;
  const float* q_scale;
  const float* w;
  const void* k;
  const float* k_scale;
  int64_t q_pos0;
  int32_t diag;
  int64_t q_stride_b, q_stride_t;
  int64_t k_stride_b;
} dsa_indexer_args;

/* Main-attention operands of one layer, multi-query form: every query head attends over
 * the same gathered key/value rows (MLA run over its shared latent KV).
 *   q  [B,T,H,d_qk] bf16                                          (16-byte aligned)
 *      query (b, t) starts at q + b*q_stride_b + t*q_stride_t; its H*d_qk values contiguous
 *   k  [B,S,k_ld] bf16; key row j of sequence b at b*k_stride_b + j*k_ld, first d_qk used
 *   v  [B,S,v_ld] bf16; row j of sequence b at b*v_stride_b + j*v_ld, first d_v used.  v may
 *      equal k (latent KV: the value is the first d_v columns of the latent row, so each
 *      gathered row serves both).
 * out = softmax(scale * q K[idx]^T) V[idx] per head.  Supported (H, d_qk, d_v):
 * (8 or 16, 64, 64) and (64, 576, 512); k_ld and v_ld multiples of 8.
 * Strides are in elements; 0 selects the dense value (q_stride_t = H*d_qk, q_stride_b =
 * T*q_stride_t, k_stride_b = S*k_ld, v_stride_b = S*v_ld).  Non-zero strides must be
 * multiples of 8 elements and q_stride_t >= H*d_qk. */
typedef struct {
  int32_t B, T, S, H, d_qk, d_v;
  float scale;
  const void* q;
  const void* k;
  int64_t k_ld;
  const void* v;
  int64_t v_ld;
  int64_t q_stride_b, q_stride_t;
  int64_t k_stride_b, v_stride_b;
} dsa_attn_args;

typedef enum { DSA_TOPK_FROM_SCORES = 0, DSA_TOPK_FROM_INDEXER = 1 } dsa_topk_kind;

/* Source of a top-k: a materialised fp32 score buffer [B,T,ld] (ld >= S; only the visible
 * prefix of each row is read), or the indexer operands.  From indexer operands with 64 indexer
 * heads, k <= 2048 and enough query rows to fill the GPU, the scores are never stored: the
 * indexer keeps, per query row, only the keys whose score reaches a threshold set from a sample
 * of the row (a few thousand (score, position) pairs in the workspace), and an exact top-k runs
 * over them; a row whose candidates could not hold its top-k (rare: a badly sampled or heavily
 * tied row) is recomputed through a score buffer in the workspace.  Other shapes (decode's few
 * rows, 4 indexer heads, larger k) pass the scores of a chunk of rows through that buffer (fp32,
 * up to 4 GiB per chunk).  Either way the result is the exact top-k. */
typedef struct {
  dsa_topk_kind kind;
  const float* scores;
  int64_t ld;
  const dsa_indexer_args* ix;
} dsa_topk_src;

/* One layer of an IndexShare group.  `ix` is read for 'F' layers only. */
typedef struct {
  dsa_indexer_args ix;
  dsa_attn_args at;
  void* out;  /* [B,T,H,d_v] bf16 */
  float* lse; /* [B,T,H] fp32 natural-log softmax normaliser, or NULL */
} dsa_layer;

/* Workspace sizes.  Every size below is the number of bytes with which the call runs its
 * fastest schedule on the current device (the split of few long rows across CTAs depends on
 * the device's SM count); the calls accept less, down to the stated minimum, and then take a
 * slower schedule with identical results.  Calls that need no scratch take DSA_WS_MIN.
 *
 * dsa_workspace_size: dsa_topk(FROM_INDEXER) for this indexer shape -- the candidate lists of
 *   the path that stores no scores when it applies (at most 1 GiB: 8,192 (score, position)
 *   pairs per row of a chunk of rows), a score buffer of fp32 rows (up to 4 GiB; at least
 *   DSA_WS_MIN plus one row of B*S*4 bytes is required) and, when a chunk has fewer query rows
 *   than the device has SMs, room for spreading each row's top-k over CTAs (a sampled
 *   threshold, a filtering pass and a candidate select; or, for k > 2,048, segments and a
 *   merge).  Without room for the candidate lists the call stores the scores of every row.
 * dsa_topk_workspace_size: dsa_topk(FROM_SCORES) over B*T rows of the given visibility --
 *   DSA_WS_MIN plus that room when the rows are few and long (0 extra otherwise).
 * dsa_attn_workspace_size: dsa_sparse_attn -- DSA_WS_MIN plus, for the 64-head latent shape
 *   with fewer query rows than half the SMs, room for each row's split parts (fp32 outputs
 *   and LSEs of up to 8 parts); with more rows, one byte per row (rounded up to 256) that
 *   marks the rows a fixed-reference softmax pass leaves to a running-maximum recompute
 *   (without it every row takes the running-maximum softmax; the two agree up to rounding).
 * indexshare_group_workspace_size: indexshare_group_forward (seqs NULL) or
 *   indexshare_group_forward_varlen (seqs given) -- the largest of the above over the
 *   group's layers ('F' layers: indexer and attention; 'S' layers: attention), including the
 *   split parts of the launches that attend several layers at once (the layers that read one
 *   index buffer, when each has few rows), and, packed, over its sequences.  Returns
 *   DSA_WS_MIN for arguments that the call would reject. */
#define DSA_WS_MIN ((size_t)256)
size_t dsa_workspace_size(const dsa_indexer_args* ix, int32_t k);
size_t dsa_topk_workspace_size(int32_t B, int32_t T, int32_t S, int64_t q_pos0, int32_t diag, int32_t k);
size_t dsa_attn_workspace_size(const dsa_attn_args* at, int32_t k);

/* Indexer scores, materialised: scores[b,i,s] (row stride ld >= S, fp32) =
 * sum_h w[b,i,h] * ReLU(q[b,i,h] . k[b,s]) for visible s, -inf for the rest of [0, S). */
dsa_status dsa_indexer_scores(const dsa_indexer_args* ix, float* scores, int64_t ld, void* ws,
                              size_t ws_bytes, void* stream);

/* Top-k per query row (IndexShare explainer, "How IndexShare Works": the full layer
 * "performs the top-k operation").  idx [B,T,k] int32 receives, for each row, the k
 * visible positions of largest score (equal scores: lower position first), listed in
 * ascending position order; rows with n < k visible keys list all n and pad with -1.
 * B, T, S, q_pos0, diag describe the rows; with FROM_INDEXER they must match src->ix.
 * 1 <= k <= 4096. */
dsa_status dsa_topk(const dsa_topk_src* src, int32_t B, int32_t T, int32_t S, int64_t q_pos0,
                    int32_t diag, int32_t k, int32_t* idx, void* ws, size_t ws_bytes,
                    void* stream);

/* Sparse attention over selected rows (explainer, "Why The Indexer Becomes Expensive":
 * "the main attention mechanism operates only on this smaller subset").
 * idx [B,T,k] int32, entries in [-1, S); -1 is skipped.  out [B,T,H,d_v] bf16;
 * lse [B,T,H] fp32 (natural log) or NULL.  A row with no valid entry gets out = 0,
 * lse = -inf. */
dsa_status dsa_sparse_attn(const dsa_attn_args* at, const int32_t* idx, int32_t k, void* out,
                           float* lse, void* ws, size_t ws_bytes, void* stream);

/* IndexShare group forward ("How IndexShare Works"; "What IndexShare reuses").
 * schedule: one 'F' or 'S' per layer, starting with 'F' (e.g. "FSSS").  For each 'F'
 * layer number f (0-based count of F layers so far), indexer + top-k write idx_bufs[f]
 * ([B,T,k] int32, caller-owned).  Every layer then attends with its own operands over the
 * most recent F layer's buffer, as dsa_sparse_attn would; the layers that read one buffer
 * share one attention launch when each has too few rows to fill the GPU (decode) and their
 * attention operands have the 64-head latent shape with equal scale and strides (results as
 * per-layer calls, up to the summation order of a decode split).  All layers share B, T, S. */
dsa_status indexshare_group_forward(const dsa_layer* layers, int32_t n_layers,
                                    const char* schedule, int32_t k, int32_t* const* idx_bufs,
                                    void* ws, size_t ws_bytes, void* stream);

/* Draft-step index reuse in the multi-token-prediction layer (GLM-5.2 article, "Reuse in the
 * MTP layer": the first draft step computes the indices; the later draft steps reuse those
 * indices and the earlier KV cache).  One call: the first step's indexer + top-k, then ONE
 * attention launch in which the n = at->T draft queries of every sequence attend over that
 * sequence's single index row.
 *   ix   the first draft step's indexer: B sequences, T = 1 query each, keys k / k_scale
 *        [B,S,...] (the layer's shared indexer-key cache).
 *   at   the draft queries as T = n query positions: q [B,n,H,d_qk] (step s of sequence b
 *        at q + b*q_stride_b + s*q_stride_t), k / v the shared latent cache [B,S,...]; B and
 *        S equal the indexer's.
 *   idx  [B,k] int32, written: the first step's selection (ascending, -1 padded); every
 *        step of sequence b reads row b (index-row stride 0 between steps).
 *   out  [B,n,H,d_v] bf16; lse [B,n,H] fp32 or NULL.
 * Results equal dsa_topk(FROM_INDEXER) on ix followed, for each step s, by dsa_sparse_attn
 * of step s's queries over idx (up to the summation order of a decode split).
 * ws: indexshare_draft_workspace_size bytes are preferred.  Errors as the two calls. */
dsa_status indexshare_draft_forward(const dsa_indexer_args* ix, const dsa_attn_args* at, int32_t k,
                                    int32_t* idx, void* out, float* lse, void* ws, size_t ws_bytes,
                                    void* stream);
size_t indexshare_draft_workspace_size(const dsa_indexer_args* ix, const dsa_attn_args* at, int32_t k);

/* Variable-length sequences packed along the row axis (host arrays).  Sequence b owns the
 * packed query rows cu_q[b] .. cu_q[b+1]-1 and the packed key rows cu_k[b] .. cu_k[b+1]-1;
 * its first query row sits at absolute position q_pos0[b] (a full prefill: q_pos0 = 0 with
 * as many rows as keys; a chunk: the last rows of a longer cache).  cu_q and cu_k hold
 * n_seqs + 1 non-decreasing entries starting at 0; every sequence has at least one key. */
typedef struct {
  int32_t n_seqs;
  const int64_t* cu_q;
  const int64_t* cu_k;
  const int64_t* q_pos0;
} dsa_varlen;

/* indexshare_group_forward over packed variable-length sequences (batched serving of
 * prompts of different lengths; the pages describe one sequence at a time, so this only
 * extends the boundary).  Every layer's operands describe the packed tensors as one
 * sequence: B = 1, T = cu_q[n_seqs] query rows, S = cu_k[n_seqs] key rows (q, w, q_scale,
 * out, lse and each idx_bufs[f] [1,T,k] packed by query row; k, k_scale and the KV packed
 * by key row); the indexer's own q_pos0 is ignored.  Each sequence runs the schedule on
 * its own rows and keys -- its scores, selections and attention never reach another
 * sequence -- with the results of indexshare_group_forward on that sequence alone.  Every
 * sequence's view is checked (shapes, alignment of its offsets, workspace) before anything
 * launches; sequences with no query rows are skipped.  ws: indexshare_group_workspace_size
 * (with seqs) bytes are preferred; dsa_workspace_size_varlen gives the indexer part alone
 * (the largest sequence's need). */
dsa_status indexshare_group_forward_varlen(const dsa_layer* layers, int32_t n_layers,
                                           const char* schedule, int32_t k,
                                           const dsa_varlen* seqs, int32_t* const* idx_bufs,
                                           void* ws, size_t ws_bytes, void* stream);
size_t dsa_workspace_size_varlen(const dsa_indexer_args* ix, const dsa_varlen* seqs, int32_t k);
size_t indexshare_group_workspace_size(const dsa_layer* layers, int32_t n_layers, const char* schedule,
                                       int32_t k, const dsa_varlen* seqs);

/* Overlap of two index buffers a, b [rows,k] (rows as written by dsa_topk: ascending valid
 * entries, then -1 padding): per_row[r] = |A_r and B_r| / |A_r| over valid entries (1 when
 * A_r is empty), fp32 device array or NULL; *mean_out (host) = mean over rows in double.
 * Synchronises `stream`.  Explainer, "Why Reusing Indices Can Work" (adjacent-layer
 * overlap). */
dsa_status topk_overlap(const int32_t* a, const int32_t* b, int32_t rows, int32_t k,
                        float* per_row, double* mean_out, void* ws, size_t ws_bytes,
                        void* stream);

/* All-pairs overlap of n index buffers of the same query rows -- the layer-overlap heatmap
 * of an all-F pass (IndexCache notes, section 2: pairwise overlap of the layers' top-k
 * sets, 70-100% between adjacent layers, with blocks of layers that pick nearly the same
 * tokens).  matrix_out[i*n + j] (host, n*n doubles) = the mean over rows of
 * |A^i_r and A^j_r| / |A^i_r| over valid entries (1 for a row whose A^i_r is empty; 1 for
 * every entry when rows = 0): what topk_overlap(bufs[i], bufs[j]) returns, for every ordered
 * pair at once; the diagonal is 1.
 *   bufs    HOST array of n DEVICE pointers, each [rows,k] int32 in the form dsa_topk
 *           writes (ascending valid entries, then -1 padding); 1 <= n <= 16.
 *   counts  DEVICE int32 [rows,n,n] receiving |A^i_r and A^j_r| (diagonal: |A^i_r|), or NULL.
 *   ws      at least topk_overlap_matrix_workspace_size(n) bytes.
 * One CTA holds a row of all n buffers in shared memory: n * (k + k/64 + 1) * 4 bytes must
 * not exceed DSA_OVERLAP_MATRIX_MAX_SMEM (n = 16 allows k <= 3,072), else
 * DSA_ERR_UNSUPPORTED.  A row not in dsa_topk's form raises DSA_FLAG_UNSORTED.  The sum over
 * rows runs in a fixed order (deterministic).  Synchronises `stream`. */
#define DSA_OVERLAP_MATRIX_MAX_SMEM ((size_t)204800)
dsa_status topk_overlap_matrix(const int32_t* const* bufs, int32_t n, int32_t rows, int32_t k,
                               int32_t* counts, double* matrix_out, void* ws, size_t ws_bytes,
                               void* stream);
size_t topk_overlap_matrix_workspace_size(int32_t n);

/* F/S schedules judged by an overlap matrix (host only, no GPU work).  A shared layer l
 * reuses the positions of the most recent full layer f(l) (f(l) = l for a full layer), so
 * the fraction of its own top-k it keeps is overlap[l*n + f(l)] (GLM-5.2 IndexShare
 * article: the released schedule repeats F,S,S,S after a few initial exceptions; IndexCache
 * notes, section 2: the first layer is always F).
 *   indexshare_schedule_score:  *score_out = mean over the n layers of overlap[l*n + f(l)].
 *   indexshare_schedule_search: among schedules with exactly n_full 'F' (the first layer
 *     one of them), one of largest score, written to schedule_out (n characters + NUL) with
 *     its score; ties go to the schedule whose later full layers sit earliest.
 * overlap: host n*n doubles, row-major (e.g. from topk_overlap_matrix).  n <=
 * DSA_SCHEDULE_MAX_LAYERS.  A bad schedule string returns DSA_ERR_SCHEDULE. */
#define DSA_SCHEDULE_MAX_LAYERS 256
dsa_status indexshare_schedule_score(const double* overlap, int32_t n, const char* schedule,
                                     double* score_out);
dsa_status indexshare_schedule_search(const double* overlap, int32_t n, int32_t n_full,
                                      char* schedule_out, double* score_out);

/* FP8 e4m3 quantisation with one fp32 scale per row, appended into an indexer cache (the
 * step before the FP8 indexer, which reads e4m3 codes with per-token scales: IndexCache notes,
 * section 1, "few heads, low-rank, FP8").  For each new row of `width` values:
 * scale = amax / 448 over the row (1 when every value is 0) and code = e4m3(x / scale), the
 * e4m3 value nearest to the fp32 quotient (ties to even), saturated to +-448; the scale and
 * the quotient are fp32 roundings (IEEE division).  A dequantised value is scale * code.
 *   x          [B, n, width] bf16; sequence b starts at x + b * x_stride_b (elements), its n
 *              rows contiguous.  8-byte aligned; x_stride_b a multiple of 4.
 *   codes      [B, S_cap, width] e4m3 cache (4-byte aligned); new row i of sequence b is
 *              written to row pos_b + i.
 *   scales     [B, S_cap] fp32 (4-byte aligned), same rows.
 *   positions  DEVICE int64 [B] giving pos_b, or NULL for pos_b = pos0 in every sequence.
 * width: a multiple of 4 in [4, 65536] -- d_I for the key cache (one scale per key), H_I * d_I
 * for queries (one scale per token over all heads).  With positions NULL, pos0 + n <= S_cap
 * is checked on the host; a device position outside [0, S_cap - n] skips that sequence and
 * raises DSA_FLAG_BAD_INDEX.  Needs DSA_WS_MIN bytes of workspace (the flag word). */
dsa_status dsa_quantize_e4m3_append(const void* x, int32_t B, int32_t n, int32_t width,
                                    int64_t x_stride_b, uint8_t* codes, float* scales,
                                    int32_t S_cap, int64_t pos0, const int64_t* positions,
                                    void* ws, size_t ws_bytes, void* stream);

/* Reads the device flag word of a workspace into *flags_out (host) and clears it.
 * Synchronises `stream`. */
dsa_status dsa_read_device_flags(void* ws, uint32_t* flags_out, void* stream);

/* Bound on every wait inside the library's kernels (a wait for a copy, a tensor-core
 * product or another warp of the same CTA), in SM clock cycles, for the kernels launched
 * after the call (all threads of the process).  0 restores the default, 2e9 cycles (about
 * one second).  A wait that runs out stops its CTA's work: the CTA lets the copies and
 * products it has started finish (those waits keep the default bound), frees its tensor
 * memory, ORs DSA_FLAG_TIMEOUT into the flag word and exits; the outputs of a call that
 * raised the flag are unspecified.  It exists to test that path: a bound of a few cycles
 * makes the waits run out on any input, without touching the GPU's state. */
void dsa_set_wait_limit(uint64_t cycles);

/* Indexer -> top-k without a caller workspace.  The paper has no counterpart to this call;
 * it exists for callers that cannot allocate device memory where they call the library
 * (allocator or memory-pool callbacks, runtimes that pre-partition all device memory,
 * code that must not grow its footprint after start-up).  Results are identical to
 * dsa_topk with a DSA_TOPK_FROM_INDEXER source.
 *   ix, k, idx  as for dsa_topk; idx [B,T,k] int32 is the caller's output buffer.
 *   flags       device uint32 the kernels OR DSA_FLAG_* bits into, or NULL: the bits that
 *               call raises (a wait that ran out, NaN scores) then go to a word inside the
 *               library's array that nothing reads back and the next call clears, so they
 *               are lost -- pass a word to observe them.
 * Scratch: a file-scope device array of 64 MiB, held by every GPU that loads the library
 * until the process exits.  B*S*4 must not exceed 64 MiB - 256 B (DSA_ERR_UNSUPPORTED
 * otherwise); no cudaMalloc/cudaFree or allocating library routine is called.  The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress); make that
 * first call before any stream capture.  All calls share the one array: calls whose work
 * overlaps on the GPU (other streams, other host threads) race on it. */
dsa_status dsa_topk_indexer_noalloc(const dsa_indexer_args* ix, int32_t k, int32_t* idx,
                                    uint32_t* flags, void* stream);

/* Name of a status code; message of the calling thread's last failure. */
const char* dsa_status_string(dsa_status s);
const char* dsa_last_error(void);

/* Number of kernels this library has launched since it was loaded (all threads). */
uint64_t dsa_launch_count(void);

/* Launch tracing, for measuring the device time of each kernel inside a larger timed region.
 * dsa_trace_enable(max_launches): creates a pool of 2*max_launches CUDA events (host call;
 *   returns DSA_ERR_INVALID_ARG unless 0 < max_launches <= 2^20, DSA_ERR_CUDA if event
 *   creation fails) and starts recording: from then on every kernel launch the library makes
 *   is bracketed by two events recorded on its stream.  Launches beyond the pool are not
 *   recorded.
 * dsa_trace_read(kinds, ms, max_records, dropped): waits for the recorded launches to finish
 *   (host synchronisation on their events), writes up to max_records entries in launch order
 *   -- kinds[i] is DSA_TRACE_INDEXER, _TOPK, _ATTENTION or _OVERLAP, ms[i] the device time in
 *   milliseconds (-1 if unavailable) -- returns the number written, stores in *dropped (may
 *   be NULL) the launches the pool could not record, and clears the records.  Host arrays
 *   are owned by the caller; kinds or ms may be NULL.
 * dsa_trace_disable(): stops recording and destroys the pool. */
enum { DSA_TRACE_INDEXER = 1, DSA_TRACE_TOPK = 2, DSA_TRACE_ATTENTION = 3, DSA_TRACE_OVERLAP = 4 };
dsa_status dsa_trace_enable(int max_launches);
int dsa_trace_read(int* kinds, float* ms, int max_records, int* dropped);
void dsa_trace_disable(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H */
