/*
 * mla.h -- C ABI of libmla.so: Multi-head Latent Attention (MLA) for
 * speculative-decoding verify steps on GB300 (sm_103a).
 *
 * What is computed.  A verify call scores L >= 1 new query rows per sequence
 * against a compressed latent KV cache (c_kv: r = kv_lora_rank values per
 * cached position, plus a shared RoPE key k_rope of rope_dim values).  The
 * pages ("One guard, 110x off the verify step", section "The defect") give two
 * mathematically equivalent ways to do it, both implemented here:
 *
 *   absorbed      q_lat = q_nope . W_UK           (fold, n -> r, per head)
 *                 s_t   = scale*(q_lat . c_kv[t] + q_rope . k_rope[t])
 *                 o_lat = softmax(s) . c_kv        (accumulated in latent space)
 *                 out   = o_lat . W_UV             (unembed, r -> v, per head)
 *
 *   materialised  K_nope[t] = c_kv[t] . W_UK^T,  V[t] = c_kv[t] . W_UV  (expand)
 *                 out = softmax(scale*([q_nope||q_rope] . [K_nope[t]||k_rope[t]])) . V
 *
 * Row l of sequence b sits at position T_b - L + l and sees cached positions
 * t <= T_b - L + l (causal among the verify rows); T_b is the cache length
 * INCLUDING the L new rows.
 *
 * Branch choice ("The threshold is not a constant" and "The change" on the same
 * page; the finite-cache form from the mlx-lm pull request "fix: Speed up
 * multi-token decode by computing the absorbed MLA threshold", opening section):
 * absorbed iff L <= floor(r*d*T / (r*d + (2r-d)*T)), d = n + v, evaluated in
 * exact integer arithmetic, never below 1, and 1 when 2r - d <= 0.
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns every buffer.  The library allocates no
 *    device memory in these calls; scratch comes from the caller's workspace.
 *  - Reads may start early: the kernels chain to the preceding kernel in the
 *    stream by programmatic dependent launch, and they may start reading
 *    W_UK, W_UV and the latent cache (never the queries, lengths or page
 *    table) before a preceding kernel that allows it has finished; a kernel
 *    that writes those buffers right before a call must not trigger early.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *    default stream).  Calls are asynchronous on it; inputs must stay alive
 *    and unmodified until the stream reaches the call's kernels.
 *  - Errors: argument errors return before anything is launched; a failed
 *    launch returns MLA_ERR_CUDA.  mla_last_error() gives a one-line detail
 *    for the calling thread's last failure.
 *  - Layouts are row-major, element strides in elements (not bytes).
 *  - Device pointers must be 16-byte aligned.
 */
#ifndef MLA_VERIFY_H_
#define MLA_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,  /* a pointer, size or geometry is out of range   */
  MLA_ERR_UNSUPPORTED = -2,  /* valid request this build has no kernel for     */
  MLA_ERR_WORKSPACE = -3,    /* workspace smaller than mla_workspace_bytes()   */
  MLA_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed              */
  MLA_ERR_TIMEOUT = -5       /* a bounded device wait ran out (status word)    */
} mla_status_t;

typedef enum {
  MLA_MODE_AUTO = 0,          /* crossover threshold decides                   */
  MLA_MODE_ABSORBED = 1,      /* force the absorbed branch                     */
  MLA_MODE_MATERIALISED = 2   /* force the materialised branch                 */
} mla_mode_t;

typedef enum {
  MLA_BRANCH_ABSORBED = 1,
  MLA_BRANCH_MATERIALISED = 2
} mla_branch_t;

typedef enum {
  MLA_DTYPE_BF16 = 0,   /* bf16 inputs/outputs, fp32 accumulation            */
  MLA_DTYPE_FP32 = 1    /* fp32 inputs/outputs, fp32 arithmetic (CUDA cores) */
} mla_dtype_t;

/* Head geometry of one MLA layer.  softmax_scale <= 0 selects
 * 1/sqrt(qk_nope_dim + rope_dim).  dtype is an mla_dtype_t. */
typedef struct {
  int32_t num_heads;      /* H                                   */
  int32_t kv_lora_rank;   /* r (latent width)                    */
  int32_t qk_nope_dim;    /* n (no-position query/key width)     */
  int32_t v_dim;          /* v (value width)                     */
  int32_t rope_dim;       /* rope (shared RoPE key width)        */
  float softmax_scale;
  int32_t dtype;
} mla_geometry_t;

/* Crossover of the pages' helper.  cache_len <= 0 asks for the long-cache
 * limit floor(r(n+v)/(2r-n-v)) ("The threshold is not a constant", table:
 * 170 for 512/128/128, 398 for 512/192/256, 512 for 512/256/256); cache_len
 * > 0 gives floor(r*d*T / (r*d + (2r-d)*T)) (pull request opening section; 379
 * for 512/192/256 at T = 8192).  Never below 1; 1 when 2r - d <= 0.  Returns
 * -1 if r, n or v is not positive.  Pure host code, no CUDA. */
int64_t mla_max_absorbed_queries(int32_t r, int32_t n, int32_t v, int64_t cache_len);

/* One decision for a batch of sequences: the summed cost model,
 * floor(r*d*S / (B*r*d + (2r-d)*S)) with S = sum of cache_lens_host[0..batch);
 * equal to mla_max_absorbed_queries for batch == 1.  Returns -1 on bad
 * arguments (NULL lengths, batch < 1, a length < 1). */
int64_t mla_max_absorbed_queries_batch(int32_t r, int32_t n, int32_t v,
                                       const int32_t* cache_lens_host, int32_t batch);

/* Branch a call would take ("The change": guard L <= max_absorbed); forced
 * modes override.  Writes an mla_branch_t to *branch.  Host only. */
mla_status_t mla_select_branch(const mla_geometry_t* geom, int32_t L,
                               const int32_t* cache_lens_host, int32_t batch,
                               int32_t mode, int32_t* branch);

/* Bytes of device workspace mla_verify_attention needs for this call
 * (branch-dependent: split-KV partials for the absorbed branch, the expanded
 * K_nope/V buffer for the materialised branch).  The workspace needs no
 * initialisation.  Host only. */
mla_status_t mla_workspace_bytes(const mla_geometry_t* geom, int32_t batch, int32_t L,
                                 const int32_t* cache_lens_host, int32_t mode,
                                 size_t* bytes);

/* One verify attention call for `batch` sequences of L rows each.
 *
 *  q_nope  device [batch, L, H, n]      query, no-position part
 *  q_rope  device [batch, L, H, rope]   query RoPE part (RoPE already applied)
 *  c_kv    device latent cache, rows of r values:
 *            contiguous (page_table == NULL): row (b, t) at
 *              c_kv + (b*seq_stride_rows + t) * c_kv_row_stride
 *            paged: row (b, t) at
 *              c_kv + (page_table[b*max_pages_per_seq + t/page_size]*page_size
 *                      + t%page_size) * c_kv_row_stride
 *  k_rope  device RoPE key cache, same addressing with k_rope_row_stride
 *          (a packed [.., r+rope] cache may pass k_rope = c_kv + r and both
 *          strides = r + rope)
 *  W_UK    device [H, n, r]   key up-projection
 *  W_UV    device [H, r, v]   value up-projection
 *  cache_lens_dev / cache_lens_host  [batch] int32, T_b with L <= T_b; the
 *          device copy is read by the kernels, the host copy for dispatch and
 *          launch sizing (they must agree)
 *  page_table  device [batch, max_pages_per_seq] int32 page ids in
 *          [0, num_pages), or NULL for a contiguous cache
 *  out     device [batch, L, H, v] in the geometry's dtype
 *  workspace / workspace_bytes  device scratch of at least
 *          mla_workspace_bytes() bytes, 256-byte aligned (may be NULL when
 *          that is 0)
 *  branch_taken  host, may be NULL; receives the mla_branch_t used
 */
mla_status_t mla_verify_attention(
    const mla_geometry_t* geom,
    const void* q_nope, const void* q_rope,
    const void* c_kv, const void* k_rope,
    int64_t c_kv_row_stride, int64_t k_rope_row_stride, int64_t seq_stride_rows,
    const void* W_UK, const void* W_UV,
    const int32_t* cache_lens_dev, const int32_t* cache_lens_host,
    int32_t batch, int32_t L,
    const int32_t* page_table, int32_t page_size, int32_t max_pages_per_seq,
    int32_t num_pages,
    int32_t mode, void* out, void* workspace, size_t workspace_bytes,
    void* stream, int32_t* branch_taken);

/* Bytes of device workspace mla_verify_attention_sparse needs for `batch`
 * sequences of L verify rows with index lists of topk_len entries (the
 * pieces of the split follow the lists, not the cache lengths).  Host only. */
mla_status_t mla_sparse_workspace_bytes(const mla_geometry_t* geom, int32_t batch, int32_t L,
                                        const int32_t* cache_lens_host, int32_t topk_len,
                                        size_t* bytes);

/* Verify attention over selected cached positions: the sparse model's top-k
 * attention ("One guard, 110x off the verify step", section "The sparse
 * model is different": an indexer picks the top 2048 cached positions and
 * attention runs over those only; mlx-lm pull request 1817, opening section,
 * on deepseek_v32's top-k gather).  Always the absorbed branch.
 *
 *  topk      device [batch, L, topk_len] int32: verify row l of sequence b
 *            attends to the positions topk[b, l, j] with
 *            0 <= topk[b, l, j] <= T_b - L + l; other entries (-1 padding,
 *            positions past the row's causal limit) are skipped.  A row whose
 *            list holds no usable position gets zeros.  The list is read as
 *            given: a position listed twice counts twice.
 *  topk_len  entries per list, >= 1
 *
 * Every other argument is that of mla_verify_attention (no mode: the
 * absorbed branch runs; no branch output).  The workspace must hold
 * mla_sparse_workspace_bytes() bytes.  bf16 calls with r = 512, rope = 64
 * and H a multiple of 128 (every 128-row tile is one verify row) run the
 * tensor-core kernels, which gather the listed cache rows tile by tile; other
 * calls run the CUDA-core kernels.  The index lists may be written by the
 * kernel right before the call: they are read only after it has finished. */
mla_status_t mla_verify_attention_sparse(
    const mla_geometry_t* geom,
    const void* q_nope, const void* q_rope,
    const void* c_kv, const void* k_rope,
    int64_t c_kv_row_stride, int64_t k_rope_row_stride, int64_t seq_stride_rows,
    const void* W_UK, const void* W_UV,
    const int32_t* cache_lens_dev, const int32_t* cache_lens_host,
    int32_t batch, int32_t L,
    const int32_t* topk, int32_t topk_len,
    const int32_t* page_table, int32_t page_size, int32_t max_pages_per_seq,
    int32_t num_pages,
    void* out, void* workspace, size_t workspace_bytes, void* stream);

/* The absorbed-branch verify call without a workspace, for callers that cannot
 * allocate device memory (a plugin host or serving engine that owns every
 * device allocation and gives its attention back-end no allocator, or a
 * latency-critical loop that must not call cudaMalloc).  The pages have no
 * counterpart: it exists for those callers only.
 *
 * Arguments are those of mla_verify_attention without mode, workspace and
 * workspace_bytes; the absorbed branch always runs.  Scratch comes from one
 * 32 MiB static device array inside the library.  A call whose scratch
 * (mla_workspace_bytes with MLA_MODE_ABSORBED) exceeds 32 MiB returns
 * MLA_ERR_WORKSPACE before launching anything.  It never calls cudaMalloc,
 * cudaFree or an allocating library routine.
 *
 * The array lives in its own CUDA module, which CUDA loads lazily: the FIRST
 * call of this entry point on a device loads it and so reserves the 32 MiB on
 * that device (kept until the process exits).  Make that first call as a
 * warm-up, before a host memory pool claims the device (otherwise the load
 * fails and the call returns MLA_ERR_WORKSPACE with a message saying so) and
 * before any stream capture starts.  Every call looks up the array's address
 * in the current context (cudaGetSymbolAddress); `stream` must belong to the
 * current device (else MLA_ERR_INVALID_ARG).
 *
 * All calls share the one array and it keeps the previous call's contents
 * (nothing in it needs to start at zero): calls that overlap on the GPU
 * (concurrent streams or threads) race on it, so issue them one at a time. */
mla_status_t mla_verify_attention_noalloc(
    const mla_geometry_t* geom,
    const void* q_nope, const void* q_rope,
    const void* c_kv, const void* k_rope,
    int64_t c_kv_row_stride, int64_t k_rope_row_stride, int64_t seq_stride_rows,
    const void* W_UK, const void* W_UV,
    const int32_t* cache_lens_dev, const int32_t* cache_lens_host,
    int32_t batch, int32_t L,
    const int32_t* page_table, int32_t page_size, int32_t max_pages_per_seq,
    int32_t num_pages,
    void* out, void* stream, int32_t* branch_taken);

/* Host-side check of a page table before it is used: for every sequence b, the table must hold
 * ceil(cache_lens_host[b] / page_size) <= max_pages_per_seq pages, and every
 * entry j < ceil(T_b / page_size) of row b of page_table_host ([batch,
 * max_pages_per_seq], host memory, row-major) must lie in [0, num_pages).
 * Entries past a sequence's last page are not read.  Returns MLA_OK, or
 * MLA_ERR_INVALID_ARG with the first offending entry in mla_last_error().
 * Pure host code, no CUDA.  The kernels guard the same range on the device:
 * an out-of-range id met there forms no address, its positions read as
 * zeros, and mla_device_status reports it (code 300). */
mla_status_t mla_check_page_table(const int32_t* page_table_host, int32_t batch,
                                  int32_t max_pages_per_seq, const int32_t* cache_lens_host,
                                  int32_t page_size, int32_t num_pages);

/* Draft cap from a measured verify-cost curve ("Draft caps and calibration",
 * the cost model "in formula form, for a cap C", and "How mlx-dspark picks
 * it"): returns the cap C in [0, limit] that maximises
 *     speedup(C) = accepted(C) * verify(1) / (drafter(C) + verify(C + 1)),
 *     accepted(C) = 1 + p + p^2 + ... + p^C,
 * where verify(w) = verify_cost[w - 1] is the measured cost of one verify
 * pass over w rows (any unit; verify(1) is one plain decode step, so costs
 * count in single-token steps), drafter(C) = drafter_cost[0] for every C
 * when n_drafter == 1, else drafter_cost[C].  C = 0 is plain decoding:
 * speedup(0) = 1.  limit = min(max_cap, n_verify - 1, n_drafter - 1 when
 * n_drafter > 1).  Ties go to the smaller cap.  speedup_out (host, may be
 * NULL) receives speedup(0..limit).  Returns -1 on bad arguments (p outside
 * [0, 1], a non-positive verify cost, a negative drafter cost, NULL arrays);
 * mla_last_error() says which.  Pure host code, double precision. */
int32_t mla_select_draft_cap(double p, const double* verify_cost, int32_t n_verify,
                             const double* drafter_cost, int32_t n_drafter, int32_t max_cap,
                             double* speedup_out);

/* ------------------------------------------------------------------------
 * Speculative-rollback state maintenance ("Over 107tok/s Qwen3.8-Flash-Next
 * on M3 Ultra").  Element i of row (h, q) of a strided buffer sits at word
 * i*strides[0] + h*strides[1] + q*strides[2] (non-negative strides, in
 * 32-bit words); words are copied as bit patterns.
 * ------------------------------------------------------------------------ */

/* One snapshot window: the s words of the concatenated row starting at
 * window_start go to cache[cache_offset + q*sequence_stride + h*s + i]. */
typedef struct {
  int32_t window_start;
  int64_t cache_offset;
  int64_t sequence_stride;
} mla_snapshot_window_t;

/* Section "A later extension: load snapshot history once", Algorithms 4 and
 * 5: X = S || T row by row (S: s state words, T: n new words per row; H
 * channels, Q sequences; 1 <= s <= 8, 1 <= n, s + n <= 16, Q <= 65535,
 * H*(s + n) <= 2^30) and the k <= 8
 * snapshot windows of X into `cache` (cache_words words long).  All buffers
 * are device memory.  When 2 <= k <= 8 and the windows' destinations are
 * pairwise disjoint and lie outside S, T and X, one kernel loads each row
 * once and writes X and every window from that load (*fused_out = 1);
 * otherwise the ordinary path runs: X, then one copy per window that reads X
 * back (*fused_out = 0; the windows are written in order).  X may share
 * words with S or T only row for row (then each row is read before it is
 * written).  A window outside the row or a destination outside the cache is
 * MLA_ERR_INVALID_ARG.
 * Asynchronous on `stream`.  fused_out is host memory and may be NULL. */
mla_status_t mla_concat_snapshots(const uint32_t* S, const int64_t* s_strides, const uint32_t* T,
                                  const int64_t* t_strides, uint32_t* X,
                                  const int64_t* x_strides, int32_t s, int32_t n, int32_t H,
                                  int32_t Q, uint32_t* cache, int64_t cache_words,
                                  const mla_snapshot_window_t* windows, int32_t k, void* stream,
                                  int32_t* fused_out);

/* Section "Keep the pooled keys; score them again", ValidBlock and Algorithm
 * 1: how many leading pooled blocks of ratio r survive a rollback that
 * removes positions from p0 on.  blocks: device [n_blocks, 8 + r] int32 rows
 * {stream, start, n_src, key_cell, pos[0..3], src_cell[0..r)}; cell_pos:
 * device [n_cells] logical positions (negative: empty cell); cell_seq:
 * device [n_cells] owner bit masks (bit q: sequence q).  A block is valid
 * when n_src == r, stream == 0, start >= 0, start + r <= p0, key_cell is one
 * of its source cells, all four pos[] equal start, and source cell i is in
 * [0, n_cells), live, owned by sequence 0 alone and at position start + i.
 * *prefix_out (device int32) receives the index of the first invalid block
 * (n_blocks when all are valid), or 0 when a global guard fails: n_streams
 * != 1, seq != 0, p0 < 0, or a bounded removal (p1 >= 0).  Asynchronous. */
mla_status_t mla_rollback_valid_prefix(const int32_t* blocks, int32_t n_blocks, int32_t r,
                                       const int32_t* cell_pos, const uint64_t* cell_seq,
                                       int32_t n_cells, int32_t p0, int32_t p1, int32_t seq,
                                       int32_t n_streams, int32_t* prefix_out, void* stream);

/* ------------------------------------------------------------------------
 * Indexer key pooling for the sparse model ("One guard, 110x off the verify
 * step", sections "The same bug, one layer over" and "The sparse model is
 * different").  Window w of a sequence covers cache positions 4w..4w+3; its
 * pooled key is the mean of the keys it holds (the last window of a cache
 * whose length is not a multiple of four holds fewer).
 * ------------------------------------------------------------------------ */

/* What a pool describes: the cache length it was computed for (-1: no pool
 * yet; a caller starts from {-1, 0, 0}), the batch and the key width. */
typedef struct {
  int64_t length;
  int32_t batch;
  int32_t dim;
} mla_indexer_pool_state_t;

/* One indexer step: the cache now holds cache_len tokens per sequence,
 * new_tokens of them appended since the last step.  keys: device, dtype
 * bf16 or fp32 (an mla_dtype_t), key (b, t) at
 * keys + (b*seq_stride_rows + t)*key_row_stride; dim a multiple of 32 up to
 * 512.  pooled: device fp32 [batch, pooled_windows_cap, dim] with
 * pooled_windows_cap >= ceil(cache_len/4); *state (host) says what it holds.
 *
 * When every guard of the page holds -- the pool exists (state->length >= 0),
 * there is no padding (padded == 0), the batch shape matches (state->batch ==
 * batch, state->dim == dim) and the cache is exactly as long as the pool
 * remembers (state->length == cache_len - new_tokens) -- only windows
 * floor(state->length/4) .. ceil(cache_len/4)-1 are recomputed, for any
 * new_tokens >= 1 (*incremental_out = 1).  Otherwise (for instance after a
 * speculative rejection trimmed the cache) every window is recomputed
 * (*incremental_out = 0).  Either way each window is computed by the same
 * code, so a wide step pools bit for bit as the same tokens fed one at a
 * time.  *state is updated on return.  Asynchronous on `stream`;
 * incremental_out is host memory and may be NULL. */
mla_status_t mla_indexer_pool_update(const void* keys, int32_t dtype, int64_t key_row_stride,
                                     int64_t seq_stride_rows, int32_t batch, int32_t dim,
                                     int64_t cache_len, int32_t new_tokens, int32_t padded,
                                     float* pooled, int64_t pooled_windows_cap,
                                     mla_indexer_pool_state_t* state, int32_t* incremental_out,
                                     void* stream);

/* Workspace bytes of mla_indexer_select (the scores of every window). */
mla_status_t mla_indexer_select_workspace_bytes(int32_t batch, int32_t new_tokens,
                                                int64_t cache_len, size_t* bytes);

/* Top-k windows for each new token.  q: device fp32 [batch, new_tokens,
 * dim] (one indexer query per new token, 1 <= new_tokens <= 32,
 * new_tokens*dim*4 <= 48 KB).  Token s of a step sits at position
 * p = cache_len - new_tokens + s and may pick window w when 4w <= p; score
 * = q . pooled key (fp32).  It keeps the k_windows highest scores (ties to
 * the lower window) and writes them in ascending window order to
 * windows_out (device [batch, new_tokens, k_windows] int32, may be NULL)
 * and their positions 4w+i (only those <= p) to positions_out (device
 * [batch, new_tokens, 4*k_windows] int32), -1 padded: positions_out is the
 * index list mla_verify_attention_sparse takes with L = new_tokens and
 * topk_len = 4*k_windows (512 windows make the page's 2048 positions). */
mla_status_t mla_indexer_select(const float* q, const float* pooled, int64_t pooled_windows_cap,
                                int32_t batch, int32_t dim, int64_t cache_len,
                                int32_t new_tokens, int32_t k_windows, int32_t* windows_out,
                                int32_t* positions_out, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Per-kernel timing, for benchmarks.  While enabled, every kernel launch the
 * library makes is bracketed by a pair of CUDA events recorded on the call's
 * stream (events come from a library-owned pool; no device memory).  Do not
 * enable it while a stream is being captured into a CUDA graph.  Not part of
 * the method: instrumentation only. */
mla_status_t mla_kernel_timing_enable(int32_t on);

/* Waits for every recorded event pair, folds them into per-kernel totals and
 * reports them: names receives the kernel names separated by ';' (truncated
 * to names_len bytes including the terminator), launches[i] and total_ms[i]
 * the launch count and summed device milliseconds of kernel i, for up to
 * max_kernels kernels; *n_kernels receives how many kernels have totals.
 * With reset != 0 the totals are cleared after reading. */
mla_status_t mla_kernel_timing_read(char* names, size_t names_len, int32_t* launches,
                                    double* total_ms, int32_t max_kernels,
                                    int32_t* n_kernels, int32_t reset);

/* Waits for the device to go idle, then reads the kernels' status word:
 * MLA_OK when nothing was recorded since the last clear; MLA_ERR_TIMEOUT
 * when a bounded wait inside a kernel ran out (*code receives the site that
 * gave up, 1..299); MLA_ERR_INVALID_ARG when a kernel met a page id outside
 * [0, num_pages) (*code = 300; that page's positions were read as zeros).
 * The kernels never hang on a missing signal: each wait gives up after about
 * a second, records its site here and lets the kernel finish (its outputs are
 * then undefined).  clear != 0 resets the word.
 *
 * With MLA_DEBUG_CHECKS=1 in the environment, mla_verify_attention also
 * synchronises the stream, copies cache_lens_dev (and the page table) to the
 * host and checks them against cache_lens_host and [0, num_pages) before it
 * launches anything (not while a stream is being captured). */
mla_status_t mla_device_status(int32_t* code, int32_t clear);

/* Failure-path self-test: launches one CTA on `stream` (cudaStream_t, NULL =
 * default stream) whose bounded wait on a barrier that nothing signals runs
 * out after about a second and records site 99 in the status word, as a
 * kernel whose signal never arrived would.  It touches no caller buffer and
 * leaves the context usable; mla_device_status then returns MLA_ERR_TIMEOUT
 * with *code == 99.  Returns MLA_ERR_CUDA if the launch fails. */
mla_status_t mla_selftest_bounded_wait(void* stream);

/* Static name of a status code. */
const char* mla_status_string(int32_t status);

/* One-line detail of the calling thread's last failed call ("" if none). */
const char* mla_last_error(void);

/* Library ABI version (major*100 + minor). */
int32_t mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_VERIFY_H_ */
