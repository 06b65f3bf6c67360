/*
 * specverify.h -- C ABI of the GB300 (sm_103a) batched speculative-decoding
 * verification library (libspecverify.so).
 *
 * What one call computes.  A batch holds B requests.  Request b drafted k_b
 * tokens x_0..x_{k_b-1} (0 <= k_b <= 32).  The target model supplied logits at
 * k_b + 1 positions (after 0, 1, .., k_b drafted tokens: "Speculative decoding
 * and multi-token prediction", section "Draft and verify", step Two; "DFlash"
 * §4 step 4, p_1..p_{gamma+1}) and the drafter supplied logits at k_b
 * positions.  Each row is turned into a temperature-scaled softmax ("FlashMap:
 * Flow Map Speculative Decoding…" §5, draft_block step 5), optionally
 * filtered by top-k and top-p, applied identically to target and draft rows
 * ("Speculative decoding and multi-token prediction", "Why the output is
 * identical").  Then:
 *   - temperature 0 (greedy): the longest prefix of drafts equal to the target
 *     argmax (lowest index on ties) is accepted and the target's own argmax
 *     token is emitted at the first disagreement, or as the bonus token after
 *     a full acceptance ("DFlash" §4 step 5; "Speculative decoding…",
 *     "Draft and verify", step Three);
 *   - temperature > 0 (sampling): draft i is accepted iff u_i < p_i(x_i) /
 *     q_i(x_i) and verification stops at the first rejection ("FlashMap…" §4
 *     "The Rejection Sampling Invariant", steps 1-2).  After a rejection at
 *     position L one token is drawn from the normalised residual
 *     max(0, p_L - q_L) ("FlashMap…" §4 step 3; "DFlash" §4); after a full
 *     acceptance a bonus token is drawn from p_k.  Both draws use the
 *     uniform u_k by inverse CDF in vocabulary-index order:
 *     y* = min{ y : C_y > u_k * S }.
 *
 * Row layout.  Request b owns target rows t_off[b] .. t_off[b] + k_b with
 * t_off[b] = sum_{j<b} (k_j + 1), and draft rows d_off[b] .. d_off[b] + k_b - 1
 * with d_off[b] = t_off[b] - b (ragged batches are packed contiguously).
 * draft_tokens[d_off[b] + i] is x_i; uniforms[t_off[b] + i] is u_i for i < k_b
 * and uniforms[t_off[b] + k_b] drives the final draw; out_tokens uses the
 * target-row layout: out_tokens[t_off[b] + j] is the j-th emitted token of
 * request b, -1 after the last emitted one.  For a fixed k this is exactly a
 * [B, k+1] matrix.
 *
 * Ownership and synchronisation.  Every pointer handed to spec_verify is a
 * device pointer owned by the caller, including the workspace.  The library
 * allocates nothing, frees nothing and never synchronises inside spec_verify:
 * all work is enqueued on the caller's stream (a cudaStream_t passed as void*;
 * NULL is the legacy default stream) and results are visible in stream order.
 * Concurrent calls are safe when they use distinct workspaces.
 *
 * Errors.  Argument errors that the host can see (null pointers, bad sizes,
 * misalignment, unsupported dtype, workspace too small) return a nonzero
 * SV_ERR_* code before anything is enqueued.  Data errors live in device
 * memory and are found by the kernels: the first one is recorded in the
 * workspace (read it with spec_verify_get_error) and every affected request
 * gets out_accept_len = -1 and out_tokens = -1.  Kernels never trap.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define SV_OK 0
#define SV_ERR_ARG 1          /* null pointer, negative or inconsistent size   */
#define SV_ERR_UNSUPPORTED 2  /* dtype, vocabulary size, alignment, stride    */
#define SV_ERR_CUDA 3         /* a CUDA runtime call or launch failed          */
#define SV_ERR_WORKSPACE 4    /* workspace missing, too small or misaligned    */
/* data errors, found on the device (one request each unless stated) */
#define SV_ERR_DATA_K 16            /* k_b outside [0, SV_MAX_K]                 */
#define SV_ERR_DATA_TEMPERATURE 17  /* temperature negative, NaN or infinite     */
#define SV_ERR_DATA_TOP_P 18        /* top_p outside (0, 1]                      */
#define SV_ERR_DATA_TOP_K 19        /* top_k < 0                                 */
#define SV_ERR_DATA_TOKEN 20        /* a draft token outside [0, V)              */
#define SV_ERR_DATA_ROWS 21         /* sum(k+1) != target rows or sum(k) !=      */
                                    /* draft rows (whole batch)                  */
#define SV_ERR_DATA_LOGIT 22        /* NaN or +inf logit, or (sampling) a row    */
                                    /* with no finite logit                      */
#define SV_ERR_DATA_NO_DRAFT 23     /* temperature > 0 but draft logits absent   */
#define SV_ERR_TIMEOUT 24           /* an internal bounded wait expired (each    */
                                    /* wait gives up after 100 ms of GPU time)   */
#define SV_ERR_INTERNAL 25          /* an internal capacity invariant failed     */
#define SV_ERR_DATA_ACCEPT 26       /* KV commit: accept length above k_b         */
#define SV_ERR_DATA_PAGE 27         /* KV commit: a destination page missing from */
                                    /* the block table, or a negative kv_len      */

/* ---- limits -------------------------------------------------------------- */
#define SV_MAX_K 32              /* drafts per request (one warp ballot)       */
#define SV_TOPK_MAX 256          /* largest top-k whose kept set is listed     */
                                 /* (spec_verify_dump_rows); larger top-k and   */
                                 /* top-p alone keep a threshold instead        */
#define SV_VOCAB_MAX (1 << 22)   /* largest vocabulary                         */

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* A [rows, vocab] logit matrix in device memory.  `data` must be 16-byte
 * aligned and row_stride * element_size must be a multiple of 16 bytes
 * (row_stride >= vocab, in elements).  Target and draft share one dtype. */
typedef struct {
  const void* data;
  int32_t dtype;      /* sv_dtype */
  int32_t vocab;      /* V, 1 <= V <= SV_VOCAB_MAX */
  int64_t rows;
  int64_t row_stride; /* elements */
} sv_logits;

/* Optional extras of spec_verify; pass NULL for none. */
typedef struct {
  /* [draft_rows, 2] device doubles: (p_i(x_i), q_i(x_i)) of sampled requests
   * at every position the decision examined (0 .. min(L, k-1)); positions
   * after the first rejection may be NaN (filtered requests never evaluate
   * them).  NaN for greedy and failed requests (parity / diagnostics). */
  double* out_pq;
  /* cudaEvent_t handles recorded on the stream right before and right after
   * the row-streaming kernel (profiling); NULL to skip. */
  void* event_rowpass_begin;
  void* event_rowpass_end;
  /* Test of the timeout path (0 in normal use): nonzero makes one bounded
   * wait of the row pass expire, as a stalled copy's would; the request of
   * the first listed row then fails with SV_ERR_TIMEOUT and every other
   * request is verified as usual.  spec_verify only. */
  int32_t test_expire_wait;
  int32_t reserved;
} sv_options;

/* Bytes of device workspace spec_verify needs for this shape; 0 on bad
 * arguments.  The workspace must be 256-byte aligned and must not be used by
 * two calls that can run concurrently. */
size_t spec_verify_workspace_size(int32_t batch, int64_t target_rows, int64_t draft_rows);

/* Batched verification (see the file comment for what it computes).
 *   target_logits  [R_t, V]  R_t = sum_b (k_b + 1)
 *   draft_logits   [R_d, V]  R_d = sum_b k_b; the descriptor is required, its
 *                  `data` may be NULL when every temperature is 0
 *   draft_tokens   [R_d] int32            k_per_req   [B] int32, 0..SV_MAX_K
 *   temperature    [B] float, 0 = greedy
 *   top_k          [B] int32 or NULL; 0 or >= V switches top-k off; any
 *                  value in [1, V) is supported
 *   top_p          [B] float or NULL; 1 switches top-p off; (0, 1]; top-k
 *                  and top-p switch on and off independently; with both
 *                  NULL no row is filtered and the call launches one
 *                  kernel fewer (the row pass over threshold-filtered rows)
 *   uniforms       [R_t] float in [0, 1)
 *   out_accept_len [B] int32 (L, or -1 on a data error)
 *   out_tokens     [R_t] int32
 *   stream         cudaStream_t
 *   batch          B >= 0
 *   workspace      >= spec_verify_workspace_size(B, R_t, R_d) bytes
 * Returns SV_OK once the work is enqueued, else an SV_ERR_* code. */
int spec_verify(const sv_logits* target_logits, const sv_logits* draft_logits,
                const int32_t* draft_tokens, const int32_t* k_per_req,
                const float* temperature, const int32_t* top_k, const float* top_p,
                const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                void* stream, int32_t batch, void* workspace, size_t workspace_bytes,
                const sv_options* options);

/* Synchronises `stream`, then reads the first data error recorded by the last
 * call that used `workspace`: *code (SV_OK if none), *request and *row (-1
 * when not applicable).  Test / debug use. */
int spec_verify_get_error(const void* workspace, void* stream, int32_t* code,
                          int32_t* request, int64_t* row);

/* Synchronises `stream` and copies the per-row intermediate results of the
 * last call into host buffers (test / debug use).  Rows are numbered target
 * rows first (0 .. R_t-1), then draft rows (R_t .. R_t+R_d-1).
 *   stats      [R, 5] doubles: row max logit, softmax normaliser (sampling rows:
 *              sum of exp((x - max)/T) for unfiltered rows; the kept set's
 *              sum for rows filtered by top-p alone or a top-k above
 *              SV_TOPK_MAX; the kept weight for other filtered rows), p(x) of
 *              the row's draft token (NaN if none), greedy argmax (-1 if not
 *              computed), and the last kept token (in logit-descending,
 *              index-ascending order) of a row filtered by top-p alone or a
 *              top-k above SV_TOPK_MAX (-1 otherwise)
 *   kept_count [R] int32: size of the kept set after top-k / top-p (0 if the
 *              row was not filtered)
 *   kept_idx   [R, SV_TOPK_MAX] int32 and kept_p [R, SV_TOPK_MAX] doubles:
 *              the kept tokens in (logit desc, index asc) order and their
 *              renormalised probabilities, for rows whose top-k is active and
 *              at most SV_TOPK_MAX.  Those requests evaluate only the rows up
 *              to their first rejection (and the bonus row after k
 *              acceptances); other rows' entries are unspecified.
 * Any output pointer may be NULL. */
int spec_verify_dump_rows(const void* workspace, size_t workspace_bytes, int32_t batch,
                          int64_t target_rows, int64_t draft_rows, void* stream,
                          double* stats, int32_t* kept_count, int32_t* kept_idx,
                          double* kept_p);

/* ---- allocation-free variant ----------------------------------------------
 * The pages describe no counterpart of this entry point: it is a convenience of
 * this library for callers that cannot allocate device memory where they
 * verify (a C host program that links only this library and owns no device
 * allocator; a serving loop whose device memory is planned once and which must
 * not allocate inside its decode step).
 *
 * spec_verify_noalloc computes exactly what spec_verify computes, with the
 * same arguments minus the workspace: the workspace is a fixed buffer of
 * SV_NOALLOC_SCRATCH_BYTES inside the library (one per device).
 *   - A batch whose spec_verify_workspace_size exceeds SV_NOALLOC_SCRATCH_BYTES
 *     returns SV_ERR_WORKSPACE before anything is enqueued (16 MiB holds about
 *     1,400 logit rows, e.g. 32 requests with k = 15).
 *   - The buffer is shared: calls that can overlap on one device race on it.
 *     Order them on one stream or with events.
 *   - The buffer's address is looked up once per device, with that device
 *     current, on the first call; make that first call before any stream
 *     capture begins.
 *   - Nothing in the buffer has to start at zero.
 * Returns SV_OK once the work is enqueued, else an SV_ERR_* code. */
#define SV_NOALLOC_SCRATCH_BYTES (16u << 20)

int spec_verify_noalloc(const sv_logits* target_logits, const sv_logits* draft_logits,
                        const int32_t* draft_tokens, const int32_t* k_per_req,
                        const float* temperature, const int32_t* top_k, const float* top_p,
                        const float* uniforms, int32_t* out_accept_len, int32_t* out_tokens,
                        void* stream, int32_t batch, const sv_options* options);

/* Device address and size of the current device's spec_verify_noalloc buffer,
 * so that spec_verify_get_error / spec_verify_dump_rows can read the last
 * allocation-free call. */
int spec_verify_noalloc_scratch(void** scratch, size_t* bytes);

/* ---- draft-side sampler ---------------------------------------------------
 * The drafter's token choice that produces the drafts verified above
 * ("FlashMap: Flow Map Speculative Decoding…", §5 draft_block step 5: logits
 * divided by the temperature, softmax, a multinomial draw; the argmax at
 * temperature 0), for a batch of drafter rows laid out like spec_verify's
 * draft rows: request b owns rows d_off[b] .. d_off[b] + k_b - 1 with
 * d_off[b] = sum_{j<b} k_j.
 *   Row i of request b draws x_i = min{ y : C_y > u_i * S } by inverse CDF in
 *   vocabulary-index order over the row's distribution at the request's
 *   temperature, filtered by its top-k / top-p exactly as spec_verify filters
 *   p and q (so the q that verification recomputes is the one drawn from);
 *   temperature 0 takes the argmax of the raw logits, lowest index on ties.
 *   draft_logits  [R, V], R = sum_b k_b; same alignment rules as spec_verify
 *   k_per_req     [B] int32, 0 .. SV_MAX_K
 *   temperature   [B] float, 0 = greedy
 *   top_k, top_p  [B] or NULL, as in spec_verify
 *   uniforms      [R] float in [0, 1): row d_off[b] + i draws with u_i
 *   out_tokens    [R] int32: x_i; -1 for every row of a request with a data
 *                 error (bad parameters, NaN / +inf logit)
 *   out_q         [R] float or NULL: q_i(x_i), the drawn token's probability
 *                 (NaN for greedy and failed rows)
 *   workspace     >= spec_draft_sample_workspace_size(B, R) bytes, 256-byte
 *                 aligned, owned by the caller
 *   options       NULL, or row-pass events as in spec_verify (out_pq ignored)
 * Same ownership, stream and error conventions as spec_verify (errors are read
 * back with spec_verify_get_error on this workspace).  Returns SV_OK once the
 * work is enqueued, else an SV_ERR_* code. */
size_t spec_draft_sample_workspace_size(int32_t batch, int64_t rows);

int spec_draft_sample(const sv_logits* draft_logits, const int32_t* k_per_req,
                      const float* temperature, const int32_t* top_k, const float* top_p,
                      const float* uniforms, int32_t* out_tokens, float* out_q, void* stream,
                      int32_t batch, void* workspace, size_t workspace_bytes,
                      const sv_options* options);

/* ---- KV-cache commit after verification ------------------------------------
 * The verification stage of the serving pipeline updates the paged KV cache
 * with the accepted tokens ("FlashMap: Flow Map Speculative Decoding…",
 * section "Architecture"), and the rollback truncates on rejection
 * ("Speculative decoding and multi-token prediction", "Practical guidance").
 * The pages define no layout; this one is chosen:
 *   cache  [num_pages, n_layers, 2, page_size, E]  (K, then V), E elements of
 *          elem_bytes each per token per layer
 *   spec   [B, spec_slots, n_layers, 2, E]: the K/V the verification pass
 *          wrote for its k_b + 1 inputs, entry 0 the last emitted token (not in
 *          the cache yet), entries 1..k_b the drafts
 *   position p of request b lives in page block_table[b * max_pages + p /
 *   page_size] at slot p % page_size.
 * With accept length L = accept_len[b] >= 0 (spec_verify's output), entries
 * 0..L are written to positions kv_len[b] .. kv_len[b] + L and kv_len[b]
 * grows by L + 1; the entries of rejected drafts are not written.  L = -1 (a
 * request that failed verification) leaves the request untouched.  A request
 * with L > k_b (or L + 1 > spec_slots) fails with SV_ERR_DATA_ACCEPT, one
 * whose destination page is missing (entry < 0 or >= num_pages, or a column
 * past max_pages) or whose kv_len is negative with SV_ERR_DATA_PAGE: nothing
 * of a failed request is written and its kv_len is unchanged.  The first data
 * error is read back with spec_verify_get_error on this workspace.
 * E * elem_bytes must be a multiple of 16 and both base pointers 16-byte
 * aligned (SV_ERR_UNSUPPORTED otherwise).  All pointers are device pointers
 * owned by the caller; the call is asynchronous on `stream`. */
typedef struct {
  void* data;
  int64_t num_pages;
  int32_t n_layers;
  int32_t page_size;    /* tokens per page */
  int32_t entry_elems;  /* E */
  int32_t elem_bytes;   /* 2 or 4 */
} sv_kv_cache;

size_t spec_kv_commit_workspace_size(int32_t batch);

int spec_kv_commit(const sv_kv_cache* cache, const void* spec, int32_t spec_slots,
                   const int32_t* accept_len, const int32_t* k_per_req, int32_t* kv_len,
                   const int32_t* block_table, int32_t max_pages, void* stream, int32_t batch,
                   void* workspace, size_t workspace_bytes);

/* ---- LM-head GEMM with fused verification statistics ----------------------
 * The target's logits are its final hidden states times the unembedding
 * matrix, z = H W^T ("FlashMap: Flow Map Speculative Decoding…", section 1),
 * and verification needs of each logit row only its softmax statistics at the
 * row's temperature, its argmax and the logit of its token (§5 draft_block
 * step 5; §4).  spec_lmhead_stats computes them in the GEMM's epilogue on the
 * tensor cores (bf16 inputs, f32 accumulation), so the logits never reach
 * memory.  Per row r, with T_r = temperature[r] (1 is used when it is 0) and
 * x_r = tokens[r] (or -1):
 *   out_max[r]    = max_y z[r][y]                         (float)
 *   out_sum[r]    = sum_y exp((z[r][y] - out_max[r]) / T_r)  (double)
 *   out_argmax[r] = the first y with z[r][y] = out_max[r]
 *   out_token[r]  = z[r][x_r], NaN when x_r < 0 or tokens is NULL
 * so that p_r(x_r) = exp((out_token[r] - out_max[r]) / T_r) / out_sum[r].
 *   hidden   [rows, d] bf16, row-major, 16-byte aligned, d a multiple of 8
 *   unembed  [vocab, d] bf16, row-major, 16-byte aligned
 *   workspace >= spec_lmhead_stats_workspace_size(rows, vocab) bytes
 * All pointers are device pointers owned by the caller; asynchronous on
 * `stream`.  A bounded internal wait that expires is recorded as
 * SV_ERR_TIMEOUT (spec_verify_get_error on this workspace). */
size_t spec_lmhead_stats_workspace_size(int32_t rows, int32_t vocab);

int spec_lmhead_stats(const void* hidden, const void* unembed, int32_t rows, int32_t vocab,
                      int32_t d, const float* temperature, const int32_t* tokens,
                      float* out_max, double* out_sum, int32_t* out_argmax, float* out_token,
                      void* stream, void* workspace, size_t workspace_bytes);

/* ---- greedy verification from the target rows' argmax ----------------------
 * At temperature 0 verification needs of each target row only its argmax
 * (lowest index on ties): the longest prefix of drafts equal to it is accepted
 * and the argmax at the first disagreement, or after a full acceptance, is
 * emitted ("DFlash" §4 step 5; "Speculative decoding and multi-token
 * prediction", "Draft and verify", step Three).  Fed by spec_lmhead_stats'
 * out_argmax, a greedy request never needs its logits in memory.  Same row
 * layout as spec_verify:
 *   target_argmax  [R_t] int32, the argmax of target row t_off[b] + i
 *   draft_tokens   [R_d] int32 (R_d = R_t - B)    k_per_req [B] int32
 *   out_accept_len [B] int32 (L, or -1)           out_tokens [R_t] int32
 *   vocab          V: tokens and argmax values must lie in [0, V)
 *   workspace      >= spec_verify_greedy_workspace_size() bytes, 256-byte
 *                  aligned; spec_verify_get_error reads its error record
 * A k outside [0, SV_MAX_K] or sum(k + 1) != R_t fails the whole batch (all
 * outputs -1, SV_ERR_DATA_K / SV_ERR_DATA_ROWS); a token or argmax outside
 * [0, V) fails its request (SV_ERR_DATA_TOKEN).  Device pointers owned by the
 * caller; asynchronous on `stream`.  Returns SV_OK once enqueued. */
size_t spec_verify_greedy_workspace_size(void);

int spec_verify_greedy_from_argmax(const int32_t* target_argmax, const int32_t* draft_tokens,
                                   const int32_t* k_per_req, int32_t* out_accept_len,
                                   int32_t* out_tokens, void* stream, int32_t batch,
                                   int64_t target_rows, int32_t vocab, void* workspace,
                                   size_t workspace_bytes);

/* ---- adaptive speculation length -------------------------------------------
 * "Speculative decoding and multi-token prediction", section "Acceptance rate
 * is the whole economics": a drafted position beyond k is worth alpha^k tokens
 * for a draft step's cost c (a fraction of a target step), so speculation
 * pays while alpha^k stays above c; alpha varies per request and within a
 * response.  spec_adapt_k updates, per request, decayed counts of accepted
 * and rejected positions from the last pass's accept length and picks the next
 * k, on the stream right after spec_verify:
 *   succ[b] = decay * succ[b] + L_b,  fail[b] = decay * fail[b] + (L_b < k_b)
 *   alpha_b = (succ[b] + 1) / (succ[b] + fail[b] + 2)
 *   k_next[b] = the largest k in [k_min, k_max] with alpha_b^k > c, else k_min
 * A request with L_b = -1 keeps its counts and k_next[b] = k_used[b].
 *   accept_len, k_used [B] int32; succ, fail [B] double, in / out (start at 0);
 *   k_next [B] int32 out; alpha [B] float out or NULL.
 * 0 <= k_min <= k_max <= SV_MAX_K, 0 <= decay <= 1, c >= 0 (SV_ERR_ARG
 * otherwise).  Device pointers; asynchronous on `stream`. */
int spec_adapt_k(const int32_t* accept_len, const int32_t* k_used, double* succ, double* fail,
                 double decay, double c, int32_t k_min, int32_t k_max, int32_t* k_next,
                 float* alpha, void* stream, int32_t batch);

/* Human-readable text of a status code. */
const char* spec_verify_strerror(int code);

/* Library version, major * 10000 + minor * 100 + patch. */
int spec_verify_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
