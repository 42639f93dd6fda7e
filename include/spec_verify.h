/*
 * spec_verify.h -- C ABI of libspecverify, the batched verify step of greedy
 * (lossless) speculative decoding with an MTP / NextN draft head, for GB300
 * (sm_103a).
 *
 * One verify step, for B branches with k draft tokens each (R = B*(k+1) rows,
 * row r = b*(k+1)+j sits at position p = pos[b]+j):
 *
 *   spec_kv_append      write the k+1 new K/V rows of every branch in place
 *   spec_verify_attn    causal GQA attention of the R rows over their pages
 *   spec_lmhead_argmax  logits = hidden . W^T with a fused per-row argmax
 *   spec_accept         greedy chain acceptance
 *   spec_accept_stop    greedy chain acceptance with stop tokens and a generation budget
 *   spec_accept_sample  speculative sampling acceptance (random numbers as inputs)
 *   spec_verify_attn_tree, spec_accept_tree, spec_kv_compact   tree / star verify
 *   spec_h_gather, spec_h_scatter   the draft head's remembered hidden rows (slot pool)
 *   spec_mtp_input      the draft head's input  fc([rmsnorm(E[tok]), rmsnorm(h)])
 *
 * The method follows the span-02 page `engine/crates/model/src/spec.rs`
 * (module documentation and `Spec::body_inner`): draft chain, ONE batched
 * verify forward of B(k+1) rows with the KV appended in place at pos..pos+k,
 * greedy acceptance, and rollback by advancing `pos` only.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer named as "device" is a device pointer owned by the caller;
 *    the library never allocates, frees or retains one past the call.
 *    `spec_kv_desc` itself is a HOST struct that is read during the call only.
 *  - Every call is asynchronous and ordered on `stream` (a cudaStream_t; 0 is
 *    the legacy default stream). No call synchronises the device or the host.
 *  - Return value: SPEC_OK (0) or a negative SPEC_ERR_* code. Host-side
 *    argument errors are found before any launch, in which case nothing was
 *    enqueued. `spec_strerror` names a code. The library never prints and
 *    never aborts.
 *  - Device-side errors (a bad page id, a position the page table does not
 *    cover, a token id outside the vocabulary, a d2t entry outside the target
 *    vocabulary, a bounded wait that gave up) are reported through an
 *    optional `dev_err` device word: the kernel ORs a SPEC_DEVERR_* bit into
 *    it with an atomic and skips the offending write. It never traps. The
 *    caller zeroes the word and reads it at its own synchronisation point.
 *  - bf16 means IEEE bfloat16 stored as 2 bytes; all matrices are row-major.
 *
 * KV pool layout (one of each for K and V):
 *    pool[num_pages][n_kv_heads][page_size][head_dim]
 *  so that one (page, kv head) block of page_size*head_dim elements is one
 *  contiguous run. Element type: bf16 (kv_dtype 0) or FP8 E4M3 codes
 *  (kv_dtype 1, one byte each) with fp32 dequantisation scales
 *  scale[num_pages][n_kv_heads]; value = decode(code) * scale.
 *  The page table is int32 [B][max_pages]; position p of branch b lives in
 *  page page_table[b*max_pages + p/page_size], slot p % page_size
 *  (span-02 spec.rs, `SpecReq`: "its KV slot is page pages[pos/16]").
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that the header needs no CUDA include. */
typedef struct CUstream_st *spec_stream_t;

/* ---- status codes --------------------------------------------------------------- */
#define SPEC_OK               0
#define SPEC_ERR_NULL        -1  /* a required pointer is NULL                           */
#define SPEC_ERR_ARG         -2  /* a size or count is out of range                      */
#define SPEC_ERR_UNSUPPORTED -3  /* valid but not implemented (e.g. head_dim 96)         */
#define SPEC_ERR_WORKSPACE   -4  /* workspace pointer NULL or smaller than required     */
#define SPEC_ERR_CUDA        -5  /* a CUDA runtime call failed (launch, attribute, ...)  */
#define SPEC_ERR_ALIGN       -6  /* a pointer or row stride breaks a 16-byte alignment  */

/* ---- device error bits (OR-ed into *dev_err) ------------------------------------- */
#define SPEC_DEVERR_PAGE     1   /* page id outside [0, num_pages)                      */
#define SPEC_DEVERR_COVER    2   /* position p with p/page_size >= max_pages            */
#define SPEC_DEVERR_TOKEN    4   /* token id outside [0, V)                             */
#define SPEC_DEVERR_D2T      8   /* d2t entry outside [0, d2t_limit)                    */
#define SPEC_DEVERR_POS      16  /* pos[b] < 0, or pos[b]+k+1 > max_pos                 */
#define SPEC_DEVERR_TIMEOUT  32  /* a bounded pipeline wait gave up (results invalid)   */
#define SPEC_DEVERR_INTERNAL 64  /* an internal consistency check failed; the access was skipped */
#define SPEC_DEVERR_TREE     128 /* a tree parent outside [0, row) or a path entry out of order */
#define SPEC_DEVERR_SLOT     256 /* a hidden-pool slot outside [0, n_slots)             */

/* ---- limits ------------------------------------------------------------------------ */
#define SPEC_KMAX            15  /* k <= 15: at most 16 verify rows per branch          */
#define SPEC_KV_BF16         0
#define SPEC_KV_FP8_E4M3     1

/* Paged KV pool shared by all branches (span-02 spec.rs, module documentation: the
 * branches verify "over the branches' own pages" of the scheduler's SHARED pool). */
typedef struct {
    void *k_pool;              /* device, [num_pages][n_kv_heads][page_size][head_dim]   */
    void *v_pool;              /* device, same layout                                    */
    const float *k_scale;      /* device, [num_pages][n_kv_heads] fp32; FP8 only else NULL */
    const float *v_scale;      /* device, same                                           */
    const int32_t *page_table; /* device, [B][max_pages] page ids (unused entries: -1)    */
    int32_t num_pages;         /* pages in the pool                                      */
    int32_t max_pages;         /* page-table row width                                   */
    int32_t page_size;         /* slots per page: a power of two, 1..1024                */
    int32_t n_kv_heads;        /* Hkv >= 1                                                */
    int32_t head_dim;          /* d in {64, 128, 256}                                     */
    int32_t kv_dtype;          /* SPEC_KV_BF16 or SPEC_KV_FP8_E4M3                         */
} spec_kv_desc;

/* Name of a status code (static string, never NULL). */
const char *spec_strerror(int status);

/* Library ABI version (major*100 + minor). */
int spec_version(void);

/* ---- a1: KV append ----------------------------------------------------------------
 * Writes, for every branch b and j = 0..k, the new K/V row of verify row
 * r = b*(k+1)+j into position p = pos[b]+j of branch b's pages.
 * Source: span-02 spec.rs, module documentation ("KV appended in place at
 * pos..pos+k"); memra-engine spec.rs, `full_attn_verify` (append of the T
 * verify tokens before the attention).
 *   pos     device int32 [B]: position of each branch's first verify row, i.e.
 *           the number of committed tokens already in the pool.
 *   k_new,
 *   v_new   device bf16 [B*(k+1)][n_kv_heads][head_dim], 16-byte aligned.
 * bf16 pools: a bit copy. FP8 pools: code = e4m3_rn_satfinite(float(x) / scale)
 * with an IEEE fp32 division and the page's (page, kv head) scale.
 * Host errors: NULL pointers, B < 1, k outside [0, SPEC_KMAX], bad descriptor.
 * Device errors: SPEC_DEVERR_PAGE, SPEC_DEVERR_COVER, SPEC_DEVERR_POS (pos < 0);
 * the offending row is skipped. dev_err may be NULL (errors then go unreported). */
int spec_kv_append(const spec_kv_desc *kv, const int32_t *pos, int B, int k,
                   const void *k_new, const void *v_new, int32_t *dev_err,
                   spec_stream_t stream);

/* General form of the append: n_rows rows, row i goes to branch row_branch[i]
 * (a page-table row) at position row_pos[i]. Used to fill a context (prefill
 * writes its KV the same way) and by spec_kv_append.
 *   row_branch, row_pos  device int32 [n_rows]
 *   k_rows, v_rows       device bf16 [n_rows][n_kv_heads][head_dim]
 * Errors as spec_kv_append. n_rows == 0 is a no-op. */
int spec_kv_write_rows(const spec_kv_desc *kv, const int32_t *row_branch,
                       const int32_t *row_pos, int n_rows, const void *k_rows,
                       const void *v_rows, int32_t *dev_err, spec_stream_t stream);

/* Diagnostic (no GPU needed, nothing launched): the launch plan spec_verify_attn would
 * use for these shapes. Only the descriptor's shape fields are read (its pointers are not
 * looked at). out[0..16] = dynamic shared memory bytes, query vectors per (branch, kv head)
 * padded to 16 (the MMAs' N), K ring stages (bf16 K, or E4M3 K), V ring stages (bf16 V;
 * on FP8 pools the converted V), raw V ring stages (FP8 only: E4M3 V as loaded), S buffers,
 * P buffers, Q buffers, O buffers, TMEM columns used, split size in positions, splits per
 * branch, work units, tiles of 128 keys per softmax step, FP8 TMA box rows (0 = bf16
 * gather), barrier bytes used, barrier bytes reserved. Returns the status the host checks
 * and the planning of spec_verify_attn would give (n_out < SPEC_ATTN_PLAN_FIELDS:
 * SPEC_ERR_ARG). */
#define SPEC_ATTN_PLAN_FIELDS 17
int spec_verify_attn_plan(const spec_kv_desc *kv, int B, int k, int n_q_heads, int max_pos,
                          int32_t *out, int n_out);

/* ---- a2: verify attention ---------------------------------------------------------
 * For every row r = b*(k+1)+j (position p = pos[b]+j) and q head h (kv head
 * g = h / (n_q_heads / n_kv_heads)):
 *     out[r][h] = sum_{t=0..p} softmax_t(scale * q[r][h] . K_t) * V_t
 * over branch b's keys 0..p inclusive (kv_hi = the row's position), never a
 * slot beyond p. Sources: span-02 spec.rs, module documentation ("never
 * attended: kv_hi = position"); memra-engine spec.rs, `full_attn_verify`
 * ("query row r attends to keys [0..base_len+r+1)"); DSSD-dev fast.py,
 * `_attention` (per-row exact key path).
 * Split-KV: keys are cut into fixed splits of 256 positions (n_kv_heads <= 2),
 * 512 (n_kv_heads <= 4), else 1024 (bf16) or 2048 (E4M3): a function of the pool's shape
 * only, independent of B, k and context, so a row's output is byte-identical
 * whatever batch it is verified in (memra-engine spec.rs, `MtpScratch`: fixed
 * split geometry). The splits are merged inside the same launch.
 *   q       device bf16 [B*(k+1)][n_q_heads][head_dim], finite values. On FP8 pools each
 *           query vector is scaled by a power of two and split into two E4M3 terms, exact
 *           for every element within 2^10 of the vector's largest (any finite magnitude).
 *   out     device bf16 [B*(k+1)][n_q_heads][head_dim]
 *   scale   softmax scale (normally 1/sqrt(head_dim))
 *   max_pos host bound: pos[b]+k+1 <= max_pos for every b (sizes the grid and
 *           the workspace; rows beyond it are a device error SPEC_DEVERR_POS).
 *   ws      device workspace of spec_verify_attn_workspace(...) bytes, 256-byte
 *           aligned, ZERO-filled before its first call. Every call that completes leaves
 *           the parts that must start at zero (the scheduler and merge counters) at zero
 *           again, so a workspace is zeroed once, not per call; after a call that reported
 *           SPEC_DEVERR_TIMEOUT, zero it again. Calls sharing a workspace must not overlap
 *           in time.
 * Host errors: NULL, B < 1, k out of range, n_q_heads % n_kv_heads != 0,
 * head_dim not 64/128/256, max_pos < k+1, workspace too small; SPEC_ERR_UNSUPPORTED
 * when (k+1)*G, the query vectors sharing one kv head, exceeds 128, when FP8 pages hold
 * fewer than 8 positions, or when no shared-memory / TMEM plan fits the shapes
 * (spec_verify_attn_plan tells which).
 * Device errors: as spec_kv_append (the row's output is then left unwritten). */
size_t spec_verify_attn_workspace(const spec_kv_desc *kv, int B, int k, int n_q_heads,
                                  int max_pos);
int spec_verify_attn(const spec_kv_desc *kv, const int32_t *pos, int B, int k,
                     int n_q_heads, const void *q, float scale, void *out,
                     void *ws, size_t ws_bytes, int max_pos, int32_t *dev_err,
                     spec_stream_t stream);

/* ---- f2: tree / star verify attention --------------------------------------------
 * The verify rows of branch b own the slots pos_b .. pos_b+k (row j is written at slot
 * pos_b + j by spec_kv_append); row j attends to every committed position (< pos_b) and to
 * the slot pos_b + i exactly when bit i of anc_mask[b*(k+1)+j] is set (its ancestors in the
 * draft tree and itself). A chain is the mask with bits 0..j (then the result is that of
 * spec_verify_attn, bit for bit). Sources: DSSD-dev `_set_rows` / `_star_cycle` (a tree row
 * reads the contiguous committed prefix and then the slots of its own path).
 *   anc_mask  device int32 [B*(k+1)]; the other arguments, the workspace, the launch plan
 *             and the errors are those of spec_verify_attn.
 * Device errors: also SPEC_DEVERR_TREE for a row j whose mask lacks bit j or has a bit above
 * j (a tree row sees itself and only earlier rows); that row's output is left unwritten. */
int spec_verify_attn_tree(const spec_kv_desc *kv, const int32_t *pos, int B, int k,
                          int n_q_heads, const void *q, float scale, const int32_t *anc_mask,
                          void *out, void *ws, size_t ws_bytes, int max_pos, int32_t *dev_err,
                          spec_stream_t stream);

/* ---- a3: LM head with fused argmax ------------------------------------------------
 *   logit[m][v] = sum_h hidden[m][h] * W[v][h]   (fp32 accumulation)
 *   ids[m]      = the lowest v attaining max_v logit[m][v]; with d2t, d2t[that v]
 * The logits never reach global memory. W is streamed once per call for all
 * M rows. Sources: span-02 spec.rs, `Spec::body_inner` (`lm_head_argmax`) and
 * `greedy_logprob` (first maximum wins); flashrt-structures whole_step.py,
 * `generate_speculative` (argmax of the fp32 logits).
 *   hidden  device bf16 [M][H];  W  device bf16 [V][H];  16-byte aligned, H % 8 == 0
 *   d2t     device int32 [V] or NULL: trimmed draft vocabulary -> target id
 *           (oxinfer qwen_mtp.rs, module documentation of the trimmed head)
 *   d2t_limit  target vocabulary size; a d2t entry outside [0, d2t_limit) is
 *           SPEC_DEVERR_D2T and that row's id is written as -1.
 *   ids     device int32 [M];  max_logit  device fp32 [M] or NULL
 *   ws      device workspace of spec_lmhead_workspace(M, V, H) bytes. Its first
 *           256 bytes must be ZERO before the first call; every call leaves
 *           them zero again, so a workspace is zeroed once, not per call.
 *           Calls that share one workspace must not overlap on the GPU.
 * Limits: 1 <= M <= 256, V >= 1, H >= 8.  */
size_t spec_lmhead_workspace(int M, int V, int H);
int spec_lmhead_argmax(const void *hidden, const void *W, int M, int V, int H,
                       const int32_t *d2t, int d2t_limit, int32_t *ids, float *max_logit,
                       void *ws, size_t ws_bytes, int32_t *dev_err, spec_stream_t stream);

/* Test hook: the same kernel, K order and accumulators as spec_lmhead_argmax, which
 * also stores the fp32 logits [M][V] (row-invariance checks). Same workspace rules. */
int spec_lmhead_logits(const void *hidden, const void *W, int M, int V, int H,
                       float *logits, int32_t *ids, void *ws, size_t ws_bytes,
                       spec_stream_t stream);

/* ---- a3 without a workspace ---------------------------------------------------------
 * The source pages have no counterpart of this entry point. It computes exactly what
 * spec_lmhead_argmax computes (same kernel, same ids and max_logit) for callers that
 * cannot allocate device memory, e.g. an engine that gives its whole HBM budget to its own
 * pool up front, or glue code that can only pass the call's tensors. The kernel's scratch
 * (a launch counter and the per-CTA argmax keys) is a library-owned device array of
 * SPEC_LMHEAD_STATIC_SCRATCH_BYTES bytes per device; no memory is allocated or freed.
 *   arguments as spec_lmhead_argmax, without ws / ws_bytes.
 * Limits: the call's spec_lmhead_workspace(M, V, H) must not exceed
 * SPEC_LMHEAD_STATIC_SCRATCH_BYTES (always true for M <= 64); otherwise SPEC_ERR_WORKSPACE
 * and nothing is launched.
 * Set-up: the first call on a device (the current device) looks the array up and zeroes
 * its counter with a synchronous cudaMemset; make that first call before any stream
 * capture. Every completed call leaves the counter zero again.
 * Concurrency: all calls on a device share the one array; calls that may be in flight at
 * the same time race on it and may return wrong ids: order them on one stream or with
 * events. */
#define SPEC_LMHEAD_STATIC_SCRATCH_BYTES ((size_t)256 + (size_t)1024 * 64 * 8)
int spec_lmhead_argmax_static(const void *hidden, const void *W, int M, int V, int H,
                              const int32_t *d2t, int d2t_limit, int32_t *ids,
                              float *max_logit, int32_t *dev_err, spec_stream_t stream);

/* ---- a4: greedy chain acceptance --------------------------------------------------
 * Per branch b, with target ids g_j = ids[b*(k+1)+j]:
 *   a = the largest a <= k with drafts[b][i] == g_i for every i < a
 *   emitted = drafts[b][0..a) followed by the bonus token g_a;  n = a+1
 *   new pos = pos[b] + a + 1 (rollback is the position advance alone)
 * Sources: span-02 spec.rs, module documentation ("a token is emitted only if it
 * equals the target's argmax at the verify row before it"); DSSD-dev fast.py,
 * `generate_spec` (accept loop then correction/bonus token); flashrt-structures
 * whole_step.py, `generate_speculative` (device-side prefix match).
 *   drafts      device int32 [B][k]  (may be NULL when k == 0)
 *   ids         device int32 [B*(k+1)]
 *   pos         device int32 [B]
 *   out_tokens  device int32 [B][k+1]: the n emitted tokens, then -1
 *   out_n, out_accepted, out_pos, out_next   device int32 [B] (out_next = bonus)
 *   out_pos may be pos itself: the positions then advance in place, and a decode loop
 *   captured in a CUDA graph keeps its step state (positions, next fed token in out_next,
 *   the draft head's hidden row in h_out) on the device across replays. The same holds
 *   for spec_accept_stop.
 *   hidden, H, h_out   optional (all three or none): h_out[b][:] =
 *       hidden[b*(k+1)+a][:], bf16 [B][H], the target hidden state of the row that
 *       produced the bonus token -- the next draft step's h (span-02 spec.rs,
 *       `Spec::body_inner`, `spec_accept` writing h0).
 * Host errors: NULL, B < 1, k out of range. */
int spec_accept(const int32_t *drafts, const int32_t *ids, const int32_t *pos, int B,
                int k, int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted,
                int32_t *out_pos, int32_t *out_next, const void *hidden, int H,
                void *h_out, spec_stream_t stream);

/* ---- a4 with stop tokens and a generation budget ------------------------------------
 * The greedy run of branch b (drafts[b][0..a) followed by g_a) is cut right after its
 * first token that is in the stop set, then to at most budget[b] tokens:
 *   n = min(first stop index + 1 (or a+1 without one), max(budget[b], 0))
 *   emitted = the first n run tokens;  accepted = min(a, n);  new pos = pos[b] + n
 *   next = the last emitted token (-1 when n == 0)
 *   done = the emitted run ends on a stop token, or n reached budget[b]
 * With no stop ids and no budget it returns exactly what spec_accept returns.
 * Sources: DSSD-dev dssd/fast.py, `_commit` (a cycle's committed tokens are appended until
 * the stop rule fires on one, which is kept, or the output reaches the generation limit);
 * span-02 engine/crates/model/src/spec.rs, `Spec::body_inner` (the device acceptance call
 * takes a stop-id buffer whose unused entries are -1, and a token limit).
 *   stop_ids   device int32 [n_stop] (entries < 0 are unused); NULL when n_stop == 0;
 *              0 <= n_stop <= SPEC_MAX_STOP
 *   budget     device int32 [B]: tokens branch b may still emit, or NULL (no limit)
 *   out_done   device int32 [B] (0/1), or NULL
 *   the other arguments are those of spec_accept; h_out[b] is the hidden row of the
 *   last emitted token (row b*(k+1) + n-1) and is left unwritten when n == 0.
 * Host errors: those of spec_accept; n_stop out of range; n_stop > 0 with NULL stop_ids. */
#define SPEC_MAX_STOP 32
int spec_accept_stop(const int32_t *drafts, const int32_t *ids, const int32_t *pos, int B,
                     int k, const int32_t *stop_ids, int n_stop, const int32_t *budget,
                     int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted,
                     int32_t *out_pos, int32_t *out_next, int32_t *out_done,
                     const void *hidden, int H, void *h_out, spec_stream_t stream);

/* ---- f2: greedy tree walk and KV compaction --------------------------------------
 * spec_accept_tree: per branch, rows 0..k form a tree (parent[b*(k+1)+j] < j for j >= 1;
 * row 0 the root). From the root, repeatedly move to the first child c (in row order) with
 * drafts[b][c-1] == ids[b*(k+1)+cur]; emitted = the drafts of the walked rows, then the
 * target of the last row (the bonus); n = a+1 with a the rows walked; new pos = pos[b]+a+1;
 * out_path[b][0] = 0, out_path[b][i] = the i-th walked row, then -1. With parent[j] = j-1 it
 * is spec_accept. out_pos may be pos.
 * spec_kv_compact: after the walk, row out_path[b][i] (written at slot pos_b + out_path[b][i])
 * is moved to slot pos_b + i for i = 1..accepted[b] (pos = the position before the step),
 * in ascending i; bf16 pools copy the bits, FP8 pools decode with the source page's scale
 * and re-encode (round to nearest even, saturating) with the destination page's.
 * Sources: DSSD-dev `_star_cycle` (walk the star / tree, copy the accepted child's K/V to
 * slot pos0 + 1).
 * Host errors: NULL, B < 1, k out of range, bad descriptor. Device errors: SPEC_DEVERR_TREE
 * for a parent outside [0, j) (that row is never walked to) or a path entry out of order
 * (that move is skipped); the page errors of spec_kv_append. */
int spec_accept_tree(const int32_t *drafts, const int32_t *ids, const int32_t *pos,
                     const int32_t *parent, int B, int k, int32_t *out_tokens, int32_t *out_n,
                     int32_t *out_accepted, int32_t *out_pos, int32_t *out_next, int32_t *out_path,
                     int32_t *dev_err, spec_stream_t stream);
int spec_kv_compact(const spec_kv_desc *kv, const int32_t *pos, const int32_t *path,
                    const int32_t *accepted, int B, int k, int32_t *dev_err, spec_stream_t stream);

/* ---- f4: speculative sampling acceptance ------------------------------------------
 * Per branch b, rows j = 0..k with p_j = softmax(logits[b*(k+1)+j] / temperature):
 *   draft i (drafts[b][i], drawn by the draft model from q[b][i]) is kept when
 *   p_i(d) >= q_i(d) or u_acc[b][i] < p_i(d) / q_i(d); the walk stops at the first draft
 *   not kept (a = its index), whose replacement is drawn from max(0, p_a - q_a)
 *   normalised (from p_a when that is all zero); after a full acceptance (a = k) the bonus
 *   token is drawn from p_k. A draw from weights w takes the smallest index t whose running
 *   sum (in index order) exceeds u_res[b] * sum(w).
 *   emitted = drafts[b][0..a) followed by the drawn token; n = a+1; new pos = pos[b]+a+1.
 * Sources: oxinfer `speculative_accept` (keep with probability min(1, p/q), else resample
 * from the normalised positive part of p - q); DSSD-dev `_sample_verify` (stop at the first
 * rejection; the bonus from the last row after a full acceptance). The random numbers are
 * inputs, uniform in [0, 1).
 *   drafts   device int32 [B][k];  logits  device fp32 [B*(k+1)][V];  q  device fp32 [B][k][V]
 *            (probabilities);  u_acc  device fp32 [B][k];  u_res  device fp32 [B]
 *   out_*    as spec_accept (out_pos may be pos);  temperature > 0
 *   workspace  device scratch of spec_accept_sample_workspace(B, k, V) bytes, 16-byte
 *            aligned (per row and chunk of the vocabulary: the softmax statistics; per
 *            branch: the draw weights' chunk sums and a counter). Zero it before its first
 *            use; every call leaves it zeroed again. Calls sharing one must not overlap.
 * Every verify row's softmax statistics are computed (all rows at once, spread over the
 * GPU), then the walk and the draw; rows past the first rejection are read but unused.
 * Precision: probabilities in fp32 (exp2); sums as double-floats (pairs of fp32 values,
 * about 48 significant bits, from compensated fp32 partial sums), each in a fixed order, so
 * results are deterministic. A decision can differ from an exact evaluation only when its
 * test value lies within that rounding (about 2^-24 relative) of the boundary.
 * Host errors: NULL, B < 1, k out of range, V < 1 or V >= 2^24, temperature not positive
 * and finite, SPEC_ERR_WORKSPACE (NULL or too small), SPEC_ERR_ALIGN (workspace).
 * Device errors: SPEC_DEVERR_TOKEN for a draft outside [0, V) or with q_i(d) <= 0 (not a
 * sample of q) that the walk reaches: that draft is treated as rejected. */
size_t spec_accept_sample_workspace(int B, int k, int V); /* 0 for invalid sizes */
int spec_accept_sample(const int32_t *drafts, const float *logits, const float *q, const int32_t *pos, int B,
                       int k, int V, float temperature, const float *u_acc, const float *u_res,
                       int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted, int32_t *out_pos,
                       int32_t *out_next, void *workspace, size_t ws_bytes, int32_t *dev_err,
                       spec_stream_t stream);

/* ---- f1: the draft head's remembered hidden rows ----------------------------------
 * Each branch b owns slot hslot[b] of a pool of hidden rows. A step gathers the draft
 * head's input rows h[b] = hpool[hslot[b]] before drafting, and scatters the rows the
 * acceptance wrote (spec_accept's h_out) back, hpool[hslot[b]] = h[b], after it. Sources:
 * span-02 engine/crates/model/src/spec.rs, `Spec::body_inner` (`spec_h_gather` at the start
 * of a step, `spec_h_scatter` at its end).
 *   hpool  device bf16 [n_slots][H];  hslot  device int32 [B];  h_out / h_in  device bf16
 *          [B][H] (16-byte aligned rows with H % 8 == 0 copy by 16-byte vectors)
 *   spec_h_scatter: slots must be distinct (with a repeated slot, which row lands there is
 *   unspecified).
 * Host errors: NULL, B < 1, H < 1, n_slots < 1.
 * Device errors: SPEC_DEVERR_SLOT for a slot outside [0, n_slots); that row is skipped. */
int spec_h_gather(void *h_out, const void *hpool, const int32_t *hslot, int B, int H, int n_slots,
                  int32_t *dev_err, spec_stream_t stream);
int spec_h_scatter(void *hpool, const void *h_in, const int32_t *hslot, int B, int H, int n_slots,
                   int32_t *dev_err, spec_stream_t stream);

/* ---- a5: MTP draft-head input -----------------------------------------------------
 *   c[m]  = [ rmsnorm(E[tok[m]]; g_emb) ; rmsnorm(h[m]; g_hid) ]  rounded to bf16
 *   x[m]  = W_fc . c[m]   (fp32 accumulation, stored as bf16)
 *   rmsnorm(y; g)_i = y_i / sqrt(mean_j y_j^2 + eps) * g_i   (fp32)
 * Source: oxinfer qwen_mtp.rs, module documentation (x = fc([rmsnorm_emb(embed
 * (x_{i+1})), rmsnorm_hidden(h_i)]), fc: [H, 2H], embedding first).
 *   tok    device int32 [M];  E  device bf16 [V][H];  h  device bf16 [M][H]
 *   g_emb, g_hid  device fp32 [H];  W_fc  device bf16 [H][2H];  x_out  device bf16 [M][H]
 *   ws     device workspace of spec_mtp_input_workspace(M, H) bytes; its first 256
 *          bytes follow the same zero rule as spec_lmhead_workspace.
 * Limits: 1 <= M <= 256, H % 64 == 0; E, h, g_emb, g_hid, W_fc and x_out 16-byte
 * aligned (SPEC_ERR_ALIGN otherwise). Device error SPEC_DEVERR_TOKEN for tok[m]
 * outside [0, V) (that row's c is written as zeros). */
size_t spec_mtp_input_workspace(int M, int H);
int spec_mtp_input(const int32_t *tok, const void *E, const void *h, const float *g_emb,
                   const float *g_hid, float eps, const void *W_fc, int M, int H, int V,
                   void *x_out, void *ws, size_t ws_bytes, int32_t *dev_err,
                   spec_stream_t stream);

/* ---- test hook: bounded waits ---------------------------------------------------------
 * The source pages have no counterpart of this entry point. Every wait inside the
 * tcgen05 kernels (spec_verify_attn, spec_lmhead_argmax, spec_lmhead_logits,
 * spec_lmhead_argmax_static and the fc of spec_mtp_input) gives up after a time limit,
 * normally one second, and the kernel then reports SPEC_DEVERR_TIMEOUT, lets the copies and
 * MMAs it has issued land, frees its tensor memory and returns. This sets that limit, in
 * nanoseconds, for the launches made after the call (0 restores one second), so that a test
 * can make a wait run out on purpose and check that the error is reported and the context
 * stays usable. The waits that drain a kernel's own copies before it exits keep the full
 * second. Process-wide; not synchronised with launches from other threads. */
void spec_test_set_wait_limit(uint64_t ns);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
