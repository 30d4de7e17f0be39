/*
 * kap.h - C ABI of the selected-KV sparse decode hot path (GB300, sm_103a).
 *
 * The operations follow the runtime access plan A = (U, M, pos, rho_access, rho_verify) of
 * "KAP: Bridging the Knowledge Selection-Runtime Consumption Gap in LLM Systems" (the arXiv paper and
 * its agifrontier.github.io tutorial, section on the runtime access plan):
 *   U           - units: KV pages (16 tokens) or token spans,
 *   M           - page map: block table from logical page to physical page, plus lengths,
 *   pos         - logical positions, kept on both the proposal and the verification path,
 *   rho_access  - sparse-access policy: the A<a>R<r>K<k> split of the KRI page (knlp.io, "The A<a>R<r>K<k> tag"),
 *   rho_verify  - verification policy: the short causal query window of the full-context verifier.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument named *_dev, and every pointer inside the structs below, is DEVICE memory owned by
 *     the caller. The library never allocates, frees or synchronises on these calls; all launches go to `stream`
 *     (NULL = the legacy default stream), so the calls that take their workspace from the caller can be captured
 *     in a CUDA graph.
 *   - KV pool layout: K and V are separate arrays [num_pages][num_kv_heads][16][head_dim] of the pool dtype.
 *     One (page, head) chunk is 16*head_dim*elem bytes and contiguous.
 *   - Query head hq reads KV head hq / (num_q_heads / num_kv_heads) (grouped-query attention).
 *   - Attention logits are (q . k) / sqrt(head_dim); lse is the natural-log log-sum-exp of those logits (fp32).
 *   - K in the pool is post-RoPE; queries passed to attention are post-RoPE at their logical positions.
 *   - Errors are returned as kap_status; nothing is thrown across the ABI. Host-side argument checks always run.
 *     Kernels that meet an inconsistent device-side value (a page id outside the pool, a selection larger than its
 *     capacity) skip that access and record a code readable with kap_device_error().
 */
#ifndef KAP_H
#define KAP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *kap_stream; /* same type as cudaStream_t */

typedef enum {
  KAP_OK = 0,
  KAP_FALLBACK_FULL = 1,   /* plan infeasible for selected access: use full-context attention (KAP paper, fallback) */
  KAP_EINVAL = -1,         /* a NULL pointer, a negative size, or an out-of-range scalar */
  KAP_ESHAPE = -2,         /* shapes that are inconsistent with one another */
  KAP_ECAPACITY = -3,      /* a caller buffer (capacity, workspace) is too small */
  KAP_ECUDA = -4,          /* a CUDA runtime call failed; see kap_last_cuda_error() */
  KAP_EUNSUPPORTED = -5    /* a shape this build has no kernel for (head_dim, group size, dtype) */
} kap_status;

typedef enum { KAP_BF16 = 0, KAP_F32 = 1 } kap_dtype;

/* Paged KV pool. All pointers are device memory owned by the caller. */
typedef struct {
  int32_t num_pages;    /* physical pages in the pool */
  int32_t page_size;    /* tokens per page; must be 16 */
  int32_t num_kv_heads; /* Hkv */
  int32_t num_q_heads;  /* Hq, a multiple of Hkv; G = Hq / Hkv in 1..8 */
  int32_t head_dim;     /* d: 64 or 128 */
  int32_t dtype;        /* kap_dtype of K, V, queries and attention outputs */
  void *k_pages;        /* [num_pages][Hkv][16][d] post-RoPE keys */
  void *v_pages;        /* [num_pages][Hkv][16][d] values */
  float *k_summary;     /* [num_pages][Hkv][d] fp32 block-mean keys (K-summary cache); may be NULL if unused */
} kap_kv_pool;

/* Page map M and lengths. Logical page j of request r covers positions 16j .. 16j+15. */
typedef struct {
  int32_t num_seqs;           /* R */
  int32_t max_pages;          /* row stride of block_table */
  const int32_t *block_table; /* [R][max_pages] physical page of each logical page */
  const int32_t *ctx_len;     /* [R] prompt tokens: positions < ctx_len are the selectable prompt */
  const int32_t *seq_len;     /* [R] tokens present (prompt + generated); a decode query sits at seq_len-1 */
} kap_page_map;

/* rho_access: the A<a>R<r>K<k> split. Prompt pages [0,a) and the last r prompt pages are pinned; k more pages
 * are chosen from the middle by score (ties to the lower page id). */
typedef struct {
  int32_t anchor, recent, topk;  /* a, r, k used for every request when per_seq_ark is NULL */
  int32_t per_kv_head;           /* 1: one selection per KV head; 0: one selection shared by all heads */
  int32_t cap;                   /* capacity of one selection row (entries) */
  const int32_t *per_seq_ark;    /* optional device [R][3] = (a, r, k) per request; overrides the scalars */
} kap_access_policy;

/* Compact selected-KV view, written by kap_compile_view and read by kap_attn_propose.
 * Row (r, v) with v < rows_per_seq lists the visible pages of request r for KV head v (or for all heads when
 * rows_per_seq == 1): first the n_selected selected prompt pages in ascending logical order (the order in which
 * they are accessed), then the tail pages holding positions >= ctx_len, up to the horizon given at compile time. */
typedef struct {
  int32_t rows_per_seq;   /* Hkv (per-head views) or 1 (one view shared by all heads) */
  int32_t cap;            /* entries per row */
  int32_t *block_table;   /* [R][rows_per_seq][cap] physical page of each entry */
  int32_t *logical_page;  /* [R][rows_per_seq][cap] logical page of each entry (keeps logical positions) */
  int32_t *n_entries;     /* [R][rows_per_seq] entries in use */
  int32_t *n_selected;    /* [R][rows_per_seq] leading entries that are selected prompt pages */
  /* Read by kap_attn_propose and kap_append_propose only; ignored (and left unchanged) by the calls that write a
   * view. Nonzero is the caller's promise that this view, the page map, the prompt tokens of the pool
   * (positions < ctx_len) and the rotary frequencies were last written before the kernel launched just ahead of
   * the call on the same stream. The call may then read them, and start streaming the selected prompt pages, while that kernel is
   * still finishing; it waits for it before reading anything else or writing anything. Zero: the call waits for
   * the previous kernel before its first memory access. The promise does not hold for a call that directly
   * follows the kernel that wrote the view. */
  int32_t settled;
} kap_view;

/* rho_verify: the verification window. Request r owns query rows q_offsets[r] .. q_offsets[r+1]-1; row i of
 * request r sits at logical position q_start_pos[r] + i and sees every position <= its own (full context,
 * causal among the candidates). */
typedef struct {
  int32_t max_q;              /* upper bound on q_offsets[r+1]-q_offsets[r]; G*max_q <= 64 */
  int32_t total_q;            /* q_offsets[R] */
  const int32_t *q_offsets;   /* [R+1] */
  const int32_t *q_start_pos; /* [R] */
} kap_verify_policy;

/* ---------------------------------------------------------------------------------------------------------
 * K-summary cache. EarlySelectKV page (routing over a K-summary cache) and the KRI page's KRI-Q row
 * (block-mean K). For every request r and prompt page j < ceil(ctx_len[r]/16), with n = min(16, ctx_len-16j)
 * valid tokens: k_summary[page][h][i] = (sum over t < n of K[page][h][t][i], fp32, t ascending) / n.
 * Requires pool->k_summary. Pages shared between requests must agree on n. */
kap_status kap_build_summaries(const kap_kv_pool *pool, const kap_page_map *map, kap_stream stream);

/* Refresh of the K summaries of listed pages: for each i < num_listed, the physical page pages_dev[i] with
 * n = n_valid_dev[i] valid tokens (1 <= n <= 16) gets k_summary[page][h][:] = (sum over t < n of K[page][h][t][:],
 * fp32, t ascending) / n, the same arithmetic as kap_build_summaries, so a refreshed page equals a full rebuild bit
 * for bit. EarlySelectKV page: routing scores pages against a K-summary cache held beside the KV pool; the page
 * does not say when that cache is updated. Here it changes only when committed tokens enter the prompt (ctx_len
 * grows): list the partial last prompt page and any new prompt pages; a full rebuild would re-read every prompt
 * page. Appends of generated tokens need no refresh, since summaries cover prompt tokens only. Listed pages must be
 * distinct (two CTAs would write one summary).
 *   pages_dev, n_valid_dev [num_listed] int32, device.
 * Errors: KAP_EINVAL for a null pointer or num_listed < 0; the pool checks of kap_build_summaries. A page outside the
 * pool or a count outside [1, 16] is skipped on the device and reported through kap_device_error. */
kap_status kap_refresh_summaries(const kap_kv_pool *pool, const int32_t *pages_dev, const int32_t *n_valid_dev,
                                 int32_t num_listed, kap_stream stream);

/* Page scoring and A/R/K top-K. KRI page (KRI-Q row; A<a>R<r>K<k> tag and its 128-block example) and
 * EarlySelectKV page (routing ranks pages by their K summaries, possibly against a proxy query).
 *   q_dev     [R][Hq][d] pool dtype: the routing query (the real query or a proxy).
 *   qbar[h]   = sum over g < G of q[h*G+g] (fp32, g ascending).
 *   score     = dot(qbar[h], k_summary[page][h]) in the fixed 32-lane order: lane l accumulates fmaf over
 *               i = l, l+32, ...; then lanes are combined by xor-butterfly 16, 8, 4, 2, 1 (a + b).
 *               Shared selection (per_kv_head = 0): score = sum over h ascending of the per-head scores.
 *   sel_ids   [R][rows][cap] out: selected prompt pages ascending; rows = Hkv or 1.
 *   n_sel     [R][rows] out: count = min(N, a + r + k) with N = ceil(ctx_len/16).
 *   workspace >= kap_score_workspace_size(...) bytes of device memory. On completion it holds the page scores,
 *             fp32 [R][rows][max_pages] from its first byte: entry (r, v, j) for j < N is the score above, entries
 *             at or past N are unspecified.
 * Errors: KAP_EINVAL for a null or misaligned pointer or a negative a, r or k; KAP_ECAPACITY for a workspace or a
 * cap too small; KAP_EUNSUPPORTED when R * rows > 65535 or the top-K row (4 bytes per page) exceeds 200 KiB. */
kap_status kap_score_topk(const kap_kv_pool *pool, const kap_page_map *map, const void *q_dev,
                          const kap_access_policy *policy, int32_t *sel_ids, int32_t *n_sel,
                          void *workspace, size_t workspace_bytes, kap_stream stream);
size_t kap_score_workspace_size(int32_t num_seqs, int32_t rows_per_seq, int32_t max_pages);

/* Page scoring, A/R/K top-K and view compilation in one call: the same outputs as kap_score_topk followed by
 * kap_compile_view(map, sel_ids, n_sel, rows, policy->cap, horizon_tokens, view, fallback_dev, s_max, slot_out,
 * pos_out), where rows = Hkv (per_kv_head) or 1. The top-K kernel compiles each row's view right after selecting
 * it, which saves the view kernel's launch and its reload of the selection. Needs map->seq_len; view->rows_per_seq
 * must equal rows and view->cap >= policy->cap + ceil(horizon_tokens/16) + 1. */
kap_status kap_score_topk_view(const kap_kv_pool *pool, const kap_page_map *map, const void *q_dev,
                               const kap_access_policy *policy, int32_t *sel_ids, int32_t *n_sel, void *workspace,
                               size_t workspace_bytes, int32_t horizon_tokens, const kap_view *view,
                               int32_t *fallback_dev, float s_max, int64_t *slot_out, int32_t *pos_out,
                               kap_stream stream);

/* External-prior selection. KRI page, prior schema and connector: a baked prior block_affinities[L][H][N] per
 * request prefix is mean-pooled across layers and heads and the top-K is taken per request (one selection row
 * shared by all heads), here under the A<a>R<r>K<k> split of `policy`, whose per_kv_head must be 0.
 *   affinities_dev [R][L][H][max_pages] fp32: the prior's block scores of each request; columns at or past
 *                  ceil(ctx_len/16) are ignored. L * H <= 2048.
 *   pooled score   = (sum over rows i = l*H + h, in chunks of 32 consecutive rows each summed from 0 with i
 *                    ascending, the chunk sums added in ascending order, all in fp32) / (L*H), one rounding.
 *                    The page states no order; this one is fixed so that selections reproduce bit for bit.
 *   sel_ids [R][1][policy->cap] out, ascending; n_sel [R][1] out (same rule and ties as kap_score_topk).
 *   workspace >= kap_score_workspace_size(R, 1, max_pages) bytes (the pooled scores).
 * Errors: KAP_EINVAL for a null pointer, L or H < 1, L*H > 2048 or per_kv_head != 0; KAP_ECAPACITY for a cap or
 * workspace that is too small. Follow with kap_compile_view (sel_rows_per_seq = 1) for the compact view. */
kap_status kap_prior_topk(const kap_page_map *map, const float *affinities_dev, int32_t num_layers,
                          int32_t num_heads, const kap_access_policy *policy, int32_t *sel_ids, int32_t *n_sel,
                          void *workspace, size_t workspace_bytes, kap_stream stream);

/* Materialised compact workspace. KAP paper, compiler (the selected spans are resolved to KV pages and materialised
 * as a compact physical view that keeps logical positions) and fallback (full-context access when the plan exceeds
 * the compact workspace). Request r owns the ws_pages_per_seq pool pages from ws_first_page + r * ws_pages_per_seq,
 * pages that no block table or view may reference otherwise (e.g. pages reserved at the end of the pool).
 * For every row (r, v) of `view`, selected entry i is copied to workspace page i of request r when all its tokens
 * are prompt tokens (16 * (logical page + 1) <= map->ctx_len[r]): K and V of head v for a per-head view
 * (rows_per_seq = Hkv), of every head for a shared view (rows_per_seq = 1). A selected page that also holds
 * positions >= ctx_len keeps its own page: generated tokens are written into it through the full table later.
 * out_view gets the row with the copied entries pointing at the workspace; tail entries, logical pages and counts
 * are copied unchanged. out_view may be `view` itself (rewritten in place); its cap >= view->cap.
 * A row whose n_selected exceeds ws_pages_per_seq is copied unchanged (attention over it stays correct, reading the
 * pool's own pages) and sets fallback_dev[r] = 1 when fallback_dev is given; the call never clears a flag.
 * Proposal attention over out_view equals attention over `view` bit for bit.
 * Errors: KAP_EINVAL for null pointers or sizes < 1; KAP_ESHAPE when rows_per_seq is neither 1 nor Hkv or the two
 * views differ in it; KAP_ECAPACITY when the workspace pages run past the pool or out_view->cap < view->cap. */
kap_status kap_materialize_view(const kap_kv_pool *pool, const kap_page_map *map, const kap_view *view,
                                int32_t ws_first_page, int32_t ws_pages_per_seq, const kap_view *out_view,
                                int32_t *fallback_dev, kap_stream stream);

/* Tolerant acceptance and commit of verify windows. KAP paper, verifier: the window is the verifier-approved carry
 * token followed by the k proposals; a proposal is accepted when it lies within the target's top-n candidates under
 * the full context (the Top-3 rule: top_n = 3; top_n = 1 is greedy exact match); m counts the proposals accepted
 * consecutively from the start; the same transition emits the next carry and advances the committed state.
 *   logits_dev         [total_rows][vocab] of logits_dtype (KAP_BF16 or KAP_F32): row j is the verifier's prediction
 *                      after window token j (the verify attention's window rows, through the model's head).
 *   window_offsets_dev [num_seqs+1] int32: request r owns rows [off[r], off[r+1]); every window holds 1 to 32 rows
 *                      and off[num_seqs] = total_rows (rows past 32 are not judged and set device error bit 4).
 *   tokens_dev         [total_rows] int32: the window's tokens; row off[r] is the carry, the rest are proposals.
 *   Rank order of a row: logit descending, lower token id first, NaN last. Proposal j passes when fewer than top_n
 *   tokens of row j - 1 come before it; a token outside [0, vocab) fails.
 *   accepted_out [num_seqs] = m; carry_out [num_seqs] = the first token of row m (the next carry);
 *   seq_len_out [num_seqs] (may be NULL, may alias a page map's seq_len) = start_pos[r] + 1 + m, the committed length:
 *   the carry at start_pos[r] and the accepted proposals after it, whose KV the window append already wrote.
 *   workspace >= kap_accept_workspace_size(num_seqs, total_rows, vocab) bytes, zeroed once before the first call
 *   (the call leaves its counters at zero).
 * Errors: KAP_EINVAL for null pointers, vocab or top_n < 1, total_rows < num_seqs; KAP_EUNSUPPORTED for another
 * dtype or more than 65535 rows; KAP_ECAPACITY for a small workspace. */
kap_status kap_accept_commit(const void *logits_dev, int32_t logits_dtype, int32_t vocab, int32_t num_seqs,
                             int32_t total_rows, const int32_t *window_offsets_dev, const int32_t *tokens_dev,
                             const int32_t *start_pos_dev, int32_t top_n, int32_t *accepted_out,
                             int32_t *carry_out, int32_t *seq_len_out, void *workspace, size_t workspace_bytes,
                             kap_stream stream);
size_t kap_accept_workspace_size(int32_t num_seqs, int32_t total_rows, int32_t vocab);

/* Span selection. KAP paper, compiler stage 3 (selected spans resolved to KV pages): a prompt page is kept when
 * any token of a selected span falls in it; pinned anchor/recent pages (policy a, r) are added. One row per
 * request (shared by all heads).
 *   spans_dev        [S][2] int32 (first token, length); span_offsets_dev [R+1] splits them by request.
 *   sel_ids          [R][1][policy->cap] out, ascending; n_sel [R][1] out. */
kap_status kap_select_spans(const kap_page_map *map, const int32_t *spans_dev, const int32_t *span_offsets_dev,
                            const kap_access_policy *policy, int32_t *sel_ids, int32_t *n_sel, kap_stream stream);

/* View compilation. KAP paper, compiler stage 3 and "selected-KV view" (selected pages compacted in access
 * order, logical positions preserved through block tables). For each row: entries 0..n_sel-1 are the selected
 * pages (block_table[i] = map->block_table[r][sel[i]], logical_page[i] = sel[i]); then tail pages: every page
 * j >= floor(ctx_len/16) with 16j < seq_len + horizon_tokens that is not already selected.
 *   sel_rows_per_seq/sel_cap give the layout of sel_ids; view->rows_per_seq must equal sel_rows_per_seq.
 *   fallback_dev     optional [R] out: 1 when request r's retained prompt fraction n_sel/N exceeds s_max,
 *                    else 0 (KAP paper, fallback: the plan keeps too large a share of the KV).
 *   slot_out/pos_out optional [R][horizon_tokens] out: the slot mapping of the tokens the cycle will append,
 *                    at positions seq_len[r] + i (same rule as kap_slot_mapping); NULL to skip.
 * Returns KAP_ECAPACITY when view->cap < sel_cap + ceil(horizon/16) + 1. */
kap_status kap_compile_view(const kap_page_map *map, const int32_t *sel_ids, const int32_t *n_sel,
                            int32_t sel_rows_per_seq, int32_t sel_cap, int32_t horizon_tokens,
                            const kap_view *view, int32_t *fallback_dev, float s_max, int64_t *slot_out,
                            int32_t *pos_out, kap_stream stream);

/* Slot mapping. KAP paper, selected-KV view (each newly scheduled token is sent to its physical KV slot).
 * Request r owns tokens tok_offsets[r] .. tok_offsets[r+1]-1; token j sits at pos = start_pos[r] + (j -
 * tok_offsets[r]) and slot = block_table[r][pos/16]*16 + pos%16 (-1 when the page is outside the table or
 * negative). Writes slot_out[j] and pos_out[j]. */
kap_status kap_slot_mapping(const kap_page_map *map, const int32_t *tok_offsets_dev, const int32_t *start_pos_dev,
                            int32_t num_tokens, int64_t *slot_out, int32_t *pos_out, kap_stream stream);

/* RoPE inverse frequencies. KAP paper, selected-KV view: the proposal and the verifier keep the same logical
 * positions, so every call that rotates (kap_append_kv, kap_append_propose) takes the one table this fills.
 * Writes inv_freq_host[i] = theta^(-2i/d) for 0 <= i < d/2, formed in double precision and rounded once to fp32,
 * into HOST memory of d/2 floats owned by the caller (who copies it to the device). No device work, no stream.
 * Returns KAP_EINVAL for a NULL pointer, d <= 0, odd d, or theta not finite and > 0. */
kap_status kap_rope_inv_freq(int32_t head_dim, double theta, float *inv_freq_host);

/* KV append with RoPE. KAP paper, executor (proposal KV written through the slot mapping; the verifier advances
 * the full-context KV state). For token t (0 <= t < T) with p = pos[t*tok_stride], s = slots[t*tok_stride]:
 * when s >= 0, K[s] = RoPE(k_new[t], p), V[s] = v_new[t] (fp32 math, round-to-nearest into the pool dtype);
 * when q_inout is not NULL, q_inout[t] = RoPE(q_inout[t], p) in place.
 * RoPE: pairs (i, i + d/2), angle = (float)p * inv_freq[i] (fp32), x' = x*cos - y*sin, y' = x*sin + y*cos.
 *   k_new, v_new [T][Hkv][d], q_inout [T][Hq][d] in the pool dtype; inv_freq_dev [d/2] fp32. */
kap_status kap_append_kv(const kap_kv_pool *pool, const void *k_new, const void *v_new, void *q_inout,
                         const int32_t *pos_dev, const int64_t *slots_dev, int32_t num_tokens, int32_t tok_stride,
                         const float *inv_freq_dev, kap_stream stream);

/* Selected-KV proposal attention, q = 1 per request. KAP paper, executor (proposal: a decode-like step with
 * q_prop = 1 over the compact view; only prompt-side KV is restricted) and EarlySelectKV (sparse attention with
 * the real query on precomputed page indices).
 * Query of request r, head hq sits at position P = seq_len[r]-1. A token at position p of view entry i is
 * visible when p <= P and (i < n_selected or p >= ctx_len).
 *   q_dev [R][Hq][d], out [R][Hq][d] (pool dtype), lse [R][Hq] fp32.
 *   workspace >= kap_propose_workspace_size(...) bytes, zero-filled once before first use (the kernels leave
 *   their counters at zero again on completion). */
kap_status kap_attn_propose(const kap_kv_pool *pool, const kap_page_map *map, const kap_view *view,
                            const void *q_dev, void *out, float *lse, void *workspace, size_t workspace_bytes,
                            kap_stream stream);
size_t kap_propose_workspace_size(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads, int32_t head_dim);

/* One proposal step with the step token's KV append fused in. KAP paper, executor (a proposal step writes its own
 * token's KV at that token's logical position through the view's slots and attends over the compact view).
 * Same pool, map, view, outputs and workspace as kap_attn_propose; in addition, for every request r:
 *   - the step token sits at position P = seq_len[r] - 1, which must lie on a page of the view (view compiled with
 *     a horizon that covers the step); a request whose P lies on no view page gets no append and sets device error
 *     bit 4;
 *   - k_new, v_new [R][Hkv][d] (pool dtype): the token's key before RoPE and its value. K = RoPE(k_new, P) and
 *     V = v_new are written into the pool at P's slot and take part in this step's attention;
 *   - q_dev [R][Hq][d] holds the step's queries BEFORE RoPE; they are rotated at P inside the call (the buffer is
 *     only read);
 *   - inv_freq_dev [d/2] fp32, as for kap_append_kv.
 * The result equals kap_append_kv at positions seq_len-1 (q rotated) followed by kap_attn_propose: the rotation
 * and its rounding into the pool dtype are the same. */
kap_status kap_append_propose(const kap_kv_pool *pool, const kap_page_map *map, const kap_view *view,
                              const void *q_dev, const void *k_new, const void *v_new, const float *inv_freq_dev,
                              void *out, float *lse, void *workspace, size_t workspace_bytes, kap_stream stream);

/* Full-context verification attention, q = n_q per request, causal among the candidates. KAP paper, verifier
 * (short contiguous query window over the full KV cache, full block table and original positions).
 *   q_dev [total_q][Hq][d], out [total_q][Hq][d] (pool dtype), lse [total_q][Hq] fp32.
 *   workspace >= kap_verify_workspace_size(...) bytes, zero-filled once before first use. */
kap_status kap_attn_verify(const kap_kv_pool *pool, const kap_page_map *map, const kap_verify_policy *vp,
                           const void *q_dev, void *out, float *lse, void *workspace, size_t workspace_bytes,
                           kap_stream stream);
size_t kap_verify_workspace_size(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_q);

/* Proposal attention without a caller workspace, for callers that cannot allocate device memory (a serving host
 * that fixes its device memory budget at start-up and owns the only allocator, a plug-in without access to that
 * allocator, or a loop where an allocation and its implicit device synchronisation are not allowed). The pages have
 * no counterpart to this call: it is a deployment variant of kap_attn_propose with identical arguments and results,
 * minus the workspace.
 *   - Scratch: a fixed array of kap_noalloc_scratch_bytes() = 16 MiB inside the library, present on every GPU that
 *     loads the library until the process exits. Shapes whose kap_propose_workspace_size exceeds it are rejected
 *     with KAP_ECAPACITY.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. Each call clears the scratch's
 *     counters with cudaMemsetAsync on `stream`, then launches the same kernel as kap_attn_propose.
 *   - The first call on a device looks up the scratch's device address (cudaGetSymbolAddress) with that device
 *     current; make that first call before any stream capture. The address is kept for the life of the process:
 *     after a cudaDeviceReset of that device the library must not be called on it again in the same process.
 *   - A failed CUDA call (the address lookup, the clearing of the counters, the launch) returns KAP_ECUDA with its
 *     text in kap_last_cuda_error, as for every other call.
 *   - Every call on a device shares the one scratch array and it keeps the last call's contents: calls that overlap
 *     on the GPU (different streams, no ordering between them) race and give wrong results. */
kap_status kap_attn_propose_noalloc(const kap_kv_pool *pool, const kap_page_map *map, const kap_view *view,
                                    const void *q_dev, void *out, float *lse, kap_stream stream);
size_t kap_noalloc_scratch_bytes(void);

/* Check of the bounded waits. Every wait of a kernel on an mbarrier (a copy landing, a slot freed, an MMA done)
 * gives up after at most about a second, sets bit 8 of the device error word and lets the kernel return, so that a
 * lost arrival cannot hang the GPU. This call runs the same bounded wait, on a barrier that nothing completes and
 * with nothing in flight, for `polls` polls of at most `suspend_ns` each (1 <= polls <= 1024,
 * 1 <= suspend_ns <= 2^20), and writes 1 to *timed_out_dev (device int32) when the wait gave up, 0 otherwise. The
 * pages have no counterpart: this is a diagnostic of the library. KAP_EINVAL for out-of-range arguments. */
kap_status kap_selftest_wait_timeout(uint32_t polls, uint32_t suspend_ns, int32_t *timed_out_dev, kap_stream stream);

/* Diagnostics. */
const char *kap_status_str(kap_status s);
const char *kap_last_cuda_error(void);   /* text of the last CUDA error seen by this thread, "" if none */
/* Reads (with a device synchronisation) and clears the device-side error word of the current device.
 * 0 = no error; otherwise a bit set: 1 page id out of the pool, 2 selection over capacity, 4 bad page length,
 * 8 a bounded wait in a kernel ran out. */
kap_status kap_device_error(int32_t *code_out);

#ifdef __cplusplus
}
#endif
#endif /* KAP_H */
