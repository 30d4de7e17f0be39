// kap_launch.h - host-side launch functions of the kernels (internal to the library; the public ABI is kap.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kap {

struct PoolArgs {
  int num_pages, hkv, hq, d, dtype;  // dtype: 0 bf16, 1 fp32
  const void *k, *v;
  float *ksum;
};

struct MapArgs {
  int R, max_pages;
  const int32_t *bt, *ctx_len, *seq_len;
};

struct ViewArgs {
  int rows_per_seq, cap;
  const int32_t *bt, *lp, *n_entries, *n_selected;
  int settled;  // the view, lengths and prompt tokens predate the previous kernel on the stream
};

// selection kernels (k_select.cu)
cudaError_t launch_build_summaries(const PoolArgs &p, const MapArgs &m, int *err, cudaStream_t s);
cudaError_t launch_refresh_summaries(const PoolArgs &p, const int32_t *pages, const int32_t *n_valid, int n, int *err,
                                     cudaStream_t s);
cudaError_t launch_score(const PoolArgs &p, const MapArgs &m, const void *q, int per_head, float *scores,
                         int *err, cudaStream_t s);
// Outputs of view compilation fused into top-K (see kap_score_topk_view).
struct ViewArgsOut {
  int32_t *vbt, *vlp, *vn, *vnsel;
  int vcap, horizon;
  int32_t *fallback;
  float s_max;
  int64_t *slot_out;
  int32_t *pos_out;
};
// view non-null: the top-K CTA of each row also compiles that row's view
cudaError_t launch_topk(const MapArgs &m, const float *scores, int rows, int a, int r, int k,
                        const int32_t *per_seq_ark, int cap, int32_t *sel, int32_t *n_sel, const ViewArgsOut *view,
                        int *err, cudaStream_t s);
// external-prior scores [R][L][H][max_pages] pooled into scores [R][max_pages], then the per-request top-K
cudaError_t launch_prior_topk(const MapArgs &m, const float *aff, int L, int H, int a, int r, int k,
                              const int32_t *per_seq_ark, int cap, int32_t *sel, int32_t *n_sel, float *scores,
                              int *err, cudaStream_t s);
cudaError_t launch_select_spans(const MapArgs &m, const int32_t *spans, const int32_t *span_offsets, int a, int r,
                                const int32_t *per_seq_ark, int cap, int32_t *sel, int32_t *n_sel, int *err,
                                cudaStream_t s);
cudaError_t launch_compile_view(const MapArgs &m, const int32_t *sel, const int32_t *n_sel, int rows, int sel_cap,
                                int horizon, int32_t *vbt, int32_t *vlp, int32_t *vn, int32_t *vnsel, int vcap,
                                int32_t *fallback, float s_max, int64_t *slot_out, int32_t *pos_out, int *err,
                                cudaStream_t s);
cudaError_t launch_slot_mapping(const MapArgs &m, const int32_t *tok_offsets, const int32_t *start_pos, int T,
                                int64_t *slot_out, int32_t *pos_out, cudaStream_t s);

// materialised compact workspace (k_materialize.cu): selected entries of `in` copied to the workspace pages
cudaError_t launch_materialize(const PoolArgs &p, int R, const int32_t *ctx_len, const ViewArgs &in, int32_t *obt,
                               int32_t *olp, int32_t *on,
                               int32_t *onsel, int ocap, int ws_first, int ws_pages, int32_t *fallback, int *err,
                               cudaStream_t s);

// tolerant acceptance and commit of verify windows (k_accept.cu)
size_t accept_workspace_bytes(int num_seqs, int total_rows, int vocab);
cudaError_t launch_accept(const void *logits, int dtype, int V, const int32_t *woff, int R, int total_rows,
                          const int32_t *tokens, const int32_t *start_pos, int top_n, void *ws, int32_t *m_out,
                          int32_t *carry_out, int32_t *seq_out, int *err, cudaStream_t s);

// KV append (k_append.cu)
cudaError_t launch_append(const PoolArgs &p, const void *k_new, const void *v_new, void *q_inout,
                          const int32_t *pos, const int64_t *slots, int T, int tok_stride, const float *inv_freq,
                          int *err, cudaStream_t s);

// proposal attention (k_propose.cu)
size_t propose_workspace_bytes(int R, int hkv, int hq, int d);
// k_new/v_new/inv_freq non-null: fused append of the step token at seq_len-1 (q is then taken before RoPE)
cudaError_t launch_propose(const PoolArgs &p, const MapArgs &m, const ViewArgs &v, const void *q, void *out,
                           float *lse, void *ws, size_t ws_bytes, const void *k_new, const void *v_new,
                           const float *inv_freq, int *err, cudaStream_t s);

// verification attention (k_verify.cu)
size_t verify_workspace_bytes(int R, int hkv, int hq, int d, int max_q);
cudaError_t launch_verify(const PoolArgs &p, const MapArgs &m, int max_q, int total_q, const int32_t *q_offsets,
                          const int32_t *q_start, const void *q, void *out, float *lse, void *ws, size_t ws_bytes,
                          int *err, cudaStream_t s);

// number of SMs of the current device (cached per device)
int device_sm_count();

// bounded-wait check (k_selftest.cu): one bounded mbarrier wait that nothing completes
cudaError_t launch_wait_probe(uint32_t polls, uint32_t suspend_ns, int *err, int32_t *timed_out, cudaStream_t s);

// Records the text of a failed CUDA call for kap_last_cuda_error (this thread) and returns true when e is an error.
bool record_cuda_error(cudaError_t e);

}  // namespace kap
