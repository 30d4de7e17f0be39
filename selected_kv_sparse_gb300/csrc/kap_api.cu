// kap_api.cu - the C ABI of include/kap.h: argument validation, dispatch to the kernels, status codes.
#include "../../include/kap.h"
#include "kap_launch.h"

#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <string>

namespace kap {

// One device-wide error word per GPU; kernels OR error bits into it.
__device__ int g_error_word;

namespace {
thread_local std::string g_last_cuda_error;
}  // namespace

bool record_cuda_error(cudaError_t e) {
  if (e == cudaSuccess) return false;
  g_last_cuda_error = cudaGetErrorString(e);
  return true;
}

namespace {

constexpr int kMaxDevices = 64;

int *error_word() {
  static int *ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int *>(p);
  }
  return ptrs[dev];
}

kap_status cuda_status(cudaError_t e) { return record_cuda_error(e) ? KAP_ECUDA : KAP_OK; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kap_status check_pool(const kap_kv_pool *p, bool need_summary) {
  if (!p) return KAP_EINVAL;
  if (p->page_size != 16) return KAP_EUNSUPPORTED;
  if (p->num_pages <= 0 || p->num_kv_heads <= 0 || p->num_q_heads <= 0) return KAP_EINVAL;
  if (p->num_q_heads % p->num_kv_heads != 0) return KAP_ESHAPE;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (G > 8) return KAP_EUNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128) return KAP_EUNSUPPORTED;
  if (p->dtype != KAP_BF16 && p->dtype != KAP_F32) return KAP_EUNSUPPORTED;
  if (!p->k_pages || !p->v_pages) return KAP_EINVAL;
  if (!aligned16(p->k_pages) || !aligned16(p->v_pages)) return KAP_EINVAL;
  if (need_summary && !p->k_summary) return KAP_EINVAL;
  if (static_cast<int64_t>(p->num_pages) * p->num_kv_heads * 16 >= (int64_t(1) << 31)) return KAP_EUNSUPPORTED;
  return KAP_OK;
}

kap_status check_map(const kap_page_map *m, bool need_seq) {
  if (!m) return KAP_EINVAL;
  if (m->num_seqs <= 0 || m->max_pages <= 0) return KAP_EINVAL;
  if (m->num_seqs > 65535) return KAP_EUNSUPPORTED;
  if (!m->block_table || !m->ctx_len) return KAP_EINVAL;
  if (need_seq && !m->seq_len) return KAP_EINVAL;
  return KAP_OK;
}

PoolArgs pool_args(const kap_kv_pool *p) {
  PoolArgs a;
  a.num_pages = p->num_pages;
  a.hkv = p->num_kv_heads;
  a.hq = p->num_q_heads;
  a.d = p->head_dim;
  a.dtype = p->dtype;
  a.k = p->k_pages;
  a.v = p->v_pages;
  a.ksum = p->k_summary;
  return a;
}

MapArgs map_args(const kap_page_map *m) {
  MapArgs a;
  a.R = m->num_seqs;
  a.max_pages = m->max_pages;
  a.bt = m->block_table;
  a.ctx_len = m->ctx_len;
  a.seq_len = m->seq_len;
  return a;
}

cudaStream_t cs(kap_stream s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

int device_sm_count() {
  static int counts[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  if (counts[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    counts[dev] = n > 0 ? n : 1;
  }
  return counts[dev];
}

}  // namespace kap

using namespace kap;

extern "C" {

kap_status kap_build_summaries(const kap_kv_pool *pool, const kap_page_map *map, kap_stream stream) {
  kap_status st = check_pool(pool, true);
  if (st != KAP_OK) return st;
  if ((st = check_map(map, false)) != KAP_OK) return st;
  return cuda_status(launch_build_summaries(pool_args(pool), map_args(map), error_word(), cs(stream)));
}

kap_status kap_refresh_summaries(const kap_kv_pool *pool, const int32_t *pages_dev, const int32_t *n_valid_dev,
                                 int32_t num_listed, kap_stream stream) {
  kap_status st = check_pool(pool, true);
  if (st != KAP_OK) return st;
  if (num_listed < 0) return KAP_EINVAL;
  if (num_listed == 0) return KAP_OK;
  if (!pages_dev || !n_valid_dev) return KAP_EINVAL;
  return cuda_status(
      launch_refresh_summaries(pool_args(pool), pages_dev, n_valid_dev, num_listed, error_word(), cs(stream)));
}

size_t kap_score_workspace_size(int32_t num_seqs, int32_t rows_per_seq, int32_t max_pages) {
  if (num_seqs <= 0 || rows_per_seq <= 0 || max_pages <= 0) return 0;
  return static_cast<size_t>(num_seqs) * rows_per_seq * max_pages * sizeof(float);
}

namespace {
kap_status score_topk_common(const kap_kv_pool *pool, const kap_page_map *map, const void *q_dev,
                             const kap_access_policy *policy, int32_t *sel_ids, int32_t *n_sel, void *workspace,
                             size_t workspace_bytes, const ViewArgsOut *vw, kap_stream stream) {
  kap_status st = check_pool(pool, true);
  if (st != KAP_OK) return st;
  if ((st = check_map(map, vw != nullptr)) != KAP_OK) return st;
  if (!q_dev || !policy || !sel_ids || !n_sel || !workspace) return KAP_EINVAL;
  if (!aligned16(q_dev)) return KAP_EINVAL;
  if (policy->anchor < 0 || policy->recent < 0 || policy->topk < 0 || policy->cap <= 0) return KAP_EINVAL;
  if (policy->per_kv_head != 0 && policy->per_kv_head != 1) return KAP_EINVAL;
  if (!policy->per_seq_ark &&
      static_cast<int64_t>(policy->anchor) + policy->recent + policy->topk > policy->cap &&
      policy->cap < map->max_pages)
    return KAP_ECAPACITY;
  if (!policy->per_kv_head && pool->num_kv_heads > 16) return KAP_EUNSUPPORTED;
  const size_t topk_smem = static_cast<size_t>(map->max_pages) * 4 + (vw ? static_cast<size_t>(policy->cap) * 4 : 0);
  if (topk_smem > 200 * 1024) return KAP_EUNSUPPORTED;
  const int rows = policy->per_kv_head ? pool->num_kv_heads : 1;
  if (static_cast<int64_t>(map->num_seqs) * rows > 65535) return KAP_EUNSUPPORTED;  // score grid rows
  if (workspace_bytes < kap_score_workspace_size(map->num_seqs, rows, map->max_pages)) return KAP_ECAPACITY;
  const PoolArgs pa = pool_args(pool);
  const MapArgs ma = map_args(map);
  int *err = error_word();
  float *scores = static_cast<float *>(workspace);
  cudaError_t e = launch_score(pa, ma, q_dev, policy->per_kv_head, scores, err, cs(stream));
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_topk(ma, scores, rows, policy->anchor, policy->recent, policy->topk, policy->per_seq_ark,
                                 policy->cap, sel_ids, n_sel, vw, err, cs(stream)));
}
}  // namespace

kap_status kap_score_topk(const kap_kv_pool *pool, const kap_page_map *map, const void *q_dev,
                          const kap_access_policy *policy, int32_t *sel_ids, int32_t *n_sel, void *workspace,
                          size_t workspace_bytes, kap_stream stream) {
  return score_topk_common(pool, map, q_dev, policy, sel_ids, n_sel, workspace, workspace_bytes, nullptr, stream);
}

kap_status kap_score_topk_view(const kap_kv_pool *pool, const kap_page_map *map, const void *q_dev,
                               const kap_access_policy *policy, int32_t *sel_ids, int32_t *n_sel, void *workspace,
                               size_t workspace_bytes, int32_t horizon_tokens, const kap_view *view,
                               int32_t *fallback_dev, float s_max, int64_t *slot_out, int32_t *pos_out,
                               kap_stream stream) {
  if (!policy || !view || horizon_tokens < 0) return KAP_EINVAL;
  if (!view->block_table || !view->logical_page || !view->n_entries || !view->n_selected) return KAP_EINVAL;
  const int rows = policy->per_kv_head ? (pool ? pool->num_kv_heads : 0) : 1;
  if (view->rows_per_seq != rows) return KAP_ESHAPE;
  if (static_cast<int64_t>(view->cap) < static_cast<int64_t>(policy->cap) + (horizon_tokens + 15) / 16 + 1)
    return KAP_ECAPACITY;
  const ViewArgsOut vw{view->block_table, view->logical_page, view->n_entries, view->n_selected, view->cap,
                       horizon_tokens, fallback_dev, s_max, slot_out, pos_out};
  return score_topk_common(pool, map, q_dev, policy, sel_ids, n_sel, workspace, workspace_bytes, &vw, stream);
}

kap_status kap_prior_topk(const kap_page_map *map, const float *affinities_dev, int32_t num_layers,
                          int32_t num_heads, const kap_access_policy *policy, int32_t *sel_ids, int32_t *n_sel,
                          void *workspace, size_t workspace_bytes, kap_stream stream) {
  kap_status st = check_map(map, false);
  if (st != KAP_OK) return st;
  if (!affinities_dev || !policy || !sel_ids || !n_sel || !workspace) return KAP_EINVAL;
  if (num_layers < 1 || num_heads < 1 || static_cast<int64_t>(num_layers) * num_heads > 2048) return KAP_EINVAL;
  if (policy->anchor < 0 || policy->recent < 0 || policy->topk < 0 || policy->cap <= 0) return KAP_EINVAL;
  if (policy->per_kv_head != 0) return KAP_EINVAL;
  if (!policy->per_seq_ark &&
      static_cast<int64_t>(policy->anchor) + policy->recent + policy->topk > policy->cap &&
      policy->cap < map->max_pages)
    return KAP_ECAPACITY;
  if (static_cast<size_t>(map->max_pages) * 4 > 200 * 1024) return KAP_EUNSUPPORTED;
  if (workspace_bytes < kap_score_workspace_size(map->num_seqs, 1, map->max_pages)) return KAP_ECAPACITY;
  return cuda_status(launch_prior_topk(map_args(map), affinities_dev, num_layers, num_heads, policy->anchor,
                                       policy->recent, policy->topk, policy->per_seq_ark, policy->cap, sel_ids,
                                       n_sel, static_cast<float *>(workspace), error_word(), cs(stream)));
}

kap_status kap_materialize_view(const kap_kv_pool *pool, const kap_page_map *map, const kap_view *view,
                                int32_t ws_first_page, int32_t ws_pages_per_seq, const kap_view *out_view,
                                int32_t *fallback_dev, kap_stream stream) {
  kap_status st = check_pool(pool, false);
  if (st != KAP_OK) return st;
  if ((st = check_map(map, false)) != KAP_OK) return st;
  if (!view || !out_view) return KAP_EINVAL;
  const int32_t num_seqs = map->num_seqs;
  if (!view->block_table || !view->logical_page || !view->n_entries || !view->n_selected) return KAP_EINVAL;
  if (!out_view->block_table || !out_view->logical_page || !out_view->n_entries || !out_view->n_selected)
    return KAP_EINVAL;
  if (view->rows_per_seq != 1 && view->rows_per_seq != pool->num_kv_heads) return KAP_ESHAPE;
  if (out_view->rows_per_seq != view->rows_per_seq || view->cap <= 0) return KAP_ESHAPE;
  if (out_view->cap < view->cap) return KAP_ECAPACITY;
  if (ws_first_page < 0 || ws_pages_per_seq <= 0) return KAP_EINVAL;
  if (static_cast<int64_t>(ws_first_page) + static_cast<int64_t>(num_seqs) * ws_pages_per_seq > pool->num_pages)
    return KAP_ECAPACITY;
  if (static_cast<int64_t>(num_seqs) * view->rows_per_seq > 65535) return KAP_EUNSUPPORTED;
  const ViewArgs in{view->rows_per_seq, view->cap, view->block_table, view->logical_page, view->n_entries,
                    view->n_selected, 0};
  return cuda_status(launch_materialize(pool_args(pool), num_seqs, map->ctx_len, in, out_view->block_table,
                                        out_view->logical_page, out_view->n_entries, out_view->n_selected,
                                        out_view->cap, ws_first_page, ws_pages_per_seq, fallback_dev, error_word(),
                                        cs(stream)));
}

size_t kap_accept_workspace_size(int32_t num_seqs, int32_t total_rows, int32_t vocab) {
  if (num_seqs <= 0 || total_rows <= 0 || vocab <= 0) return 0;
  return accept_workspace_bytes(num_seqs, total_rows, vocab);
}

kap_status kap_accept_commit(const void *logits_dev, int32_t logits_dtype, int32_t vocab, int32_t num_seqs,
                             int32_t total_rows, const int32_t *window_offsets_dev, const int32_t *tokens_dev,
                             const int32_t *start_pos_dev, int32_t top_n, int32_t *accepted_out,
                             int32_t *carry_out, int32_t *seq_len_out, void *workspace, size_t workspace_bytes,
                             kap_stream stream) {
  if (!logits_dev || !window_offsets_dev || !tokens_dev || !accepted_out || !carry_out || !workspace)
    return KAP_EINVAL;
  if (seq_len_out && !start_pos_dev) return KAP_EINVAL;
  if (logits_dtype != KAP_BF16 && logits_dtype != KAP_F32) return KAP_EUNSUPPORTED;
  if (vocab <= 0 || num_seqs <= 0 || total_rows < num_seqs || top_n <= 0) return KAP_EINVAL;
  if (total_rows > 65535) return KAP_EUNSUPPORTED;  // grid rows
  if (workspace_bytes < accept_workspace_bytes(num_seqs, total_rows, vocab)) return KAP_ECAPACITY;
  return cuda_status(launch_accept(logits_dev, logits_dtype, vocab, window_offsets_dev, num_seqs, total_rows,
                                   tokens_dev, start_pos_dev, top_n, workspace, accepted_out, carry_out, seq_len_out,
                                   error_word(), cs(stream)));
}

kap_status kap_select_spans(const kap_page_map *map, const int32_t *spans_dev, const int32_t *span_offsets_dev,
                            const kap_access_policy *policy, int32_t *sel_ids, int32_t *n_sel, kap_stream stream) {
  kap_status st = check_map(map, false);
  if (st != KAP_OK) return st;
  if (!span_offsets_dev || !policy || !sel_ids || !n_sel) return KAP_EINVAL;
  if (policy->anchor < 0 || policy->recent < 0 || policy->cap <= 0) return KAP_EINVAL;
  if (map->max_pages > 200 * 1024) return KAP_EUNSUPPORTED;
  return cuda_status(launch_select_spans(map_args(map), spans_dev, span_offsets_dev, policy->anchor, policy->recent,
                                         policy->per_seq_ark, policy->cap, sel_ids, n_sel, error_word(),
                                         cs(stream)));
}

kap_status kap_compile_view(const kap_page_map *map, const int32_t *sel_ids, const int32_t *n_sel,
                            int32_t sel_rows_per_seq, int32_t sel_cap, int32_t horizon_tokens, const kap_view *view,
                            int32_t *fallback_dev, float s_max, int64_t *slot_out, int32_t *pos_out,
                            kap_stream stream) {
  kap_status st = check_map(map, true);
  if (st != KAP_OK) return st;
  if (!sel_ids || !n_sel || !view) return KAP_EINVAL;
  if (sel_rows_per_seq <= 0 || sel_cap <= 0 || horizon_tokens < 0) return KAP_EINVAL;
  if (!view->block_table || !view->logical_page || !view->n_entries || !view->n_selected) return KAP_EINVAL;
  if (view->rows_per_seq != sel_rows_per_seq) return KAP_ESHAPE;
  if (static_cast<int64_t>(view->cap) < static_cast<int64_t>(sel_cap) + (horizon_tokens + 15) / 16 + 1)
    return KAP_ECAPACITY;
  return cuda_status(launch_compile_view(map_args(map), sel_ids, n_sel, sel_rows_per_seq, sel_cap, horizon_tokens,
                                         view->block_table, view->logical_page, view->n_entries, view->n_selected,
                                         view->cap, fallback_dev, s_max, slot_out, pos_out, error_word(),
                                         cs(stream)));
}

kap_status kap_slot_mapping(const kap_page_map *map, const int32_t *tok_offsets_dev, const int32_t *start_pos_dev,
                            int32_t num_tokens, int64_t *slot_out, int32_t *pos_out, kap_stream stream) {
  kap_status st = check_map(map, false);
  if (st != KAP_OK) return st;
  if (num_tokens < 0) return KAP_EINVAL;
  if (num_tokens == 0) return KAP_OK;
  if (!tok_offsets_dev || !start_pos_dev || !slot_out) return KAP_EINVAL;
  return cuda_status(launch_slot_mapping(map_args(map), tok_offsets_dev, start_pos_dev, num_tokens, slot_out, pos_out,
                                         cs(stream)));
}

kap_status kap_append_kv(const kap_kv_pool *pool, const void *k_new, const void *v_new, void *q_inout,
                         const int32_t *pos_dev, const int64_t *slots_dev, int32_t num_tokens, int32_t tok_stride,
                         const float *inv_freq_dev, kap_stream stream) {
  kap_status st = check_pool(pool, false);
  if (st != KAP_OK) return st;
  if (num_tokens < 0 || tok_stride < 1) return KAP_EINVAL;
  if (num_tokens == 0) return KAP_OK;
  if (!k_new || !v_new || !pos_dev || !slots_dev || !inv_freq_dev) return KAP_EINVAL;
  return cuda_status(launch_append(pool_args(pool), k_new, v_new, q_inout, pos_dev, slots_dev, num_tokens, tok_stride,
                                   inv_freq_dev, error_word(), cs(stream)));
}

size_t kap_propose_workspace_size(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads, int32_t head_dim) {
  if (num_seqs <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  return propose_workspace_bytes(num_seqs, num_kv_heads, num_q_heads, head_dim);
}

namespace {
kap_status propose_common(const kap_kv_pool *pool, const kap_page_map *map, const kap_view *view, const void *q_dev,
                          void *out, float *lse, void *workspace, size_t workspace_bytes, const void *k_new,
                          const void *v_new, const float *inv_freq_dev, kap_stream stream) {
  kap_status st = check_pool(pool, false);
  if (st != KAP_OK) return st;
  if ((st = check_map(map, true)) != KAP_OK) return st;
  if (!view || !q_dev || !out || !lse || !workspace) return KAP_EINVAL;
  if (!view->block_table || !view->logical_page || !view->n_entries || !view->n_selected) return KAP_EINVAL;
  if (view->cap <= 0) return KAP_EINVAL;
  if (view->rows_per_seq != 1 && view->rows_per_seq != pool->num_kv_heads) return KAP_ESHAPE;
  if (!aligned16(q_dev) || !aligned16(out)) return KAP_EINVAL;
  if (k_new && (!aligned16(k_new) || !aligned16(v_new) || !aligned16(inv_freq_dev))) return KAP_EINVAL;
  const int G = pool->num_q_heads / pool->num_kv_heads;
  if (!(G == 1 || G == 2 || G == 4 || G == 5 || G == 8)) return KAP_EUNSUPPORTED;
  if (workspace_bytes <
      propose_workspace_bytes(map->num_seqs, pool->num_kv_heads, pool->num_q_heads, pool->head_dim))
    return KAP_ECAPACITY;
  ViewArgs va;
  va.rows_per_seq = view->rows_per_seq;
  va.cap = view->cap;
  va.bt = view->block_table;
  va.lp = view->logical_page;
  va.n_entries = view->n_entries;
  va.n_selected = view->n_selected;
  va.settled = view->settled != 0;
  return cuda_status(launch_propose(pool_args(pool), map_args(map), va, q_dev, out, lse, workspace, workspace_bytes,
                                    k_new, v_new, inv_freq_dev, error_word(), cs(stream)));
}
}  // namespace

kap_status kap_attn_propose(const kap_kv_pool *pool, const kap_page_map *map, const kap_view *view, const void *q_dev,
                            void *out, float *lse, void *workspace, size_t workspace_bytes, kap_stream stream) {
  return propose_common(pool, map, view, q_dev, out, lse, workspace, workspace_bytes, nullptr, nullptr, nullptr,
                        stream);
}

kap_status kap_append_propose(const kap_kv_pool *pool, const kap_page_map *map, const kap_view *view,
                              const void *q_dev, const void *k_new, const void *v_new, const float *inv_freq_dev,
                              void *out, float *lse, void *workspace, size_t workspace_bytes, kap_stream stream) {
  if (!k_new || !v_new || !inv_freq_dev) return KAP_EINVAL;
  return propose_common(pool, map, view, q_dev, out, lse, workspace, workspace_bytes, k_new, v_new, inv_freq_dev,
                        stream);
}

size_t kap_verify_workspace_size(int32_t num_seqs, int32_t num_kv_heads, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_q) {
  if (num_seqs <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_q <= 0) return 0;
  return verify_workspace_bytes(num_seqs, num_kv_heads, num_q_heads, head_dim, max_q);
}

kap_status kap_attn_verify(const kap_kv_pool *pool, const kap_page_map *map, const kap_verify_policy *vp,
                           const void *q_dev, void *out, float *lse, void *workspace, size_t workspace_bytes,
                           kap_stream stream) {
  kap_status st = check_pool(pool, false);
  if (st != KAP_OK) return st;
  if ((st = check_map(map, false)) != KAP_OK) return st;
  if (!vp || !q_dev || !out || !lse || !workspace) return KAP_EINVAL;
  if (!vp->q_offsets || !vp->q_start_pos) return KAP_EINVAL;
  if (vp->max_q <= 0 || vp->total_q < 0) return KAP_EINVAL;
  const int G = pool->num_q_heads / pool->num_kv_heads;
  if (G * vp->max_q > 64) return KAP_EUNSUPPORTED;
  if (!aligned16(q_dev) || !aligned16(out)) return KAP_EINVAL;
  if (workspace_bytes < verify_workspace_bytes(map->num_seqs, pool->num_kv_heads, pool->num_q_heads, pool->head_dim,
                                               vp->max_q))
    return KAP_ECAPACITY;
  return cuda_status(launch_verify(pool_args(pool), map_args(map), vp->max_q, vp->total_q, vp->q_offsets,
                                   vp->q_start_pos, q_dev, out, lse, workspace, workspace_bytes, error_word(),
                                   cs(stream)));
}

const char *kap_status_str(kap_status s) {
  switch (s) {
    case KAP_OK: return "ok";
    case KAP_FALLBACK_FULL: return "plan infeasible for selected access: use full-context attention";
    case KAP_EINVAL: return "invalid argument (NULL pointer, negative size, misaligned buffer)";
    case KAP_ESHAPE: return "inconsistent shapes";
    case KAP_ECAPACITY: return "buffer or capacity too small";
    case KAP_ECUDA: return "CUDA runtime error";
    case KAP_EUNSUPPORTED: return "shape or dtype without a kernel in this build";
  }
  return "unknown status";
}

kap_status kap_rope_inv_freq(int32_t head_dim, double theta, float *inv_freq_host) {
  if (!inv_freq_host || head_dim <= 0 || (head_dim & 1) || !std::isfinite(theta) || !(theta > 0.0)) return KAP_EINVAL;
  for (int32_t i = 0; i < head_dim / 2; ++i)
    inv_freq_host[i] = static_cast<float>(std::pow(theta, -2.0 * i / head_dim));
  return KAP_OK;
}

const char *kap_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

kap_status kap_selftest_wait_timeout(uint32_t polls, uint32_t suspend_ns, int32_t *timed_out_dev, kap_stream stream) {
  if (!timed_out_dev || polls == 0 || polls > 1024u || suspend_ns == 0 || suspend_ns > (1u << 20)) return KAP_EINVAL;
  int *err = error_word();
  if (!err) return KAP_ECUDA;
  return cuda_status(launch_wait_probe(polls, suspend_ns, err, timed_out_dev, cs(stream)));
}

kap_status kap_device_error(int32_t *code_out) {
  if (!code_out) return KAP_EINVAL;
  int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
  if (e != cudaSuccess) return cuda_status(e);
  *code_out = v;
  return KAP_OK;
}

}  // extern "C"
