// k_select.cu - K-summary cache, page scoring, A<a>R<r>K<k> top-K, span selection, compact view compilation and
// slot mapping for the selected-KV hot path (sm_103a).
//
// Sources: EarlySelectKV news page (pages ranked by their K summaries, proxy query allowed), KRI page (KRI-Q:
// Q . block-mean K; the A<a>R<r>K<k> tag), KAP paper (compiler: spans resolved to KV pages, compact view in access
// order with logical positions, block tables and slot mappings).
#include "kap_device.cuh"
#include "kap_launch.h"

namespace kap {
namespace {

// ------------------------------------------------------------------------------------------ summaries
// One CTA per (logical prompt page, request). Sum in fp32 over valid tokens (t ascending), one RN division.
template <class T>
__global__ void __launch_bounds__(128) summaries_kernel(const T *__restrict__ K, float *__restrict__ S,
                                                        int num_pages, int hkv, int d,
                                                        const int32_t *__restrict__ bt, int max_pages,
                                                        const int32_t *__restrict__ ctx_len, int *err) {
  grid_dependency_sync();
  const int r = blockIdx.y, j = blockIdx.x;
  const int L = ctx_len[r];
  const int N = min((L + kPage - 1) / kPage, max_pages);
  if (j >= N) return;
  const int page = bt[static_cast<size_t>(r) * max_pages + j];
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0) set_error(err, kErrPage);
    return;
  }
  const int n = min(kPage, L - kPage * j);
  for (int idx = threadIdx.x; idx < hkv * d; idx += blockDim.x) {
    const int h = idx / d, i = idx - h * d;
    const T *base = K + (static_cast<size_t>(page) * hkv + h) * kPage * d + i;
    float acc = 0.0f;
    for (int t = 0; t < n; ++t) acc = __fadd_rn(acc, to_f(base[static_cast<size_t>(t) * d]));
    S[(static_cast<size_t>(page) * hkv + h) * d + i] = __fdiv_rn(acc, static_cast<float>(n));
  }
}

// ---------------------------------------------------------------------------------------------- scores
// grid.x: chunks of 64 logical pages; grid.y: (request, selection row). 8 warps; each warp scores 8 pages with all
// of their summary loads in flight at once. Dot products follow the fixed order: lane l accumulates fmaf over
// i = l, l+32, ...; then an xor-butterfly 16, 8, 4, 2, 1.
constexpr int kScorePagesPerWarp = 8;
constexpr int kScorePagesPerCta = 8 * kScorePagesPerWarp;
constexpr int kMaxPooledHeads = 16;

template <class T, int D>
__global__ void __launch_bounds__(256) score_kernel(const T *__restrict__ q, const float *__restrict__ S, int hkv,
                                                    int hq, int num_pages, const int32_t *__restrict__ bt,
                                                    int max_pages, const int32_t *__restrict__ ctx_len,
                                                    int per_head, float *__restrict__ scores, int *err) {
  __shared__ float qbar[kMaxPooledHeads][D];
  grid_dependency_sync();
  const int rows = per_head ? hkv : 1;
  const int row = blockIdx.y;
  const int r = row / rows, v = row - r * rows;
  const int G = hq / hkv;
  const int N = min((ctx_len[r] + kPage - 1) / kPage, max_pages);
  const int j0 = blockIdx.x * kScorePagesPerCta;
  if (j0 >= N) return;
  const int h_lo = per_head ? v : 0, h_hi = per_head ? v + 1 : hkv;
  for (int idx = threadIdx.x; idx < (h_hi - h_lo) * D; idx += blockDim.x) {
    const int hh = h_lo + idx / D, i = idx % D;
    float acc = 0.0f;
    for (int g = 0; g < G; ++g) acc = __fadd_rn(acc, to_f(q[(static_cast<size_t>(r) * hq + hh * G + g) * D + i]));
    qbar[hh - h_lo][i] = acc;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int jb = j0 + warp * kScorePagesPerWarp;
  if (jb >= N) return;
  const int32_t *btr = bt + static_cast<size_t>(r) * max_pages;
  int pg[kScorePagesPerWarp];
  bool ok[kScorePagesPerWarp];
#pragma unroll
  for (int u = 0; u < kScorePagesPerWarp; ++u) {
    const int j = jb + u;
    ok[u] = j < N;
    pg[u] = ok[u] ? btr[j] : 0;
    if (ok[u] && (pg[u] < 0 || pg[u] >= num_pages)) {
      ok[u] = false;
      if (lane == 0) set_error(err, kErrPage);
    }
  }
  float tot[kScorePagesPerWarp];
  for (int hh = h_lo; hh < h_hi; ++hh) {
    float sv[kScorePagesPerWarp][D / 32];
#pragma unroll
    for (int u = 0; u < kScorePagesPerWarp; ++u)
#pragma unroll
      for (int c = 0; c < D / 32; ++c)
        sv[u][c] = ok[u] ? __ldg(S + (static_cast<size_t>(pg[u]) * hkv + hh) * D + lane + 32 * c) : 0.0f;
#pragma unroll
    for (int u = 0; u < kScorePagesPerWarp; ++u) {
      float a = 0.0f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) a = __fmaf_rn(qbar[hh - h_lo][lane + 32 * c], sv[u][c], a);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, o));
      tot[u] = (hh == h_lo) ? a : __fadd_rn(tot[u], a);
    }
  }
  if (lane < kScorePagesPerWarp && ok[lane]) {
    float val = tot[0];
#pragma unroll
    for (int u = 1; u < kScorePagesPerWarp; ++u)
      if (lane == u) val = tot[u];
    scores[static_cast<size_t>(row) * max_pages + jb + lane] = val;
  }
}

// ------------------------------------------------------------------------------------ compaction helper
// Writes, in ascending order, every id in [0, N) whose flag is set; the flags come from `flag(j)`. Each thread
// owns a contiguous range of ids. Returns the total count (to every thread).
template <class F>
__device__ int compact_ascending(int N, F flag, int32_t *out, int cap, int *scan_scratch, int *err) {
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int lo = min(N, static_cast<int>(threadIdx.x) * per), hi = min(N, lo + per);
  int cnt = 0;
  for (int j = lo; j < hi; ++j) cnt += flag(j) ? 1 : 0;
  const int incl = block_inclusive_scan(cnt, scan_scratch);
  int pos = incl - cnt;
  for (int j = lo; j < hi; ++j)
    if (flag(j)) {
      if (pos < cap) out[pos] = j;
      ++pos;
    }
  __shared__ int total;
  if (threadIdx.x == blockDim.x - 1) total = incl;
  __syncthreads();
  const int t = total;
  if (t > cap && threadIdx.x == 0) set_error(err, kErrCapacity);
  __syncthreads();
  return t;
}

__device__ __forceinline__ void read_ark(const int32_t *per_seq_ark, int r, int &a, int &rr, int &k) {
  if (per_seq_ark) {
    a = per_seq_ark[3 * r];
    rr = per_seq_ark[3 * r + 1];
    k = per_seq_ark[3 * r + 2];
  }
  a = max(a, 0);
  rr = max(rr, 0);
  k = max(k, 0);
}

// ---------------------------------------------------------------------------------------------- top-K
// One CTA per selection row. Pinned pages [0, a) and [N-r, N); from the middle the k largest scores by a 4-pass
// 8-bit radix select on order keys, ties resolved toward the lower page id; output ascending.
constexpr int kTopkThreads = 512;

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float *__restrict__ scores, int rows,
                                                             const int32_t *__restrict__ ctx_len, int max_pages,
                                                             int a_def, int r_def, int k_def,
                                                             const int32_t *__restrict__ per_seq_ark, int cap,
                                                             int32_t *__restrict__ sel, int32_t *__restrict__ n_sel,
                                                             int *err) {
  extern __shared__ uint32_t keys[];  // [max_pages]
  __shared__ int hist[256];
  __shared__ int scan_scratch[32];
  __shared__ int s_bin, s_remaining;
  grid_dependency_sync();
  const int row = blockIdx.x;
  const int r = row / rows;
  int a = a_def, rr = r_def, k = k_def;
  read_ark(per_seq_ark, r, a, rr, k);
  int N = (ctx_len[r] + kPage - 1) / kPage;
  if (N > max_pages) {
    if (threadIdx.x == 0) set_error(err, kErrLength);
    N = max_pages;
  }
  const int a_end = min(a, N), r_begin = max(0, N - rr);
  const int M = max(0, r_begin - a_end);
  const int kk = min(k, M);
  const float *sc = scores + static_cast<size_t>(row) * max_pages;
  for (int j = a_end + threadIdx.x; j < r_begin; j += blockDim.x) keys[j] = order_key(sc[j]);
  __syncthreads();

  // Radix select of the kk-th largest key among the middle pages.
  uint32_t prefix = 0, mask = 0;
  int remaining = kk;
  const bool all_middle = (kk == M);
  if (kk > 0 && !all_middle) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0;
      __syncthreads();
      for (int j = a_end + threadIdx.x; j < r_begin; j += blockDim.x) {
        const uint32_t key = keys[j];
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int c = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) c += hist[lane * 8 + b];
        // inclusive suffix sum over lanes: sum of c over lanes >= lane
        int suf = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_down_sync(0xffffffffu, suf, o);
          if (lane + o < 32) suf += n;
        }
        const int above = suf - c;  // keys in bins of higher lanes
        if (above < remaining && suf >= remaining) {
          int cum = above;
          for (int b = lane * 8 + 7; b >= lane * 8; --b) {
            if (cum + hist[b] >= remaining) {
              s_bin = b;
              s_remaining = remaining - cum;
              break;
            }
            cum += hist[b];
          }
        }
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(s_bin) << shift;
      mask |= 0xFFu << shift;
      remaining = s_remaining;
      __syncthreads();
    }
  }
  const uint32_t T = prefix;
  const int need = remaining;  // how many keys equal to T are taken (lowest ids first)

  // Rank of each middle page among the pages whose key equals T, in id order.
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int lo = min(N, static_cast<int>(threadIdx.x) * per), hi = min(N, lo + per);
  int eq = 0;
  if (kk > 0 && !all_middle)
    for (int j = max(lo, a_end); j < min(hi, r_begin); ++j) eq += (keys[j] == T) ? 1 : 0;
  const int eq_incl = block_inclusive_scan(eq, scan_scratch);
  const int eq_base = eq_incl - eq;
  // Selection flags, then ascending compaction.
  auto chosen = [&](int j, int &eq_seen) -> bool {
    if (j < a_end || j >= r_begin) return true;
    if (kk == 0) return false;
    if (all_middle) return true;
    const uint32_t key = keys[j];
    if (key > T) return true;
    if (key == T) return (eq_seen++) < need;
    return false;
  };
  int cnt = 0;
  {
    int eq_seen = eq_base;
    for (int j = lo; j < hi; ++j) cnt += chosen(j, eq_seen) ? 1 : 0;
  }
  const int incl = block_inclusive_scan(cnt, scan_scratch);
  int pos = incl - cnt;
  int32_t *out = sel + static_cast<size_t>(row) * cap;
  {
    int eq_seen = eq_base;
    for (int j = lo; j < hi; ++j)
      if (chosen(j, eq_seen)) {
        if (pos < cap) out[pos] = j;
        ++pos;
      }
  }
  if (threadIdx.x == blockDim.x - 1) {
    if (incl > cap) set_error(err, kErrCapacity);
    n_sel[row] = min(incl, cap);
  }
}

// -------------------------------------------------------------------------------------------- spans
// One CTA per request: a prompt page is kept when a token of a span falls in it, plus anchors and recents.
__global__ void __launch_bounds__(512) spans_kernel(const int32_t *__restrict__ ctx_len, int max_pages,
                                                    const int32_t *__restrict__ spans,
                                                    const int32_t *__restrict__ span_offsets, int a_def, int r_def,
                                                    const int32_t *__restrict__ per_seq_ark, int cap,
                                                    int32_t *__restrict__ sel, int32_t *__restrict__ n_sel,
                                                    int *err) {
  extern __shared__ unsigned char keep[];
  __shared__ int scan_scratch[32];
  grid_dependency_sync();
  const int r = blockIdx.x;
  int a = a_def, rr = r_def, k = 0;
  read_ark(per_seq_ark, r, a, rr, k);
  int N = (ctx_len[r] + kPage - 1) / kPage;
  if (N > max_pages) {
    if (threadIdx.x == 0) set_error(err, kErrLength);
    N = max_pages;
  }
  for (int j = threadIdx.x; j < N; j += blockDim.x) keep[j] = (j < a || j >= N - rr) ? 1 : 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int64_t end_tok = static_cast<int64_t>(N) * kPage;
  for (int s = span_offsets[r] + warp; s < span_offsets[r + 1]; s += nw) {
    const int64_t first = spans[2 * s], len = spans[2 * s + 1];
    const int64_t t0 = first > 0 ? first : 0;
    const int64_t t1 = (first + len < end_tok) ? first + len : end_tok;
    if (len <= 0 || t0 >= t1) continue;
    const int p0 = static_cast<int>(t0 / kPage), p1 = static_cast<int>((t1 - 1) / kPage);
    for (int p = p0 + lane; p <= p1; p += 32) keep[p] = 1;
  }
  __syncthreads();
  const int total = compact_ascending(
      N, [&](int j) { return keep[j] != 0; }, sel + static_cast<size_t>(r) * cap, cap, scan_scratch, err);
  if (threadIdx.x == 0) n_sel[r] = min(total, cap);
}

// --------------------------------------------------------------------------------------- compile view
// One CTA per view row: selected pages (ascending) then tail pages, physical ids from the full block table.
__global__ void __launch_bounds__(128) view_kernel(const int32_t *__restrict__ bt, int max_pages,
                                                   const int32_t *__restrict__ ctx_len,
                                                   const int32_t *__restrict__ seq_len,
                                                   const int32_t *__restrict__ sel, const int32_t *__restrict__ n_sel,
                                                   int rows, int sel_cap, int horizon, int32_t *__restrict__ vbt,
                                                   int32_t *__restrict__ vlp, int32_t *__restrict__ vn,
                                                   int32_t *__restrict__ vnsel, int vcap,
                                                   int32_t *__restrict__ fallback, float s_max,
                                                   int64_t *__restrict__ slot_out, int32_t *__restrict__ pos_out,
                                                   int *err) {
  grid_dependency_sync();
  const int row = blockIdx.x;
  const int r = row / rows;
  const int L = ctx_len[r];
  const int N = min((L + kPage - 1) / kPage, max_pages);
  int n = n_sel[row];
  if (n > sel_cap || n < 0) {
    if (threadIdx.x == 0) set_error(err, kErrCapacity);
    n = min(max(n, 0), sel_cap);
  }
  const int32_t *srow = sel + static_cast<size_t>(row) * sel_cap;
  const int32_t *btr = bt + static_cast<size_t>(r) * max_pages;
  const int first_tail = min(L / kPage, max_pages);
  int end_page = static_cast<int>((static_cast<int64_t>(seq_len[r]) + horizon + kPage - 1) / kPage);
  if (end_page > max_pages) {
    if (threadIdx.x == 0) set_error(err, kErrCapacity);
    end_page = max_pages;
  }
  const int last_sel = n > 0 ? srow[n - 1] : -1;
  const int skip = (last_sel == first_tail) ? 1 : 0;
  int n_tail = max(0, end_page - first_tail - skip);
  int n_keep = n;
  if (n_keep > vcap) n_keep = vcap;
  if (n_keep + n_tail > vcap) {
    if (threadIdx.x == 0) set_error(err, kErrCapacity);
    n_tail = vcap - n_keep;
  }
  int32_t *obt = vbt + static_cast<size_t>(row) * vcap;
  int32_t *olp = vlp + static_cast<size_t>(row) * vcap;
  for (int i = threadIdx.x; i < n_keep; i += blockDim.x) {
    const int j = srow[i];
    const bool ok = j >= 0 && j < max_pages;
    if (!ok) set_error(err, kErrPage);
    olp[i] = ok ? j : 0;
    obt[i] = ok ? btr[j] : -1;
  }
  for (int t = threadIdx.x; t < n_tail; t += blockDim.x) {
    const int j = first_tail + skip + t;
    olp[n_keep + t] = j;
    obt[n_keep + t] = btr[j];
  }
  if (slot_out && row % rows == 0) {  // slot mapping of the horizon tokens, once per request
    for (int t = threadIdx.x; t < horizon; t += blockDim.x) {
      const int pos = seq_len[r] + t;
      int64_t slot = -1;
      if (pos >= 0 && pos / kPage < max_pages) {
        const int page = btr[pos / kPage];
        if (page >= 0) slot = static_cast<int64_t>(page) * kPage + pos % kPage;
      }
      slot_out[static_cast<size_t>(r) * horizon + t] = slot;
      if (pos_out) pos_out[static_cast<size_t>(r) * horizon + t] = pos;
    }
  }
  if (threadIdx.x == 0) {
    vn[row] = n_keep + n_tail;
    vnsel[row] = n_keep;
    if (fallback && row % rows == 0) {
      int fb = 0;
      for (int v = 0; v < rows; ++v) {
        const float ratio = static_cast<float>(n_sel[r * rows + v]) / static_cast<float>(max(N, 1));
        fb |= (ratio > s_max) ? 1 : 0;
      }
      fallback[r] = fb;
    }
  }
}

// --------------------------------------------------------------------------------------- slot mapping
__global__ void slot_kernel(const int32_t *__restrict__ bt, int max_pages, int R,
                            const int32_t *__restrict__ tok_offsets, const int32_t *__restrict__ start_pos, int T,
                            int64_t *__restrict__ slot_out, int32_t *__restrict__ pos_out) {
  grid_dependency_sync();
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= T) return;
  int lo = 0, hi = R - 1;  // request r with tok_offsets[r] <= j < tok_offsets[r+1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tok_offsets[mid] <= j) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  const int pos = start_pos[r] + (j - tok_offsets[r]);
  int64_t slot = -1;
  if (pos >= 0 && pos / kPage < max_pages) {
    const int page = bt[static_cast<size_t>(r) * max_pages + pos / kPage];
    if (page >= 0) slot = static_cast<int64_t>(page) * kPage + pos % kPage;
  }
  slot_out[j] = slot;
  if (pos_out) pos_out[j] = pos;
}

}  // namespace

// =============================================================================================== launchers
cudaError_t launch_build_summaries(const PoolArgs &p, const MapArgs &m, int *err, cudaStream_t s) {
  dim3 grid(m.max_pages, m.R);
  if (p.dtype == 0)
    launch_pdl(summaries_kernel<__nv_bfloat16>, grid, dim3(128), 0, s, static_cast<const __nv_bfloat16 *>(p.k),
               p.ksum, p.num_pages, p.hkv, p.d, m.bt, m.max_pages, m.ctx_len, err);
  else
    launch_pdl(summaries_kernel<float>, grid, dim3(128), 0, s, static_cast<const float *>(p.k), p.ksum, p.num_pages,
               p.hkv, p.d, m.bt, m.max_pages, m.ctx_len, err);
  return cudaGetLastError();
}

cudaError_t launch_score(const PoolArgs &p, const MapArgs &m, const void *q, int per_head, float *scores, int *err,
                         cudaStream_t s) {
  const int rows = per_head ? p.hkv : 1;
  dim3 grid((m.max_pages + kScorePagesPerCta - 1) / kScorePagesPerCta, m.R * rows);
#define KAP_SCORE(T, D)                                                                                    \
  launch_pdl(score_kernel<T, D>, grid, dim3(256), 0, s, static_cast<const T *>(q), p.ksum, p.hkv, p.hq,     \
             p.num_pages, m.bt, m.max_pages, m.ctx_len, per_head, scores, err)
  if (p.dtype == 0 && p.d == 128) KAP_SCORE(__nv_bfloat16, 128);
  else if (p.dtype == 0 && p.d == 64) KAP_SCORE(__nv_bfloat16, 64);
  else if (p.dtype == 1 && p.d == 128) KAP_SCORE(float, 128);
  else KAP_SCORE(float, 64);
#undef KAP_SCORE
  return cudaGetLastError();
}

cudaError_t launch_topk(const MapArgs &m, const float *scores, int rows, int a, int r, int k,
                        const int32_t *per_seq_ark, int cap, int32_t *sel, int32_t *n_sel, int *err, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(m.max_pages) * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  launch_pdl(topk_kernel, dim3(m.R * rows), dim3(kTopkThreads), smem, s, scores, rows, m.ctx_len, m.max_pages, a, r,
             k, per_seq_ark, cap, sel, n_sel, err);
  return cudaGetLastError();
}

cudaError_t launch_select_spans(const MapArgs &m, const int32_t *spans, const int32_t *span_offsets, int a, int r,
                                const int32_t *per_seq_ark, int cap, int32_t *sel, int32_t *n_sel, int *err,
                                cudaStream_t s) {
  const size_t smem = static_cast<size_t>(m.max_pages);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(spans_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  launch_pdl(spans_kernel, dim3(m.R), dim3(512), smem, s, m.ctx_len, m.max_pages, spans, span_offsets, a, r,
             per_seq_ark, cap, sel, n_sel, err);
  return cudaGetLastError();
}

cudaError_t launch_compile_view(const MapArgs &m, const int32_t *sel, const int32_t *n_sel, int rows, int sel_cap,
                                int horizon, int32_t *vbt, int32_t *vlp, int32_t *vn, int32_t *vnsel, int vcap,
                                int32_t *fallback, float s_max, int64_t *slot_out, int32_t *pos_out, int *err,
                                cudaStream_t s) {
  launch_pdl(view_kernel, dim3(m.R * rows), dim3(128), 0, s, m.bt, m.max_pages, m.ctx_len, m.seq_len, sel, n_sel,
             rows, sel_cap, horizon, vbt, vlp, vn, vnsel, vcap, fallback, s_max, slot_out, pos_out, err);
  return cudaGetLastError();
}

cudaError_t launch_slot_mapping(const MapArgs &m, const int32_t *tok_offsets, const int32_t *start_pos, int T,
                                int64_t *slot_out, int32_t *pos_out, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  launch_pdl(slot_kernel, dim3((T + 255) / 256), dim3(256), 0, s, m.bt, m.max_pages, m.R, tok_offsets, start_pos, T,
             slot_out, pos_out);
  return cudaGetLastError();
}

}  // namespace kap
