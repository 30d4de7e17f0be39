// k_select.cu - K-summary cache, page scoring, A<a>R<r>K<k> top-K, span selection, compact view compilation and
// slot mapping for the selected-KV hot path (sm_103a).
//
// Sources: EarlySelectKV news page (pages ranked by their K summaries, proxy query allowed), KRI page (KRI-Q:
// Q . block-mean K; the A<a>R<r>K<k> tag), KAP paper (compiler: spans resolved to KV pages, compact view in access
// order with logical positions, block tables and slot mappings).
#include <algorithm>
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

// Refresh of listed pages: one CTA per (physical page, valid-token count) pair, the same arithmetic as
// summaries_kernel, so a refreshed page equals a full rebuild of it bit for bit.
template <class T>
__global__ void __launch_bounds__(128) refresh_summaries_kernel(const T *__restrict__ K, float *__restrict__ S,
                                                                int num_pages, int hkv, int d,
                                                                const int32_t *__restrict__ pages,
                                                                const int32_t *__restrict__ n_valid, int *err) {
  grid_dependency_sync();
  const int page = pages[blockIdx.x];
  const int n = n_valid[blockIdx.x];
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0) set_error(err, kErrPage);
    return;
  }
  if (n < 1 || n > kPage) {
    if (threadIdx.x == 0) set_error(err, kErrLength);
    return;
  }
  for (int idx = threadIdx.x; idx < hkv * d; idx += blockDim.x) {
    const int h = idx / d, i = idx - h * d;
    const T *base = K + (static_cast<size_t>(page) * hkv + h) * kPage * d + i;
    float acc = 0.0f;
    for (int t = 0; t < n; ++t) acc = __fadd_rn(acc, to_f(base[static_cast<size_t>(t) * d]));
    S[(static_cast<size_t>(page) * hkv + h) * d + i] = __fdiv_rn(acc, static_cast<float>(n));
  }
}

// ---------------------------------------------------------------------------------------------- scores
// Work items are (request, selection row, chunk of 32 logical pages); only chunks that hold prompt pages exist. A
// grid of a few CTAs per SM walks them. With kScoreFlatMin < R <= kScoreScanMax requests, every CTA scans the
// requests' item counts into shared memory and takes a contiguous range of items in request, row, chunk order (so
// ragged prompts balance over the SMs and no CTA is spent on pages past a prompt's end). Otherwise grid row r takes
// request r's items, chunk-major, in a strided loop: a CTA then loads its first item's block-table entries and query
// together with the prompt length (one round trip fewer for a small batch). Per item, warp w scores 4 pages. The
// next item's block-table entries and, when its row changes, its query elements are loaded while the current item's
// summaries are in flight.
// Dot products follow the fixed order: lane l accumulates fmaf over i = l, l+32, ...; then an xor-butterfly
// 16, 8, 4, 2, 1. The query of a row is summed over its G heads in ascending order (fp32), once per row.
constexpr int kScorePagesPerWarp = 4;
constexpr int kScorePagesPerCta = 8 * kScorePagesPerWarp;
constexpr int kMaxPooledHeads = 16;
constexpr int kScoreCtasPerSm = 4;
constexpr int kScoreScanMax = 2048;
constexpr int kScoreFlatMin = 8;  // with at most this many requests, each request's items go to its own grid row

struct ScoreItem {
  int r, v, j0, N;  // request, row within the request, first page, prompt pages of the request
};

template <class T, int D, bool PER_HEAD>
__global__ void __launch_bounds__(256, kScoreCtasPerSm) score_kernel(
    const T *__restrict__ q, const float *__restrict__ S, int hkv, int hq, int num_pages,
    const int32_t *__restrict__ bt, int max_pages, const int32_t *__restrict__ ctx_len, int R,
    float *__restrict__ scores, int *err) {
  constexpr int C = D / 32;
  // query elements a thread sums: one head's row, or the pooled heads' rows
  constexpr int QPT = ((PER_HEAD ? 1 : kMaxPooledHeads) * D + 255) / 256;
  constexpr bool per_head = PER_HEAD;
  __shared__ float qbar[kMaxPooledHeads][D];
  __shared__ int s_cum[kScoreScanMax + 1];  // items before request r
  __shared__ int s_np[kScoreScanMax];       // prompt pages of request r
  __shared__ int scan_scratch[32];
  grid_dependency_sync();
  const int rows = per_head ? hkv : 1;
  const int G = hq / hkv;
  const int nh = per_head ? 1 : hkv;  // heads pooled into one row
  const int nq = nh * D;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool flat = R > kScoreFlatMin && R <= kScoreScanMax;  // uniform over the grid
  auto pages_of = [&](int r) { return min((ctx_len[r] + kPage - 1) / kPage, max_pages); };

  int64_t t = 0, t_end = 0, t_step = 1;
  int r_cur = 0;
  if (flat) {
    const int per = (R + 255) / 256;
    const int lo = min(R, static_cast<int>(threadIdx.x) * per), hi = min(R, lo + per);
    auto items_of = [&](int n) { return rows * ((n + kScorePagesPerCta - 1) / kScorePagesPerCta); };
    int cnt = 0;
    for (int r = lo; r < hi; ++r) {
      const int n = pages_of(r);
      s_np[r] = n;
      cnt += items_of(n);
    }
    const int incl = block_inclusive_scan(cnt, scan_scratch);
    int run = incl - cnt;
    for (int r = lo; r < hi; ++r) {
      s_cum[r] = run;
      run += items_of(s_np[r]);
    }
    if (threadIdx.x == 255) s_cum[R] = incl;
    __syncthreads();
    const int64_t W = s_cum[R];
    t = static_cast<int64_t>(blockIdx.x) * W / gridDim.x;
    t_end = static_cast<int64_t>(blockIdx.x + 1) * W / gridDim.x;
    int lo_r = 0, hi_r = R - 1;  // the request holding item t: the last r with s_cum[r] <= t
    while (lo_r < hi_r) {
      const int mid = (lo_r + hi_r + 1) >> 1;
      if (s_cum[mid] <= t) lo_r = mid; else hi_r = mid - 1;
    }
    r_cur = lo_r;
  }
  int n_req = 0;  // per-request mode: the request's prompt pages
  if (!flat) {
    // items chunk-major (t = chunk * rows + row), so that an item's pages are known before the prompt length
    r_cur = blockIdx.y;
    n_req = pages_of(r_cur);  // in flight while the first item's loads are issued
    t = blockIdx.x;
    t_step = gridDim.x;
  }
  auto decode = [&](int64_t ti) {
    ScoreItem it;
    if (flat) {
      while (ti >= s_cum[r_cur + 1]) ++r_cur;  // items are visited in ascending order
      it.r = r_cur;
      it.N = s_np[r_cur];
      const int within = static_cast<int>(ti - s_cum[r_cur]);
      const int nch = (it.N + kScorePagesPerCta - 1) / kScorePagesPerCta;
      it.v = within / nch;
      it.j0 = (within - it.v * nch) * kScorePagesPerCta;
    } else {
      it.r = r_cur;
      it.N = n_req;
      it.v = static_cast<int>(ti % rows);
      it.j0 = static_cast<int>(ti / rows) * kScorePagesPerCta;
    }
    return it;
  };
  // this warp's block-table entries of an item (masked to the prompt where the scores are formed)
  auto load_pages = [&](const ScoreItem &it, int (&pg)[kScorePagesPerWarp]) {
    const int jb = it.j0 + warp * kScorePagesPerWarp;
    const int32_t *btr = bt + static_cast<size_t>(it.r) * max_pages;
#pragma unroll
    for (int u = 0; u < kScorePagesPerWarp; ++u) pg[u] = (jb + u < max_pages) ? btr[jb + u] : -1;
  };
  // this thread's elements of the row's group-summed query (heads ascending, fp32)
  auto load_query = [&](const ScoreItem &it, float (&qs)[QPT]) {
    const int h_lo = per_head ? it.v : 0;
#pragma unroll
    for (int e = 0; e < QPT; ++e) {
      const int i = static_cast<int>(threadIdx.x) + 256 * e;
      float acc = 0.0f;
      if (i < nq) {
        const T *qr = q + (static_cast<size_t>(it.r) * hq + (h_lo + i / D) * G) * D + i % D;
        for (int g = 0; g < G; ++g) acc = __fadd_rn(acc, to_f(qr[static_cast<size_t>(g) * D]));
      }
      qs[e] = acc;
    }
  };

  ScoreItem cur = decode(t);
  int pg[kScorePagesPerWarp];
  float qs[QPT];
  if (!flat) {
    load_pages(cur, pg);
    load_query(cur, qs);
    cur.N = n_req;  // the first use of the prompt length
    t_end = static_cast<int64_t>(rows) * ((n_req + kScorePagesPerCta - 1) / kScorePagesPerCta);
  }
  if (t >= t_end) return;
  if (flat) {
    load_pages(cur, pg);
    load_query(cur, qs);
  }
  int qrow = -1;  // the row whose query sits in qbar
  while (true) {
    const int row = cur.r * rows + cur.v;
    const int h_lo = per_head ? cur.v : 0;
    const int jb = cur.j0 + warp * kScorePagesPerWarp;
    bool ok[kScorePagesPerWarp];
    int pc[kScorePagesPerWarp];
#pragma unroll
    for (int u = 0; u < kScorePagesPerWarp; ++u) {
      ok[u] = jb + u < cur.N;
      if (ok[u] && (pg[u] < 0 || pg[u] >= num_pages)) {
        ok[u] = false;
        if (lane == 0) set_error(err, kErrPage);
      }
      pc[u] = ok[u] ? pg[u] : 0;  // a valid page: the loads below are unconditional
    }
    float sv[kScorePagesPerWarp][C];
#pragma unroll
    for (int u = 0; u < kScorePagesPerWarp; ++u)
#pragma unroll
      for (int c = 0; c < C; ++c) sv[u][c] = __ldg(S + (static_cast<size_t>(pc[u]) * hkv + h_lo) * D + lane + 32 * c);
    // the next item's block-table entries, and its query when its row differs, while the summaries are in flight
    const int64_t tn = t + t_step;
    const bool more = tn < t_end;
    ScoreItem nxt = cur;
    int pgn[kScorePagesPerWarp];
    float qsn[QPT];
    if (more) {
      nxt = decode(tn);
      load_pages(nxt, pgn);
      if (nxt.r * rows + nxt.v != row) load_query(nxt, qsn);
    }
    if (row != qrow) {  // uniform over the CTA
      __syncthreads();  // every warp is done with the previous row's query
#pragma unroll
      for (int e = 0; e < QPT; ++e) {
        const int i = static_cast<int>(threadIdx.x) + 256 * e;
        if (i < nq) qbar[i / D][i % D] = qs[e];
      }
      __syncthreads();
      qrow = row;
    }
    float tot[kScorePagesPerWarp];
    for (int hh = 0; hh < nh; ++hh) {
      if (hh > 0) {
#pragma unroll
        for (int u = 0; u < kScorePagesPerWarp; ++u)
#pragma unroll
          for (int c = 0; c < C; ++c)
            sv[u][c] = __ldg(S + (static_cast<size_t>(pc[u]) * hkv + h_lo + hh) * D + lane + 32 * c);
      }
#pragma unroll
      for (int u = 0; u < kScorePagesPerWarp; ++u) {
        float acc = 0.0f;
#pragma unroll
        for (int c = 0; c < C; ++c) acc = __fmaf_rn(qbar[hh][lane + 32 * c], sv[u][c], acc);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
        tot[u] = (hh == 0) ? acc : __fadd_rn(tot[u], acc);
      }
    }
    float val = tot[0];
    bool okl = ok[0];
#pragma unroll
    for (int u = 1; u < kScorePagesPerWarp; ++u)
      if (lane == u) {
        val = tot[u];
        okl = ok[u];
      }
    if (lane < kScorePagesPerWarp && okl) scores[static_cast<size_t>(row) * max_pages + jb + lane] = val;
    if (!more) break;
    t = tn;
    cur = nxt;
#pragma unroll
    for (int u = 0; u < kScorePagesPerWarp; ++u) pg[u] = pgn[u];
    if (nxt.r * rows + nxt.v != row) {
#pragma unroll
      for (int e = 0; e < QPT; ++e) qs[e] = qsn[e];
    }
  }
}

// ------------------------------------------------------------------------------------ compaction helper
// Writes, in ascending order, every id in [0, N) whose flag is set; the flags come from `flag(j)`. Each thread
// owns a contiguous range of ids. Returns the total count (to every thread).
// ------------------------------------------------------------------------------ external-prior scores
// KRI page, prior schema: a baked block_affinities[L][H][N] per request is mean-pooled over layers and heads before
// the per-request top-K. The page fixes no summation order; this one is fixed so selections reproduce bit for bit:
// rows i = l*H + h are summed in chunks of 32 (each chunk from 0, i ascending), the chunk sums are added in
// ascending order (from 0), and the total is divided by L*H once (round to nearest). One CTA covers 32 consecutive
// blocks of one request: lane = block, so each load is one 128-byte row segment; warp w sums chunks w, w+8, ...
// with all 32 loads of a chunk in flight; warp 0 adds the chunk sums in order.
constexpr int kPriorWarps = 8;
constexpr int kPriorMaxChunks = 64;  // L*H <= 2048

__global__ void __launch_bounds__(kPriorWarps * 32) prior_score_kernel(const float *__restrict__ aff, int M,
                                                                       int max_pages,
                                                                       const int32_t *__restrict__ ctx_len,
                                                                       float *__restrict__ scores) {
  __shared__ float csum[kPriorMaxChunks][32];
  grid_dependency_sync();
  const int r = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = blockIdx.x * 32 + lane;
  const int N = min(max_pages, (ctx_len[r] + kPage - 1) / kPage);
  const bool ok = n < N;
  const int nch = (M + 31) / 32;
  const float *col = aff + static_cast<size_t>(r) * M * max_pages + (ok ? n : 0);  // clamped: always in bounds
  for (int c = warp; c < nch; c += kPriorWarps) {
    const int i0 = c * 32;
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = (i0 + j < M) ? __ldcs(col + static_cast<size_t>(i0 + j) * max_pages) : 0.0f;
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (i0 + j < M) sum = __fadd_rn(sum, x[j]);
    csum[c][lane] = sum;
  }
  __syncthreads();
  if (warp == 0 && ok) {
    float t = 0.0f;
    for (int c = 0; c < nch; ++c) t = __fadd_rn(t, csum[c][lane]);
    scores[static_cast<size_t>(r) * max_pages + n] = __fdiv_rn(t, static_cast<float>(M));
  }
}

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

// --------------------------------------------------------------------------------------- compile view
// One view row: the n selected pages (ascending, sel_at(i)) then the tail pages, physical ids from the full block
// table; the horizon's slot mapping and the request's fallback flag come with the request's first row.
struct ViewOut {
  int32_t *vbt, *vlp, *vn, *vnsel;
  int vcap, sel_cap, horizon;
  int32_t *fallback;
  float s_max;
  int64_t *slot_out;
  int32_t *pos_out;
};

template <class SelAt, class NselOf>
__device__ void compile_view_row(int row, int rows, const int32_t *__restrict__ bt, int max_pages, int L, int S,
                                 int n, SelAt sel_at, NselOf nsel_of, const ViewOut &vo, int *err) {
  const int r = row / rows;
  const int N = min((L + kPage - 1) / kPage, max_pages);
  if (n > vo.sel_cap || n < 0) {
    if (threadIdx.x == 0) set_error(err, kErrCapacity);
    n = min(max(n, 0), vo.sel_cap);
  }
  const int32_t *btr = bt + static_cast<size_t>(r) * max_pages;
  const int first_tail = min(L / kPage, max_pages);
  int end_page = static_cast<int>((static_cast<int64_t>(S) + vo.horizon + kPage - 1) / kPage);
  if (end_page > max_pages) {
    if (threadIdx.x == 0) set_error(err, kErrCapacity);
    end_page = max_pages;
  }
  const int last_sel = n > 0 ? sel_at(n - 1) : -1;
  const int skip = (last_sel == first_tail) ? 1 : 0;
  int n_tail = max(0, end_page - first_tail - skip);
  int n_keep = n;
  if (n_keep > vo.vcap) n_keep = vo.vcap;
  if (n_keep + n_tail > vo.vcap) {
    if (threadIdx.x == 0) set_error(err, kErrCapacity);
    n_tail = vo.vcap - n_keep;
  }
  int32_t *obt = vo.vbt + static_cast<size_t>(row) * vo.vcap;
  int32_t *olp = vo.vlp + static_cast<size_t>(row) * vo.vcap;
  for (int i = threadIdx.x; i < n_keep; i += blockDim.x) {
    const int j = sel_at(i);
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
  if (vo.slot_out && row % rows == 0) {  // slot mapping of the horizon tokens, once per request
    for (int t = threadIdx.x; t < vo.horizon; t += blockDim.x) {
      const int pos = S + t;
      int64_t slot = -1;
      if (pos >= 0 && pos / kPage < max_pages) {
        const int page = btr[pos / kPage];
        if (page >= 0) slot = static_cast<int64_t>(page) * kPage + pos % kPage;
      }
      vo.slot_out[static_cast<size_t>(r) * vo.horizon + t] = slot;
      if (vo.pos_out) vo.pos_out[static_cast<size_t>(r) * vo.horizon + t] = pos;
    }
  }
  if (threadIdx.x == 0) {
    vo.vn[row] = n_keep + n_tail;
    vo.vnsel[row] = n_keep;
    if (vo.fallback && row % rows == 0) {
      int fb = 0;
      for (int v = 0; v < rows; ++v) {
        const float ratio = static_cast<float>(nsel_of(r * rows + v)) / static_cast<float>(max(N, 1));
        fb |= (ratio > vo.s_max) ? 1 : 0;
      }
      vo.fallback[r] = fb;
    }
  }
}

// ---------------------------------------------------------------------------------------------- top-K
// One CTA per selection row. Pinned pages [0, a) and [N-r, N); from the middle the k largest scores by a 4-pass
// 8-bit radix select on order keys, ties resolved toward the lower page id; output ascending. With VIEW the CTA also
// compiles its view row from the selection it just made (every row of a request selects the same number of pages,
// so the request's fallback flag needs no other row).
constexpr int kTopkThreads = 512;
constexpr int kCandMax = 64;  // once at most this many keys share the selected prefix, they are ranked directly

template <bool VIEW>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float *__restrict__ scores, int rows,
                                                             const int32_t *__restrict__ ctx_len, int max_pages,
                                                             int a_def, int r_def, int k_def,
                                                             const int32_t *__restrict__ per_seq_ark, int cap,
                                                             int32_t *__restrict__ sel, int32_t *__restrict__ n_sel,
                                                             const int32_t *__restrict__ bt,
                                                             const int32_t *__restrict__ seq_len, const ViewOut vo,
                                                             int *err) {
  extern __shared__ uint32_t keys[];  // [max_pages], then (VIEW) the selection [cap]
  int32_t *sel_s = reinterpret_cast<int32_t *>(keys + max_pages);
  __shared__ int s_nsel;
  __shared__ int hist2[2][256];  // pass p counts into hist2[p & 1] while hist2[(p + 1) & 1] is cleared
  __shared__ unsigned long long scan_scratch[32];
  __shared__ int s_bin, s_remaining, s_cnt, s_ncand, s_need;
  __shared__ uint32_t s_cand[kCandMax], s_T;
  if (threadIdx.x == 0) s_ncand = 0;
  grid_dependency_sync();
  const int row = blockIdx.x;
  const int r = row / rows;
  int a = a_def, rr = r_def, k = k_def;
  read_ark(per_seq_ark, r, a, rr, k);
  const int Lr = ctx_len[r];
  const int Sr = VIEW ? seq_len[r] : 0;
  int N = (Lr + kPage - 1) / kPage;
  if (N > max_pages) {
    if (threadIdx.x == 0) set_error(err, kErrLength);
    N = max_pages;
  }
  const int a_end = min(a, N), r_begin = max(0, N - rr);
  const int M = max(0, r_begin - a_end);
  const int kk = min(k, M);
  const float *sc = scores + static_cast<size_t>(row) * max_pages;
  // middle-page keys, four loads in flight per thread (clamped indices: every load is issued)
  for (int base = a_end; base < r_begin; base += 4 * static_cast<int>(blockDim.x)) {
    float vals[4];
    int js[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      js[u] = base + u * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x);
      vals[u] = sc[min(js[u], r_begin - 1)];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (js[u] < r_begin) keys[js[u]] = order_key(vals[u]);
  }
  __syncthreads();

  // Radix select of the kk-th largest key among the middle pages.
  uint32_t prefix = 0, mask = 0;
  int remaining = kk;
  const bool all_middle = (kk == M);
  if (kk > 0 && !all_middle) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist2[0][b] = 0;
    __syncthreads();
    const int lane_id = threadIdx.x & 31;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      int *hist = hist2[pass & 1];
      for (int b = threadIdx.x; b < 256; b += blockDim.x) hist2[(pass + 1) & 1][b] = 0;
      // Scores of similar magnitude share few leading key bytes: lanes of a warp with equal bins are merged into
      // one shared-memory atomic (the loop trip count is uniform over the block, so the warp stays converged).
      for (int jj = a_end; jj < r_begin; jj += blockDim.x) {
        const int j = jj + static_cast<int>(threadIdx.x);
        const uint32_t key = j < r_begin ? keys[j] : 0u;
        const bool take = j < r_begin && (key & mask) == prefix;
        const unsigned tm = __ballot_sync(0xffffffffu, take);
        if (take) {
          const int bin = static_cast<int>((key >> shift) & 255u);
          const unsigned grp = __match_any_sync(tm, bin);
          if (lane_id == __ffs(grp) - 1) atomicAdd(&hist[bin], __popc(grp));
        }
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
              s_cnt = hist[b];
              break;
            }
            cum += hist[b];
          }
        }
      }
      __syncthreads();
      // s_bin / s_remaining are rewritten only after the next pass's first barrier
      prefix |= static_cast<uint32_t>(s_bin) << shift;
      mask |= 0xFFu << shift;
      remaining = s_remaining;
      if (pass < 3 && s_cnt <= kCandMax) {
        // Few keys left with this prefix: gather them and take the remaining-th largest exactly. T is the key with
        // fewer than `remaining` candidates above it and at least `remaining` at or above it.
        for (int jj = a_end; jj < r_begin; jj += blockDim.x) {
          const int j = jj + static_cast<int>(threadIdx.x);
          if (j < r_begin) {
            const uint32_t key = keys[j];
            if ((key & mask) == prefix) s_cand[atomicAdd(&s_ncand, 1)] = key;
          }
        }
        __syncthreads();
        if (threadIdx.x < 32) {
          const int nc = s_ncand;
          for (int c0 = lane_id; c0 < nc; c0 += 32) {
            const uint32_t x = s_cand[c0];
            int gt = 0, ge = 0;
            for (int i = 0; i < nc; ++i) {
              const uint32_t y = s_cand[i];
              gt += y > x ? 1 : 0;
              ge += y >= x ? 1 : 0;
            }
            if (gt < remaining && remaining <= ge) {  // equal candidates write equal values
              s_T = x;
              s_need = remaining - gt;
            }
          }
        }
        __syncthreads();
        prefix = s_T;
        mask = 0xFFFFFFFFu;
        remaining = s_need;
        break;
      }
    }
  }
  const uint32_t T = prefix;
  const int need = remaining;  // how many keys equal to T are taken (lowest ids first)

  // One block scan of packed counts per thread's id range: low half the pages taken for certain (pinned, or key
  // above T), high half the middle pages whose key equals T. In id order, the first `need` of the latter are taken.
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int lo = min(N, static_cast<int>(threadIdx.x) * per), hi = min(N, lo + per);
  const bool radix = kk > 0 && !all_middle;
  int c_sure = 0, c_eq = 0;
  for (int j = lo; j < hi; ++j) {
    if (j < a_end || j >= r_begin || (kk > 0 && all_middle)) {
      ++c_sure;
    } else if (radix) {
      const uint32_t key = keys[j];
      c_sure += key > T ? 1 : 0;
      c_eq += key == T ? 1 : 0;
    }
  }
  const unsigned long long mine = static_cast<unsigned long long>(c_sure) |
                                  (static_cast<unsigned long long>(c_eq) << 32);
  const unsigned long long incl = block_inclusive_scan(mine, scan_scratch);
  const unsigned long long excl = incl - mine;
  const int sure_before = static_cast<int>(excl & 0xffffffffull), eq_before = static_cast<int>(excl >> 32);
  int pos = sure_before + min(eq_before, need);
  int eq_seen = eq_before;
  int32_t *out = sel + static_cast<size_t>(row) * cap;
  for (int j = lo; j < hi; ++j) {
    bool take;
    if (j < a_end || j >= r_begin || (kk > 0 && all_middle)) {
      take = true;
    } else if (radix) {
      const uint32_t key = keys[j];
      take = key > T || (key == T && (eq_seen++) < need);
    } else {
      take = false;
    }
    if (take) {
      if (pos < cap) {
        out[pos] = j;
        if (VIEW) sel_s[pos] = j;
      }
      ++pos;
    }
  }
  if (threadIdx.x == blockDim.x - 1) {
    const int total = static_cast<int>(incl & 0xffffffffull) + min(static_cast<int>(incl >> 32), need);
    if (total > cap) set_error(err, kErrCapacity);
    n_sel[row] = min(total, cap);
    s_nsel = min(total, cap);
  }
  if (VIEW) {
    __syncthreads();
    const int n = s_nsel;
    compile_view_row(
        row, rows, bt, max_pages, Lr, Sr, n, [&](int i) { return sel_s[i]; }, [&](int) { return n; }, vo, err);
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

// One CTA per view row, reading a selection made by an earlier kernel.
__global__ void __launch_bounds__(128) view_kernel(const int32_t *__restrict__ bt, int max_pages,
                                                   const int32_t *__restrict__ ctx_len,
                                                   const int32_t *__restrict__ seq_len,
                                                   const int32_t *__restrict__ sel, const int32_t *__restrict__ n_sel,
                                                   int rows, const ViewOut vo, int *err) {
  grid_dependency_sync();
  const int row = blockIdx.x;
  const int r = row / rows;
  const int32_t *srow = sel + static_cast<size_t>(row) * vo.sel_cap;
  compile_view_row(
      row, rows, bt, max_pages, ctx_len[r], seq_len[r], n_sel[row], [&](int i) { return srow[i]; },
      [&](int rr) { return n_sel[rr]; }, vo, err);
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

cudaError_t launch_refresh_summaries(const PoolArgs &p, const int32_t *pages, const int32_t *n_valid, int n, int *err,
                                     cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (p.dtype == 0)
    launch_pdl(refresh_summaries_kernel<__nv_bfloat16>, dim3(n), dim3(128), 0, s,
               static_cast<const __nv_bfloat16 *>(p.k), p.ksum, p.num_pages, p.hkv, p.d, pages, n_valid, err);
  else
    launch_pdl(refresh_summaries_kernel<float>, dim3(n), dim3(128), 0, s, static_cast<const float *>(p.k), p.ksum,
               p.num_pages, p.hkv, p.d, pages, n_valid, err);
  return cudaGetLastError();
}

template <class T, int D>
void launch_score_td(const PoolArgs &p, const MapArgs &m, const void *q, int per_head, float *scores, int *err,
                     dim3 grid, cudaStream_t s) {
  const T *qt = static_cast<const T *>(q);
  if (per_head)
    launch_pdl(score_kernel<T, D, true>, grid, dim3(256), 0, s, qt, p.ksum, p.hkv, p.hq, p.num_pages, m.bt,
               m.max_pages, m.ctx_len, m.R, scores, err);
  else
    launch_pdl(score_kernel<T, D, false>, grid, dim3(256), 0, s, qt, p.ksum, p.hkv, p.hq, p.num_pages, m.bt,
               m.max_pages, m.ctx_len, m.R, scores, err);
}

cudaError_t launch_score(const PoolArgs &p, const MapArgs &m, const void *q, int per_head, float *scores, int *err,
                         cudaStream_t s) {
  const int rows = per_head ? p.hkv : 1;
  // Items: at most rows * ceil(max_pages / 32) per request. A few CTAs per SM, never more than there are items.
  const int64_t per_req = static_cast<int64_t>(rows) * ((m.max_pages + kScorePagesPerCta - 1) / kScorePagesPerCta);
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * kScoreCtasPerSm;
  dim3 grid;
  if (m.R > kScoreFlatMin && m.R <= kScoreScanMax) {
    grid = dim3(static_cast<unsigned>(std::min<int64_t>(cap, per_req * m.R)));
  } else {
    grid = dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(per_req, cap / m.R))), m.R);
  }
  if (p.dtype == 0 && p.d == 128) launch_score_td<__nv_bfloat16, 128>(p, m, q, per_head, scores, err, grid, s);
  else if (p.dtype == 0 && p.d == 64) launch_score_td<__nv_bfloat16, 64>(p, m, q, per_head, scores, err, grid, s);
  else if (p.dtype == 1 && p.d == 128) launch_score_td<float, 128>(p, m, q, per_head, scores, err, grid, s);
  else launch_score_td<float, 64>(p, m, q, per_head, scores, err, grid, s);
  return cudaGetLastError();
}

cudaError_t launch_topk(const MapArgs &m, const float *scores, int rows, int a, int r, int k,
                        const int32_t *per_seq_ark, int cap, int32_t *sel, int32_t *n_sel, const ViewArgsOut *view,
                        int *err, cudaStream_t s) {
  const bool with_view = view != nullptr;
  const size_t smem = static_cast<size_t>(m.max_pages) * sizeof(uint32_t) + (with_view ? cap * sizeof(int32_t) : 0);
  auto kern = with_view ? topk_kernel<true> : topk_kernel<false>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  ViewOut vo{};
  if (with_view)
    vo = ViewOut{view->vbt, view->vlp, view->vn, view->vnsel, view->vcap, cap, view->horizon, view->fallback,
                 view->s_max, view->slot_out, view->pos_out};
  launch_pdl(kern, dim3(m.R * rows), dim3(kTopkThreads), smem, s, scores, rows, m.ctx_len, m.max_pages, a, r, k,
             per_seq_ark, cap, sel, n_sel, m.bt, m.seq_len, vo, err);
  return cudaGetLastError();
}

cudaError_t launch_prior_topk(const MapArgs &m, const float *aff, int L, int H, int a, int r, int k,
                              const int32_t *per_seq_ark, int cap, int32_t *sel, int32_t *n_sel, float *scores,
                              int *err, cudaStream_t s) {
  const int M = L * H;
  if (M < 1 || M > 32 * kPriorMaxChunks) return cudaErrorInvalidValue;
  dim3 grid((m.max_pages + 31) / 32, m.R);
  launch_pdl(prior_score_kernel, grid, dim3(kPriorWarps * 32), 0, s, aff, M, m.max_pages, m.ctx_len, scores);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_topk(m, scores, 1, a, r, k, per_seq_ark, cap, sel, n_sel, nullptr, err, s);
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
  const ViewOut vo{vbt, vlp, vn, vnsel, vcap, sel_cap, horizon, fallback, s_max, slot_out, pos_out};
  launch_pdl(view_kernel, dim3(m.R * rows), dim3(128), 0, s, m.bt, m.max_pages, m.ctx_len, m.seq_len, sel, n_sel,
             rows, vo, err);
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
