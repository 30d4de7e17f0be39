// kap_oracle.cpp - plain, slow CPU oracle of the selected-KV sparse decode hot path.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path may call this file: only the tests, the smoke check and
// the benchmark's CPU-baseline leg load it. It shares no code, header or constant with the CUDA library.
//
// Every function is the plain definition of its step, written straight from the pages:
//   * "KAP: Bridging the Knowledge Selection-Runtime Consumption Gap in LLM Systems" (arXiv paper and the
//     agifrontier.github.io tutorial): selected-KV view, slot mapping, proposal q=1, verifier window, cost model.
//   * KRI page (knlp.io/kri.html): A<a>R<r>K<k> tag with its 128-block example; KRI-Q (Q . block-mean K);
//     skip-list semantics of the connector.
//   * EarlySelectKV news page: score and top-k over a K-summary cache, with a proxy query.
// Attention is an explicit enumeration of the visible (token, position) pairs followed by a softmax in fp64; there
// is no paging trick, no online softmax and no split. Inputs arrive as fp32 arrays (bf16 values are exact in fp32).
//
// Where floating point decides an integer (page scores decide the top-K), the oracle computes in fp32 in the
// one fixed order the library specifies (sequential token sum for the block mean; the 32-lane fmaf order and
// xor-butterfly for the dot product), so that both sides take the decision on identical numbers.
//
// Built with -ffp-contract=off so that the compiler does not fuse a*b+c behind the oracle's back.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr int kPage = 16;  // tokens per KV page (all configurations)

inline const float *kv_row(const float *pool, int page, int head, int tok, int hkv, int d) {
  return pool + ((static_cast<int64_t>(page) * hkv + head) * kPage + tok) * d;
}

// Runs f(unit) for unit in [0, n) on up to nthreads threads.
template <class F>
void parallel_units(int n, int nthreads, F f) {
  if (nthreads <= 1 || n <= 1) {
    for (int u = 0; u < n; ++u) f(u);
    return;
  }
  int nt = std::min(nthreads, n);
  std::vector<std::thread> ts;
  for (int t = 0; t < nt; ++t)
    ts.emplace_back([=]() {
      for (int u = t; u < n; u += nt) f(u);
    });
  for (auto &th : ts) th.join();
}

// Softmax-weighted sum over an explicit list of visible positions, in fp64.
// logits_j = (q . k_j) / sqrt(d); out = sum_j softmax_j * v_j; lse = log sum_j exp(logit_j).
void attend(const float *q, const std::vector<const float *> &ks, const std::vector<const float *> &vs, int d,
            double *out, double *lse) {
  const size_t n = ks.size();
  std::vector<double> logit(n);
  const double scale = 1.0 / std::sqrt(static_cast<double>(d));
  double mx = -INFINITY;
  for (size_t j = 0; j < n; ++j) {
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += static_cast<double>(q[i]) * static_cast<double>(ks[j][i]);
    logit[j] = s * scale;
    mx = std::max(mx, logit[j]);
  }
  double denom = 0.0;
  for (size_t j = 0; j < n; ++j) denom += std::exp(logit[j] - mx);
  for (int i = 0; i < d; ++i) out[i] = 0.0;
  for (size_t j = 0; j < n; ++j) {
    const double w = std::exp(logit[j] - mx) / denom;
    for (int i = 0; i < d; ++i) out[i] += w * static_cast<double>(vs[j][i]);
  }
  *lse = mx + std::log(denom);
}

// Monotone map of a float score onto an unsigned key: larger score -> larger key. -0 and +0 map to the same key;
// NaN maps to 0, below every number.
uint32_t order_key(float f) {
  if (std::isnan(f)) return 0u;
  if (f == 0.0f) f = 0.0f;
  uint32_t b;
  std::memcpy(&b, &f, 4);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------------------------------------------
// K-summary cache: block-mean K per (page, KV head) over the page's valid prompt tokens.
// EarlySelectKV page (K-summary cache) and the KRI page (KRI-Q: block-mean K). Sum in fp32, t ascending,
// then one IEEE division by the count.
int orc_build_summaries(const float *K, int num_pages, int hkv, int d, const int32_t *block_table, int R,
                        int max_pages, const int32_t *ctx_len, float *S) {
  for (int r = 0; r < R; ++r) {
    const int L = ctx_len[r];
    const int N = (L + kPage - 1) / kPage;
    for (int j = 0; j < N; ++j) {
      const int page = block_table[static_cast<int64_t>(r) * max_pages + j];
      if (page < 0 || page >= num_pages) return -1;
      const int n = std::min(kPage, L - kPage * j);
      for (int h = 0; h < hkv; ++h) {
        for (int i = 0; i < d; ++i) {
          float acc = 0.0f;
          for (int t = 0; t < n; ++t) acc += kv_row(K, page, h, t, hkv, d)[i];
          S[(static_cast<int64_t>(page) * hkv + h) * d + i] = acc / static_cast<float>(n);
        }
      }
    }
  }
  return 0;
}

// Dot product of two length-d fp32 vectors in the library's fixed order: 32 partial sums, partial l taking
// i = l, l+32, ... with fmaf, then pairwise combination by xor distance 16, 8, 4, 2, 1; partial 0 is the result.
float orc_dot_fixed_order(const float *a, const float *b, int d) {
  float part[32];
  for (int l = 0; l < 32; ++l) {
    float acc = 0.0f;
    for (int i = l; i < d; i += 32) acc = std::fma(a[i], b[i], acc);
    part[l] = acc;
  }
  for (int off = 16; off >= 1; off >>= 1) {
    float next[32];
    for (int l = 0; l < 32; ++l) next[l] = part[l] + part[l ^ off];
    std::memcpy(part, next, sizeof(part));
  }
  return part[0];
}

// Page scores against the group-summed query (KRI-Q on the KRI page; EarlySelectKV's selector on a
// K-summary cache). qbar[h] = sum_g q[h*G+g] (fp32, g ascending). Per-head rows: score[r][h][j]; shared rows
// (per_head = 0): score[r][0][j] = sum over h ascending of the per-head scores. Also the fp64 value of the same
// quantity (for diagnosing near ties). Entries j >= N are left untouched.
int orc_scores(const float *q, const float *S, int hq, int hkv, int d, const int32_t *block_table, int R,
               int max_pages, const int32_t *ctx_len, int per_head, float *scores, double *scores64) {
  const int G = hq / hkv;
  const int rows = per_head ? hkv : 1;
  std::vector<float> qbar(static_cast<size_t>(hkv) * d);
  for (int r = 0; r < R; ++r) {
    for (int h = 0; h < hkv; ++h)
      for (int i = 0; i < d; ++i) {
        float acc = 0.0f;
        for (int g = 0; g < G; ++g) acc += q[(static_cast<int64_t>(r) * hq + h * G + g) * d + i];
        qbar[static_cast<size_t>(h) * d + i] = acc;
      }
    const int N = (ctx_len[r] + kPage - 1) / kPage;
    for (int j = 0; j < N; ++j) {
      const int page = block_table[static_cast<int64_t>(r) * max_pages + j];
      float pooled = 0.0f;
      double pooled64 = 0.0;
      for (int h = 0; h < hkv; ++h) {
        const float *s = S + (static_cast<int64_t>(page) * hkv + h) * d;
        const float v = orc_dot_fixed_order(&qbar[static_cast<size_t>(h) * d], s, d);
        double v64 = 0.0;
        for (int i = 0; i < d; ++i) v64 += static_cast<double>(qbar[static_cast<size_t>(h) * d + i]) * s[i];
        if (per_head) {
          const int64_t o = (static_cast<int64_t>(r) * rows + h) * max_pages + j;
          scores[o] = v;
          if (scores64) scores64[o] = v64;
        } else {
          pooled = (h == 0) ? v : pooled + v;
          pooled64 += v64;
        }
      }
      if (!per_head) {
        const int64_t o = static_cast<int64_t>(r) * max_pages + j;
        scores[o] = pooled;
        if (scores64) scores64[o] = pooled64;
      }
    }
  }
  return 0;
}

// External-prior page scores (KRI page, "Required output shape" and the prior schema: a baked
// block_affinities[L][H][N] tensor that the connector mean-pools across layers and heads before taking the top-K of
// each request). aff holds M = L*H rows of N block scores, row i = l*H + h. The page is silent on the summation
// order, so the library fixes one and this function states it plainly in fp32: the M values of a block are summed
// in chunks of 32 consecutive rows (each chunk from 0.0f, rows ascending), the chunk sums are added in ascending
// chunk order (from 0.0f), and the total is divided by M once. out[N].
int orc_prior_scores(const float *aff, int L, int H, int N, float *out) {
  const int M = L * H;
  if (L <= 0 || H <= 0 || N < 0) return -1;
  for (int n = 0; n < N; ++n) {
    float total = 0.0f;
    for (int c0 = 0; c0 < M; c0 += 32) {
      float chunk = 0.0f;
      for (int i = c0; i < std::min(c0 + 32, M); ++i) chunk = chunk + aff[static_cast<size_t>(i) * N + n];
      total = total + chunk;
    }
    out[n] = total / static_cast<float>(M);
  }
  return 0;
}

// A<a>R<r>K<k> selection over N prompt pages (KRI page, "The A<a>R<r>K<k> tag"): pages [0, a) and the last r
// pages are pinned; from the middle [a, N-r) the k best by score are chosen, ties to the lower page id. The
// result is written ascending; the return value is its length. Plain full sort, no selection algorithm.
int orc_topk_ark(const float *scores, int N, int a, int r, int k, int32_t *out_ids) {
  std::vector<char> keep(N, 0);
  const int a_end = std::min(a, N);
  const int r_begin = std::max(0, N - r);
  for (int j = 0; j < a_end; ++j) keep[j] = 1;
  for (int j = r_begin; j < N; ++j) keep[j] = 1;
  std::vector<int> middle;
  for (int j = a_end; j < r_begin; ++j) middle.push_back(j);
  std::stable_sort(middle.begin(), middle.end(), [&](int x, int y) {
    const uint32_t kx = order_key(scores[x]), ky = order_key(scores[y]);
    if (kx != ky) return kx > ky;
    return x < y;
  });
  const int take = std::min<int>(k, static_cast<int>(middle.size()));
  for (int t = 0; t < take; ++t) keep[middle[t]] = 1;
  int n = 0;
  for (int j = 0; j < N; ++j)
    if (keep[j]) out_ids[n++] = j;
  return n;
}

// Span selection (KAP paper, compiler: selected token spans resolved to KV pages): a page is kept if any token of
// any span lies in it, plus the pinned anchor/recent pages. spans = [nspans][2] (first token, length); tokens at
// or beyond 16*N are ignored. Ascending output; returns the count.
int orc_select_spans(int N, const int32_t *spans, int nspans, int a, int r, int32_t *out_ids) {
  std::vector<char> keep(N, 0);
  for (int j = 0; j < std::min(a, N); ++j) keep[j] = 1;
  for (int j = std::max(0, N - r); j < N; ++j) keep[j] = 1;
  for (int s = 0; s < nspans; ++s) {
    const int64_t first = spans[2 * s], len = spans[2 * s + 1];
    for (int64_t t = first; t < first + len; ++t)
      if (t >= 0 && t < static_cast<int64_t>(N) * kPage) keep[t / kPage] = 1;
  }
  int n = 0;
  for (int j = 0; j < N; ++j)
    if (keep[j]) out_ids[n++] = j;
  return n;
}

// Compact view of one row (KAP paper, selected-KV view): the selected pages in ascending logical order, each with
// its physical page from the full block table, followed by the tail pages (logical pages j >= floor(ctx_len/16)
// with 16j < seq_len + horizon) that are not already selected. Returns the entry count.
int orc_compile_view_row(const int32_t *block_table_row, int ctx_len, int seq_len, int horizon, const int32_t *sel,
                         int nsel, int32_t *cbt, int32_t *clog, int32_t *n_selected) {
  int n = 0;
  for (int i = 0; i < nsel; ++i) {
    clog[n] = sel[i];
    cbt[n] = block_table_row[sel[i]];
    ++n;
  }
  *n_selected = nsel;
  const int first_tail = ctx_len / kPage;
  const int64_t end_tok = static_cast<int64_t>(seq_len) + horizon;
  for (int j = first_tail; static_cast<int64_t>(j) * kPage < end_tok; ++j) {
    bool already = false;
    for (int i = 0; i < nsel; ++i) already = already || (sel[i] == j);
    if (already) continue;
    clog[n] = j;
    cbt[n] = block_table_row[j];
    ++n;
  }
  return n;
}

// Slot of a token at logical position pos: physical page of logical page pos/16, times 16, plus pos%16.
int64_t orc_slot(const int32_t *block_table_row, int max_pages, int pos) {
  const int j = pos / kPage;
  if (pos < 0 || j >= max_pages) return -1;
  const int page = block_table_row[j];
  if (page < 0) return -1;
  return static_cast<int64_t>(page) * kPage + pos % kPage;
}

// RoPE inverse frequencies: theta^(-2i/d) in fp64, rounded once to fp32.
void orc_inv_freq(int d, double theta, float *out) {
  for (int i = 0; i < d / 2; ++i) out[i] = static_cast<float>(std::pow(theta, -2.0 * i / d));
}

// Rotary embedding of x [T][H][d] at positions pos[T] (half-split pairs (i, i+d/2)). The angle is formed in
// fp32 as (float)pos * inv_freq[i], as the library specifies; sin and cos are then taken in fp64.
void orc_rope(const float *x, int T, int H, int d, const int32_t *pos, const float *inv_freq, double *out) {
  const int half = d / 2;
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      const float *xr = x + (static_cast<int64_t>(t) * H + h) * d;
      double *o = out + (static_cast<int64_t>(t) * H + h) * d;
      for (int i = 0; i < half; ++i) {
        const float ang = static_cast<float>(pos[t]) * inv_freq[i];
        const double c = std::cos(static_cast<double>(ang)), s = std::sin(static_cast<double>(ang));
        const double a = xr[i], b = xr[i + half];
        o[i] = a * c - b * s;
        o[i + half] = a * s + b * c;
      }
    }
}

// Proposal attention (KAP paper, executor: q_prop = 1 over the selected view, same logical positions; only
// prompt-side KV is restricted). For request r and query head hq at position P = seq_len[r]-1, the visible
// positions are: prompt positions p < ctx_len whose page is in the selection row of KV head hq/G (or the shared
// row), and every generated position ctx_len <= p <= P. K and V are read through the full block table.
int orc_attn_propose(const float *q, const float *K, const float *V, int num_pages, int hq, int hkv, int d,
                     const int32_t *block_table, int R, int max_pages, const int32_t *ctx_len, const int32_t *seq_len,
                     const int32_t *sel, const int32_t *nsel, int rows, int cap, double *out, double *lse,
                     int nthreads) {
  const int G = hq / hkv;
  int bad = 0;
  parallel_units(R * hkv, nthreads, [&](int unit) {
    const int r = unit / hkv, h = unit % hkv;
    const int row = (rows == 1) ? 0 : h;
    const int32_t *sr = sel + (static_cast<int64_t>(r) * rows + row) * cap;
    const int n = nsel[r * rows + row];
    const int32_t *bt = block_table + static_cast<int64_t>(r) * max_pages;
    std::vector<const float *> ks, vs;
    const int L = ctx_len[r], P = seq_len[r] - 1;
    std::vector<char> selected(static_cast<size_t>(max_pages), 0);
    for (int i = 0; i < n; ++i)
      if (sr[i] >= 0 && sr[i] < max_pages) selected[sr[i]] = 1;
    for (int p = 0; p <= P; ++p) {
      const bool vis = (p >= L) || selected[p / kPage];
      if (!vis) continue;
      const int page = bt[p / kPage];
      if (page < 0 || page >= num_pages) {
        bad = 1;
        return;
      }
      ks.push_back(kv_row(K, page, h, p % kPage, hkv, d));
      vs.push_back(kv_row(V, page, h, p % kPage, hkv, d));
    }
    for (int g = 0; g < G; ++g) {
      const int hh = h * G + g;
      attend(q + (static_cast<int64_t>(r) * hq + hh) * d, ks, vs, d, out + (static_cast<int64_t>(r) * hq + hh) * d,
             lse + static_cast<int64_t>(r) * hq + hh);
    }
  });
  return bad ? -1 : 0;
}

// Verification attention (KAP paper, verifier: a short contiguous query window over the full KV cache, the
// full block table and the original positions). Row i of request r sits at position q_start[r] + i and sees every
// position <= its own: the full prompt, earlier generated tokens and candidates 0..i (causal among candidates).
int orc_attn_verify(const float *q, const float *K, const float *V, int num_pages, int hq, int hkv, int d,
                    const int32_t *block_table, int R, int max_pages, const int32_t *q_offsets,
                    const int32_t *q_start, double *out, double *lse, int nthreads) {
  const int G = hq / hkv;
  int bad = 0;
  parallel_units(R * hkv, nthreads, [&](int unit) {
    const int r = unit / hkv, h = unit % hkv;
    const int32_t *bt = block_table + static_cast<int64_t>(r) * max_pages;
    for (int row = q_offsets[r]; row < q_offsets[r + 1]; ++row) {
      const int P = q_start[r] + (row - q_offsets[r]);
      std::vector<const float *> ks, vs;
      for (int p = 0; p <= P; ++p) {
        const int page = bt[p / kPage];
        if (page < 0 || page >= num_pages) {
          bad = 1;
          return;
        }
        ks.push_back(kv_row(K, page, h, p % kPage, hkv, d));
        vs.push_back(kv_row(V, page, h, p % kPage, hkv, d));
      }
      for (int g = 0; g < G; ++g) {
        const int hh = h * G + g;
        attend(q + (static_cast<int64_t>(row) * hq + hh) * d, ks, vs, d,
               out + (static_cast<int64_t>(row) * hq + hh) * d, lse + static_cast<int64_t>(row) * hq + hh);
      }
    }
  });
  return bad ? -1 : 0;
}

// Number of hardware threads of this host (reported beside CPU timings).
// Tolerant acceptance and commit of one verify window (KAP paper, verifier: the window is the carry token followed by
// the k proposals; a proposal is accepted when it lies within the target's top-n candidates under the full context,
// the Top-3 rule being n = 3; m counts the proposals accepted consecutively from the start; the verifier then emits
// the next carry and commits). logits [rows][V]: row j is the verifier's prediction after window token j;
// tokens [rows]: token 0 is the carry, tokens 1..rows-1 the proposals. Proposal j is checked against row j - 1 by
// its rank under (logit descending, token id ascending, NaN last): accepted when fewer than n tokens come before it.
// The next carry is the first token of row m under the same order (the target's top choice after the accepted
// prefix); the committed length is start + 1 + m (the carry and the accepted proposals). Plain full sorts.
int orc_accept_commit(const float *logits, int rows, int V, const int32_t *tokens, int top_n, int start_pos,
                      int32_t *m_out, int32_t *carry_out, int32_t *seq_len_out) {
  if (rows < 1 || V < 1 || top_n < 1) return -1;
  auto ranked = [&](int j) {  // the tokens of row j in rank order
    std::vector<int> ids(V);
    for (int t = 0; t < V; ++t) ids[t] = t;
    const float *row = logits + static_cast<size_t>(j) * V;
    std::stable_sort(ids.begin(), ids.end(), [&](int x, int y) {
      const uint32_t kx = order_key(row[x]), ky = order_key(row[y]);
      if (kx != ky) return kx > ky;
      return x < y;
    });
    return ids;
  };
  int m = 0;
  for (int j = 1; j < rows; ++j) {
    const int x = tokens[j];
    if (x < 0 || x >= V) break;  // not a token of the vocabulary: rejected
    const std::vector<int> ids = ranked(j - 1);
    const int rank = static_cast<int>(std::find(ids.begin(), ids.end(), x) - ids.begin());
    if (rank >= top_n) break;
    ++m;
  }
  *m_out = m;
  *carry_out = ranked(m)[0];
  *seq_len_out = start_pos + 1 + m;
  return 0;
}

// Materialisation of one compact view row into a fixed-capacity workspace (KAP paper, compiler: the selected spans
// are resolved to KV pages and materialised as a compact physical view that keeps logical positions; a plan that
// exceeds the compact workspace falls back). The workspace of the row's request is the ws_pages pool pages from
// ws_base. The i-th selected entry is copied to page ws_base + i when all its tokens are prompt tokens (logical page
// lp with 16 * (lp + 1) <= ctx_len); a selected page that also holds positions >= ctx_len keeps its own page, since
// generated tokens are written through the full table into it after the copy. Tail entries keep their pages;
// logical pages are unchanged. Writes the new row and the (source, destination) page pairs to copy; returns their
// count, or -1 when the selection does not fit (the row is then left as it is and nothing is copied).
int orc_materialize_row(const int32_t *bt_row, const int32_t *lp_row, int n_entries, int n_selected, int ctx_len,
                        int ws_base, int ws_pages, int32_t *out_bt_row, int32_t *copy_src, int32_t *copy_dst) {
  for (int i = 0; i < n_entries; ++i) out_bt_row[i] = bt_row[i];
  if (n_selected > ws_pages) return -1;
  int n = 0;
  for (int i = 0; i < n_selected; ++i) {
    if (kPage * (lp_row[i] + 1) > ctx_len) continue;
    copy_src[n] = bt_row[i];
    copy_dst[n] = ws_base + i;
    ++n;
    out_bt_row[i] = ws_base + i;
  }
  return n;
}

int orc_hardware_threads(void) { return static_cast<int>(std::thread::hardware_concurrency()); }

}  // extern "C"
