// k_propose.cu - selected-KV proposal attention, q = 1 per request (sm_103a).
//
// KAP paper, executor: each proposal step is a decode-like step (q_prop = 1) whose attention sees only the
// selected prompt pages of the compact view, plus every generated token, at the original logical positions.
// EarlySelectKV page: the main flow gathers KV at precomputed page indices and runs sparse attention with the real
// query.
//
// Design (GB300):
//  * Work = the concatenated entry lists of all (request, KV head) rows; CTA b owns the contiguous entry range
//    [b*E/nb, (b+1)*E/nb) (stream-K), so long and short rows balance across the 152 SMs. A row split over several
//    CTAs is merged by the last CTA to finish (one atomic counter per row, no waiting).
//  * Each CTA streams its entries in chunks of CH pages through a 2-deep shared-memory ring: one thread issues a
//    1-D bulk copy (cp.async.bulk) per 4 KiB (page, head) chunk of K and of V, each completing on its own mbarrier.
//  * The G query heads of one KV head share every K/V vector read: lane l holds 16 bytes of each token row
//    (coalesced, conflict-free), computes partial dot products for G heads, and a reduce-scatter across the lanes of
//    a row leaves each lane owning a few finished logits. Softmax is exact per chunk with an online rescale across
//    chunks (base-2 exponentials on pre-scaled logits).
#include "kap_device.cuh"
#include "kap_launch.h"

namespace kap {
namespace {

constexpr int kNumWarps = 4;
constexpr int kThreads = kNumWarps * 32;
constexpr int kMaxSlotsExtraCtas = 4096;  // bound on the grid, for workspace sizing
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <class T, int D, int G, int CH>
struct Cfg {
  static constexpr int ESZ = sizeof(T);
  static constexpr int EPL = 16 / ESZ;           // elements per 16-byte vector
  static constexpr int LPT = D * ESZ / 16;       // lanes covering one token row
  static constexpr int TPI = 32 / LPT;           // token rows per warp-wide 16-byte load
  static constexpr int NI = kPage / TPI;         // 16-byte vectors per lane per (page, head) chunk
  static constexpr int CHUNK = kPage * D * ESZ;  // bytes of one (page, head) chunk
  static constexpr int NV = ((NI * G + LPT - 1) / LPT) * LPT;  // reduce-scatter values (padded)
  static constexpr int VPL = NV / LPT;           // finished logits owned by each lane
  static constexpr int LOG_LPT = LPT == 8 ? 3 : (LPT == 16 ? 4 : 5);
  // shared memory carve-up (bytes)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + 2 * CH * CHUNK;
  static constexpr int OFF_SL = OFF_V + 2 * CH * CHUNK;      // logits / probabilities [CH][G][16]
  static constexpr int OFF_RED = OFF_SL + CH * G * kPage * 4;  // output reduction [G][D]
  static constexpr int OFF_ST = OFF_RED + G * D * 4;           // m, l, alpha [3][G]
  static constexpr int OFF_BAR = ((OFF_ST + 3 * G * 4 + 7) / 8) * 8;  // barK[2][CH], barV[2][CH]
  static constexpr int OFF_META = OFF_BAR + 4 * CH * 8;
  static constexpr int SMEM = OFF_META + 2 * (40 + 8 * CH);
};

struct Params {
  const void *k, *v;
  int num_pages, hkv, hq;
  const int32_t *ctx_len, *seq_len;
  const int32_t *vbt, *vlp, *vn, *vnsel;
  int rows_per_seq, vcap;
  int nrows;  // R * Hkv
  const void *q;
  void *out;
  float *lse;
  int *counters;  // [nrows]
  float *ml;      // [slots][G][2]
  float *part;    // [slots][G][D]
  int *err;
};

__device__ __forceinline__ int view_row(const Params &p, int row) {
  const int r = row / p.hkv, h = row - r * p.hkv;
  return r * p.rows_per_seq + (p.rows_per_seq == 1 ? 0 : h);
}
__device__ __forceinline__ int row_entries(const Params &p, int row) {
  return max(0, min(p.vn[view_row(p, row)], p.vcap));
}
// CTA that owns global entry x under the static split of E entries over nb CTAs.
__device__ __forceinline__ int owner_cta(int64_t x, int64_t E, int nb) {
  return static_cast<int>(((x + 1) * nb - 1) / E);
}

template <int CH>
struct Meta {
  int64_t rb, re;  // global entry range of the chunk's row
  int n, row, l0, first, last, pad;
  int tlo[CH], thi[CH];
};

template <class T, int D, int G, int CH>
__global__ void __launch_bounds__(kThreads, 3) propose_kernel(const Params p) {
  using C = Cfg<T, D, G, CH>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *kbuf = smem + C::OFF_K;
  unsigned char *vbuf = smem + C::OFF_V;
  float *sl = reinterpret_cast<float *>(smem + C::OFF_SL);
  float *red = reinterpret_cast<float *>(smem + C::OFF_RED);
  float *st_m = reinterpret_cast<float *>(smem + C::OFF_ST);
  float *st_l = st_m + G;
  float *st_a = st_l + G;
  uint64_t *barK = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *barV = barK + 2 * CH;
  Meta<CH> *meta = reinterpret_cast<Meta<CH> *>(smem + C::OFF_META);
  __shared__ int s_flag;
  __shared__ int64_t s_total;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Total entries E (warp 0), then this CTA's range.
  if (warp == 0) {
    int64_t tot = 0;
    for (int base = 0; base < p.nrows; base += 32) {
      const int row = base + lane;
      int c = row < p.nrows ? row_entries(p, row) : 0;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      tot += c;
    }
    if (lane == 0) s_total = tot;
  }
  for (int i = tid; i < G * D; i += kThreads) red[i] = 0.0f;
  if (tid == 0) {
    for (int i = 0; i < 2 * CH; ++i) {
      mbar_init(&barK[i], 1);
      mbar_init(&barV[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int64_t E = s_total;
  // Split over nb <= E CTAs so that every participating CTA owns at least one entry (the merge counts them).
  const int nb = static_cast<int>(E < static_cast<int64_t>(gridDim.x) ? E : static_cast<int64_t>(gridDim.x));
  if (E == 0 || static_cast<int>(blockIdx.x) >= nb) return;
  const int64_t cta_begin = static_cast<int64_t>(blockIdx.x) * E / nb;
  const int64_t cta_end = static_cast<int64_t>(blockIdx.x + 1) * E / nb;
  if (cta_begin >= cta_end) return;

  // First row of this CTA's range: warp-parallel prefix over the rows' entry counts (no per-row round trips).
  __shared__ int s_row0;
  __shared__ int64_t s_rb0, s_re0;
  if (warp == 0) {
    int64_t base = 0;
    for (int b = 0; b < p.nrows; b += 32) {
      const int row = b + lane;
      const int c = row < p.nrows ? row_entries(p, row) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nb_ = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += nb_;
      }
      const int64_t rb = base + incl - c, re = base + incl;
      const unsigned hit = __ballot_sync(0xffffffffu, c > 0 && rb <= cta_begin && cta_begin < re);
      if (hit) {
        if (lane == __ffs(hit) - 1) {
          s_row0 = row;
          s_rb0 = rb;
          s_re0 = re;
        }
        break;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();

  // Producer (all lanes of warp 0, uniform control flow): plan() advances the cursor and starts the loads of the
  // next chunk's view metadata (lane e loads entry e); commit(buf) consumes them one chunk later, so the load
  // latency overlaps the compute of the chunk in between.
  int pr_row = s_row0;
  int64_t pr_row_begin = s_rb0, pr_row_end = s_re0, pr_cursor = cta_begin;
  int row_r = -1, row_h = 0, row_vr = 0, row_L = 0, row_S = 0, row_nsel = 0;
  int pl_n = 0, pl_row = 0, pl_l0 = 0, pl_first = 0, pl_last = 0, pl_lp = 0, pl_page = -1;
  int pl_L = 0, pl_S = 0, pl_nsel = 0, pl_h = 0;
  int64_t pl_rb = 0, pl_re = 0;
  const T *Kp = static_cast<const T *>(p.k);
  const T *Vp = static_cast<const T *>(p.v);

  auto plan = [&]() {
    if (pr_cursor >= cta_end) {
      pl_n = 0;
      return;
    }
    while (pr_cursor >= pr_row_end) {
      ++pr_row;
      pr_row_begin = pr_row_end;
      pr_row_end += row_entries(p, pr_row);
    }
    if (row_r != pr_row) {  // row-level metadata, loaded once per row
      row_r = pr_row;
      const int r = pr_row / p.hkv;
      row_h = pr_row - r * p.hkv;
      row_vr = view_row(p, pr_row);
      row_L = p.ctx_len[r];
      row_S = p.seq_len[r];
      row_nsel = p.vnsel[row_vr];
    }
    const int64_t seg_end = min(pr_row_end, cta_end);
    pl_n = static_cast<int>((seg_end - pr_cursor < CH) ? seg_end - pr_cursor : CH);
    pl_l0 = static_cast<int>(pr_cursor - pr_row_begin);
    pl_row = pr_row;
    pl_rb = pr_row_begin;
    pl_re = pr_row_end;
    pl_first = (pr_cursor == pr_row_begin || pr_cursor == cta_begin) ? 1 : 0;
    pl_last = (pr_cursor + pl_n == seg_end) ? 1 : 0;
    pl_L = row_L;
    pl_S = row_S;
    pl_nsel = row_nsel;
    pl_h = row_h;
    if (lane < pl_n) {
      const size_t o = static_cast<size_t>(row_vr) * p.vcap + pl_l0 + lane;
      pl_lp = p.vlp[o];
      pl_page = p.vbt[o];
    }
    pr_cursor += pl_n;
  };

  auto commit = [&](int buf) {
    Meta<CH> &m = meta[buf];
    if (lane == 0) {
      m.n = pl_n;
      m.row = pl_row;
      m.l0 = pl_l0;
      m.first = pl_first;
      m.last = pl_last;
      m.rb = pl_rb;
      m.re = pl_re;
    }
    if (pl_n == 0 || lane >= CH) return;
    const int e = lane;
    int tlo = 0, thi = 0;
    if (e < pl_n) {
      const int i = pl_l0 + e;
      const int base = pl_lp * kPage;
      thi = min(kPage, pl_S - base);
      tlo = (i < pl_nsel) ? 0 : max(0, pl_L - base);
      if (thi > tlo && (pl_page < 0 || pl_page >= p.num_pages)) {
        set_error(p.err, kErrPage);
        tlo = thi = 0;
      }
    }
    if (thi > tlo) {
      const size_t off = (static_cast<size_t>(pl_page) * p.hkv + pl_h) * kPage * D;
      mbar_arrive_expect_tx(&barK[buf * CH + e], C::CHUNK);
      bulk_g2s(kbuf + (buf * CH + e) * C::CHUNK, Kp + off, C::CHUNK, &barK[buf * CH + e]);
      mbar_arrive_expect_tx(&barV[buf * CH + e], C::CHUNK);
      bulk_g2s(vbuf + (buf * CH + e) * C::CHUNK, Vp + off, C::CHUNK, &barV[buf * CH + e]);
    } else {  // keep every slot's barrier phase in step with the ring
      tlo = thi = 0;
      mbar_arrive(&barK[buf * CH + e]);
      mbar_arrive(&barV[buf * CH + e]);
    }
    m.tlo[e] = tlo;
    m.thi[e] = thi;
  };

  if (warp == 0) {
    plan();
    commit(0);
    plan();
    commit(1);
    plan();
  }
  __syncthreads();

  const int ts = lane / C::LPT;         // token sub-row of this lane
  const int base_dim = (lane % C::LPT) * C::EPL;
  float qf[G][C::EPL];
  float o[G][C::EPL];
  const float qscale = rsqrtf(static_cast<float>(D)) * kLog2e;

  for (int c = 0;; ++c) {
    const int buf = c & 1;
    const uint32_t parity = (c >> 1) & 1;
    const Meta<CH> m = meta[buf];
    if (m.n == 0) break;
    const int r = m.row / p.hkv, h = m.row - r * p.hkv;
    if (m.first) {
      const T *qrow = static_cast<const T *>(p.q) + (static_cast<size_t>(r) * p.hq + h * G) * D + base_dim;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float tmp[C::EPL];
        Vec16<T>::unpack(*reinterpret_cast<const uint4 *>(qrow + static_cast<size_t>(g) * D), tmp);
#pragma unroll
        for (int k = 0; k < C::EPL; ++k) {
          qf[g][k] = tmp[k] * qscale;
          o[g][k] = 0.0f;
        }
      }
      if (tid < G) {
        st_m[tid] = -INFINITY;
        st_l[tid] = 0.0f;
      }
    }
    // ---- logits: q . k for every token of the chunk
    for (int e = warp; e < m.n; e += kNumWarps) {
      float part[C::NV];
#pragma unroll
      for (int v = 0; v < C::NV; ++v) part[v] = 0.0f;
      if (m.thi[e] > m.tlo[e]) {
        mbar_wait(&barK[buf * CH + e], parity, p.err);
        const uint4 *kv = reinterpret_cast<const uint4 *>(kbuf + (buf * CH + e) * C::CHUNK);
        uint4 w[C::NI];
#pragma unroll
        for (int j = 0; j < C::NI; ++j) w[j] = kv[j * 32 + lane];
#pragma unroll
        for (int j = 0; j < C::NI; ++j) {
          float kf[C::EPL];
          Vec16<T>::unpack(w[j], kf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float acc = 0.0f;
#pragma unroll
            for (int k = 0; k < C::EPL; ++k) acc = fmaf(qf[g][k], kf[k], acc);
            part[j * G + g] = acc;
          }
        }
      }
      // reduce-scatter over the LPT lanes of a token row: lane keeps values [(lane%LPT)*VPL, +VPL)
#pragma unroll
      for (int step = 0; step < C::LOG_LPT; ++step) {
        const int msk = (C::LPT >> 1) >> step;
        const int half = C::NV >> (step + 1);
        const bool upper = (lane & msk) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k) {
          const float send = upper ? part[k] : part[k + half];
          const float keep = upper ? part[k + half] : part[k];
          part[k] = keep + __shfl_xor_sync(0xffffffffu, send, msk);
        }
      }
#pragma unroll
      for (int k = 0; k < C::VPL; ++k) {
        const int v = (lane % C::LPT) * C::VPL + k;
        if (v < C::NI * G) {
          const int j = v / G, g = v - (v / G) * G;
          const int tok = j * C::TPI + ts;
          const bool vis = tok >= m.tlo[e] && tok < m.thi[e];
          sl[(e * G + g) * kPage + tok] = vis ? part[k] : -INFINITY;
        }
      }
    }
    __syncthreads();
    // ---- softmax over the chunk (exact within the chunk, online across chunks)
    for (int g = warp; g < G; g += kNumWarps) {
      const int ntok = m.n * kPage;
      float mx = -INFINITY;
      for (int tk = lane; tk < ntok; tk += 32) mx = fmaxf(mx, sl[((tk >> 4) * G + g) * kPage + (tk & 15)]);
      mx = warp_max(mx);
      const float m_old = st_m[g];
      const float m_new = fmaxf(m_old, mx);
      float alpha, sum = 0.0f;
      if (m_new == -INFINITY) {
        alpha = 1.0f;
        for (int tk = lane; tk < ntok; tk += 32) sl[((tk >> 4) * G + g) * kPage + (tk & 15)] = 0.0f;
      } else {
        alpha = exp2f(m_old - m_new);
        for (int tk = lane; tk < ntok; tk += 32) {
          float *ps = &sl[((tk >> 4) * G + g) * kPage + (tk & 15)];
          const float pv = exp2f(*ps - m_new);
          *ps = pv;
          sum += pv;
        }
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        st_m[g] = m_new;
        st_l[g] = st_l[g] * alpha + sum;
        st_a[g] = alpha;
      }
    }
    __syncthreads();
    // ---- o = o * alpha + sum_t p_t v_t
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float a = st_a[g];
#pragma unroll
      for (int k = 0; k < C::EPL; ++k) o[g][k] *= a;
    }
    for (int e = warp; e < m.n; e += kNumWarps) {
      const int tlo = m.tlo[e], thi = m.thi[e];
      if (thi <= tlo) continue;
      mbar_wait(&barV[buf * CH + e], parity, p.err);
      const uint4 *vv = reinterpret_cast<const uint4 *>(vbuf + (buf * CH + e) * C::CHUNK);
      const bool full = (tlo == 0 && thi == kPage);
#pragma unroll
      for (int j = 0; j < C::NI; ++j) {
        const int tok = j * C::TPI + ts;
        float vf[C::EPL];
        Vec16<T>::unpack(vv[j * 32 + lane], vf);
        if (!full && !(tok >= tlo && tok < thi)) {
#pragma unroll
          for (int k = 0; k < C::EPL; ++k) vf[k] = 0.0f;  // invisible slots may hold anything (even NaN)
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pw = sl[(e * G + g) * kPage + tok];
#pragma unroll
          for (int k = 0; k < C::EPL; ++k) o[g][k] = fmaf(pw, vf[k], o[g][k]);
        }
      }
    }
    __syncthreads();
    if (warp == 0) {  // refill this ring slot with chunk c + 2, then start loading chunk c + 3's metadata
      commit(buf);
      plan();
    }
    if (!m.last) continue;

    // ---- segment end: reduce o over lanes and warps, then finish or hand over a partial
#pragma unroll
    for (int msk = C::LPT; msk < 32; msk <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < C::EPL; ++k) o[g][k] += __shfl_xor_sync(0xffffffffu, o[g][k], msk);
    if (lane < C::LPT) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int k = 0; k < C::EPL; ++k) atomicAdd(&red[g * D + base_dim + k], o[g][k]);
    }
    __syncthreads();
    // contributors of this row: the CTAs owning its first and its last entry
    const int64_t rb = m.rb, re = m.re;
    const int b_first = owner_cta(rb, E, nb), b_last = owner_cta(re - 1, E, nb);
    const int n_contrib = b_last - b_first + 1;
    const size_t out_base = (static_cast<size_t>(r) * p.hq + h * G) * D;
    T *outp = static_cast<T *>(p.out);
    if (n_contrib == 1) {
      for (int i = tid; i < G * D; i += kThreads) {
        const int g = i / D;
        const float l = st_l[g];
        outp[out_base + i] = from_f<T>(l > 0.0f ? red[i] / l : 0.0f);
      }
      if (tid < G) {
        const float l = st_l[tid];
        p.lse[static_cast<size_t>(r) * p.hq + h * G + tid] = l > 0.0f ? (st_m[tid] + log2f(l)) * kLn2 : -INFINITY;
        if (!(l > 0.0f)) set_error(p.err, kErrLength);
      }
    } else {
      const int slot = static_cast<int>(blockIdx.x) + m.row;
      float *pp = p.part + static_cast<size_t>(slot) * G * D;
      for (int i = tid; i < G * D; i += kThreads) __stcg(pp + i, red[i]);
      if (tid < G) {
        __stcg(p.ml + (static_cast<size_t>(slot) * G + tid) * 2, st_m[tid]);
        __stcg(p.ml + (static_cast<size_t>(slot) * G + tid) * 2 + 1, st_l[tid]);
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int old = atomicAdd(&p.counters[m.row], 1);
        s_flag = (old == n_contrib - 1) ? 1 : 0;
        if (s_flag) p.counters[m.row] = 0;  // every contributor has arrived: leave the counter at zero
      }
      __syncthreads();
      if (s_flag) {
        // Last arriver: merge the row's partial records from CTAs b_first..b_last. The (m, l) pairs of up to 32
        // contributors are staged in shared memory by one parallel load pass; the partial outputs are loaded with
        // up to 16 loads in flight per element before any is used.
        __threadfence();
        constexpr int kElems = (G * D + kThreads - 1) / kThreads;
        float *sm_m = sl;           // [32][G]
        float *sm_w = sl + 32 * G;  // [32][G]
        float *Mg = red, *Lg = red + G, *Rg = red + 2 * G;  // red is free: its content is in the partial record
        if (tid < G) {
          Mg[tid] = -INFINITY;
          Lg[tid] = 0.0f;
        }
        float acc[kElems];
#pragma unroll
        for (int k = 0; k < kElems; ++k) acc[k] = 0.0f;
        const int nc = b_last - b_first + 1;
        for (int g0 = 0; g0 < nc; g0 += 32) {
          const int ng = min(32, nc - g0);
          __syncthreads();
          for (int q = tid; q < ng * G; q += kThreads) {
            const int bb = q / G, g = q - (q / G) * G;
            const size_t o = (static_cast<size_t>(b_first + g0 + bb + m.row) * G + g) * 2;
            sm_m[bb * G + g] = __ldcg(p.ml + o);
            sm_w[bb * G + g] = __ldcg(p.ml + o + 1);
          }
          __syncthreads();
          if (tid < G) {
            const float Mo = Mg[tid];
            float M = Mo;
            for (int bb = 0; bb < ng; ++bb) M = fmaxf(M, sm_m[bb * G + tid]);
            const float resc = (Mo == -INFINITY || M == -INFINITY) ? 0.0f : exp2f(Mo - M);
            float Ls = Lg[tid] * resc;
            for (int bb = 0; bb < ng; ++bb) {
              const float mb = sm_m[bb * G + tid];
              const float w = (mb == -INFINITY || M == -INFINITY) ? 0.0f : exp2f(mb - M);
              Ls += sm_w[bb * G + tid] * w;
              sm_w[bb * G + tid] = w;
            }
            Mg[tid] = M;
            Lg[tid] = Ls;
            Rg[tid] = resc;
          }
          __syncthreads();
#pragma unroll
          for (int k = 0; k < kElems; ++k) {
            const int i = tid + k * kThreads;
            if (i < G * D) {
              const int g = i / D;
              float a = (g0 > 0) ? acc[k] * Rg[g] : 0.0f;
              for (int b0 = 0; b0 < ng; b0 += 16) {
                float v[16];
#pragma unroll
                for (int bb = 0; bb < 16; ++bb)
                  v[bb] = (b0 + bb < ng)
                              ? __ldcg(p.part + static_cast<size_t>(b_first + g0 + b0 + bb + m.row) * G * D + i)
                              : 0.0f;
#pragma unroll
                for (int bb = 0; bb < 16; ++bb)
                  if (b0 + bb < ng) a = fmaf(v[bb], sm_w[(b0 + bb) * G + g], a);
              }
              acc[k] = a;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < kElems; ++k) {
          const int i = tid + k * kThreads;
          if (i < G * D) {
            const int g = i / D;
            const float Ls = Lg[g];
            outp[out_base + i] = from_f<T>(Ls > 0.0f ? acc[k] / Ls : 0.0f);
            if ((i % D) == 0) {
              p.lse[static_cast<size_t>(r) * p.hq + h * G + g] = Ls > 0.0f ? (Mg[g] + log2f(Ls)) * kLn2 : -INFINITY;
              if (!(Ls > 0.0f)) set_error(p.err, kErrLength);
            }
          }
        }
      }
    }
    __syncthreads();
    for (int i = tid; i < G * D; i += kThreads) red[i] = 0.0f;
    __syncthreads();
  }
}

template <class T, int D, int G>
cudaError_t launch_tdg(const Params &prm, cudaStream_t s) {
  constexpr int CH = 4;
  using C = Cfg<T, D, G, CH>;
  auto kern = propose_kernel<T, D, G, CH>;
  static int occ_cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int &occ = occ_cache[dev & 63];
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int o = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, kThreads, C::SMEM);
    if (e != cudaSuccess) return e;
    occ = o > 0 ? o : 1;
  }
  int nb = device_sm_count() * occ;
  if (nb > kMaxSlotsExtraCtas) nb = kMaxSlotsExtraCtas;
  kern<<<nb, kThreads, C::SMEM, s>>>(prm);
  return cudaGetLastError();
}

template <class T, int D>
cudaError_t launch_td(const Params &prm, int G, cudaStream_t s) {
  switch (G) {
    case 1: return launch_tdg<T, D, 1>(prm, s);
    case 2: return launch_tdg<T, D, 2>(prm, s);
    case 4: return launch_tdg<T, D, 4>(prm, s);
    case 5: return launch_tdg<T, D, 5>(prm, s);
    case 8: return launch_tdg<T, D, 8>(prm, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool propose_supported(int dtype, int d, int G) {
  (void)dtype;
  return (d == 64 || d == 128) && (G == 1 || G == 2 || G == 4 || G == 5 || G == 8);
}

size_t propose_workspace_bytes(int R, int hkv, int hq, int d) {
  const size_t nrows = static_cast<size_t>(R) * hkv;
  const size_t G = static_cast<size_t>(hq / hkv);
  const size_t slots = nrows + kMaxSlotsExtraCtas;
  size_t b = ((nrows * 4 + 255) / 256) * 256;       // counters
  b += ((slots * G * 2 * 4 + 255) / 256) * 256;     // m, l
  b += slots * G * d * 4;                           // partial outputs
  return b;
}

cudaError_t launch_propose(const PoolArgs &pa, const MapArgs &ma, const ViewArgs &va, const void *q, void *out,
                           float *lse, void *ws, size_t ws_bytes, int *err, cudaStream_t s) {
  (void)ws_bytes;
  const int G = pa.hq / pa.hkv;
  Params prm;
  prm.k = pa.k;
  prm.v = pa.v;
  prm.num_pages = pa.num_pages;
  prm.hkv = pa.hkv;
  prm.hq = pa.hq;
  prm.ctx_len = ma.ctx_len;
  prm.seq_len = ma.seq_len;
  prm.vbt = va.bt;
  prm.vlp = va.lp;
  prm.vn = va.n_entries;
  prm.vnsel = va.n_selected;
  prm.rows_per_seq = va.rows_per_seq;
  prm.vcap = va.cap;
  prm.nrows = ma.R * pa.hkv;
  prm.q = q;
  prm.out = out;
  prm.lse = lse;
  const size_t nrows = static_cast<size_t>(prm.nrows);
  const size_t slots = nrows + kMaxSlotsExtraCtas;
  unsigned char *w = static_cast<unsigned char *>(ws);
  prm.counters = reinterpret_cast<int *>(w);
  w += ((nrows * 4 + 255) / 256) * 256;
  prm.ml = reinterpret_cast<float *>(w);
  w += ((slots * G * 2 * 4 + 255) / 256) * 256;
  prm.part = reinterpret_cast<float *>(w);
  prm.err = err;
  if (pa.dtype == 0 && pa.d == 128) return launch_td<__nv_bfloat16, 128>(prm, G, s);
  if (pa.dtype == 0 && pa.d == 64) return launch_td<__nv_bfloat16, 64>(prm, G, s);
  if (pa.dtype == 1 && pa.d == 128) return launch_td<float, 128>(prm, G, s);
  return launch_td<float, 64>(prm, G, s);
}

}  // namespace kap
