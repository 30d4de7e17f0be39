// k_propose.cu - selected-KV proposal attention, q = 1 per request (sm_103a).
//
// KAP paper, executor: each proposal step is a decode-like step (q_prop = 1) whose attention sees only the
// selected prompt pages of the compact view, plus every generated token, at the original logical positions.
// EarlySelectKV page: attention of the main flow reads only the pages the routing side chose in advance, and uses
// the true query.
//
// Design (GB300):
//  * Work = the concatenated entry lists of all (request, KV head) rows; CTA b owns the contiguous entry range
//    [b*E/nb, (b+1)*E/nb) (stream-K, one CTA per SM), so long and short rows balance across the SMs. A row split
//    over several CTAs is merged by the last CTA to finish it (one atomic counter per row, no waiting).
//  * A producer warp streams the CTA's entries through a ring of page slots: per entry one 1-D bulk copy
//    (cp.async.bulk) of the 4 KiB (page, head) chunk of K and one of V, completing on the slot's mbarrier. With
//    ~20 slots most of a CTA's range is in flight at once.
//  * Twelve consumer warps take the entries of a row segment round-robin and work independently: lane l holds 16
//    bytes of each token row (coalesced, conflict-free), computes partial dot products for the G query heads of the
//    KV head, and a reduce-scatter across the lanes of a row leaves each lane owning a few finished logits. Each
//    warp keeps its own running max, sum and output; the max is only raised (and the state rescaled) when a page
//    exceeds it by more than 2^8, which is exact. Warps meet only at the end of a row segment, where their states
//    are combined.
#include "kap_device.cuh"
#include "kap_launch.h"

namespace kap {
namespace {

constexpr int kNCW = 12;                     // consumer warps
constexpr int kThreads = (kNCW + 1) * 32;    // + the producer warp (warp kNCW)
constexpr int kMaxSlotsExtraCtas = 4096;     // bound on the grid, for workspace sizing
constexpr int kMaxSeg = 32;                  // row segments per window of a CTA's range
constexpr int kMaxRowsScan = 2048;           // rows whose entry offsets are scanned into shared memory at once
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;    // log2 units

template <class T, int D, int G>
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
  static constexpr int COMB = kNCW * (G * D + 2 * G) * 4;  // per-warp segment states
  static constexpr int WLOG = kNCW * G * kPage * 4;        // per-warp logits / probabilities of one page
  static constexpr int RES = (G * D + 4 * G) * 4;          // combined segment state (+ merge scalars)
  static constexpr int SEGB = kMaxSeg * 56;                // segment table
  static constexpr int ROWB = kMaxRowsScan * 4;            // per-row entry offsets (row scan)
  static constexpr int FIXED = COMB + WLOG + RES + SEGB + ROWB + 2048;
  static constexpr int SLOT = 2 * CHUNK;                   // K and V of one entry
  static constexpr int SLOTS_FIT = (200 * 1024 - FIXED) / SLOT;
  static constexpr int SLOTS = SLOTS_FIT > 32 ? 32 : SLOTS_FIT;
  static constexpr int BATCH = SLOTS < 16 ? SLOTS : 16;    // entries the producer handles per step
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_COMB = OFF_KV + SLOTS * SLOT;
  static constexpr int OFF_WLOG = OFF_COMB + COMB;
  static constexpr int OFF_RES = OFF_WLOG + WLOG;
  static constexpr int OFF_SEG = ((OFF_RES + RES + 15) / 16) * 16;
  static constexpr int OFF_SMETA = ((OFF_SEG + SEGB + 15) / 16) * 16;  // [SLOTS] (tlo, thi)
  static constexpr int OFF_BAR = OFF_SMETA + SLOTS * 8;                // full[SLOTS], empty[SLOTS]
  static constexpr int OFF_ROWS = OFF_BAR + 2 * SLOTS * 8;             // [kMaxRowsScan + 1] int32
  static constexpr int SMEM = OFF_ROWS + ROWB + 4;
  static_assert(SLOTS >= 4, "too few page slots");
  static_assert(WLOG >= 2 * 32 * G * 4, "merge scratch does not fit");
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

// One row segment of a CTA's range: global entries [b, e) of attention row `row` (whose own range is [rb, re)),
// with the row-level metadata the producer and the consumers need.
struct Seg {
  int64_t b, e, rb, re;
  int row, vr, L, S, nsel, pad;
};
static_assert(sizeof(Seg) == 56, "segment record size");

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
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kNCW * 32) : "memory"); }

template <class T, int D, int G>
__global__ void __launch_bounds__(kThreads, 1) propose_kernel(const Params p) {
  using C = Cfg<T, D, G>;
  constexpr int kCT = kNCW * 32;  // consumer threads
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *kv = smem + C::OFF_KV;
  float *comb = reinterpret_cast<float *>(smem + C::OFF_COMB);      // [kNCW][G*D + 2G]
  float *wlog_all = reinterpret_cast<float *>(smem + C::OFF_WLOG);  // [kNCW][G][16]
  float *res = reinterpret_cast<float *>(smem + C::OFF_RES);        // [G*D] output, then m[G], l[G], 2G scratch
  Seg *segs = reinterpret_cast<Seg *>(smem + C::OFF_SEG);
  int2 *smeta = reinterpret_cast<int2 *>(smem + C::OFF_SMETA);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::SLOTS;
  __shared__ int64_t s_total, s_rb0, s_wnext_rb;
  __shared__ int s_row0, s_nseg, s_wnext_row, s_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Entry offsets of the rows (one parallel load of every row's count, a block scan in shared memory), then E,
  // this CTA's range and the row holding its first entry. Rows beyond kMaxRowsScan use a warp scan in global order.
  int *rowoff = reinterpret_cast<int *>(smem + C::OFF_ROWS);  // [nrows + 1] when nrows <= kMaxRowsScan
  __shared__ int scan_scratch[32];
  if (tid == 0) {
    for (int i = 0; i < C::SLOTS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_barrier_init();
  }
  const bool small_rows = p.nrows <= kMaxRowsScan;
  if (small_rows) {
    // thread t owns rows [t*per, (t+1)*per)
    const int per = (p.nrows + kThreads - 1) / kThreads;
    const int lo = min(p.nrows, tid * per), hi = min(p.nrows, lo + per);
    int cnt = 0;
    for (int rr = lo; rr < hi; ++rr) {
      const int c = row_entries(p, rr);
      rowoff[rr] = c;
      cnt += c;
    }
    const int incl = block_inclusive_scan(cnt, scan_scratch);
    int run = incl - cnt;
    for (int rr = lo; rr < hi; ++rr) {
      const int c = rowoff[rr];
      rowoff[rr] = run;
      run += c;
    }
    if (tid == kThreads - 1) {
      rowoff[p.nrows] = incl;
      s_total = incl;
    }
  } else if (warp == 0) {
    int64_t tot = 0;
    for (int base = 0; base < p.nrows; base += 32) {
      int c = (base + lane < p.nrows) ? row_entries(p, base + lane) : 0;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      tot += c;
    }
    if (lane == 0) s_total = tot;
  }
  __syncthreads();
  const int64_t E = s_total;
  // Split over nb <= E CTAs so that every participating CTA owns at least one entry (the merge counts them).
  const int nb = static_cast<int>(E < static_cast<int64_t>(gridDim.x) ? E : static_cast<int64_t>(gridDim.x));
  if (E == 0 || static_cast<int>(blockIdx.x) >= nb) return;
  const int64_t cta_begin = static_cast<int64_t>(blockIdx.x) * E / nb;
  const int64_t cta_end = static_cast<int64_t>(blockIdx.x + 1) * E / nb;

  // First row of the range.
  if (small_rows) {
    if (tid == 0) {  // last row whose start is <= cta_begin (and which is not empty)
      int lo = 0, hi = p.nrows - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (rowoff[mid] <= cta_begin) lo = mid; else hi = mid - 1;
      }
      s_row0 = lo;
      s_rb0 = rowoff[lo];
    }
  } else if (warp == 0) {
    int64_t base = 0;
    for (int b = 0; b < p.nrows; b += 32) {
      const int row = b + lane;
      const int c = row < p.nrows ? row_entries(p, row) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int64_t rb = base + incl - c, re = base + incl;
      const unsigned hit = __ballot_sync(0xffffffffu, c > 0 && rb <= cta_begin && cta_begin < re);
      if (hit) {
        if (lane == __ffs(hit) - 1) {
          s_row0 = row;
          s_rb0 = rb;
        }
        break;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();

  const T *Kp = static_cast<const T *>(p.k);
  const T *Vp = static_cast<const T *>(p.v);
  const int ts = lane / C::LPT;  // token sub-row of this lane
  const int base_dim = (lane % C::LPT) * C::EPL;
  const float qscale = rsqrtf(static_cast<float>(D)) * kLog2e;
  int w_row = s_row0;
  int64_t w_rb = s_rb0;

  // The range is processed in windows of up to kMaxSeg row segments (one warp-wide scan of 32 rows each).
  for (int64_t cur = cta_begin; cur < cta_end;) {
    if (warp == kNCW) {
      // segment table of this window: rows w_row .. w_row+31 intersected with [cur, cta_end)
      const int row = w_row + lane;
      const int c = row < p.nrows ? (small_rows ? rowoff[row + 1] - rowoff[row] : row_entries(p, row)) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int64_t rb = w_rb + incl - c, re = w_rb + incl;
      const int64_t sb = rb > cur ? rb : cur, se = re < cta_end ? re : cta_end;
      const bool nonempty = c > 0 && sb < se;
      const unsigned mask = __ballot_sync(0xffffffffu, nonempty);
      if (nonempty) {
        const int idx = __popc(mask & ((1u << lane) - 1u));
        Seg sg;
        sg.b = sb;
        sg.e = se;
        sg.rb = rb;
        sg.re = re;
        sg.row = row;
        const int r = row / p.hkv;
        sg.vr = view_row(p, row);
        sg.L = p.ctx_len[r];
        sg.S = p.seq_len[r];
        sg.nsel = p.vnsel[sg.vr];
        sg.pad = 0;
        segs[idx] = sg;
      }
      const int tot = __shfl_sync(0xffffffffu, incl, 31);
      if (lane == 0) {
        s_nseg = __popc(mask);
        s_wnext_row = w_row + 32;
        s_wnext_rb = w_rb + tot;
      }
    }
    __syncthreads();
    const int nseg = s_nseg;
    const int64_t win_end = (nseg > 0) ? segs[nseg - 1].e : cur;  // a window of empty rows only moves the rows on

    if (warp == kNCW) {
      // ============================================================================================== producer
      for (int si = 0; si < nseg; ++si) {
        const Seg sg = segs[si];
        const int h = sg.row - (sg.row / p.hkv) * p.hkv;
        for (int64_t e0 = sg.b; e0 < sg.e; e0 += C::BATCH) {
          const int64_t e = e0 + lane;
          if (lane < C::BATCH && e < sg.e) {
            const int i = static_cast<int>(e - sg.rb);  // entry index within the row's view
            const size_t o = static_cast<size_t>(sg.vr) * p.vcap + i;
            const int lp = p.vlp[o];
            const int page = p.vbt[o];
            const int base = lp * kPage;
            int thi = min(kPage, sg.S - base);
            int tlo = (i < sg.nsel) ? 0 : max(0, sg.L - base);
            if (thi > tlo && (page < 0 || page >= p.num_pages)) {
              set_error(p.err, kErrPage);
              tlo = thi = 0;
            }
            if (thi <= tlo) tlo = thi = 0;
            const int64_t k = e - cta_begin;
            const int slot = static_cast<int>(k % C::SLOTS);
            if (k >= C::SLOTS) mbar_wait(&empty[slot], static_cast<uint32_t>((k / C::SLOTS) - 1) & 1u, p.err);
            smeta[slot] = make_int2(tlo, thi);
            if (thi > tlo) {
              const size_t off = (static_cast<size_t>(page) * p.hkv + h) * kPage * D;
              mbar_arrive_expect_tx(&full[slot], 2 * C::CHUNK);
              bulk_g2s(kv + slot * C::SLOT, Kp + off, C::CHUNK, &full[slot]);
              bulk_g2s(kv + slot * C::SLOT + C::CHUNK, Vp + off, C::CHUNK, &full[slot]);
            } else {
              mbar_arrive(&full[slot]);
            }
          }
          __syncwarp();
        }
      }
    } else {
      // ============================================================================================= consumers
      float *wlog = wlog_all + warp * G * kPage;
      for (int si = 0; si < nseg; ++si) {
        const Seg sg = segs[si];
        const int r = sg.row / p.hkv, h = sg.row - r * p.hkv;
        float qf[G][C::EPL], o[G][C::EPL], m_run[G], l_own[C::VPL];
        {
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
            m_run[g] = -INFINITY;
          }
#pragma unroll
          for (int k = 0; k < C::VPL; ++k) l_own[k] = 0.0f;
        }
        // owned (token, head) pairs after the reduce-scatter: value v = j*G + g is token j*TPI + ts of head g
        int g_own[C::VPL], tok_own[C::VPL];
        bool ok_own[C::VPL];
#pragma unroll
        for (int k = 0; k < C::VPL; ++k) {
          const int v = (lane % C::LPT) * C::VPL + k;
          const int j = v / G;
          g_own[k] = v - j * G;
          tok_own[k] = j * C::TPI + ts;
          ok_own[k] = v < C::NI * G;
        }
        for (int64_t e = sg.b + warp; e < sg.e; e += kNCW) {
          const int64_t kk = e - cta_begin;
          const int slot = static_cast<int>(kk % C::SLOTS);
          mbar_wait(&full[slot], static_cast<uint32_t>(kk / C::SLOTS) & 1u, p.err);
          const int2 tt = smeta[slot];
          const int tlo = tt.x, thi = tt.y;
          const unsigned char *kb = kv + slot * C::SLOT;
          // ---- logits of the page's 16 tokens for the G heads
          float part[C::NV];
#pragma unroll
          for (int v = 0; v < C::NV; ++v) part[v] = 0.0f;
          if (thi > tlo) {
            const uint4 *kvec = reinterpret_cast<const uint4 *>(kb);
            uint4 w4[C::NI];
#pragma unroll
            for (int j = 0; j < C::NI; ++j) w4[j] = kvec[j * 32 + lane];
#pragma unroll
            for (int j = 0; j < C::NI; ++j) {
              float kf[C::EPL];
              Vec16<T>::unpack(w4[j], kf);
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
          float s_own[C::VPL], mr_own[C::VPL];
          bool over = false;
#pragma unroll
          for (int k = 0; k < C::VPL; ++k) {
            const bool vis = ok_own[k] && tok_own[k] >= tlo && tok_own[k] < thi;
            s_own[k] = vis ? part[k] : -INFINITY;
            float mr = -INFINITY;
#pragma unroll
            for (int g = 0; g < G; ++g)
              if (g == g_own[k]) mr = m_run[g];
            mr_own[k] = mr;
            over |= vis && (s_own[k] > mr + kRescaleThreshold);
          }
          if (__any_sync(0xffffffffu, over)) {
            // raise the running max of every head to this page's max, rescaling the state accumulated so far
#pragma unroll
            for (int k = 0; k < C::VPL; ++k)
              if (ok_own[k]) wlog[g_own[k] * kPage + tok_own[k]] = s_own[k];
            __syncwarp();
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float pm = warp_max(lane < kPage ? wlog[g * kPage + lane] : -INFINITY);
              const float mn = fmaxf(m_run[g], pm);
              const float a = (m_run[g] == -INFINITY) ? (mn == -INFINITY ? 1.0f : 0.0f) : exp2f(m_run[g] - mn);
              m_run[g] = mn;
#pragma unroll
              for (int k = 0; k < C::EPL; ++k) o[g][k] *= a;
#pragma unroll
              for (int k = 0; k < C::VPL; ++k)
                if (g_own[k] == g) {
                  l_own[k] *= a;
                  mr_own[k] = mn;
                }
            }
            __syncwarp();
          }
          // probabilities of the owned logits, shared with the warp through wlog[g][token]
#pragma unroll
          for (int k = 0; k < C::VPL; ++k) {
            if (ok_own[k]) {
              const float pv = (s_own[k] == -INFINITY) ? 0.0f : exp2f(s_own[k] - mr_own[k]);
              l_own[k] += pv;
              wlog[g_own[k] * kPage + tok_own[k]] = pv;
            }
          }
          __syncwarp();
          // ---- o += p v
          if (thi > tlo) {
            const uint4 *vvec = reinterpret_cast<const uint4 *>(kb + C::CHUNK);
            const bool fullpage = (tlo == 0 && thi == kPage);
#pragma unroll
            for (int j = 0; j < C::NI; ++j) {
              const int tok = j * C::TPI + ts;
              float vf[C::EPL];
              Vec16<T>::unpack(vvec[j * 32 + lane], vf);
              if (!fullpage && !(tok >= tlo && tok < thi)) {
#pragma unroll
                for (int k = 0; k < C::EPL; ++k) vf[k] = 0.0f;  // invisible slots may hold anything (even NaN)
              }
#pragma unroll
              for (int g = 0; g < G; ++g) {
                const float pw = wlog[g * kPage + tok];
#pragma unroll
                for (int k = 0; k < C::EPL; ++k) o[g][k] = fmaf(pw, vf[k], o[g][k]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // ---- end of the segment: this warp's state into comb[warp], then combine across warps
        float *cw = comb + warp * (G * D + 2 * G);
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
            for (int k = 0; k < C::EPL; ++k) cw[g * D + base_dim + k] = o[g][k];
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float lsum = 0.0f;
#pragma unroll
          for (int k = 0; k < C::VPL; ++k)
            if (ok_own[k] && g_own[k] == g) lsum += l_own[k];
          lsum = warp_sum(lsum);
          if (lane == 0) {
            cw[G * D + g] = m_run[g];
            cw[G * D + G + g] = lsum;
          }
        }
        consumer_sync();
        // combine the kNCW warp states: res[0, G*D) output, res[G*D + g] max, res[G*D + G + g] sum
        const int ctid = tid;  // 0 .. kCT-1
        if (ctid < G) {
          float M = -INFINITY;
          for (int w = 0; w < kNCW; ++w) M = fmaxf(M, comb[w * (G * D + 2 * G) + G * D + ctid]);
          float L = 0.0f;
          for (int w = 0; w < kNCW; ++w) {
            const float mw = comb[w * (G * D + 2 * G) + G * D + ctid];
            L += (mw == -INFINITY) ? 0.0f : comb[w * (G * D + 2 * G) + G * D + G + ctid] * exp2f(mw - M);
          }
          res[G * D + ctid] = M;
          res[G * D + G + ctid] = L;
        }
        consumer_sync();
        for (int i = ctid; i < G * D; i += kCT) {
          const int g = i / D;
          const float M = res[G * D + g];
          float acc = 0.0f;
          if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kNCW; ++w) {
              const float mw = comb[w * (G * D + 2 * G) + G * D + g];
              if (mw != -INFINITY) acc = fmaf(comb[w * (G * D + 2 * G) + i], exp2f(mw - M), acc);
            }
          }
          res[i] = acc;
        }
        consumer_sync();

        // ---- finish the row, or hand over a partial record (the last CTA to finish the row merges)
        const int b_first = owner_cta(sg.rb, E, nb), b_last = owner_cta(sg.re - 1, E, nb);
        const int n_contrib = b_last - b_first + 1;
        const size_t out_base = (static_cast<size_t>(r) * p.hq + h * G) * D;
        T *outp = static_cast<T *>(p.out);
        if (n_contrib == 1) {
          for (int i = ctid; i < G * D; i += kCT) {
            const float l = res[G * D + G + i / D];
            outp[out_base + i] = from_f<T>(l > 0.0f ? res[i] / l : 0.0f);
          }
          if (ctid < G) {
            const float l = res[G * D + G + ctid];
            p.lse[static_cast<size_t>(r) * p.hq + h * G + ctid] =
                l > 0.0f ? (res[G * D + ctid] + log2f(l)) * kLn2 : -INFINITY;
            if (!(l > 0.0f)) set_error(p.err, kErrLength);
          }
        } else {
          const int pslot = static_cast<int>(blockIdx.x) + sg.row;
          float *pp = p.part + static_cast<size_t>(pslot) * G * D;
          for (int i = ctid; i < G * D; i += kCT) __stcg(pp + i, res[i]);
          if (ctid < G) {
            __stcg(p.ml + (static_cast<size_t>(pslot) * G + ctid) * 2, res[G * D + ctid]);
            __stcg(p.ml + (static_cast<size_t>(pslot) * G + ctid) * 2 + 1, res[G * D + G + ctid]);
          }
          __threadfence();
          consumer_sync();
          if (ctid == 0) {
            const int old = atomicAdd(&p.counters[sg.row], 1);
            s_flag = (old == n_contrib - 1) ? 1 : 0;
            if (s_flag) p.counters[sg.row] = 0;  // every contributor has arrived: leave the counter at zero
          }
          consumer_sync();
          if (s_flag) {
            // Last arriver: merge the row's partial records from CTAs b_first..b_last. The (m, l) pairs of up to
            // 32 contributors are staged in shared memory by one parallel load pass; the partial outputs are loaded
            // with up to 16 loads in flight per element before any is used.
            __threadfence();
            constexpr int kElems = (G * D + kCT - 1) / kCT;
            float *sm_m = wlog_all;           // [32][G] (every warp is past its pages)
            float *sm_w = wlog_all + 32 * G;  // [32][G]
            float *Mg = res + G * D + 2 * G, *Rg = res + G * D + 3 * G, *Lg = res + G * D + G;
            if (ctid < G) {
              Mg[ctid] = -INFINITY;
              Lg[ctid] = 0.0f;
            }
            float acc[kElems];
#pragma unroll
            for (int k = 0; k < kElems; ++k) acc[k] = 0.0f;
            const int nc = b_last - b_first + 1;
            for (int g0 = 0; g0 < nc; g0 += 32) {
              const int ng = min(32, nc - g0);
              consumer_sync();
              for (int q = ctid; q < ng * G; q += kCT) {
                const int bb = q / G, g = q - (q / G) * G;
                const size_t o2 = (static_cast<size_t>(b_first + g0 + bb + sg.row) * G + g) * 2;
                sm_m[bb * G + g] = __ldcg(p.ml + o2);
                sm_w[bb * G + g] = __ldcg(p.ml + o2 + 1);
              }
              consumer_sync();
              if (ctid < G) {
                const float Mo = Mg[ctid];
                float M = Mo;
                for (int bb = 0; bb < ng; ++bb) M = fmaxf(M, sm_m[bb * G + ctid]);
                const float resc = (Mo == -INFINITY || M == -INFINITY) ? 0.0f : exp2f(Mo - M);
                float Ls = Lg[ctid] * resc;
                for (int bb = 0; bb < ng; ++bb) {
                  const float mb = sm_m[bb * G + ctid];
                  const float w = (mb == -INFINITY || M == -INFINITY) ? 0.0f : exp2f(mb - M);
                  Ls += sm_w[bb * G + ctid] * w;
                  sm_w[bb * G + ctid] = w;
                }
                Mg[ctid] = M;
                Lg[ctid] = Ls;
                Rg[ctid] = resc;
              }
              consumer_sync();
#pragma unroll
              for (int k = 0; k < kElems; ++k) {
                const int i = ctid + k * kCT;
                if (i < G * D) {
                  const int g = i / D;
                  float a = (g0 > 0) ? acc[k] * Rg[g] : 0.0f;
                  for (int b0 = 0; b0 < ng; b0 += 16) {
                    float v[16];
#pragma unroll
                    for (int bb = 0; bb < 16; ++bb)
                      v[bb] = (b0 + bb < ng)
                                  ? __ldcg(p.part + static_cast<size_t>(b_first + g0 + b0 + bb + sg.row) * G * D + i)
                                  : 0.0f;
#pragma unroll
                    for (int bb = 0; bb < 16; ++bb)
                      if (b0 + bb < ng) a = fmaf(v[bb], sm_w[(b0 + bb) * G + g], a);
                  }
                  acc[k] = a;
                }
              }
            }
            consumer_sync();
#pragma unroll
            for (int k = 0; k < kElems; ++k) {
              const int i = ctid + k * kCT;
              if (i < G * D) {
                const int g = i / D;
                const float Ls = Lg[g];
                outp[out_base + i] = from_f<T>(Ls > 0.0f ? acc[k] / Ls : 0.0f);
                if ((i % D) == 0) {
                  p.lse[static_cast<size_t>(r) * p.hq + h * G + g] =
                      Ls > 0.0f ? (Mg[g] + log2f(Ls)) * kLn2 : -INFINITY;
                  if (!(Ls > 0.0f)) set_error(p.err, kErrLength);
                }
              }
            }
          }
        }
        consumer_sync();
      }
    }
    __syncthreads();
    cur = win_end;
    w_row = s_wnext_row;
    w_rb = s_wnext_rb;
    __syncthreads();
    if (w_row >= p.nrows) break;
  }
}

template <class T, int D, int G>
cudaError_t launch_tdg(const Params &prm, cudaStream_t s) {
  using C = Cfg<T, D, G>;
  auto kern = propose_kernel<T, D, G>;
  static bool attr[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr[dev & 63] = true;
  }
  int nb = device_sm_count();
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
