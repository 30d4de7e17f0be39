// k_propose.cu - selected-KV proposal attention, q = 1 per request (sm_103a), optionally fused with the step's
// KV append.
//
// KAP paper, executor: each proposal step is a decode-like step (q_prop = 1) whose attention sees only the
// selected prompt pages of the compact view, plus every generated token, at the original logical positions; the
// step writes its own token's KV at that token's logical position.
// EarlySelectKV page: attention of the main flow reads only the pages the routing side chose in advance, and uses
// the true query.
//
// Design (GB300):
//  * Work = the concatenated entry lists of all (request, KV head) rows; CTA b owns the contiguous entry range
//    [b*E/nb, (b+1)*E/nb) (stream-K, one CTA per SM), so long and short rows balance across the SMs. A row split
//    over several CTAs is merged by the last CTA to finish it (one atomic counter per row, no waiting). A short
//    launch leaves the grid's last CTAs idle, since they start last, on the SMs the previous kernel frees last.
//  * A producer warp streams the CTA's entries through a ring of page slots: per entry one 1-D bulk copy
//    (cp.async.bulk) of the 4 KiB (page, head) chunk of K and one of V, completing on the slot's mbarrier. A view
//    entry and its row's lengths are loaded together, so a copy leaves two dependent loads after the kernel starts.
//    Once the ring's first fill is out, the window's next entries are prefetched into L2.
//  * The range is cut into windows of at most NSEG row segments. Each segment gets its own group of consumer warps
//    (one at least, the others in proportion to its entries) that takes the segment's entries round-robin, so all
//    segments of a window stream at once. The group's first warp prepares the segment's query once (rotated,
//    rounded, scaled) and, fused, the step token's key and value, in shared memory for the whole group. Lane l
//    holds 16 bytes of each token row; packed fp32 pair FMAs form the G heads' partial dot products, a few vector
//    rows at a time, and a reduce-scatter across the lanes of a token row leaves each lane a few finished logits.
//    Each warp keeps its own running max, sum and output; the max is only raised (and the state rescaled) when a
//    page exceeds it by more than 2^8, which is exact.
//  * A group that has finished its segment combines its warps' states behind its own named barrier and writes the
//    row's output, or hands a partial record to the row's last CTA, while the other groups keep streaming.
//  * With a settled view (lengths and prompt pages older than the previous kernel), the row scan, the segment
//    tables, the copies of pure prompt pages and the query's rotation angles all run before the dependency wait.
//  * Fused append: the step token of request r sits at position P = seq_len[r] - 1. The warp that consumes the page
//    holding P writes the prepared K and V into the pool and patches its shared-memory copy of the page first.
#include "kap_device.cuh"
#include "kap_launch.h"

namespace kap {
namespace {

constexpr int kMaxSlotsExtraCtas = 4096;     // bound on the grid, for workspace sizing
constexpr int kMaxRowsScan = 256;            // rows whose entry offsets are scanned into shared memory at once
constexpr int kBarSeg0 = 1;                  // named barriers kBarSeg0 .. kBarSeg0 + NSEG - 1, one per segment
constexpr int kMergeChunk = 8;               // partial records loaded at once by a merging CTA
constexpr int kPrefetchAhead = 32;           // entries beyond the ring prefetched into L2 per window
constexpr int kShortEntries = 64;            // entries per CTA up to which a launch leaves spare SMs
constexpr int kSpareDiv = 19;                // ... 1/kSpareDiv of its grid (8 of 152 SMs)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;    // log2 units

// Consumer warps per CTA (one CTA per SM). A CTA's warps are a multiple of 4 less the producer's share: each of
// the SM's four sub-partitions holds a quarter of the register file and warps are dealt to them in turn, so 12
// warps leave 168 registers a lane. fp32 pages of d = 128 (twice the bytes per slot) keep 8 warps so that the ring
// still holds more slots than there are consumers. (Half-SM CTAs, which let the next launch's CTA start beside
// this one, and 15 consumer warps at 128 registers were measured slower.)
template <class T, int D, int G> struct Shape {
  static constexpr int NCW = (sizeof(T) == 4 && D == 128) ? 7 : 11;
  static constexpr int MINB = 1;
  static constexpr int THREADS = (NCW + 1) * 32;  // + the producer warp (warp NCW)
  // registers per thread: the SM's 64K over the resident threads, a multiple of 8, at most 248
  static constexpr int MAXREG = ((65536 / (MINB * THREADS)) / 8) * 8 > 248 ? 248 : ((65536 / (MINB * THREADS)) / 8) * 8;
};

template <class T, int D, int G>
struct Cfg {
  static constexpr int NCW = Shape<T, D, G>::NCW;
  static constexpr int MINB = Shape<T, D, G>::MINB;
  static constexpr int THREADS = Shape<T, D, G>::THREADS;
  static constexpr int ESZ = sizeof(T);
  static constexpr int EPL = 16 / ESZ;           // elements per 16-byte vector
  static constexpr int EP2 = EPL / 2;            // fp32 pairs per vector
  static constexpr int LPT = D * ESZ / 16;       // lanes covering one token row
  static constexpr int TPI = 32 / LPT;           // token rows per warp-wide 16-byte load
  static constexpr int NI = kPage / TPI;         // 16-byte vectors per lane per (page, head) chunk
  static constexpr int CHUNK = kPage * D * ESZ;  // bytes of one (page, head) chunk
  static constexpr int LOG_LPT = LPT == 8 ? 3 : (LPT == 16 ? 4 : 5);
  static constexpr bool POW2G = (G & (G - 1)) == 0;
  static constexpr int LOG_G = G == 1 ? 0 : (G == 2 ? 1 : (G == 4 ? 2 : 3));
  // The logits of a page are formed RC vector rows at a time (RC * G partial values per lane, reduce-scattered over
  // the LPT lanes of a token row), so that few partial sums are live at once.
  static constexpr int RC = (POW2G && NI * G > LPT) ? LPT / G : NI;
  static constexpr int NCH = NI / RC;                          // chunks per page
  static constexpr int NVC = ((RC * G + LPT - 1) / LPT) * LPT;  // reduce-scatter values per chunk (padded)
  static constexpr int VPC = NVC / LPT;                        // finished logits a lane owns per chunk
  static constexpr int VPL = NCH * VPC;                        // ... per page
  static constexpr int REC = G * D + 2 * G;      // floats of one warp's state record (o, m, l)
  static constexpr int NSEG = NCW < 4 ? NCW : 4;  // row segments per window (each gets at least one warp)
  // per segment: the group's query, rotated, rounded to T and scaled (fp32 [G][D]), then the step token's K
  // (rotated) and V as T
  static constexpr int QPB = G * D * 4 + 2 * D * ESZ;
  // Select-free reduce-scatter: when the RC*G values of a chunk are a power of two (G a power of two) and at least
  // LPT, a lane keeps logical value v in register v ^ PERM(lane), so every butterfly level sends the upper half of
  // the registers and keeps the lower half. The lane loads vector row j ^ PJ(lane) and query head g ^ PG(lane).
  static constexpr bool XPERM = POW2G && RC * G >= LPT;
  // shared memory carve-up (bytes)
  static constexpr int COMB = NCW * REC * 4;              // per-warp state records
  static constexpr int WLOG = NCW * G * kPage * 8;        // per-warp logits, or probability pairs, of one page
  static constexpr int SEGB = NSEG * 48;                  // segment table
  static constexpr int QPREP = NSEG * QPB;                // per-segment query and step token
  static constexpr int ROWB = (kMaxRowsScan + 1) * 4;     // per-row entry offsets (row scan)
  static constexpr int FIXED = COMB + WLOG + SEGB + QPREP + ROWB + 256;
  static constexpr int SLOT = 2 * CHUNK;                  // K and V of one entry
  // per CTA: 227 KB alone on an SM, else its share of the SM's 228 KB less the 1 KB each CTA reserves
  static constexpr int BUDGET = MINB == 1 ? 226 * 1024 : (228 / MINB - 2) * 1024;
  static constexpr int SLOTS_FIT = (BUDGET - FIXED) / (SLOT + 32);
  static constexpr int SLOTS = SLOTS_FIT > 32 ? 32 : SLOTS_FIT;
  // entries the producer handles per step: small enough that a step waiting on one slot's consumer holds back few
  // copies (8 measured best against 2, 4 and 16)
  static constexpr int BATCH = SLOTS < 8 ? SLOTS : 8;
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_COMB = OFF_KV + SLOTS * SLOT;
  static constexpr int OFF_WLOG = OFF_COMB + COMB;
  static constexpr int OFF_SEG = ((OFF_WLOG + WLOG + 15) / 16) * 16;
  static constexpr int OFF_QP = OFF_SEG + SEGB;          // [NSEG][QPB]
  static constexpr int OFF_SMETA = OFF_QP + QPREP;        // [SLOTS] int4 (tlo | thi << 16, step token, page, entry)
  static constexpr int OFF_BAR = OFF_SMETA + SLOTS * 16;  // full[SLOTS], empty[SLOTS]
  static constexpr int OFF_ROWS = OFF_BAR + 2 * SLOTS * 8;
  static constexpr int SMEM = OFF_ROWS + ROWB;
  static_assert(SLOTS >= 4, "too few page slots");
  static_assert(SMEM + 256 <= BUDGET, "shared memory per CTA");
  static_assert(EPL % 2 == 0 && (D / 2) % EPL == 0, "vector layout");
  static_assert(NI % RC == 0, "chunk rows");
  static_assert(kBarSeg0 + NSEG <= 16, "named barriers");
  static_assert(QPB % 16 == 0, "query area alignment");
  static_assert(NCW <= SLOTS, "a round of issues fits in the ring");
};

struct Params {
  const void *k, *v;  // pool; written only by the fused append
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
  const void *k_new, *v_new;  // fused append: [R][Hkv][D] step-token keys (before RoPE) and values, or null
  const float *inv_freq;      // [D/2]
  int settled;                // view, lengths and prompt tokens predate the previous kernel on the stream
};

// One row segment of a window: global entries [b, e) of attention row `row` (whose own range is [rb, re)),
// consumed by warps [w0, w0 + nw).
struct Seg {
  int64_t b, e, rb, re;
  int row, vr, w0, nw;
};
static_assert(sizeof(Seg) == 48, "segment record size");

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
__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ int ld_acquire_shared(const int *p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// Waits until ring entry kk (this CTA's entry sequence number) has landed in its slot. The slot's barrier completes
// one phase per entry issued to it, in order (entry kk is phase kk / SLOTS of its slot), and a warp may reach its
// entry while an earlier phase of the slot is still pending, when a parity wait alone can return for that earlier
// phase. The producer stamps the slot with kk before it issues kk's copy, and it issues kk only after the slot's
// previous phase has completed and been consumed. So once the stamp reads kk, the pending phase is kk's own (or it
// has completed) and the parity wait is exact. Until then the warp waits on the parity of each earlier phase in turn
// (each attempt that fails moves the slot on by a phase; at most kk / SLOTS phases precede kk's). All waits suspend
// in hardware and are bounded.
template <int SLOTS>
__device__ __forceinline__ bool wait_entry(const int *stamp, uint64_t *full, int kk, uint32_t parity, int *err) {
  const int attempts = kk / SLOTS + 2;
  for (int attempt = 0; attempt < attempts; ++attempt) {
    if (ld_acquire_shared(stamp) == kk) return mbar_wait(full, parity, err);
    if (!mbar_wait(full, parity, err)) return false;
    if (ld_acquire_shared(stamp) == kk) return mbar_wait(full, parity, err);
    if (!mbar_wait(full, parity ^ 1u, err)) return false;
  }
  set_error(err, kErrTimeout);
  return false;
}

// Four consecutive output elements, rounded to the output type, in one store (8 bytes bf16, 16 bytes fp32).
template <class T>
__device__ __forceinline__ void store4(T *dst, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *dst, float a, float b, float c, float d) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  *reinterpret_cast<uint2 *>(dst) =
      make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}
template <>
__device__ __forceinline__ void store4<float>(float *dst, float a, float b, float c, float d) {
  *reinterpret_cast<float4 *>(dst) = make_float4(a, b, c, d);
}

// Two consecutive elements of T in one load or store.
template <class T> struct Vec2;
template <> struct Vec2<__nv_bfloat16> {
  using type = __nv_bfloat162;
  __device__ static float get(type v, int t) { return t == 0 ? __low2float(v) : __high2float(v); }
  __device__ static type make(float a, float b) { return __floats2bfloat162_rn(a, b); }
};
template <> struct Vec2<float> {
  using type = float2;
  __device__ static float get(type v, int t) { return t == 0 ? v.x : v.y; }
  __device__ static type make(float a, float b) { return make_float2(a, b); }
};

template <class T, int D, int G>
__global__ void __launch_bounds__((Shape<T, D, G>::THREADS)) __maxnreg__((Shape<T, D, G>::MAXREG)) propose_kernel(
    const Params p) {
  using C = Cfg<T, D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *kv = smem + C::OFF_KV;
  float *comb = reinterpret_cast<float *>(smem + C::OFF_COMB);      // [C::NCW][REC]
  float *wlog_all = reinterpret_cast<float *>(smem + C::OFF_WLOG);  // [C::NCW][16][G] float2 (or [G][16] float)
  unsigned char *qprep_all = smem + C::OFF_QP;                       // [NSEG][QPB]
  Seg *segs = reinterpret_cast<Seg *>(smem + C::OFF_SEG);
  int4 *smeta = reinterpret_cast<int4 *>(smem + C::OFF_SMETA);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::SLOTS;
  int *rowoff = reinterpret_cast<int *>(smem + C::OFF_ROWS);  // [nrows + 1] when nrows <= kMaxRowsScan
  __shared__ int64_t s_total, s_rb0, s_wnext_rb;
  __shared__ int s_row0, s_nseg, s_wnext_row;
  __shared__ int s_last[C::NSEG];
  __shared__ int scan_scratch[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool fused = p.k_new != nullptr;

  // Entry offsets of the rows (one parallel load of every row's count, a block scan in shared memory), then E,
  // this CTA's range and the row holding its first entry. Rows beyond kMaxRowsScan use a warp scan in global order.
  if (tid < C::SLOTS) {  // one slot's barriers per thread
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], 1);
    fence_barrier_init();
    smeta[tid].w = -1;  // no entry issued yet (shared memory keeps an earlier launch's stamps)
  }
  // A settled view lets the row scan, the segment tables and the copies of pure prompt pages run while the previous
  // kernel finishes; everything else waits for it (consumers below, the producer at its first other entry).
  if (!p.settled) grid_dependency_sync();
  const bool small_rows = p.nrows <= kMaxRowsScan;
  if (small_rows) {
    const int per = (p.nrows + C::THREADS - 1) / C::THREADS;  // thread t owns rows [t*per, (t+1)*per)
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
    if (tid == C::THREADS - 1) {
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
  // Split over nb <= E CTAs so that every participating CTA owns at least one entry (the merge counts them). A short
  // launch (at most kShortEntries per CTA) leaves the grid's last CTAs idle: they are dispatched last, onto the SMs
  // that the previous kernel frees last, and waiting for those SMs would hold up the whole launch (as long as the
  // rest of the launch takes, the SMs freed first then take the next launch's first CTAs).
  int nb = static_cast<int>(E < static_cast<int64_t>(gridDim.x) ? E : static_cast<int64_t>(gridDim.x));
  if (E <= static_cast<int64_t>(kShortEntries) * gridDim.x)
    nb = min(nb, static_cast<int>(gridDim.x - gridDim.x / kSpareDiv));
  if (E == 0 || static_cast<int>(blockIdx.x) >= nb) {
    // With nothing to do at all, a CTA still orders its dependents after the previous kernel; beside working CTAs,
    // whose triggers follow their own waits, an idle CTA just leaves.
    if (p.settled && E == 0) grid_dependency_sync();
    return;
  }
  const int64_t cta_begin = static_cast<int64_t>(blockIdx.x) * E / nb;
  const int64_t cta_end = static_cast<int64_t>(blockIdx.x + 1) * E / nb;

  if (small_rows) {
    if (tid == 0) {  // last row whose start is <= cta_begin
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
  // With a settled view the dependency wait comes later: consumers take it before their first read of q (after the
  // first window's segment table, so that the producer's copies are not held at that barrier), the producer before
  // its first entry that is not pure prompt.
  bool waited = !p.settled;

  for (int64_t cur = cta_begin; cur < cta_end;) {
    if (warp == C::NCW) {
      // ---- segment table of this window: rows w_row .. w_row+31 intersected with [cur, cta_end), at most
      // NSEG non-empty segments; each gets one warp plus a share of the spare warps by its entry count.
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
      const int idx = __popc(mask & ((1u << lane) - 1u));
      const int nseg = min(__popc(mask), C::NSEG);
      const bool keep = nonempty && idx < C::NSEG;
      const int cnt = keep ? static_cast<int>(se - sb) : 0;
      int cinc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, cinc, o);
        if (lane >= o) cinc += v;
      }
      const int n = __shfl_sync(0xffffffffu, cinc, 31);
      if (keep) {
        const int64_t cum = cinc - cnt;
        const int64_t spare = C::NCW - nseg;
        Seg sg;
        sg.b = sb;
        sg.e = se;
        sg.rb = rb;
        sg.re = re;
        sg.row = row;
        sg.vr = view_row(p, row);
        sg.w0 = idx + static_cast<int>(spare * cum / n);
        sg.nw = idx + 1 + static_cast<int>(spare * (cum + cnt) / n) - sg.w0;
        segs[idx] = sg;
      }
      const unsigned dmask = __ballot_sync(0xffffffffu, nonempty && idx == C::NSEG);  // first row left over
      const int tot = __shfl_sync(0xffffffffu, incl, 31);
      if (dmask) {
        const int dl = __ffs(dmask) - 1;
        const int64_t drb = __shfl_sync(0xffffffffu, rb, dl);
        if (lane == 0) {
          s_wnext_row = w_row + dl;
          s_wnext_rb = drb;
        }
      } else if (lane == 0) {
        s_wnext_row = w_row + 32;
        s_wnext_rb = w_rb + tot;
      }
      if (lane == 0) s_nseg = nseg;
    }
    __syncthreads();
    const int nseg = s_nseg;
    const int64_t win_end = (nseg > 0) ? segs[nseg - 1].e : cur;  // a window of empty rows only moves the rows on

    if (warp == C::NCW) {
      // ============================================================================================== producer
      const uint64_t pol = l2_evict_first_policy();  // the selected pages are streamed once per launch
      // Issue order: the window's segments take turns, each issuing in round j the entries j*nw .. j*nw + nw - 1
      // of its own range (nw = its warps), so that all groups stream at once and every warp's next entry is about
      // one ring length ahead at most. Entry u of a round, counted over the segments in order, gets the sequence
      // number (kacc + u) of this CTA: its ring slot and the stamp the consumer checks.
      // The entries past the ring's first fill (up to kPrefetchAhead, in each segment's share) are prefetched into
      // L2 once the ring is full, so that it refills from L2 when the consumers free their slots; before the
      // dependency wait, only pages whose visible tokens are all prompt tokens. (Issued before the first fill, their
      // metadata loads would hold back the first copies by a round trip per segment.)
      auto prefetch_window = [&]() {
        for (int si = 0; si < nseg; ++si) {
          const Seg sg = segs[si];
          const int64_t n = sg.e - sg.b;
          const int64_t lo = sg.b + (static_cast<int64_t>(C::SLOTS) * sg.nw) / C::NCW;
          const int64_t hi = min(sg.e, sg.b + (static_cast<int64_t>(C::SLOTS + kPrefetchAhead) * sg.nw) / C::NCW);
          if (n <= 0 || lo >= hi) continue;
          const int r = sg.row / p.hkv, h = sg.row - r * p.hkv;
          const int L = p.ctx_len[r], S = p.seq_len[r], nsel = p.vnsel[sg.vr];
          for (int64_t e = lo + lane; e < hi; e += 32) {
            const int i = static_cast<int>(e - sg.rb);
            const size_t o = static_cast<size_t>(sg.vr) * p.vcap + i;
            const int page = p.vbt[o], base = p.vlp[o] * kPage;
            const int thi = min(kPage, S - base), tlo = (i < nsel) ? 0 : max(0, L - base);
            if (thi > tlo && page >= 0 && page < p.num_pages && (waited || base + thi <= L)) {
              const size_t off = (static_cast<size_t>(page) * p.hkv + h) * kPage * D;
              bulk_prefetch_l2(Kp + off, C::CHUNK);
              bulk_prefetch_l2(Vp + off, C::CHUNK);
            }
          }
        }
      };
      int64_t kacc = (nseg > 0) ? segs[0].b - cta_begin : 0;
      bool prefetched = false;
      for (int j = 0;; ++j) {
        // this round's share of every segment; lane u < total takes entry u of the round
        int total = 0, my_si = -1, my_u = 0;
#pragma unroll
        for (int s2 = 0; s2 < C::NSEG; ++s2) {
          if (s2 < nseg) {
            const int64_t left = (segs[s2].e - segs[s2].b) - static_cast<int64_t>(j) * segs[s2].nw;
            const int c = left <= 0 ? 0 : (left < segs[s2].nw ? static_cast<int>(left) : segs[s2].nw);
            if (lane >= total && lane < total + c) {
              my_si = s2;
              my_u = lane - total;
            }
            total += c;
          }
        }
        if (total == 0) break;
        if (!prefetched && kacc + total > C::SLOTS) {  // this round waits for freed slots
          prefetch_window();
          prefetched = true;
        }
        const bool act = my_si >= 0;
        int i = 0, page = 0, base = 0, tlo = 0, thi = 0, L = 0, S = 0, h = 0, rn = 0;
        if (act) {
          const Seg sg = segs[my_si];
          const int r = sg.row / p.hkv;
          h = sg.row - r * p.hkv;
          L = p.ctx_len[r];
          S = p.seq_len[r];
          const int nsel = p.vnsel[sg.vr];
          rn = static_cast<int>(sg.re - sg.rb);
          const int64_t e = sg.b + static_cast<int64_t>(j) * sg.nw + my_u;
          i = static_cast<int>(e - sg.rb);  // entry index within the row's view
          const size_t o = static_cast<size_t>(sg.vr) * p.vcap + i;
          const int lp = p.vlp[o];
          page = p.vbt[o];
          base = lp * kPage;
          thi = min(kPage, S - base);
          tlo = (i < nsel) ? 0 : max(0, L - base);
          if (thi > tlo && (page < 0 || page >= p.num_pages)) {
            set_error(p.err, kErrPage);
            tlo = thi = 0;
          }
          if (thi <= tlo) tlo = thi = 0;
        }
        // Before the dependency wait only pages whose visible tokens are all prompt tokens are copied: a later
        // position of a page (a generated token) may have been written by the previous kernel.
        if (!waited && __any_sync(0xffffffffu, act && thi > tlo && base + thi > L)) {
          grid_dependency_wait();
          waited = true;
        }
        if (act) {
          int step_tok = -1;
          if (fused) {
            const int tk = S - 1 - base;
            if (tk >= tlo && tk < thi) step_tok = tk;
            if (i == rn - 1 && base + kPage <= S - 1) set_error(p.err, kErrLength);  // the view misses P
          }
          const int64_t k = kacc + lane;
          const int slot = static_cast<int>(k % C::SLOTS);
          if (k >= C::SLOTS) mbar_wait(&empty[slot], static_cast<uint32_t>((k / C::SLOTS) - 1) & 1u, p.err);
          smeta[slot] = make_int4(tlo | (thi << 16), step_tok, page, static_cast<int>(k));
          if (thi > tlo) {
            const size_t off = (static_cast<size_t>(page) * p.hkv + h) * kPage * D;
            mbar_arrive_expect_tx(&full[slot], 2 * C::CHUNK);
            bulk_g2s_stream(kv + slot * C::SLOT, Kp + off, C::CHUNK, &full[slot], pol);
            bulk_g2s_stream(kv + slot * C::SLOT + C::CHUNK, Vp + off, C::CHUNK, &full[slot], pol);
          } else {
            mbar_arrive(&full[slot]);
          }
        }
        __syncwarp();
        kacc += total;
      }
    } else if (nseg > 0) {
      // ============================================================================================= consumers
      int si = 0;
      while (si + 1 < nseg && segs[si + 1].w0 <= warp) ++si;
      const Seg sg = segs[si];
      const int gw = warp - sg.w0, nw = sg.nw;
      const int r = sg.row / p.hkv, h = sg.row - r * p.hkv;
      const int bar_id = kBarSeg0 + si, bar_n = nw * 32;
      float *wlog = wlog_all + warp * G * kPage * 2;  // logits [g][token] for a rescale, then (p, p) [token][g]
      float2 *wpair = reinterpret_cast<float2 *>(wlog);
      unsigned char *qp = qprep_all + si * C::QPB;
      float *qprep = reinterpret_cast<float *>(qp);          // [G][D] query of the group, ready for the dot products
      T *stepkv = reinterpret_cast<T *>(qp + G * D * 4);     // [D] step key (rotated), then [D] step value
      // The group's first warp prepares what every warp of the group needs once: the G query heads, rotated at the
      // step position P (fused form), rounded to T as a stored query would be and scaled by log2(e)/sqrt(D); in the
      // fused form also the step token's key (rotated by the same angles) and value. Lane l takes the rotary pairs
      // (i, i + D/2) for i = 2l and 2l + 1 (lanes with 2l >= D/2 idle). The angles depend on the lengths only, which
      // a settled view lets the warp read before the dependency wait; after it, the loads of q and of the step token
      // (two elements each) are all issued before the first is used (one round trip).
      const int i2 = 2 * lane;
      const bool rot_lane = gw == 0 && i2 < D / 2;
      if (rot_lane && fused) {
        // cos and sin of the lane's two angles, parked in the lane's own elements of head 0's query row
        const int P = p.seq_len[r] - 1;
        rope_factors(P, p.inv_freq[i2], qprep[i2], qprep[i2 + D / 2]);
        rope_factors(P, p.inv_freq[i2 + 1], qprep[i2 + 1], qprep[i2 + 1 + D / 2]);
      }
      if (!waited) {
        grid_dependency_sync();  // before q, the step token, outputs and the workspace
        waited = true;
      }
      if (rot_lane) {
        using P2 = typename Vec2<T>::type;
        const P2 *qrow = reinterpret_cast<const P2 *>(static_cast<const T *>(p.q) +
                                                      (static_cast<size_t>(r) * p.hq + h * G) * D + i2);
        const size_t src = (static_cast<size_t>(r) * p.hkv + h) * D + i2;
        P2 qx[G], qy[G], kx, ky, vx, vy;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          qx[g] = qrow[g * D / 2];
          qy[g] = qrow[g * D / 2 + D / 4];
        }
        if (fused) {
          const P2 *kn = reinterpret_cast<const P2 *>(static_cast<const T *>(p.k_new) + src);
          const P2 *vn = reinterpret_cast<const P2 *>(static_cast<const T *>(p.v_new) + src);
          kx = kn[0];
          ky = kn[D / 4];
          vx = vn[0];
          vy = vn[D / 4];
        }
        float c[2] = {1.0f, 1.0f}, sn2[2] = {0.0f, 0.0f};
        if (fused) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            c[t] = qprep[i2 + t];
            sn2[t] = qprep[i2 + t + D / 2];
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            float x = Vec2<T>::get(qx[g], t), y = Vec2<T>::get(qy[g], t);
            if (fused) {
              float xr, yr;
              rope_rotate(x, y, c[t], sn2[t], xr, yr);
              x = to_f(from_f<T>(xr));
              y = to_f(from_f<T>(yr));
            }
            qprep[g * D + i2 + t] = x * qscale;
            qprep[g * D + i2 + t + D / 2] = y * qscale;
          }
        }
        if (fused) {
          float xr[2], yr[2];
#pragma unroll
          for (int t = 0; t < 2; ++t)
            rope_rotate(Vec2<T>::get(kx, t), Vec2<T>::get(ky, t), c[t], sn2[t], xr[t], yr[t]);
          *reinterpret_cast<P2 *>(stepkv + i2) = Vec2<T>::make(xr[0], xr[1]);
          *reinterpret_cast<P2 *>(stepkv + i2 + D / 2) = Vec2<T>::make(yr[0], yr[1]);
          *reinterpret_cast<P2 *>(stepkv + D + i2) = vx;
          *reinterpret_cast<P2 *>(stepkv + D + i2 + D / 2) = vy;
        }
      }
      group_sync(bar_id, bar_n);
      float2 qf[G][C::EP2], o[G][C::EP2];
      float m_run[G], m_own[C::VPL], l_own[C::VPL];
      {
        const int pg = C::XPERM ? (((lane % C::LPT) * C::VPC) & (G - 1)) : 0;  // register g holds head g ^ pg
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 *src = reinterpret_cast<const float4 *>(qprep + (g ^ pg) * D + base_dim);
#pragma unroll
          for (int k = 0; k < C::EP2; k += 2) {
            const float4 f = src[k / 2];
            qf[g][k] = make_float2(f.x, f.y);
            qf[g][k + 1] = make_float2(f.z, f.w);
            o[g][k] = make_float2(0.0f, 0.0f);
            o[g][k + 1] = make_float2(0.0f, 0.0f);
          }
          m_run[g] = -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < C::VPL; ++k) {
          l_own[k] = 0.0f;
          m_own[k] = -INFINITY;
        }
      }
      // owned (token, head) pairs after the reduce-scatter: chunk c's value v = j*G + g is vector row c*RC + j,
      // i.e. token (c*RC + j)*TPI + ts, of head g; the lane keeps values [(lane%LPT)*VPC, +VPC) of every chunk
      int g_own[C::VPL], tok_own[C::VPL], wp_off[C::VPL];
      bool ok_own[C::VPL];
#pragma unroll
      for (int c = 0; c < C::NCH; ++c)
#pragma unroll
        for (int k = 0; k < C::VPC; ++k) {
          const int v = (lane % C::LPT) * C::VPC + k;
          const int j = v / G;
          g_own[c * C::VPC + k] = v - j * G;
          tok_own[c * C::VPC + k] = (c * C::RC + j) * C::TPI + ts;
          ok_own[c * C::VPC + k] = v < C::RC * G;
          wp_off[c * C::VPC + k] = tok_own[c * C::VPC + k] * G + g_own[c * C::VPC + k];
        }
      // This warp's entries are gw, gw + nw, ... of its segment: the one of round j has the sequence number
      // k0 + (entries of all segments in earlier rounds) + (entries of earlier segments in round j) + gw, the order
      // in which the producer issues them (fewer than 2^31 per CTA); slot kk % SLOTS, phase parity (kk / SLOTS) & 1.
      int sn[C::NSEG], sw[C::NSEG];
#pragma unroll
      for (int s2 = 0; s2 < C::NSEG; ++s2) {
        sn[s2] = s2 < nseg ? static_cast<int>(segs[s2].e - segs[s2].b) : 0;
        sw[s2] = s2 < nseg ? segs[s2].nw : 1;
      }
      const int n_mine = static_cast<int>(sg.e - sg.b);
      // the CTAs sharing this row (formed while the first pages are in flight: two 64-bit divisions)
      const int b_first = owner_cta(sg.rb, E, nb), b_last = owner_cta(sg.re - 1, E, nb);
      int issued = static_cast<int>(segs[0].b - cta_begin);  // sequence number of round j's first entry
      for (int j = 0; j * nw + gw < n_mine; ++j) {
        int before = 0, round = 0;
#pragma unroll
        for (int s2 = 0; s2 < C::NSEG; ++s2) {
          const int left = sn[s2] - j * sw[s2];
          const int c = left <= 0 ? 0 : (left < sw[s2] ? left : sw[s2]);
          before += (s2 < si) ? c : 0;
          round += c;
        }
        const int kk = issued + before + gw;
        issued += round;
        const int slot = kk % C::SLOTS;
        if (!wait_entry<C::SLOTS>(&smeta[slot].w, &full[slot], kk, static_cast<uint32_t>(kk / C::SLOTS) & 1u, p.err))
          break;  // timed out (error recorded): stop reading the ring
        const int4 mt = smeta[slot];
        const int tlo = mt.x & 0xffff, thi = mt.x >> 16;
        unsigned char *kb = kv + slot * C::SLOT;
        if (mt.y >= 0) {
          // the step token of this row lies in this page: its rotated key and its value into the pool and into
          // this copy of the page
          const int tok = mt.y;
          if (lane < C::LPT) {
            const uint4 kw = *reinterpret_cast<const uint4 *>(stepkv + base_dim);
            const uint4 vw = *reinterpret_cast<const uint4 *>(stepkv + D + base_dim);
            const int rowb = (tok * D + base_dim) * C::ESZ;
            *reinterpret_cast<uint4 *>(kb + rowb) = kw;
            *reinterpret_cast<uint4 *>(kb + C::CHUNK + rowb) = vw;
            const size_t dst = ((static_cast<size_t>(mt.z) * p.hkv + h) * kPage + tok) * D + base_dim;
            *reinterpret_cast<uint4 *>(const_cast<T *>(Kp) + dst) = kw;
            *reinterpret_cast<uint4 *>(const_cast<T *>(Vp) + dst) = vw;
            fence_proxy_async_smem();  // the slot is refilled by a bulk copy later
          }
          __syncwarp();
        }
        // ---- logits of the page's 16 tokens for the G heads, RC vector rows at a time. Slots of invisible tokens
        // (or of an entry with nothing to read) may hold anything: their logits are masked below.
        float s_own[C::VPL];
        {
          const uint4 *kvec = reinterpret_cast<const uint4 *>(kb);
          const int pj = C::XPERM ? (((lane % C::LPT) * C::VPC) >> C::LOG_G) : 0;  // register j: row j ^ pj
#pragma unroll
          for (int c = 0; c < C::NCH; ++c) {
            float part[C::NVC];
#pragma unroll
            for (int j = 0; j < C::RC; ++j) {
              float2 kf[C::EP2];
              Vec16<T>::unpack2(kvec[(c * C::RC + (j ^ pj)) * 32 + lane], kf);
#pragma unroll
              for (int g = 0; g < G; ++g) {
                float2 acc = __fmul2_rn(qf[g][0], kf[0]);
#pragma unroll
                for (int k = 1; k < C::EP2; ++k) acc = __ffma2_rn(qf[g][k], kf[k], acc);
                part[j * G + g] = acc.x + acc.y;
              }
            }
#pragma unroll
            for (int v = C::RC * G; v < C::NVC; ++v) part[v] = 0.0f;  // padding of the reduce-scatter
            // reduce-scatter over the LPT lanes of a token row: the lane keeps values [(lane%LPT)*VPC, +VPC)
#pragma unroll
            for (int step = 0; step < C::LOG_LPT; ++step) {
              const int msk = (C::LPT >> 1) >> step;
              const int half = C::NVC >> (step + 1);
              const bool upper = (lane & msk) != 0;
#pragma unroll
              for (int k = 0; k < half; ++k) {
                if (C::XPERM) {
                  part[k] += __shfl_xor_sync(0xffffffffu, part[k + half], msk);
                } else {
                  const float send = upper ? part[k] : part[k + half];
                  const float keep = upper ? part[k + half] : part[k];
                  part[k] = keep + __shfl_xor_sync(0xffffffffu, send, msk);
                }
              }
            }
#pragma unroll
            for (int k = 0; k < C::VPC; ++k) s_own[c * C::VPC + k] = part[k];
          }
        }
        bool over = false;
#pragma unroll
        for (int k = 0; k < C::VPL; ++k) {
          const bool vis = ok_own[k] && tok_own[k] >= tlo && tok_own[k] < thi;
          if (!vis) s_own[k] = -INFINITY;
          over |= s_own[k] > m_own[k] + kRescaleThreshold;
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
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int k = 0; k < C::EP2; ++k) o[g][k] = __fmul2_rn(o[g][k], a2);
#pragma unroll
            for (int k = 0; k < C::VPL; ++k)
              if (g_own[k] == g) {
                l_own[k] *= a;
                m_own[k] = mn;
              }
          }
          __syncwarp();
        }
        // probabilities of the owned logits, shared with the warp as (p, p) pairs in wpair[token][g]
#pragma unroll
        for (int k = 0; k < C::VPL; ++k) {
          if (ok_own[k]) {
            const float pv = (s_own[k] == -INFINITY) ? 0.0f : exp2f(s_own[k] - m_own[k]);
            l_own[k] += pv;
            wpair[wp_off[k]] = make_float2(pv, pv);
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
            float2 vf[C::EP2];
            Vec16<T>::unpack2(vvec[j * 32 + lane], vf);
            if (!fullpage && !(tok >= tlo && tok < thi)) {
#pragma unroll
              for (int k = 0; k < C::EP2; ++k) vf[k] = make_float2(0.0f, 0.0f);  // invisible slots may hold NaN
            }
            float2 pw2[G];
            if (G % 2 == 0) {
              const float4 *p4 = reinterpret_cast<const float4 *>(wpair + tok * G);
#pragma unroll
              for (int g = 0; g < G; g += 2) {
                const float4 t = p4[g / 2];
                pw2[g] = make_float2(t.x, t.y);
                pw2[g + 1 < G ? g + 1 : g] = make_float2(t.z, t.w);
              }
            } else {
#pragma unroll
              for (int g = 0; g < G; ++g) pw2[g] = wpair[tok * G + g];
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
              for (int k = 0; k < C::EP2; ++k) o[g][k] = __ffma2_rn(pw2[g], vf[k], o[g][k]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }

      // ---- end of this warp's share of the segment: its state into comb[warp]
      float *cw = comb + warp * C::REC;
#pragma unroll
      for (int msk = C::LPT; msk < 32; msk <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int k = 0; k < C::EP2; ++k) {
            o[g][k].x += __shfl_xor_sync(0xffffffffu, o[g][k].x, msk);
            o[g][k].y += __shfl_xor_sync(0xffffffffu, o[g][k].y, msk);
          }
      if (lane < C::LPT) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int k = 0; k < C::EP2; ++k) *reinterpret_cast<float2 *>(cw + g * D + base_dim + 2 * k) = o[g][k];
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
      group_sync(bar_id, bar_n);

      // ---- the group combines its warps' states: for each of its elements (head g), the max M over the group's
      // warps, their weights 2^(m_w - M), the weighted sum L and the weighted output, with no further barrier. The
      // 32 elements a warp takes at once share their head (D is a multiple of 32), so lane j forms warp j's weight
      // once and every lane reads the weights by shuffle.
      const int gt = gw * 32 + lane, GT = nw * 32;
      auto combined = [&](int i, int g, float &M, float &Ls) {
        const float *rec = comb + sg.w0 * C::REC;
        const float *rl = rec + min(lane, nw - 1) * C::REC;
        const float mj = lane < nw ? rl[G * D + g] : -INFINITY;
        const float lj = lane < nw ? rl[G * D + G + g] : 0.0f;
        float ow[C::NCW];  // every load issued up front (past the group's last warp: its record, weighted out)
#pragma unroll
        for (int j = 0; j < C::NCW; ++j) ow[j] = rec[min(j, nw - 1) * C::REC + i];
        M = warp_max(mj);
        const float wj = (mj == -INFINITY) ? 0.0f : exp2f(mj - M);
        Ls = warp_sum(lj * wj);
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < C::NCW; ++j) {
          const float w = __shfl_sync(0xffffffffu, wj, j);
          acc = j < nw ? fmaf(ow[j], w, acc) : acc;
        }
        return acc;
      };

      // ---- finish the row, or hand over a partial record (the last CTA to finish the row merges)
      const size_t out_base = (static_cast<size_t>(r) * p.hq + h * G) * D;
      T *outp = static_cast<T *>(p.out);
      float *lse_row = p.lse + static_cast<size_t>(r) * p.hq + h * G;
      if (b_first == b_last) {
        for (int i = gt; i < G * D; i += GT) {
          const int g = i / D;
          float M, Ls;
          const float acc = combined(i, g, M, Ls);
          outp[out_base + i] = from_f<T>(Ls > 0.0f ? acc / Ls : 0.0f);
          if (i - g * D == 0) {
            lse_row[g] = Ls > 0.0f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
            if (!(Ls > 0.0f)) set_error(p.err, kErrLength);
          }
        }
      } else {
        const size_t pslot = static_cast<size_t>(blockIdx.x) + sg.row;
        for (int i = gt; i < G * D; i += GT) {
          const int g = i / D;
          float M, Ls;
          __stcg(p.part + pslot * G * D + i, combined(i, g, M, Ls));
          if (i - g * D == 0) {
            __stcg(reinterpret_cast<float2 *>(p.ml) + pslot * G + g, make_float2(M, Ls));
          }
        }
        // One thread publishes the group's record and counts it in: the group barrier orders every thread's stores
        // before its acquire-release atomic, which also makes the other contributors' records visible to the last
        // arriver (and, through the second barrier, to its whole group).
        group_sync(bar_id, bar_n);
        if (gt == 0) {
          const int old = atom_add_acq_rel_gpu(&p.counters[sg.row], 1);
          const int last = (old == b_last - b_first) ? 1 : 0;
          if (last) p.counters[sg.row] = 0;  // every contributor has arrived: leave the counter at zero
          s_last[si] = last;
        }
        group_sync(bar_id, bar_n);
        if (s_last[si]) {
          // Last arriver: merge the partial records of CTAs b_first..b_last. A thread owns 4 consecutive elements of
          // one head; the kW = D/4 threads (at most a warp) that share a head form each contributor's weight once
          // (thread c of the group for contributor c) and read the weights by shuffle. Per chunk of kMergeChunk
          // contributors every load (an (m, l) pair per thread c, a 16-byte piece of the partial output per
          // contributor) is issued before any is used: one round trip per chunk.
          constexpr int kW = (D / 4 < 32) ? D / 4 : 32;
          static_assert(kMergeChunk <= kW, "one contributor per thread of a head's group");
          const int sub = lane % kW;
          // a warp-uniform trip count (whole warps take part in the shuffles); past the last element a lane repeats
          // the last one and stores nothing
          for (int i4w = gt - lane; i4w < G * D / 4; i4w += GT) {
            const bool act = i4w + lane < G * D / 4;
            const int i4 = act ? i4w + lane : G * D / 4 - 1;
            const int i0 = i4 * 4, g = i0 / D;
            float M = -INFINITY, Ls = 0.0f;
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int b0 = b_first; b0 <= b_last; b0 += kMergeChunk) {
              float4 pv[kMergeChunk];
#pragma unroll
              for (int c = 0; c < kMergeChunk; ++c) {
                const size_t ps = static_cast<size_t>(min(b0 + c, b_last)) + sg.row;  // clamped: always valid
                pv[c] = __ldcg(reinterpret_cast<const float4 *>(p.part + ps * G * D + i0));
              }
              const bool mine = sub < kMergeChunk && b0 + sub <= b_last;  // this thread's contributor exists
              const size_t pc = static_cast<size_t>(min(b0 + min(sub, kMergeChunk - 1), b_last)) + sg.row;
              float2 mlc = __ldcg(reinterpret_cast<const float2 *>(p.ml) + pc * G + g);
              if (!mine) mlc = make_float2(-INFINITY, 0.0f);
              float Mc = mlc.x;
#pragma unroll
              for (int o = kW / 2; o >= 1; o >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, o, kW));
              Mc = fmaxf(Mc, M);
              // with no finite maximum yet everything stays zero: the weights below are 0 and rs is 0
              const float rs = (M == -INFINITY) ? 0.0f : exp2f(M - Mc);
              const float wc = (mlc.x == -INFINITY) ? 0.0f : exp2f(mlc.x - Mc);
              float lw = mlc.y * wc;
#pragma unroll
              for (int o = kW / 2; o >= 1; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o, kW);
              Ls = fmaf(Ls, rs, lw);
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[e] *= rs;
#pragma unroll
              for (int c = 0; c < kMergeChunk; ++c) {
                const float w = __shfl_sync(0xffffffffu, wc, c, kW);
                acc[0] = fmaf(pv[c].x, w, acc[0]);
                acc[1] = fmaf(pv[c].y, w, acc[1]);
                acc[2] = fmaf(pv[c].z, w, acc[2]);
                acc[3] = fmaf(pv[c].w, w, acc[3]);
              }
              M = Mc;
            }
            if (!act) continue;
            const float inv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
            store4<T>(outp + out_base + i0, acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
            if (i0 - g * D == 0) {
              lse_row[g] = Ls > 0.0f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
              if (!(Ls > 0.0f)) set_error(p.err, kErrLength);
            }
          }
        }
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
    // The whole unified L1 as shared memory (MINB CTAs of this shape fit on one SM only with it).
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    attr[dev & 63] = true;
  }
  // One CTA per SM, but no more CTAs than the view can feed with a page per consumer warp (its capacity bounds
  // the entries): a small launch then leaves SMs free for work on other streams, at the same latency, since a
  // CTA's warps take its pages in parallel.
  int nb = device_sm_count();
  const int64_t feed = (static_cast<int64_t>(prm.nrows) * prm.vcap + C::NCW - 1) / C::NCW;
  if (feed < nb) nb = static_cast<int>(feed < 1 ? 1 : feed);
  if (nb > kMaxSlotsExtraCtas) nb = kMaxSlotsExtraCtas;
  launch_pdl(kern, dim3(nb), dim3(C::THREADS), C::SMEM, s, prm);
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
                           float *lse, void *ws, size_t ws_bytes, const void *k_new, const void *v_new,
                           const float *inv_freq, int *err, cudaStream_t s) {
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
  prm.k_new = k_new;
  prm.v_new = v_new;
  prm.inv_freq = inv_freq;
  prm.settled = va.settled;
  if (pa.dtype == 0 && pa.d == 128) return launch_td<__nv_bfloat16, 128>(prm, G, s);
  if (pa.dtype == 0 && pa.d == 64) return launch_td<__nv_bfloat16, 64>(prm, G, s);
  if (pa.dtype == 1 && pa.d == 128) return launch_td<float, 128>(prm, G, s);
  return launch_td<float, 64>(prm, G, s);
}

}  // namespace kap
