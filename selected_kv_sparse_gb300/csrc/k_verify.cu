// k_verify.cu - full-context verification attention with a causal query window (sm_103a).
//
// KAP paper, verifier: after k proposals the window (carry token and/or candidates) is verified in one forward
// pass over the full KV cache, the full block table and the original logical positions; row i of the window sees
// every earlier position and candidates 0..i.
//
// bf16, head_dim 128 (the tensor-core path): the G query heads of a KV head times the n_q window rows form a dense
// contraction of N = G*n_q (padded to 16) query columns against 128-token tiles (8 pages) of K and V.
//   S^T[128 tok x N] = K_tile[128 x 128] . Q^T         (tcgen05.mma, M = 128, K-major A and B, fp32 in TMEM)
//   softmax over tokens per column (thread = token), P^T written to shared memory as bf16 (128-byte swizzle)
//   O^T[128 d x N]   = V_tile^T[128 x 128 tok] . P^T     (tcgen05.mma, A = V read MN-major, fp32 in TMEM)
// K and V pages arrive by tiled TMA (two 64-column boxes per (page, head), 128-byte swizzle) into a 3-stage ring.
// Work is split stream-K over the concatenated tile lists of all (request, KV head) rows; the last CTA to finish
// a split row merges the partial (m, l, O) records.
// Other shapes (fp32 pools, head_dim 64) use a plain FFMA kernel, one warp per (query row, query head).
#include "kap_device.cuh"
#include "kap_launch.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace kap {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxCtas = 4096;
constexpr int kMaxDeferred = 16;  // row segments whose hand-off a CTA postpones to the end of its tiles

struct VParams {
  int num_pages, hkv, hq;
  const int32_t *bt;
  int max_pages;
  const int32_t *q_offsets, *q_start;
  int R, nrows;
  const void *q;
  void *out;
  float *lse;
  int *counters;
  float *ml;
  float *part;
  int npad_ws;  // padded query columns per partial record
  int *err;
};

__device__ __forceinline__ int row_nq(const VParams &p, int r) { return p.q_offsets[r + 1] - p.q_offsets[r]; }
// 128-token tiles of row (r, h): the pages holding positions 0 .. q_start + n_q - 1.
__device__ __forceinline__ int row_tiles(const VParams &p, int row) {
  const int r = row / p.hkv;
  const int nq = row_nq(p, r);
  if (nq <= 0) return 0;
  const int pages = (p.q_start[r] + nq + kPage - 1) / kPage;
  return (pages + 7) / 8;
}
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ int owner_cta(int64_t x, int64_t E, int nb) {
  return static_cast<int>(((x + 1) * nb - 1) / E);
}
__device__ __forceinline__ int fkey(float x) {
  const int b = __float_as_int(x);
  return b >= 0 ? b : (b ^ 0x7fffffff);
}
__device__ __forceinline__ float ffrom(int k) { return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff)); }

// ============================================================================================ tensor cores
// Warp roles (224 threads): warps 0-3 softmax + output merge (thread = token row of a tile for the softmax,
// thread = head-dim row for the merge), warps 4 and 6 TMA producers (K and V), warp 5 tcgen05 issuer. S, P and O are double
// buffered so that MMA1 of tile t+1 and MMA2 of tile t overlap the softmax of tile t and the merge of tile t-1.
constexpr int kTileTok = 128;
constexpr int kHalfBytes = 8 * kPage * 128;  // one 64-column half of a tile: 8 pages x 16 rows x 128 B = 16 KiB
constexpr int kStageBytes = 2 * kHalfBytes;   // 32 KiB of K (or V) per stage
constexpr int kTcThreads = 224;
constexpr float kRescaleThreshold = 8.0f;     // log2 units: keep a running max until a tile exceeds it by 2^8

struct TileMeta {
  int64_t rb, re;
  int valid, row, tile, first, last, npg, seg, nq, qpos0, qoff, pad;
};

template <int NPMAX>
struct TcSmem {
  static constexpr int KATOM = NPMAX * 128;  // bytes of one 64-column K-atom of an [NPMAX x 128] bf16 operand
  static constexpr int QP_BYTES = 4 * 2 * KATOM;  // Q[2] and P[2]
  static constexpr int kStages = (3 * 2 * kStageBytes + QP_BYTES + 4096 <= 227 * 1024) ? 3 : 2;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + kStages * kStageBytes;
  static constexpr int OFF_Q = OFF_V + kStages * kStageBytes;     // Q[2] (segment parity)
  static constexpr int OFF_P = OFF_Q + 2 * 2 * KATOM;              // P[2] (tile parity)
  static constexpr int OFF_CM = OFF_P + 2 * 2 * KATOM;             // column maxima [4][NPMAX]
  static constexpr int OFF_ST = OFF_CM + 4 * NPMAX * 4;            // m_run, lsum, alpha[2], m_sub, thr : [6][NPMAX]
  static constexpr int OFF_FLAG = OFF_ST + 6 * NPMAX * 4;          // rescale flag per tile parity [2]
  static constexpr int OFF_BAR = OFF_FLAG + 16;
  static constexpr int kMetaRing = 2 * kStages;  // tile metadata outlives its K stage (read until MMA2 and softmax)
  // kfull, vfull, kempty, vempty [kStages]; sfull, sfree, pfull, ofull, ofree, qfull, qempty [2];
  // mfull, mfree [kMetaRing]
  static constexpr int NBAR = 4 * kStages + 14 + 2 * kMetaRing;
  static constexpr int OFF_META = OFF_BAR + NBAR * 8;
  static constexpr int OFF_TMEM = OFF_META + kMetaRing * static_cast<int>(sizeof(TileMeta));
  static constexpr int BYTES = OFF_TMEM + 16;
  static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 bytes
  static constexpr int TMEM_COLS = (4 * NPMAX <= 32) ? 32 : (4 * NPMAX <= 64 ? 64 : (4 * NPMAX <= 128 ? 128 : 256));
  static_assert(ALLOC <= 227 * 1024, "shared memory per CTA");
};

// 2^x with the hardware approximation (relative error about 2^-22; the result is rounded to bf16 for P anyway).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_sync_128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// 16 consecutive floats from shared memory (16-byte aligned) in four 16-byte loads, ordered after earlier barriers
__device__ __forceinline__ void load16_shared(const float *src, float *v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float4 f;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                 : "r"(smem_u32(src + 4 * q)) : "memory");
    v[4 * q] = f.x;
    v[4 * q + 1] = f.y;
    v[4 * q + 2] = f.z;
    v[4 * q + 3] = f.w;
  }
}
__device__ __forceinline__ bool named_or_128(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

template <int NPMAX>
__global__ void __launch_bounds__(kTcThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const VParams p) {
  using L = TcSmem<NPMAX>;
  constexpr int kStages = L::kStages;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  unsigned char *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  unsigned char *Ks = sm + L::OFF_K;
  unsigned char *Vs = sm + L::OFF_V;
  unsigned char *Qs = sm + L::OFF_Q;
  unsigned char *Ps = sm + L::OFF_P;
  float *colmax = reinterpret_cast<float *>(sm + L::OFF_CM);
  float *m_run = reinterpret_cast<float *>(sm + L::OFF_ST);
  float *lsum = m_run + NPMAX;
  float *alpha_s = lsum + NPMAX;  // [2][NPMAX]
  // the running maxima as subtracted from the logits: m_run, or 0 while a column has seen no visible token (its
  // logits are then all -inf, and -inf - 0 gives the weight 0 where -inf - m_run would give NaN)
  float *m_sub = alpha_s + 2 * NPMAX;
  // the raw logit above which a column's running max must be raised: (m_run + 8) / scale (-inf before any)
  float *thr = m_sub + NPMAX;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
  constexpr int kMR = L::kMetaRing;
  uint64_t *kfull = bars, *vfull = bars + kStages, *kempty = bars + 2 * kStages, *vempty = bars + 3 * kStages;
  uint64_t *sfull = bars + 4 * kStages, *sfree = sfull + 2, *pfull = sfree + 2, *ofull = pfull + 2;
  uint64_t *ofree = ofull + 2, *qfull = ofree + 2, *qempty = qfull + 2, *mfree = qempty + 2;
  uint64_t *mfull = mfree + kMR;
  TileMeta *meta = reinterpret_cast<TileMeta *>(sm + L::OFF_META);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::OFF_TMEM);
  __shared__ int64_t s_total;
  __shared__ int s_abort, s_row0;
  __shared__ int4 s_def[kMaxDeferred];  // row segments whose partial record awaits counting in: row, b_first,
  __shared__ int s_defn[kMaxDeferred];  // b_last, first window row; and the row's query columns
  __shared__ int s_deflast[kMaxDeferred];
  __shared__ int s_ndef;
  volatile int *abort_flag = &s_abort;
  __shared__ int64_t s_rb0, s_re0;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.hq / p.hkv;
  grid_dependency_sync();

  if (warp == 0) {
    int64_t tot = 0;
    for (int base = 0; base < p.nrows; base += 32) {
      int c = (base + lane < p.nrows) ? row_tiles(p, base + lane) : 0;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      tot += c;
    }
    if (lane == 0) s_total = tot;
  }
  if (tid == 0) {
    s_abort = 0;
    s_ndef = 0;
    for (int i = 0; i < L::NBAR; ++i) mbar_init(&bars[i], 1);
    for (int b = 0; b < 2; ++b) {  // barriers the 4 softmax warps arrive on (one elected lane per warp)
      mbar_init(&sfree[b], 4);
      mbar_init(&pfull[b], 4);
      mbar_init(&ofree[b], 4);
    }
    for (int i = 0; i < kMR; ++i) mbar_init(&mfree[i], 5);  // 4 softmax warps + the MMA issuer
    fence_barrier_init();
  }
  __syncthreads();
  const int64_t E = s_total;
  // Split over nb <= E CTAs so that every participating CTA owns at least one tile (the merge counts them).
  const int nb = static_cast<int>(E < static_cast<int64_t>(gridDim.x) ? E : static_cast<int64_t>(gridDim.x));
  if (E == 0 || static_cast<int>(blockIdx.x) >= nb) return;
  const int64_t cta_begin = static_cast<int64_t>(blockIdx.x) * E / nb;
  const int64_t cta_end = static_cast<int64_t>(blockIdx.x + 1) * E / nb;

  // First row of this CTA's range: warp-parallel prefix over the rows' tile counts.
  if (warp == 0) {
    int64_t base = 0;
    for (int b = 0; b < p.nrows; b += 32) {
      const int row = b + lane;
      const int c = row < p.nrows ? row_tiles(p, row) : 0;
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
          s_re0 = re;
        }
        break;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4 || warp == 6) {
    // ============================================================================================== producers
    // Warp 4 issues the K boxes of each tile (and writes the tile metadata and the Q operand), warp 6 the V
    // boxes: both walk the same tile sequence, so their 16 TMA requests per tile are issued in parallel.
    const bool kprod = (warp == 4);
    const uint64_t pol = l2_evict_first_policy();  // the full KV is streamed once per launch
    int pr_row = s_row0, seg = -1;
    int64_t pr_rb = s_rb0, pr_re = s_re0, pr_cur = cta_begin;
    int row_r = -1, row_kvp = 0, row_nq_ = 0, row_qpos0 = 0, row_qoff = 0;
    int pl_row = 0, pl_tile = 0, pl_first = 0, pl_last = 0, pl_npg = 0, pl_h = 0, pl_page = -1, pl_valid = 0;
    int64_t pl_rb = 0, pl_re = 0;
    auto plan = [&]() {
      if (pr_cur >= cta_end) {
        pl_valid = 0;
        return;
      }
      while (pr_cur >= pr_re) {
        ++pr_row;
        pr_rb = pr_re;
        pr_re += row_tiles(p, pr_row);
      }
      const int r = pr_row / p.hkv;
      if (row_r != r) {
        row_r = r;
        row_nq_ = row_nq(p, r);
        row_qpos0 = p.q_start[r];
        row_qoff = p.q_offsets[r];
        row_kvp = (row_qpos0 + row_nq_ + kPage - 1) / kPage;
      }
      const int64_t seg_end = min(pr_re, cta_end);
      pl_valid = 1;
      pl_row = pr_row;
      pl_h = pr_row - r * p.hkv;
      pl_tile = static_cast<int>(pr_cur - pr_rb);
      pl_rb = pr_rb;
      pl_re = pr_re;
      pl_first = (pr_cur == pr_rb || pr_cur == cta_begin) ? 1 : 0;
      pl_last = (pr_cur + 1 == seg_end) ? 1 : 0;
      pl_npg = min(8, row_kvp - pl_tile * 8);
      pl_page = -1;
      if (lane < pl_npg && pl_tile * 8 + lane < p.max_pages)
        pl_page = p.bt[static_cast<size_t>(r) * p.max_pages + pl_tile * 8 + lane];
      ++pr_cur;
    };
    plan();
    int t = 0;
    for (;; ++t) {
      const int st = t % kStages, mi = t % kMR;
      if (t >= kStages && !mbar_wait(kprod ? &kempty[st] : &vempty[st], ((t / kStages) - 1) & 1, p.err)) {
        *abort_flag = 1;
        break;
      }
      if (kprod && t >= kMR && !mbar_wait(&mfree[mi], ((t / kMR) - 1) & 1, p.err)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      TileMeta &m = meta[mi];
      if (!pl_valid) {
        if (kprod && lane == 0) {
          m.valid = 0;
          mbar_arrive(&mfull[mi]);
          mbar_arrive(&kfull[st]);
        }
        break;
      }
      if (pl_first && kprod) {
        // Q rows n = i*G + g of this (request, KV head) into Q[seg parity], K-major with 128-byte swizzle.
        ++seg;
        const int qb = seg & 1;
        if (seg >= 2 && !mbar_wait(&qempty[qb], ((seg >> 1) - 1) & 1, p.err)) {
          *abort_flag = 1;
          break;
        }
        const int nreal = row_nq_ * G;
        const int qoff = row_qoff;
        const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
        unsigned char *qd = Qs + qb * 2 * L::KATOM;
        // 16-byte pieces idx = lane + 32 u of the [NPMAX x 128] operand, loaded 8 at a time (one round trip)
        // before any is stored
        constexpr int kQPieces = NPMAX * 16 / 32;  // per lane
        for (int u0 = 0; u0 < kQPieces; u0 += 8) {
          uint4 val[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int idx = lane + 32 * (u0 + u);
            const int n = idx >> 4, c = idx & 15;
            const int nc_ = n < nreal ? n : 0;  // clamped row: the load is always issued
            const int i = nc_ / G, g = nc_ - (nc_ / G) * G;
            val[u] = *reinterpret_cast<const uint4 *>(qg + (static_cast<size_t>(qoff + i) * p.hq + pl_h * G + g) * 128 +
                                                      c * 8);
            if (n >= nreal) val[u] = make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int idx = lane + 32 * (u0 + u);
            const int n = idx >> 4, c = idx & 15;
            const int katom = c >> 3, cc = c & 7;
            *reinterpret_cast<uint4 *>(qd + katom * L::KATOM + (n >> 3) * 1024 + (n & 7) * 128 +
                                       ((cc ^ (n & 7)) << 4)) = val[u];
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&qfull[qb]);
      }
      const bool in_tile = lane < pl_npg;
      const bool ok = in_tile && pl_page >= 0 && pl_page < p.num_pages;
      if (in_tile && !ok) set_error(p.err, kErrPage);
      const int nvalid = __popc(__ballot_sync(0xffffffffu, ok));
      if (!kprod) {
        if (lane == 0) mbar_arrive_expect_tx(&vfull[st], nvalid * 2 * 2048);
        __syncwarp();
        if (ok) {
          unsigned char *vd = Vs + st * kStageBytes;
          const int row0 = (pl_page * p.hkv + pl_h) * kPage;
          tma_load_2d_stream(vd + lane * 2048, &tmV, 0, row0, &vfull[st], pol);
          tma_load_2d_stream(vd + kHalfBytes + lane * 2048, &tmV, 64, row0, &vfull[st], pol);
        }
        plan();
        continue;
      }
      if (lane == 0) {
        m.valid = 1;
        m.rb = pl_rb;
        m.re = pl_re;
        m.row = pl_row;
        m.tile = pl_tile;
        m.first = pl_first;
        m.last = pl_last;
        m.npg = pl_npg;
        m.seg = seg;
        m.nq = row_nq_;
        m.qpos0 = row_qpos0;
        m.qoff = row_qoff;
        mbar_arrive(&mfull[mi]);
        mbar_arrive_expect_tx(&kfull[st], nvalid * 2 * 2048);
      }
      __syncwarp();
      if (ok) {
        unsigned char *kd = Ks + st * kStageBytes;
        const int row0 = (pl_page * p.hkv + pl_h) * kPage;
        tma_load_2d_stream(kd + lane * 2048, &tmK, 0, row0, &kfull[st], pol);
        tma_load_2d_stream(kd + kHalfBytes + lane * 2048, &tmK, 64, row0, &kfull[st], pol);
      }
      plan();
    }
    // copies still in flight after an abort are waited for (bounded) before the CTA leaves
    if (*abort_flag && lane == 0)
      for (int u = max(0, t - kStages + 1); u <= t; ++u)
        mbar_wait(kprod ? &kfull[u % kStages] : &vfull[u % kStages], (u / kStages) & 1, nullptr);
  } else if (warp == 5) {
    // ============================================================================================ MMA issuer
    // Issues whichever MMA is ready first: MMA1(t1) as soon as K(t1) has landed and S[t1 parity] is free, MMA2(t2)
    // as soon as P(t2) is written. Issuing MMA2 early frees the K/V stage (kvempty) for the producer sooner.
    if (lane == 0) {
      int seg = -1, t1 = 0, t2 = 0;
      bool done1 = false, okrun = true;
      uint32_t idle = 0;
      while (true) {
        if (*abort_flag) {
          okrun = false;
          break;
        }
        bool progressed = false;
        if (!done1) {
          const int st = t1 % kStages, b = t1 & 1;
          if (mbar_test(&kfull[st], (t1 / kStages) & 1)) {
            const TileMeta m = meta[t1 % kMR];
            if (!m.valid) {
              done1 = true;
              progressed = true;
            } else if ((!m.first || mbar_test(&qfull[(seg + 1) & 1], ((seg + 1) >> 1) & 1)) &&
                       (t1 < 2 || mbar_test(&sfree[b], ((t1 >> 1) - 1) & 1))) {
              if (m.first) ++seg;
              tc_fence_after();
              const int npad = (m.nq * G + 15) & ~15;
              const uint32_t idesc = idesc_bf16(128, npad, 0, 0);
              const uint32_t kb = smem_u32(Ks + st * kStageBytes), qb = smem_u32(Qs + (seg & 1) * 2 * L::KATOM);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = smem_desc(kb + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024, 2);
                const uint64_t bd = smem_desc(qb + (kk >> 2) * L::KATOM + (kk & 3) * 32, 16, 1024, 2);
                umma_bf16(tmem + b * NPMAX, ad, bd, idesc, kk > 0 ? 1u : 0u);
              }
              umma_commit(&sfull[b]);
              umma_commit(&kempty[st]);
              if (m.last) umma_commit(&qempty[seg & 1]);
              ++t1;
              progressed = true;
            }
          }
        }
        if (t2 < t1) {
          const int su = t2 % kStages, b = t2 & 1;
          if (mbar_test(&pfull[b], (t2 >> 1) & 1) && mbar_test(&vfull[su], (t2 / kStages) & 1) &&
              (t2 < 2 || mbar_test(&ofree[b], ((t2 >> 1) - 1) & 1))) {
            tc_fence_after();
            // meta of tile t2 stays valid until this issuer (and the softmax warps) release its ring slot
            const int npad = (meta[t2 % kMR].nq * G + 15) & ~15;
            const uint32_t idesc = idesc_bf16(128, npad, 1, 0);
            const uint32_t vb = smem_u32(Vs + su * kStageBytes), pb = smem_u32(Ps + b * 2 * L::KATOM);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t ad = smem_desc(vb + kk * 2048, kHalfBytes, 1024, 2);
              const uint64_t bd = smem_desc(pb + (kk >> 2) * L::KATOM + (kk & 3) * 32, 16, 1024, 2);
              umma_bf16(tmem + 2 * NPMAX + b * NPMAX, ad, bd, idesc, kk > 0 ? 1u : 0u);
            }
            umma_commit(&ofull[b]);
            umma_commit(&vempty[su]);
            mbar_arrive(&mfree[t2 % kMR]);
            ++t2;
            progressed = true;
          }
        }
        if (done1 && t2 == t1) break;
        if (progressed) {
          idle = 0;
        } else if (++idle > kSpinPolls) {
          set_error(p.err, kErrTimeout);
          okrun = false;
          break;
        }
      }
      if (!okrun) *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp < 4) {
    // ==================================================================================== softmax and merge
    const float scale2 = rsqrtf(128.0f) * kLog2e;
    const float inv_scale2 = 1.0f / scale2;
    constexpr bool kRawLogits = NPMAX >= 48;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float lt[NPMAX];    // softmax role (thread = token): this token's share of each column's sum
    float oreg[NPMAX];  // merge role (thread = head-dim row): running output of each column
#pragma unroll
    for (int n = 0; n < NPMAX; ++n) {
      lt[n] = 0.0f;
      oreg[n] = 0.0f;
    }
    auto merge = [&](int u, int npad_u, bool resc_u) -> bool {
      const int b = u & 1;
      if (!mbar_wait(&ofull[b], (u >> 1) & 1, p.err)) return false;
      tc_fence_after();
      // 16 columns at a time, so that only one chunk of the tile is held in registers beside the running output
#pragma unroll
      for (int c = 0; c < NPMAX / 16; ++c) {
        if (c * 16 < npad_u) {
          float ot[16];
          tmem_ld16(tmem + 2 * NPMAX + b * NPMAX + lane_base + c * 16, ot);
          tmem_wait_ld();
          if (resc_u) {
#pragma unroll
            for (int e = 0; e < 16; ++e) oreg[c * 16 + e] = fmaf(oreg[c * 16 + e], alpha_s[b * NPMAX + c * 16 + e], ot[e]);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) oreg[c * 16 + e] += ot[e];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ofree[b]);
      return true;
    };
    // Last arriver of a row: merges the partial records of CTAs b_first..b_last and writes the row's output.
    // Thread t owns 16 consecutive head dims of one query column (8 threads per column, 16 columns at a time); for
    // every chunk of kMergeChunkV contributors it issues all its loads (four 16-byte pieces of the partial output
    // per contributor, and one contributor's (m, l) pair) before using any, so a chunk costs one round trip and no
    // barrier. Wide tiles take fewer contributors per chunk: their running state already holds most of the
    // registers.
    constexpr int kMergeChunkV = NPMAX <= 16 ? 8 : 4;
    auto merge_row = [&](int row, int b_first, int b_last, int qoff, int nreal) {
      const int h = row - (row / p.hkv) * p.hkv;
      __nv_bfloat16 *outp = static_cast<__nv_bfloat16 *>(p.out);
      const int nc = b_last - b_first + 1;
      const int d0 = (tid & 7) * 16;
      for (int n0 = 0; n0 < nreal; n0 += 16) {
        const int n = n0 + (tid >> 3);
        const int nn = n < nreal ? n : n0;  // clamped column: every load below is issued
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
        float M = -INFINITY, Ls = 0.0f;
        // the 8 threads of a column form each contributor's weight once (thread c for contributor c) and read the
        // weights by shuffle within their group of 8
        const int sub = tid & 7;
        for (int b0 = 0; b0 < nc; b0 += kMergeChunkV) {
          float4 pv[kMergeChunkV][4];
#pragma unroll
          for (int c = 0; c < kMergeChunkV; ++c) {
            const size_t sl = static_cast<size_t>(b_first + min(b0 + c, nc - 1) + row);
            const float4 *pp = reinterpret_cast<const float4 *>(p.part + (sl * p.npad_ws + nn) * 128 + d0);
#pragma unroll
            for (int q = 0; q < 4; ++q) pv[c][q] = __ldcg(pp + q);
          }
          const bool mine = sub < kMergeChunkV && b0 + sub < nc;
          const size_t slc = static_cast<size_t>(b_first + min(b0 + min(sub, kMergeChunkV - 1), nc - 1) + row);
          float2 mlc = __ldcg(reinterpret_cast<const float2 *>(p.ml) + slc * p.npad_ws + nn);
          if (!mine) mlc = make_float2(-INFINITY, 0.0f);
          float Mc = mlc.x;
#pragma unroll
          for (int o = 4; o >= 1; o >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, o, 8));
          Mc = fmaxf(Mc, M);
          // with no finite maximum yet everything stays zero: the weights are 0 and rs is 0
          const float rs = (M == -INFINITY) ? 0.0f : exp2f(M - Mc);
          const float wc = (mlc.x == -INFINITY) ? 0.0f : exp2f(mlc.x - Mc);
          float lw = mlc.y * wc;
#pragma unroll
          for (int o = 4; o >= 1; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o, 8);
          Ls = fmaf(Ls, rs, lw);
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[e] *= rs;
#pragma unroll
          for (int c = 0; c < kMergeChunkV; ++c) {
            const float w = __shfl_sync(0xffffffffu, wc, c, 8);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[4 * q] = fmaf(pv[c][q].x, w, acc[4 * q]);
              acc[4 * q + 1] = fmaf(pv[c][q].y, w, acc[4 * q + 1]);
              acc[4 * q + 2] = fmaf(pv[c][q].z, w, acc[4 * q + 2]);
              acc[4 * q + 3] = fmaf(pv[c][q].w, w, acc[4 * q + 3]);
            }
          }
          M = Mc;
        }
        if (n < nreal) {
          const int i = n / G, g = n - (n / G) * G;
          const float inv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
          uint32_t wd[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
            wd[e] = *reinterpret_cast<const uint32_t *>(&b2);
          }
          uint4 *dst = reinterpret_cast<uint4 *>(outp + (static_cast<size_t>(qoff + i) * p.hq + h * G + g) * 128 + d0);
          dst[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
          dst[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
          if ((tid & 7) == 0)
            p.lse[static_cast<size_t>(qoff + i) * p.hq + h * G + g] = Ls > 0.0f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
        }
      }
    };
    // Counts the noted row segments in: one thread's acquire-release atomic per row publishes this CTA's records
    // (ordered before it by the group barrier) and, for the row's last arriver, makes the others' records visible.
    auto flush_deferred = [&]() {
      named_sync_128();
      const int nd = s_ndef;
      if (tid == 0)
        for (int d = 0; d < nd; ++d) {
          const int4 e = s_def[d];
          const int old = atom_add_acq_rel_gpu(&p.counters[e.x], 1);
          const int last = (old == e.z - e.y) ? 1 : 0;
          if (last) p.counters[e.x] = 0;  // every contributor has arrived: leave the counter at zero
          s_deflast[d] = last;
        }
      named_sync_128();
      for (int d = 0; d < nd; ++d)
        if (s_deflast[d]) {
          const int4 e = s_def[d];
          merge_row(e.x, e.y, e.z, e.w, s_defn[d]);
        }
      named_sync_128();
      if (tid == 0) s_ndef = 0;
      named_sync_128();
    };
    int pending = -1, pending_npad = 16;  // tile whose O is not merged yet
    bool pending_resc = false;
    bool okrun = true;
    for (int t = 0;; ++t) {
      const int st = t % kStages, b = t & 1;
      if (*abort_flag || !mbar_wait(&mfull[t % kMR], (t / kMR) & 1, p.err)) {
        okrun = false;
        break;
      }
      const TileMeta m = meta[t % kMR];
      if (!m.valid) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&mfree[t % kMR]);
      const int r = m.row / p.hkv, h = m.row - r * p.hkv;
      const int nq = m.nq;
      const int nreal = nq * G;
      const int npad = (nreal + 15) & ~15;
      const int qpos0 = m.qpos0;
      const int qoff = m.qoff;
      if (m.first) {
        if (tid < NPMAX) {
          m_run[tid] = -INFINITY;
          m_sub[tid] = 0.0f;
          thr[tid] = -INFINITY;
          lsum[tid] = 0.0f;
        }
#pragma unroll
        for (int n = 0; n < NPMAX; ++n) {
          lt[n] = 0.0f;
          oreg[n] = 0.0f;
        }
        named_sync_128();
      }
      // ---- S tile from TMEM (thread = token)
      if (!mbar_wait(&sfull[b], (t >> 1) & 1, p.err)) {
        okrun = false;
        break;
      }
      tc_fence_after();
      float x[NPMAX];
#pragma unroll
      for (int c = 0; c < NPMAX / 16; ++c)
        if (c * 16 < npad) {
          tmem_ld16(tmem + b * NPMAX + lane_base + c * 16, x + c * 16);
        } else {  // columns past this row's padded width: no logits, weight 0
#pragma unroll
          for (int e = 0; e < 16; ++e) x[c * 16 + e] = -INFINITY;
        }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[b]);
      const int pos = m.tile * kTileTok + tid;
      // the running maxima are read from shared memory 16 columns at a time (not all held in registers beside x,
      // lt and oreg)
      bool over = false;
      // column n is window row n / G: visible when this token's position is at most qpos0 + n / G
      const int rel = pos - qpos0;  // the token is visible to window rows i >= rel
      const int n_first = rel <= 0 ? 0 : rel * G;
      // Columns past nreal (padding) need no mask: their query rows are zero and their outputs are never written.
      // Only a tile that reaches the window has masked entries; a warp without any scales its logits only.
      if (kRawLogits) {
        // Wide tiles keep the logits unscaled: the scale enters the max test through each column's threshold and
        // the exponent through one fused multiply-add (two instructions fewer per logit on the softmax path that
        // bounds them). Narrow tiles measured faster with the scaled form below.
        if (!__all_sync(0xffffffffu, n_first == 0)) {
#pragma unroll
          for (int n = 0; n < NPMAX; ++n)
            if (n < n_first) x[n] = -INFINITY;
        }
#pragma unroll
        for (int c = 0; c < NPMAX / 16; ++c) {
          float th[16];
          load16_shared(thr + c * 16, th);
#pragma unroll
          for (int e = 0; e < 16; ++e) over |= x[c * 16 + e] > th[e];
        }
      } else {
        if (__all_sync(0xffffffffu, n_first == 0)) {
#pragma unroll
          for (int n = 0; n < NPMAX; ++n) x[n] *= scale2;
        } else {
#pragma unroll
          for (int n = 0; n < NPMAX; ++n) x[n] = (n >= n_first) ? x[n] * scale2 : -INFINITY;
        }
#pragma unroll
        for (int c = 0; c < NPMAX / 16; ++c) {
          float mr[16];
          load16_shared(m_run + c * 16, mr);
#pragma unroll
          for (int e = 0; e < 16; ++e) over |= x[c * 16 + e] > mr[e] + kRescaleThreshold;
        }
      }
      // ---- running max: only when some logit of this tile exceeds it by more than 2^8
      const bool rescale = named_or_128(over);
      if (rescale) {
#pragma unroll
        for (int n = 0; n < NPMAX; ++n) {
          const int wmax = __reduce_max_sync(0xffffffffu, fkey(x[n]));
          if (lane == 0) colmax[warp * NPMAX + n] = ffrom(wmax);
        }
        named_sync_128();
        if (tid < NPMAX) {
          // the column's largest scaled logit (scaling by a positive factor keeps the order and the maximum)
          const float cm = fmaxf(fmaxf(colmax[tid], colmax[NPMAX + tid]),
                                 fmaxf(colmax[2 * NPMAX + tid], colmax[3 * NPMAX + tid])) *
                           (kRawLogits ? scale2 : 1.0f);
          const float mo = m_run[tid];
          const float mn = fmaxf(mo, cm);
          alpha_s[b * NPMAX + tid] = (mn == -INFINITY) ? 1.0f : exp2f(mo - mn);
          m_run[tid] = mn;
          m_sub[tid] = (mn == -INFINITY) ? 0.0f : mn;
          thr[tid] = (mn == -INFINITY) ? -INFINITY : (mn + kRescaleThreshold) * inv_scale2;
        }
        named_sync_128();
        // this thread's running sums follow the raised maxima (the tile's weights are added below)
#pragma unroll
        for (int cc = 0; cc < NPMAX / 16; ++cc) {
          float al[16];
          load16_shared(alpha_s + b * NPMAX + cc * 16, al);
#pragma unroll
          for (int ee = 0; ee < 16; ++ee) lt[cc * 16 + ee] *= al[ee];
        }
      }
      // ---- P = exp2(x - m_run) as bf16, K-major with 128-byte swizzle (row n, column = token); a masked logit
      // (-inf) gives 0 since m_sub is finite
      {
        unsigned char *pd = Ps + b * 2 * L::KATOM;
        const int katom = tid >> 6, c = (tid & 63) >> 3, e = tid & 7;
#pragma unroll
        for (int cc = 0; cc < NPMAX / 16; ++cc) {
          float mr[16];
          load16_shared(m_sub + cc * 16, mr);
#pragma unroll
          for (int ee = 0; ee < 16; ++ee) {
            const int n = cc * 16 + ee;
            const float pv = kRawLogits ? fast_exp2(fmaf(x[n], scale2, -mr[ee])) : fast_exp2(x[n] - mr[ee]);
            lt[n] += pv;
            *reinterpret_cast<__nv_bfloat16 *>(pd + katom * L::KATOM + (n >> 3) * 1024 + (n & 7) * 128 +
                                              ((c ^ (n & 7)) << 4) + e * 2) = __float2bfloat16_rn(pv);
          }
        }
      }
      // tokens past the last query position carry no weight; their V rows may hold anything (even NaN) and must
      // not reach the tensor core: zero them
      if (pos > qpos0 + nq - 1) {
        if (!mbar_wait(&vfull[st], (t / kStages) & 1, p.err)) okrun = false;
        unsigned char *vrow0 = Vs + st * kStageBytes + (tid >> 4) * 2048 + (tid & 15) * 128;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4 *>(vrow0 + hh * kHalfBytes + c * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[b]);
      // ---- merge the previous tile's O (its MMA2 overlapped this softmax)
      if (pending >= 0) {
        if (!merge(pending, pending_npad, pending_resc)) {
          okrun = false;
          break;
        }
        pending = -1;
      }
      pending = t;
      pending_npad = npad;
      pending_resc = rescale;
      if (!m.last) continue;

      // ---- end of this row segment: drain, column sums, then finish or hand over a partial record
      if (!merge(pending, pending_npad, pending_resc)) {
        okrun = false;
        break;
      }
      pending = -1;
#pragma unroll
      for (int n = 0; n < NPMAX; ++n) {
        if (n < npad) {
          const float v = warp_sum(lt[n]);
          if (lane == 0) atomicAdd(&lsum[n], v);
        }
      }
      named_sync_128();
      const int b_first = owner_cta(m.rb, E, nb), b_last = owner_cta(m.re - 1, E, nb);
      const int ncontrib = b_last - b_first + 1;
      __nv_bfloat16 *outp = static_cast<__nv_bfloat16 *>(p.out);
      if (ncontrib == 1) {
#pragma unroll
        for (int n = 0; n < NPMAX; ++n) {
          if (n < nreal) {
            const int i = n / G, g = n - (n / G) * G;
            const float l = lsum[n];
            outp[(static_cast<size_t>(qoff + i) * p.hq + h * G + g) * 128 + tid] =
                __float2bfloat16_rn(l > 0.0f ? oreg[n] / l : 0.0f);
          }
        }
        if (tid < nreal) {
          const int i = tid / G, g = tid - (tid / G) * G;
          const float l = lsum[tid];
          p.lse[static_cast<size_t>(qoff + i) * p.hq + h * G + g] =
              l > 0.0f ? (m_run[tid] + log2f(l)) * kLn2 : -INFINITY;
        }
      } else {
        // Partial record of this row segment. The row is counted in (and merged, by its last arriver) only once
        // this CTA's tiles are done, so the pipeline never waits here on other CTAs' progress.
        const int slot = static_cast<int>(blockIdx.x) + m.row;
        float *pp = p.part + static_cast<size_t>(slot) * p.npad_ws * 128;
#pragma unroll
        for (int n = 0; n < NPMAX; ++n)
          if (n < npad) __stcg(pp + n * 128 + tid, oreg[n]);
        if (tid < npad)
          __stcg(reinterpret_cast<float2 *>(p.ml) + static_cast<size_t>(slot) * p.npad_ws + tid,
                 make_float2(m_run[tid], lsum[tid]));
        if (tid == 0) {
          s_def[s_ndef] = make_int4(m.row, b_first, b_last, qoff);
          s_defn[s_ndef] = nreal;
          ++s_ndef;
        }
        named_sync_128();
        if (s_ndef == kMaxDeferred) flush_deferred();
      }
      named_sync_128();
    }
    // every softmax thread gets here; the hand-offs run only when none of them gave up on a wait
    if (!named_or_128(!okrun)) flush_deferred();
    if (!okrun) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

// ================================================================================================ FFMA path
// One warp per (query row, query head); online softmax over every visible position, in fp32.
template <class T, int D>
__global__ void __launch_bounds__(256) verify_ffma_kernel(const T *__restrict__ K, const T *__restrict__ V,
                                                          const VParams p, int total_q) {
  grid_dependency_sync();
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= static_cast<int64_t>(total_q) * p.hq) return;
  const int row = static_cast<int>(wid / p.hq), hq = static_cast<int>(wid - static_cast<int64_t>(row) * p.hq);
  int lo = 0, hi = p.R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.q_offsets[mid] <= row) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  const int G = p.hq / p.hkv, h = hq / G;
  const int P = p.q_start[r] + (row - p.q_offsets[r]);
  constexpr int PL = D / 32;
  float qv[PL], ov[PL];
  const T *qrow = static_cast<const T *>(p.q) + (static_cast<size_t>(row) * p.hq + hq) * D;
  const float sc = rsqrtf(static_cast<float>(D)) * kLog2e;
#pragma unroll
  for (int k = 0; k < PL; ++k) {
    qv[k] = to_f(qrow[lane + 32 * k]) * sc;
    ov[k] = 0.0f;
  }
  float mx = -INFINITY, l = 0.0f;
  const int32_t *btr = p.bt + static_cast<size_t>(r) * p.max_pages;
  for (int pos = 0; pos <= P; ++pos) {
    if (pos / kPage >= p.max_pages) {
      if (lane == 0) set_error(p.err, kErrPage);
      break;
    }
    const int pg = btr[pos / kPage];
    if (pg < 0 || pg >= p.num_pages) {
      if (lane == 0) set_error(p.err, kErrPage);
      continue;
    }
    const size_t o = ((static_cast<size_t>(pg) * p.hkv + h) * kPage + pos % kPage) * D;
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < PL; ++k) s = fmaf(qv[k], to_f(K[o + lane + 32 * k]), s);
    s = warp_sum(s);
    const float mn = fmaxf(mx, s);
    const float a = exp2f(mx - mn), w = exp2f(s - mn);
    l = l * a + w;
#pragma unroll
    for (int k = 0; k < PL; ++k) ov[k] = ov[k] * a + w * to_f(V[o + lane + 32 * k]);
    mx = mn;
  }
  T *op = static_cast<T *>(p.out) + (static_cast<size_t>(row) * p.hq + hq) * D;
#pragma unroll
  for (int k = 0; k < PL; ++k) op[lane + 32 * k] = from_f<T>(l > 0.0f ? ov[k] / l : 0.0f);
  if (lane == 0) p.lse[static_cast<size_t>(row) * p.hq + hq] = l > 0.0f ? (mx + log2f(l)) * kLn2 : -INFINITY;
}

// ============================================================================================== host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D view [num_pages * Hkv * 16 rows][128 columns] of a bf16 pool; boxes of 64 columns x 16 rows, 128B swizzle.
bool make_pool_map(CUtensorMap *map, const void *base, int num_pages, int hkv) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(num_pages) * hkv * kPage};
  cuuint64_t strides[1] = {128 * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t estr[2] = {1, 1};
  CUresult rc = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

template <int NPMAX>
cudaError_t launch_tc(const PoolArgs &pa, const VParams &prm, cudaStream_t s) {
  using L = TcSmem<NPMAX>;
  static_assert(L::ALLOC <= 227 * 1024, "shared memory over the per-CTA limit");
  CUtensorMap tmK, tmV;
  if (!make_pool_map(&tmK, pa.k, pa.num_pages, pa.hkv) || !make_pool_map(&tmV, pa.v, pa.num_pages, pa.hkv))
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(verify_tc_kernel<NPMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::ALLOC);
    if (e != cudaSuccess) return e;
    attr_set[dev & 63] = true;
  }
  const int nb = device_sm_count();
  launch_pdl(verify_tc_kernel<NPMAX>, dim3(nb), dim3(kTcThreads), L::ALLOC, s, tmK, tmV, prm);
  return cudaGetLastError();
}

}  // namespace

int verify_npad(int hq, int hkv, int max_q) {
  const int n = (hq / hkv) * max_q;
  return (n + 15) & ~15;
}

size_t verify_workspace_bytes(int R, int hkv, int hq, int d, int max_q) {
  const size_t nrows = static_cast<size_t>(R) * hkv;
  const size_t np = static_cast<size_t>(verify_npad(hq, hkv, max_q));
  const size_t slots = nrows + kMaxCtas;
  size_t b = ((nrows * 4 + 255) / 256) * 256;
  b += ((slots * np * 2 * 4 + 255) / 256) * 256;
  b += slots * np * d * 4;
  return b;
}

cudaError_t launch_verify(const PoolArgs &pa, const MapArgs &ma, int max_q, int total_q, const int32_t *q_offsets,
                          const int32_t *q_start, const void *q, void *out, float *lse, void *ws, size_t ws_bytes,
                          int *err, cudaStream_t s) {
  (void)ws_bytes;
  VParams prm;
  prm.num_pages = pa.num_pages;
  prm.hkv = pa.hkv;
  prm.hq = pa.hq;
  prm.bt = ma.bt;
  prm.max_pages = ma.max_pages;
  prm.q_offsets = q_offsets;
  prm.q_start = q_start;
  prm.R = ma.R;
  prm.nrows = ma.R * pa.hkv;
  prm.q = q;
  prm.out = out;
  prm.lse = lse;
  prm.err = err;
  const int npad = verify_npad(pa.hq, pa.hkv, max_q);
  prm.npad_ws = npad;
  const size_t nrows = static_cast<size_t>(prm.nrows);
  const size_t slots = nrows + kMaxCtas;
  unsigned char *w = static_cast<unsigned char *>(ws);
  prm.counters = reinterpret_cast<int *>(w);
  w += ((nrows * 4 + 255) / 256) * 256;
  prm.ml = reinterpret_cast<float *>(w);
  w += ((slots * npad * 2 * 4 + 255) / 256) * 256;
  prm.part = reinterpret_cast<float *>(w);
  if (total_q <= 0) return cudaSuccess;
  if (pa.dtype == 0 && pa.d == 128) {
    if (npad <= 16) return launch_tc<16>(pa, prm, s);
    if (npad <= 32) return launch_tc<32>(pa, prm, s);
    if (npad <= 48) return launch_tc<48>(pa, prm, s);
    return launch_tc<64>(pa, prm, s);
  }
  const int64_t warps = static_cast<int64_t>(total_q) * pa.hq;
  const int blocks = static_cast<int>((warps + 7) / 8);
  if (pa.dtype == 0)
    launch_pdl(verify_ffma_kernel<__nv_bfloat16, 64>, dim3(blocks), dim3(256), 0, s,
               static_cast<const __nv_bfloat16 *>(pa.k), static_cast<const __nv_bfloat16 *>(pa.v), prm, total_q);
  else if (pa.d == 128)
    launch_pdl(verify_ffma_kernel<float, 128>, dim3(blocks), dim3(256), 0, s, static_cast<const float *>(pa.k),
               static_cast<const float *>(pa.v), prm, total_q);
  else
    launch_pdl(verify_ffma_kernel<float, 64>, dim3(blocks), dim3(256), 0, s, static_cast<const float *>(pa.k),
               static_cast<const float *>(pa.v), prm, total_q);
  return cudaGetLastError();
}

}  // namespace kap
