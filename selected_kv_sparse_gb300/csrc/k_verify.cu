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
__device__ __forceinline__ int owner_cta(int64_t x, int64_t E, int nb) {
  return static_cast<int>(((x + 1) * nb - 1) / E);
}
__device__ __forceinline__ int fkey(float x) {
  const int b = __float_as_int(x);
  return b >= 0 ? b : (b ^ 0x7fffffff);
}
__device__ __forceinline__ float ffrom(int k) { return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff)); }

// ============================================================================================ tensor cores
constexpr int kTileTok = 128;
constexpr int kHalfBytes = 8 * kPage * 128;  // one 64-column half of a tile: 8 pages x 16 rows x 128 B = 16 KiB
constexpr int kStageBytes = 2 * kHalfBytes;   // 32 KiB of K (or V) per stage

struct TileMeta {
  int64_t rb, re;
  int valid, row, tile, first, last, npg, seq;
};

template <int NPMAX>
struct TcSmem {
  static constexpr int kStages = NPMAX <= 48 ? 3 : 2;  // stay under 227 KB of shared memory
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + kStages * kStageBytes;
  static constexpr int OFF_Q = OFF_V + kStages * kStageBytes;
  static constexpr int KATOM = NPMAX * 128;  // bytes of one 64-column K-atom of an [NPMAX x 128] operand
  static constexpr int OFF_P = OFF_Q + 2 * KATOM;
  static constexpr int OFF_CM = OFF_P + 2 * KATOM;       // column maxima [4][NPMAX]
  static constexpr int OFF_ST = OFF_CM + 4 * NPMAX * 4;  // m_run, m_new, alpha, lsum [4][NPMAX]
  static constexpr int OFF_BAR = OFF_ST + 4 * NPMAX * 4;
  static constexpr int OFF_META = OFF_BAR + (2 * kStages + 2) * 8;
  static constexpr int OFF_TMEM = OFF_META + kStages * static_cast<int>(sizeof(TileMeta));
  static constexpr int BYTES = OFF_TMEM + 16;
  static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 bytes
  static constexpr int TMEM_COLS = (2 * NPMAX <= 32) ? 32 : (2 * NPMAX <= 64 ? 64 : 128);
};

template <int NPMAX>
__global__ void __launch_bounds__(128, 1)
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
  float *m_new = m_run + NPMAX;
  float *alpha = m_new + NPMAX;
  float *lsum = alpha + NPMAX;
  uint64_t *barK = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
  uint64_t *barV = barK + kStages;
  uint64_t *bar_s = barV + kStages;
  uint64_t *bar_o = bar_s + 1;
  TileMeta *meta = reinterpret_cast<TileMeta *>(sm + L::OFF_META);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::OFF_TMEM);
  __shared__ int64_t s_total;
  __shared__ int s_flag, s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.hq / p.hkv;
  if (tid == 0) s_abort = 0;

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
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&barK[i], 1);
      mbar_init(&barV[i], 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_barrier_init();
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  __syncthreads();
  const int64_t E = s_total;
  // Split over nb <= E CTAs so that every participating CTA owns at least one tile (the merge counts them).
  const int nb = static_cast<int>(E < static_cast<int64_t>(gridDim.x) ? E : static_cast<int64_t>(gridDim.x));
  if (E == 0 || static_cast<int>(blockIdx.x) >= nb) return;
  const int64_t cta_begin = static_cast<int64_t>(blockIdx.x) * E / nb;
  const int64_t cta_end = static_cast<int64_t>(blockIdx.x + 1) * E / nb;

  if (warp == 0) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_S = tmem;
  const uint32_t tmem_O = tmem + NPMAX;

  // producer state (thread 0)
  int pr_row = 0, pr_seq = 0;
  int64_t pr_rb = 0, pr_re = 0, pr_cur = cta_begin;
  if (tid == 0) {
    pr_re = row_tiles(p, 0);
    while (pr_re <= cta_begin) {
      ++pr_row;
      pr_rb = pr_re;
      pr_re += row_tiles(p, pr_row);
    }
  }
  auto issue = [&](int st) {
    TileMeta &m = meta[st];
    if (pr_cur >= cta_end) {
      m.valid = 0;
      return;
    }
    while (pr_cur >= pr_re) {
      ++pr_row;
      pr_rb = pr_re;
      pr_re += row_tiles(p, pr_row);
    }
    const int64_t seg_end = min(pr_re, cta_end);
    const int r = pr_row / p.hkv, h = pr_row - r * p.hkv;
    const int tile = static_cast<int>(pr_cur - pr_rb);
    const int kv_pages = (p.q_start[r] + row_nq(p, r) + kPage - 1) / kPage;
    const int npg = min(8, kv_pages - tile * 8);
    m.valid = 1;
    m.rb = pr_rb;
    m.re = pr_re;
    m.row = pr_row;
    m.tile = tile;
    m.first = (pr_cur == pr_rb || pr_cur == cta_begin) ? 1 : 0;
    m.last = (pr_cur + 1 == seg_end) ? 1 : 0;
    m.npg = npg;
    m.seq = pr_seq++;
    int pages[8];
    int nvalid = 0;
    const int32_t *btr = p.bt + static_cast<size_t>(r) * p.max_pages;
    for (int i = 0; i < 8; ++i) {
      pages[i] = -1;
      if (i < npg && tile * 8 + i < p.max_pages) {
        const int pg = btr[tile * 8 + i];
        if (pg >= 0 && pg < p.num_pages) {
          pages[i] = pg;
          ++nvalid;
        } else {
          set_error(p.err, kErrPage);
        }
      }
    }
    mbar_arrive_expect_tx(&barK[st], nvalid * 2 * 2048);
    mbar_arrive_expect_tx(&barV[st], nvalid * 2 * 2048);
    unsigned char *kd = Ks + st * kStageBytes;
    unsigned char *vd = Vs + st * kStageBytes;
    for (int i = 0; i < 8; ++i) {
      if (pages[i] < 0) continue;
      const int row0 = (pages[i] * p.hkv + h) * kPage;
      tma_load_2d(kd + i * 2048, &tmK, 0, row0, &barK[st]);
      tma_load_2d(kd + kHalfBytes + i * 2048, &tmK, 64, row0, &barK[st]);
      tma_load_2d(vd + i * 2048, &tmV, 0, row0, &barV[st]);
      tma_load_2d(vd + kHalfBytes + i * 2048, &tmV, 64, row0, &barV[st]);
    }
    ++pr_cur;
  };
  if (tid == 0)
    for (int st = 0; st < kStages; ++st) issue(st);
  __syncthreads();

  const float scale2 = rsqrtf(128.0f) * kLog2e;
  float lt[NPMAX];  // softmax role (thread = token): this token's share of each column's sum
  float oreg[NPMAX];  // merge role (thread = head-dim row): running output of each column
#pragma unroll
  for (int n = 0; n < NPMAX; ++n) {
    lt[n] = 0.0f;
    oreg[n] = 0.0f;
  }
  bool abort = false;
  int t_end = 0;

  for (int t = 0;; ++t) {
    t_end = t;
    const int st = t % kStages;
    const uint32_t ph = (t / kStages) & 1;
    const TileMeta m = meta[st];
    if (!m.valid) break;
    const int r = m.row / p.hkv, h = m.row - r * p.hkv;
    const int nq = row_nq(p, r);
    const int nreal = nq * G;
    const int npad = (nreal + 15) & ~15;
    const int qpos0 = p.q_start[r];
    const int qoff = p.q_offsets[r];
    if (m.first) {
      // Q rows n = i*G + g of this (request, KV head), K-major with 128-byte swizzle; zero padding rows.
      const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
      for (int idx = tid; idx < NPMAX * 16; idx += 128) {
        const int n = idx >> 4, c = idx & 15;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (n < nreal) {
          const int i = n / G, g = n - (n / G) * G;
          val = *reinterpret_cast<const uint4 *>(qg + (static_cast<size_t>(qoff + i) * p.hq + h * G + g) * 128 + c * 8);
        }
        const int katom = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4 *>(Qs + katom * L::KATOM + (n >> 3) * 1024 + (n & 7) * 128 + ((cc ^ (n & 7)) << 4)) = val;
      }
      fence_proxy_async_smem();
      if (tid < NPMAX) {
        m_run[tid] = -INFINITY;
        lsum[tid] = 0.0f;
      }
#pragma unroll
      for (int n = 0; n < NPMAX; ++n) {
        lt[n] = 0.0f;
        oreg[n] = 0.0f;
      }
    }
    __syncthreads();
    // ---- S^T = K . Q^T
    if (tid == 0) {
      if (!mbar_wait(&barK[st], ph, p.err)) abort = true;
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, npad, 0, 0);
      const uint32_t kb = smem_u32(Ks + st * kStageBytes), qb = smem_u32(Qs);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ad = smem_desc(kb + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024, 2);
        const uint64_t bd = smem_desc(qb + (kk >> 2) * L::KATOM + (kk & 3) * 32, 16, 1024, 2);
        umma_bf16(tmem_S, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      umma_commit(bar_s);
    }
    if (!mbar_wait(bar_s, t & 1, p.err)) abort = true;
    tc_fence_after();
    // ---- softmax over the tile's tokens (thread = token)
    const int pos = m.tile * kTileTok + tid;
    float x[NPMAX];
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
    for (int c = 0; c < NPMAX / 16; ++c)
      if (c * 16 < npad) tmem_ld16(tmem_S + lane_base + c * 16, x + c * 16);
    tmem_wait_ld();
    tc_fence_before();
#pragma unroll
    for (int n = 0; n < NPMAX; ++n) {
      const int i = n / G;
      const bool vis = n < nreal && pos <= qpos0 + i;
      x[n] = vis ? x[n] * scale2 : -INFINITY;
      const int wmax = __reduce_max_sync(0xffffffffu, fkey(x[n]));
      if (lane == 0) colmax[warp * NPMAX + n] = ffrom(wmax);
    }
    __syncthreads();
    if (tid < NPMAX) {
      const float cm = fmaxf(fmaxf(colmax[tid], colmax[NPMAX + tid]), fmaxf(colmax[2 * NPMAX + tid], colmax[3 * NPMAX + tid]));
      const float mo = m_run[tid];
      const float mn = fmaxf(mo, cm);
      alpha[tid] = (mn == -INFINITY) ? 1.0f : exp2f(mo - mn);
      m_new[tid] = mn;
      m_run[tid] = mn;
    }
    __syncthreads();
    {
      const int katom = tid >> 6, c = (tid & 63) >> 3, e = tid & 7;
#pragma unroll
      for (int n = 0; n < NPMAX; ++n) {
        const float pv = (x[n] == -INFINITY) ? 0.0f : exp2f(x[n] - m_new[n]);
        lt[n] = lt[n] * alpha[n] + pv;
        *reinterpret_cast<__nv_bfloat16 *>(Ps + katom * L::KATOM + (n >> 3) * 1024 + (n & 7) * 128 +
                                          ((c ^ (n & 7)) << 4) + e * 2) = __float2bfloat16_rn(pv);
      }
    }
    // tokens past the last query position carry no weight; their V rows may hold anything (even NaN) and
    // must not reach the tensor core: zero them
    if (pos > qpos0 + nq - 1) {
      if (!mbar_wait(&barV[st], ph, p.err)) abort = true;
      unsigned char *vrow0 = Vs + st * kStageBytes + (tid >> 4) * 2048 + (tid & 15) * 128;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4 *>(vrow0 + hh * kHalfBytes + c * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncthreads();
    // ---- O^T = V^T . P^T
    if (tid == 0) {
      if (!mbar_wait(&barV[st], ph, p.err)) abort = true;
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, npad, 1, 0);
      const uint32_t vb = smem_u32(Vs + st * kStageBytes), pb = smem_u32(Ps);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t ad = smem_desc(vb + kk * 2048, kHalfBytes, 1024, 2);
        const uint64_t bd = smem_desc(pb + (kk >> 2) * L::KATOM + (kk & 3) * 32, 16, 1024, 2);
        umma_bf16(tmem_O, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      umma_commit(bar_o);
    }
    if (!mbar_wait(bar_o, t & 1, p.err)) abort = true;
    tc_fence_after();
    {
      float ot[NPMAX];
#pragma unroll
      for (int c = 0; c < NPMAX / 16; ++c)
        if (c * 16 < npad) tmem_ld16(tmem_O + lane_base + c * 16, ot + c * 16);
      tmem_wait_ld();
      tc_fence_before();
#pragma unroll
      for (int n = 0; n < NPMAX; ++n)
        if (n < npad) oreg[n] = oreg[n] * alpha[n] + ot[n];
    }
    if (abort) s_abort = 1;
    __syncthreads();
    if (s_abort) {
      t_end = t + 1;
      break;
    }
    if (tid == 0) issue(st);  // tile t + kStages into this stage
    if (!m.last) continue;

    // ---- end of this row segment: column sums, then finish or hand over a partial record
#pragma unroll
    for (int n = 0; n < NPMAX; ++n) {
      if (n < npad) {
        const float v = warp_sum(lt[n]);
        if (lane == 0) atomicAdd(&lsum[n], v);
      }
    }
    __syncthreads();
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
        p.lse[static_cast<size_t>(qoff + i) * p.hq + h * G + g] = l > 0.0f ? (m_run[tid] + log2f(l)) * kLn2 : -INFINITY;
      }
    } else {
      const int slot = static_cast<int>(blockIdx.x) + m.row;
      float *pp = p.part + static_cast<size_t>(slot) * p.npad_ws * 128;
#pragma unroll
      for (int n = 0; n < NPMAX; ++n)
        if (n < npad) __stcg(pp + n * 128 + tid, oreg[n]);
      if (tid < npad) {
        __stcg(p.ml + (static_cast<size_t>(slot) * p.npad_ws + tid) * 2, m_run[tid]);
        __stcg(p.ml + (static_cast<size_t>(slot) * p.npad_ws + tid) * 2 + 1, lsum[tid]);
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int old = atomicAdd(&p.counters[m.row], 1);
        s_flag = (old == ncontrib - 1) ? 1 : 0;
        if (s_flag) p.counters[m.row] = 0;
      }
      __syncthreads();
      if (s_flag) {
        __threadfence();
        for (int n = 0; n < nreal; ++n) {
          float M = -INFINITY;
          for (int b = b_first; b <= b_last; ++b)
            M = fmaxf(M, __ldcg(p.ml + (static_cast<size_t>(b + m.row) * p.npad_ws + n) * 2));
          float Ls = 0.0f, acc = 0.0f;
          if (M != -INFINITY) {
            for (int b = b_first; b <= b_last; ++b) {
              const size_t s2 = static_cast<size_t>(b + m.row);
              const float mb = __ldcg(p.ml + (s2 * p.npad_ws + n) * 2);
              const float lb = __ldcg(p.ml + (s2 * p.npad_ws + n) * 2 + 1);
              const float w = (mb == -INFINITY) ? 0.0f : exp2f(mb - M);
              Ls += lb * w;
              acc += __ldcg(p.part + (s2 * p.npad_ws + n) * 128 + tid) * w;
            }
          }
          const int i = n / G, g = n - (n / G) * G;
          outp[(static_cast<size_t>(qoff + i) * p.hq + h * G + g) * 128 + tid] =
              __float2bfloat16_rn(Ls > 0.0f ? acc / Ls : 0.0f);
          if (tid == 0)
            p.lse[static_cast<size_t>(qoff + i) * p.hq + h * G + g] = Ls > 0.0f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
        }
      }
    }
    __syncthreads();
  }

  // After a bounded wait ran out, the copies still in flight (tiles issued but not consumed) are waited for,
  // again with a bound, before the CTA leaves.
  if (tid == 0 && s_abort) {
    for (int st = 0; st < kStages; ++st) {
      const TileMeta &mm = meta[st];
      if (!mm.valid || mm.seq < t_end) continue;
      const uint32_t ph = (mm.seq / kStages) & 1;
      mbar_wait(&barK[st], ph, nullptr);
      mbar_wait(&barV[st], ph, nullptr);
    }
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
  verify_tc_kernel<NPMAX><<<nb, 128, L::ALLOC, s>>>(tmK, tmV, prm);
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
    verify_ffma_kernel<__nv_bfloat16, 64><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(pa.k),
                                                                  static_cast<const __nv_bfloat16 *>(pa.v), prm, total_q);
  else if (pa.d == 128)
    verify_ffma_kernel<float, 128><<<blocks, 256, 0, s>>>(static_cast<const float *>(pa.k),
                                                          static_cast<const float *>(pa.v), prm, total_q);
  else
    verify_ffma_kernel<float, 64><<<blocks, 256, 0, s>>>(static_cast<const float *>(pa.k),
                                                         static_cast<const float *>(pa.v), prm, total_q);
  return cudaGetLastError();
}

}  // namespace kap
