// k_accept.cu - tolerant acceptance and commit of verify windows (sm_103a).
//
// KAP paper, verifier: the verification window is the verifier-approved carry token followed by the k proposed
// tokens; a proposal is accepted when it lies within the target model's top-n candidates under the full context
// (the Top-3 rule: n = 3), m counts the proposals accepted consecutively from the start of the window, and the same
// transition emits the next carry and advances the committed full-context state.
//
// Rank order of a row: logit descending, lower token id first, NaN last. Proposal j of a window is checked against
// window row j - 1: it passes when fewer than n tokens of that row come before it. The next carry is the first
// token of row m; the committed length is start + 1 + m (the carry and the accepted proposals, whose KV the window
// append has already written at their positions).
//
// Design (GB300): the pass is a stream over the logits, so the grid is (vocabulary chunks, window rows). Each CTA
// reads 4096 logits of one row with coalesced loads and reduces two things: how many of its tokens come before the
// row's candidate (the next window token), and its first token under the rank order as one 64-bit key (order key
// high, inverted id low). The last CTA of a request (one acquire-release counter per request) adds the counts of
// each row, finds m and the carry, and writes the commit. No second launch and no host round trip.
#include "kap_device.cuh"
#include "kap_launch.h"

namespace kap {
namespace {

constexpr int kAccThreads = 256;
constexpr int kAccPerThread = 16;
constexpr int kAccChunk = kAccThreads * kAccPerThread;  // logits per CTA

struct AccPart {
  unsigned long long first;  // max over the chunk of (order key << 32) | (0xffffffff - token)
  int before;                // tokens of the chunk that come before the row's candidate
  int pad;
};
static_assert(sizeof(AccPart) == 16, "partial record");

__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const unsigned long long u = __shfl_xor_sync(0xffffffffu, v, o);
    v = u > v ? u : v;
  }
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <class T>
__global__ void __launch_bounds__(kAccThreads) accept_kernel(const T *__restrict__ logits, int V, int nchunks,
                                                             const int32_t *__restrict__ woff, int R,
                                                             const int32_t *__restrict__ tokens,
                                                             const int32_t *__restrict__ start_pos, int top_n,
                                                             AccPart *__restrict__ parts, int *__restrict__ counters,
                                                             int32_t *__restrict__ m_out, int32_t *__restrict__ carry_out,
                                                             int32_t *__restrict__ seq_out, int *err) {
  __shared__ unsigned long long s_first[kAccThreads / 32];
  __shared__ int s_before[kAccThreads / 32];
  __shared__ int s_last;
  grid_dependency_sync();
  const int row = blockIdx.y, chunk = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // request of this row: the last r with woff[r] <= row
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (woff[mid] <= row) lo = mid; else hi = mid - 1;
  }
  const int r = lo, w0 = woff[r], w1 = woff[r + 1];
  if (row >= w1) {  // more rows launched than the offsets hold: this CTA judges nothing and is not counted
    if (threadIdx.x == 0) set_error(err, kErrLength);
    return;
  }
  const int x = row + 1 < w1 ? tokens[row + 1] : -1;  // the candidate this row judges (none for the last row)
  const bool has_x = x >= 0 && x < V;
  const T *lrow = logits + static_cast<size_t>(row) * V;
  const uint32_t kx = has_x ? order_key(to_f(lrow[x])) : 0u;

  int before = 0;
  unsigned long long first = 0ull;
  const int t0 = chunk * kAccChunk + threadIdx.x;
  float vals[kAccPerThread];
#pragma unroll
  for (int i = 0; i < kAccPerThread; ++i) {
    const int t = t0 + i * kAccThreads;
    vals[i] = t < V ? to_f(lrow[t]) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < kAccPerThread; ++i) {
    const int t = t0 + i * kAccThreads;
    if (t < V) {
      const uint32_t kt = order_key(vals[i]);
      before += (has_x && (kt > kx || (kt == kx && t < x))) ? 1 : 0;
      const unsigned long long key = (static_cast<unsigned long long>(kt) << 32) | (0xffffffffu - static_cast<uint32_t>(t));
      first = key > first ? key : first;
    }
  }
  before = warp_sum_i(before);
  first = warp_max_u64(first);
  if (lane == 0) {
    s_before[warp] = before;
    s_first[warp] = first;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int b = 0;
    unsigned long long f = 0ull;
    for (int i = 0; i < kAccThreads / 32; ++i) {
      b += s_before[i];
      f = s_first[i] > f ? s_first[i] : f;
    }
    AccPart pr;
    pr.first = f;
    pr.before = b;
    pr.pad = 0;
    parts[static_cast<size_t>(row) * nchunks + chunk] = pr;
    // counts the CTA in; the acquire-release atomic publishes this record and, for the last arriver, makes every
    // other CTA's record of the request visible
    const int total = (w1 - w0) * nchunks;
    const int old = atom_add_acq_rel_gpu(&counters[r], 1);
    s_last = (old == total - 1) ? 1 : 0;
    if (s_last) counters[r] = 0;  // leave the counter at zero for the next call
  }
  __syncthreads();
  if (!s_last || warp != 0) return;

  // ---- last CTA of the request: warp 0 adds each row's counts over the chunks, then m, the carry and the commit
  const int rows = w1 - w0;
  int m = 0;
  for (int j = 1; j < rows; ++j) {
    const int xj = tokens[w0 + j];
    if (xj < 0 || xj >= V) break;  // outside the vocabulary: rejected
    int b = 0;
    for (int c = lane; c < nchunks; c += 32) b += __ldcg(&parts[static_cast<size_t>(w0 + j - 1) * nchunks + c].before);
    b = warp_sum_i(b);
    if (b >= top_n) break;
    ++m;
  }
  unsigned long long f = 0ull;
  for (int c = lane; c < nchunks; c += 32) {
    const unsigned long long u = __ldcg(&parts[static_cast<size_t>(w0 + m) * nchunks + c].first);
    f = u > f ? u : f;
  }
  f = warp_max_u64(f);
  if (lane == 0) {
    m_out[r] = m;
    carry_out[r] = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(f & 0xffffffffull));
    if (seq_out) seq_out[r] = start_pos[r] + 1 + m;
  }
}

}  // namespace

size_t accept_workspace_bytes(int num_seqs, int total_rows, int vocab) {
  const size_t nchunks = (static_cast<size_t>(vocab) + kAccChunk - 1) / kAccChunk;
  return ((static_cast<size_t>(num_seqs) * 4 + 255) / 256) * 256 + static_cast<size_t>(total_rows) * nchunks * 16;
}

cudaError_t launch_accept(const void *logits, int dtype, int V, const int32_t *woff, int R, int total_rows,
                          const int32_t *tokens, const int32_t *start_pos, int top_n, void *ws, int32_t *m_out,
                          int32_t *carry_out, int32_t *seq_out, int *err, cudaStream_t s) {
  const int nchunks = (V + kAccChunk - 1) / kAccChunk;
  int *counters = static_cast<int *>(ws);
  AccPart *parts = reinterpret_cast<AccPart *>(static_cast<unsigned char *>(ws) +
                                               ((static_cast<size_t>(R) * 4 + 255) / 256) * 256);
  const dim3 grid(nchunks, total_rows);
  if (dtype == 0)
    launch_pdl(accept_kernel<__nv_bfloat16>, grid, dim3(kAccThreads), 0, s,
               static_cast<const __nv_bfloat16 *>(logits), V, nchunks, woff, R, tokens, start_pos, top_n, parts,
               counters, m_out, carry_out, seq_out, err);
  else
    launch_pdl(accept_kernel<float>, grid, dim3(kAccThreads), 0, s, static_cast<const float *>(logits), V, nchunks,
               woff, R, tokens, start_pos, top_n, parts, counters, m_out, carry_out, seq_out, err);
  return cudaGetLastError();
}

}  // namespace kap
