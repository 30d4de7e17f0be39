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
// high, inverted id low). The chunk's logits, the next window token and the window offsets (32 per warp-wide load)
// are loaded together, so only the candidate's own logit waits on a load. The last CTA of a request (one
// acquire-release counter per request) loads every (row, chunk) record at once, reduces them per row in shared
// memory, and takes m (a ballot over the rows), the carry and the commit. No second launch, no host round trip.
#include "kap_device.cuh"
#include "kap_launch.h"

namespace kap {
namespace {

constexpr int kAccThreads = 256;
constexpr int kAccPerThread = 16;
constexpr int kAccChunk = kAccThreads * kAccPerThread;  // logits per CTA
constexpr int kMaxWindowRows = 32;                      // rows a window may hold (the carry and 31 proposals)

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
                                                             const int32_t *__restrict__ woff, int R, int total_rows,
                                                             const int32_t *__restrict__ tokens,
                                                             const int32_t *__restrict__ start_pos, int top_n,
                                                             AccPart *__restrict__ parts, int *__restrict__ counters,
                                                             int32_t *__restrict__ m_out, int32_t *__restrict__ carry_out,
                                                             int32_t *__restrict__ seq_out, int *err) {
  __shared__ unsigned long long s_first[kAccThreads / 32];
  __shared__ int s_before[kAccThreads / 32];
  __shared__ int s_last;
  __shared__ int s_rb[kMaxWindowRows];                 // finalisation: per window row, tokens before its candidate
  __shared__ unsigned long long s_rf[kMaxWindowRows];  // and its first token (64-bit key)
  grid_dependency_sync();
  const int row = blockIdx.y, chunk = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Independent loads first: this chunk's logits and the next window token (used only if it is in this window)
  const T *lrow = logits + static_cast<size_t>(row) * V;
  const int t0 = chunk * kAccChunk + threadIdx.x;
  float vals[kAccPerThread];
#pragma unroll
  for (int i = 0; i < kAccPerThread; ++i) {
    const int t = t0 + i * kAccThreads;
    vals[i] = t < V ? to_f(lrow[t]) : 0.0f;
  }
  const int x_next = row + 1 < total_rows ? tokens[row + 1] : -1;
  // request of this row: offsets are nondecreasing, so {i < R : off[i] <= row} is a prefix; each warp counts it
  // 32 offsets per load (one round trip while R <= 32) and takes the window bounds from the same loads
  int r = -1, w0 = 0, w1 = 0;
  for (int base = 0; base < R; base += 32) {
    const int i = base + lane;
    const int v = i <= R ? woff[i] : 0;
    const unsigned le = __ballot_sync(0xffffffffu, i < R && v <= row);
    const int cnt = __popc(le);
    if (cnt > 0) {
      r = base + cnt - 1;
      w0 = __shfl_sync(0xffffffffu, v, cnt - 1);
      w1 = cnt < 32 ? __shfl_sync(0xffffffffu, v, cnt) : woff[r + 1];
    }
    if (cnt < 32) break;
  }
  if (r < 0 || row >= w1) {  // rows beyond the offsets: this CTA judges nothing and is not counted
    if (threadIdx.x == 0) set_error(err, kErrLength);
    return;
  }
  const int x = row + 1 < w1 ? x_next : -1;  // the candidate this row judges (none for the window's last row)
  const bool has_x = x >= 0 && x < V;
  const uint32_t kx = has_x ? order_key(to_f(lrow[x])) : 0u;

  int before = 0;
  unsigned long long first = 0ull;
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
  const int rows = w1 - w0;
  if (threadIdx.x < kMaxWindowRows) {
    s_rb[threadIdx.x] = 0;
    s_rf[threadIdx.x] = 0ull;
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
    // other CTA's record of the request visible (to the whole CTA through the barrier below)
    const int old = atom_add_acq_rel_gpu(&counters[r], 1);
    s_last = (old == rows * nchunks - 1) ? 1 : 0;
    if (s_last) counters[r] = 0;  // leave the counter at zero for the next call
  }
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA of the request: every (row, chunk) record is loaded at once and reduced per row in shared memory
  const int nr = rows < kMaxWindowRows ? rows : kMaxWindowRows;
  for (int q = threadIdx.x; q < nr * nchunks; q += kAccThreads) {
    const int j = q / nchunks, c = q - j * nchunks;
    const size_t o = static_cast<size_t>(w0 + j) * nchunks + c;
    const int bq = __ldcg(&parts[o].before);
    const unsigned long long fq = __ldcg(&parts[o].first);
    if (bq) atomicAdd(&s_rb[j], bq);
    atomicMax(&s_rf[j], fq);
  }
  const int tok_j = threadIdx.x < nr ? tokens[w0 + threadIdx.x] : -1;
  __syncthreads();
  if (warp != 0) return;
  // proposal j (window row j >= 1) passes when it is a vocabulary token and fewer than top_n tokens of row j - 1
  // come before it; m is the length of the leading run of passes
  int tj = lane < nr ? tok_j : -1;
  bool pass = lane >= 1 && lane < nr && tj >= 0 && tj < V && s_rb[lane - 1] < top_n;
  unsigned bal = __ballot_sync(0xffffffffu, pass) | 1u;  // bit 0 stands for the carry
  int m = __ffs(~bal) - 2;                             // passes 1 .. m, then the first failure
  if (m < 0) m = 31;                                   // every lane passed: at most nr - 1 anyway
  m = min(m, nr - 1);
  if (rows > kMaxWindowRows && lane == 0) set_error(err, kErrLength);  // rows past the bound are not judged
  if (lane == 0) {
    const unsigned long long f = s_rf[m];
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
               static_cast<const __nv_bfloat16 *>(logits), V, nchunks, woff, R, total_rows, tokens, start_pos, top_n, parts,
               counters, m_out, carry_out, seq_out, err);
  else
    launch_pdl(accept_kernel<float>, grid, dim3(kAccThreads), 0, s, static_cast<const float *>(logits), V, nchunks,
               woff, R, total_rows, tokens, start_pos, top_n, parts, counters, m_out, carry_out, seq_out, err);
  return cudaGetLastError();
}

}  // namespace kap
