// k_materialize.cu - materialised compact selected-KV workspace (sm_103a).
//
// KAP paper, compiler (stage 3: the selected spans are resolved to KV pages and materialised as a compact physical
// view that keeps logical positions, with the block tables and slot mappings the executor needs) and fallback (full
// access when the plan exceeds the compact workspace). Request r owns the ws_pages pool pages from
// ws_first + r * ws_pages. The i-th selected entry of a view row is copied to page ws_first + r * ws_pages + i
// (K and V; for a per-head view only that head's chunk, for a shared view every head) and the row's table entry is
// pointed there, when all its tokens are prompt tokens; a selected page that also holds positions >= ctx_len (the
// partial last prompt page) keeps its page, because generated tokens are written into it through the full table
// after the copy. Tail entries keep their pages; logical pages are unchanged. A row whose selection exceeds the
// workspace is left unchanged and flags its request.
//
// Design (GB300): a plain HBM copy. One warp moves one 4 KiB (page, head) chunk with 16-byte loads and stores,
// eight chunks in flight per CTA; the grid is (entry blocks, view rows), so every selected chunk of every row is
// in flight at once. The copy reads with streaming loads (the source pages are not read again this cycle) and
// writes with the default policy (the proposals of the cycle read the workspace next). The output view may be the
// input view itself.
#include "kap_device.cuh"
#include "kap_launch.h"

namespace kap {
namespace {

constexpr int kMatWarps = 8;
constexpr int kMatEntries = 4;  // view entries per CTA: K and V of each go to two warps

__global__ void __launch_bounds__(kMatWarps * 32) materialize_kernel(
    const uint4 *k_in, const uint4 *v_in, uint4 *k_out, uint4 *v_out, int num_pages,
    int hkv, int chunk_vecs, int rows_per_seq, const int32_t *ctx_len, const int32_t *vbt, const int32_t *vlp,
    const int32_t *vn,
    const int32_t *vnsel, int vcap, int32_t *obt, int32_t *olp, int32_t *on, int32_t *onsel, int ocap, int ws_first,
    int ws_pages, int32_t *fallback, int *err) {
  grid_dependency_sync();
  const int vrow = blockIdx.y;  // r * rows_per_seq + v
  const int r = vrow / rows_per_seq, v = vrow - r * rows_per_seq;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n_ent = min(vn[vrow], vcap);
  const int n_sel = min(vnsel[vrow], n_ent);
  const bool fits = n_sel <= ws_pages;
  const int ws_base = ws_first + r * ws_pages;
  const int i = blockIdx.x * kMatEntries + warp / 2;  // entry of this warp
  const bool is_v = (warp & 1) != 0;
  const bool active = i < n_ent;
  const size_t in_o = static_cast<size_t>(vrow) * vcap + i;
  const size_t out_o = static_cast<size_t>(vrow) * ocap + i;
  const int src = active ? vbt[in_o] : 0;
  const int lp = active ? vlp[in_o] : 0;
  __syncthreads();  // both warps of an entry have read its page before either rewrites it (the view may be in place)
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    on[vrow] = n_ent;
    onsel[vrow] = n_sel;
    if (!fits && fallback) fallback[r] = 1;  // the plan exceeds the compact workspace (never cleared here)
  }
  if (!active) return;
  const bool copy = fits && i < n_sel && kPage * (lp + 1) <= ctx_len[r];  // pure prompt pages only
  const int dst = copy ? ws_base + i : src;
  if (copy) {
    if (src < 0 || src >= num_pages) {
      if (lane == 0) set_error(err, kErrPage);
    } else {
      const uint4 *in = is_v ? v_in : k_in;
      uint4 *out = is_v ? v_out : k_out;
      // a per-head row moves its own head's chunk; a shared row moves every head of the page
      const int h_lo = rows_per_seq == 1 ? 0 : v, h_hi = rows_per_seq == 1 ? hkv : v + 1;
      for (int h = h_lo; h < h_hi; ++h) {
        const uint4 *s = in + (static_cast<size_t>(src) * hkv + h) * chunk_vecs;
        uint4 *d = out + (static_cast<size_t>(dst) * hkv + h) * chunk_vecs;
        uint4 buf[8];
        for (int c0 = 0; c0 < chunk_vecs; c0 += 8 * 32) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < chunk_vecs) buf[u] = __ldcs(s + c);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < chunk_vecs) d[c] = buf[u];
          }
        }
      }
    }
  }
  if (!is_v && lane == 0) {  // the K warp of the entry writes its table entries
    obt[out_o] = dst;
    olp[out_o] = lp;
  }
}

}  // namespace

cudaError_t launch_materialize(const PoolArgs &p, int R, const int32_t *ctx_len, const ViewArgs &in, int32_t *obt,
                               int32_t *olp, int32_t *on,
                               int32_t *onsel, int ocap, int ws_first, int ws_pages, int32_t *fallback, int *err,
                               cudaStream_t s) {
  const int elem = p.dtype == 0 ? 2 : 4;
  const int chunk_vecs = kPage * p.d * elem / 16;
  const dim3 grid((in.cap + kMatEntries - 1) / kMatEntries, R * in.rows_per_seq);
  launch_pdl(materialize_kernel, grid, dim3(kMatWarps * 32), 0, s, static_cast<const uint4 *>(p.k),
             static_cast<const uint4 *>(p.v), static_cast<uint4 *>(const_cast<void *>(p.k)),
             static_cast<uint4 *>(const_cast<void *>(p.v)), p.num_pages, p.hkv, chunk_vecs, in.rows_per_seq, ctx_len,
             in.bt,
             in.lp, in.n_entries, in.n_selected, in.cap, obt, olp, on, onsel, ocap, ws_first, ws_pages, fallback,
             err);
  return cudaGetLastError();
}

}  // namespace kap
