// k_append.cu - KV append with rotary position embedding for the selected-KV hot path (sm_103a).
//
// KAP paper, executor: proposed tokens are written through the slot mapping at their full-sequence logical
// positions, and the verifier writes the window's KV into the full-context slots. K is rotated at its logical
// position (half-split pairs (i, i + d/2), angle = (float)pos * inv_freq[i] in fp32), V is copied. Optionally the
// query rows of the same tokens are rotated in place.
#include "kap_device.cuh"
#include "kap_launch.h"

namespace kap {
namespace {

// One warp per (token, head row); rows [0, Hkv) are K/V heads, rows [Hkv, Hkv + Hq) query heads.
template <class T, int D>
__global__ void __launch_bounds__(256) append_kernel(T *__restrict__ Kp, T *__restrict__ Vp,
                                                     const T *__restrict__ k_new, const T *__restrict__ v_new,
                                                     T *__restrict__ q_inout, const int32_t *__restrict__ pos,
                                                     const int64_t *__restrict__ slots, int T_tok, int tok_stride,
                                                     const float *__restrict__ inv_freq, int hkv, int hq,
                                                     int num_pages, int *err) {
  constexpr int HALF = D / 2;
  grid_dependency_sync();
  const int warps_per_cta = blockDim.x >> 5;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int rows_per_tok = hkv + (q_inout ? hq : 0);
  if (wid >= static_cast<int64_t>(T_tok) * rows_per_tok) return;
  const int t = static_cast<int>(wid / rows_per_tok);
  const int h = static_cast<int>(wid - static_cast<int64_t>(t) * rows_per_tok);
  const int p = pos[static_cast<int64_t>(t) * tok_stride];
  const bool is_q = h >= hkv;
  const T *src;
  T *dst;
  if (is_q) {
    src = q_inout + (static_cast<size_t>(t) * hq + (h - hkv)) * D;
    dst = q_inout + (static_cast<size_t>(t) * hq + (h - hkv)) * D;
  } else {
    const int64_t s = slots[static_cast<int64_t>(t) * tok_stride];
    if (s < 0) return;
    const int64_t page = s / kPage;
    const int off = static_cast<int>(s - page * kPage);
    if (page >= num_pages) {
      if (lane == 0) set_error(err, kErrPage);
      return;
    }
    const size_t o = ((static_cast<size_t>(page) * hkv + h) * kPage + off) * D;
    src = k_new + (static_cast<size_t>(t) * hkv + h) * D;
    dst = Kp + o;
    // V is copied unchanged.
    const T *vs = v_new + (static_cast<size_t>(t) * hkv + h) * D;
    T *vd = Vp + o;
    for (int i = lane; i < D; i += 32) vd[i] = vs[i];
  }
  for (int i = lane; i < HALF; i += 32) {
    const float x = to_f(src[i]), y = to_f(src[i + HALF]);
    float xr, yr;
    rope_pair(x, y, p, inv_freq[i], xr, yr);
    dst[i] = from_f<T>(xr);
    dst[i + HALF] = from_f<T>(yr);
  }
}

}  // namespace

cudaError_t launch_append(const PoolArgs &p, const void *k_new, const void *v_new, void *q_inout,
                          const int32_t *pos, const int64_t *slots, int T, int tok_stride, const float *inv_freq,
                          int *err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int rows = p.hkv + (q_inout ? p.hq : 0);
  const int64_t warps = static_cast<int64_t>(T) * rows;
  const int blocks = static_cast<int>((warps + 7) / 8);
#define KAP_APPEND(TT, D)                                                                                       \
  launch_pdl(append_kernel<TT, D>, dim3(blocks), dim3(256), 0, s,                                               \
             static_cast<TT *>(const_cast<void *>(p.k)), static_cast<TT *>(const_cast<void *>(p.v)),             \
             static_cast<const TT *>(k_new), static_cast<const TT *>(v_new), static_cast<TT *>(q_inout), pos,     \
             slots, T, tok_stride, inv_freq, p.hkv, p.hq, p.num_pages, err)
  if (p.dtype == 0 && p.d == 128) KAP_APPEND(__nv_bfloat16, 128);
  else if (p.dtype == 0 && p.d == 64) KAP_APPEND(__nv_bfloat16, 64);
  else if (p.dtype == 1 && p.d == 128) KAP_APPEND(float, 128);
  else KAP_APPEND(float, 64);
#undef KAP_APPEND
  return cudaGetLastError();
}

}  // namespace kap
