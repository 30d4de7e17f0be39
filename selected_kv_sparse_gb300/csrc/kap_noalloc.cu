// kap_noalloc.cu - proposal attention for callers that cannot allocate device memory.
//
// Some hosts may not call cudaMalloc once they are serving: an engine that plans its whole device memory budget at
// start-up and owns the only allocator, a plug-in that has no handle on that allocator, or a latency-critical loop
// where an allocation (which may synchronise the device) is not allowed. kap_attn_propose needs a caller-provided
// workspace; this entry point instead uses a scratch array that lives in the library image itself.
//
// The array below is a file-scope device variable of fixed size. Every GPU that loads the library holds it until the
// process exits. Host code must never pass the array's name to a kernel (on the host it is only a stand-in symbol,
// not a device address): the device address is obtained with cudaGetSymbolAddress, once per device, with that
// device current, and cached.
#include "../../include/kap.h"
#include "kap_launch.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array on the current device (looked up on the first call per device and kept for
// the life of the process: a cudaDeviceReset of that device invalidates it, see kap.h).
cudaError_t scratch_address(void **out) {
  static void *addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kap_status kap_attn_propose_noalloc(const kap_kv_pool *pool, const kap_page_map *map,
                                               const kap_view *view, const void *q_dev, void *out, float *lse,
                                               kap_stream stream) {
  if (!pool || !map) return KAP_EINVAL;
  if (map->num_seqs <= 0 || pool->num_kv_heads <= 0 || pool->num_q_heads <= 0 || pool->head_dim <= 0)
    return KAP_EINVAL;
  const size_t need =
      kap_propose_workspace_size(map->num_seqs, pool->num_kv_heads, pool->num_q_heads, pool->head_dim);
  if (need == 0 || need > kScratchBytes) return KAP_ECAPACITY;  // the shape needs more than the fixed scratch
  void *scratch = nullptr;
  if (kap::record_cuda_error(scratch_address(&scratch))) return KAP_ECUDA;
  // The per-row arrival counters at the start of the scratch must be zero when the kernel starts; the array keeps
  // whatever the previous call left, so clear them on the caller's stream.
  const size_t counter_bytes = static_cast<size_t>(map->num_seqs) * pool->num_kv_heads * sizeof(int);
  if (kap::record_cuda_error(cudaMemsetAsync(scratch, 0, counter_bytes, reinterpret_cast<cudaStream_t>(stream))))
    return KAP_ECUDA;
  return kap_attn_propose(pool, map, view, q_dev, out, lse, scratch, kScratchBytes, stream);
}

extern "C" size_t kap_noalloc_scratch_bytes(void) { return kScratchBytes; }
