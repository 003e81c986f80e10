// gqa_noalloc.cu -- a decode entry point that needs no caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run attention: a
// plugin hosted by an inference engine that owns every byte of device memory and gives
// its plugins no allocator, or a latency-critical loop in which a cudaMalloc (which can
// synchronize the whole device) is not acceptable.  For them this file keeps the decode
// scratch (rotated queries, split partials, tickets) in one statically sized device array
// that the library carries itself, and forwards to gqa_attention_decode with that array as
// the workspace.  The kernels are the same; only the scratch comes from somewhere else.
#include <cuda_runtime.h>

#include <mutex>

#include "gqa.h"
#include "launch.h"

namespace {

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[GQA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device (the
// symbol's name in host code is only a host-side handle, never a device address).
gqa_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return GQA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GQA_OK;
}

}  // namespace

extern "C" gqa_status gqa_attention_decode_noalloc(const gqa_params *p, const void *q, const void *k, const void *v,
                                                   const void *past_k, const void *past_v, const int32_t *seqlens_k,
                                                   const void *cos_cache, const void *sin_cache,
                                                   const float *head_sink, void *out, void *present_k,
                                                   void *present_v, int32_t *dev_status, void *stream) {
  if (!p) return GQA_ERR_INVALID_ARG;
  // validate before anything else: the scratch layout below is only meaningful (and only
  // bounded by the array) for params that pass the checks
  const size_t need = gqa_workspace_bytes(p);  // 0 for invalid params, or when no scratch is needed
  if (need == 0)
    return gqa_attention_decode(p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, head_sink, out,
                                present_k, present_v, nullptr, 0, dev_status, stream);
  if (need > (size_t)GQA_NOALLOC_SCRATCH_BYTES) return GQA_ERR_WORKSPACE;
  const gqa::WsLayout wl = gqa::workspace_layout(*p, p->do_rotary != 0);
  if (wl.total > (size_t)GQA_NOALLOC_SCRATCH_BYTES || wl.tickets_off + wl.tickets_bytes > wl.total)
    return GQA_ERR_WORKSPACE;
  void *scratch = nullptr;
  gqa_status s = scratch_address(&scratch);
  if (s != GQA_OK) return s;
  // the split tickets must start at zero: the array keeps whatever the previous call left
  // (normally zeros, but not after a call whose waits timed out), so clear them every call
  if (wl.tickets_bytes > 0 &&
      cudaMemsetAsync(static_cast<char *>(scratch) + wl.tickets_off, 0, wl.tickets_bytes,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GQA_ERR_CUDA;
  return gqa_attention_decode(p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, head_sink, out, present_k,
                              present_v, scratch, (size_t)GQA_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
