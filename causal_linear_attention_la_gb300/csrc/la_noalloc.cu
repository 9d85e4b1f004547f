// la_forward_noalloc: the forward pass with its scratch in a static device
// array of this file, for callers that cannot allocate device memory (see
// include/la.h for who they are and for the rules of use).
#include <stdio.h>

#include <mutex>

#include "la_internal.cuh"

namespace la {
namespace {

// The scratch of every la_forward_noalloc call on a device. Sized for the
// per-segment state records of moderate problems; larger ones are rejected.
__device__ __align__(256) unsigned char g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current (the host-side name of a __device__
// array is not a device address).
la_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return set_error(LA_ERR_CUDA, "la_forward_noalloc: cudaGetDevice failed");
  }
  if (dev < 0 || dev >= kMaxDevices) return set_error(LA_ERR_UNSUPPORTED, "la_forward_noalloc: device index out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return set_error(LA_ERR_CUDA, "la_forward_noalloc: cudaGetSymbolAddress of the static scratch failed");
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return LA_OK;
}

}  // namespace
}  // namespace la

extern "C" la_status la_forward_noalloc(const void* q, const void* k, const void* v, void* out, int B, int H,
                                        int N, int dk, int dv, int causal, float eps, la_dtype dtype,
                                        float* S_final, float* z_final, la_stream_t stream) {
  void* scratch = nullptr;
  la_status st = la::scratch_address(&scratch);
  if (st != LA_OK) return st;
  const size_t need = la_forward_workspace_size(B, H, N, dk, dv, causal, dtype);
  if (need > LA_NOALLOC_SCRATCH_BYTES) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "la_forward_noalloc: problem needs %zu bytes of scratch, the static array holds %zu",
             need, (size_t)LA_NOALLOC_SCRATCH_BYTES);
    return la::set_error(LA_ERR_INVALID_ARG, msg);
  }
  return la_forward(q, k, v, out, B, H, N, dk, dv, causal, eps, dtype, S_final, z_final, scratch,
                    LA_NOALLOC_SCRATCH_BYTES, stream);
}
