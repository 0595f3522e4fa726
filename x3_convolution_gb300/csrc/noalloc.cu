// noalloc.cu -- conv3x3_wgrad_noalloc: the weight gradient for callers that
// cannot allocate device memory.
//
// conv3x3_wgrad needs caller-provided scratch for its split-K partial sums.
// Some callers have no way to provide it: a plugin running inside a host
// application or engine that owns all device memory through its own pool and
// does not let extensions allocate, or a latency-critical loop where a
// cudaMalloc (which can synchronise the whole device) is not allowed after
// start-up.  This entry point takes the scratch from a fixed array that lives
// in this library's own device memory instead, so the call allocates nothing.
//
// The array is CONV3X3_WGRAD_NOALLOC_MAX_BYTES (64 MiB) per GPU, held by
// every GPU that loads the library until the process exits.  All calls on a
// GPU share it and it keeps whatever the previous call left there; the kernels
// overwrite every partial they later read, so nothing has to be cleared, but
// two calls whose work overlaps on the GPU (different streams, no ordering
// between them) race on the array and give wrong results.
#include <cuda_runtime.h>

#include <mutex>

#include "conv3x3_internal.h"

namespace c3 {
namespace {

static __device__ __align__(256) unsigned char g_wgrad_scratch[CONV3X3_WGRAD_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 64;  // device ordinals 0..63
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of this device's copy of the array.  In host code the name
// g_wgrad_scratch is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress with the device current; done once per device.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return CONV3X3_ERR_CUDA;
  if (dev >= kMaxDevices) return CONV3X3_ERR_UNSUPPORTED;  // beyond the per-device cache
  std::lock_guard<std::mutex> g(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wgrad_scratch) != cudaSuccess || p == nullptr)
      return CONV3X3_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CONV3X3_OK;
}

}  // namespace
}  // namespace c3

extern "C" {

int conv3x3_wgrad_noalloc(const void* x, const void* dy, float* dw, float* dbias, int N, int Cin,
                          int Cout, int H, int W, void* stream) {
  // same shape rules as conv3x3_wgrad; 0 means the shape itself is invalid
  const size_t need = conv3x3_wgrad_workspace_bytes(N, Cin, Cout, H, W);
  if (need == 0) return CONV3X3_ERR_INVALID_ARG;
  if (need > (size_t)CONV3X3_WGRAD_NOALLOC_MAX_BYTES) return CONV3X3_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = c3::scratch_for_current_device(&scratch);
  if (rc != CONV3X3_OK) return rc;
  return conv3x3_wgrad(x, dy, dw, dbias, N, Cin, Cout, H, W, scratch,
                       (size_t)CONV3X3_WGRAD_NOALLOC_MAX_BYTES, stream);
}

}  // extern "C"
