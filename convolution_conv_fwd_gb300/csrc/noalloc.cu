// Weight gradient for callers that cannot allocate device memory.
//
// gbconv_bwd_filter needs a caller-provided scratch buffer (the per-chunk fp32 partial sums that the
// ordered reduction adds).  Some callers cannot obtain one: code running where cudaMalloc is not
// allowed or not wanted (inside a custom allocator's own callbacks, a plugin handed only its tensors,
// a host that pre-reserves all device memory and forbids further allocations).  For them this file
// keeps the scratch in a fixed-size array in device global memory that the library module itself
// owns.  The array exists once per GPU that loads this library and stays until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "problem.h"

namespace gbconv {
namespace {

// The shared scratch.  Its size is GBCONV_NOALLOC_WORKSPACE_BYTES (include/gbconv.h).
__device__ __align__(256) unsigned char g_noalloc_scratch[GBCONV_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// The device address of g_noalloc_scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device (with that device current)
// and cached.
gbconv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GBCONV_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GBCONV_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GBCONV_OK;
}

}  // namespace
}  // namespace gbconv

extern "C" gbconv_status gbconv_bwd_filter_noalloc(const gbconv_desc* desc, const void* x, const void* dy, void* dw,
                                                   float* db, void* stream) {
  int64_t need = 0;
  const gbconv_status s = gbconv_bwd_filter_workspace(desc, &need);
  if (s != GBCONV_OK) return s;
  if (need > int64_t(GBCONV_NOALLOC_WORKSPACE_BYTES)) return GBCONV_EUNSUPPORTED;
  if (!x || !dy || !dw) return GBCONV_EINVAL;
  void* scratch = nullptr;
  const gbconv_status a = gbconv::scratch_address(&scratch);
  if (a != GBCONV_OK) return a;
  // Every partial sum the reduction reads is written earlier in the same call, so the array's
  // leftover contents from a previous call need no clearing.
  return gbconv_bwd_filter(desc, x, dy, dw, db, scratch, int64_t(GBCONV_NOALLOC_WORKSPACE_BYTES), stream);
}
