// gdn_prefill_chunked_noalloc: the chunked prompt pass for callers that cannot allocate
// device memory (see include/gdn.h).  Its scratch is a fixed array compiled into this
// translation unit instead of a caller-supplied workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"

namespace {

// The scratch.  In host code `g_scratch` names only a host-side stand-in for the
// symbol, never its device address: the address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) unsigned char g_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up on first use).
gdn_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return GDN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_prefill_chunked_noalloc(const gdn_shape *shape, const void *q,
                                                  const void *k, const void *v, const float *g,
                                                  const float *beta, const float *state_in,
                                                  float *state_out, const int32_t *cu_seqlens,
                                                  void *o, void *stream) {
  const size_t need = gdn_workspace_size(shape, GDN_OP_PREFILL);
  if (need == (size_t)-1 || need == 0)  // invalid shape (reported by the call), or no scratch
    return gdn_prefill_chunked(shape, q, k, v, g, beta, state_in, state_out, cu_seqlens, o,
                               nullptr, 0, stream);
  if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
  void *ws = nullptr;
  const gdn_status st = scratch_address(&ws);
  if (st != GDN_OK) return st;
  // Nothing in the scratch has to start at zero: each call writes every scratch element
  // before it reads it, so what a previous call left there is never used.
  return gdn_prefill_chunked(shape, q, k, v, g, beta, state_in, state_out, cu_seqlens, o, ws,
                             (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}
