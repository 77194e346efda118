// ffa_fwd_noalloc: the forward pass without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the attention: runtimes that
// reserve all device memory at start-up and forbid any later cudaMalloc, and latency-bound
// paths that cannot afford the implicit device synchronisation cudaMalloc / cudaFree may
// perform.  This entry point takes the planner's scratch from a fixed array in device
// memory that the library owns instead of from the caller.  The array exists once per
// device that loads the library and stays allocated until the process exits.
//
// The planner writes every scratch word it later reads (slice count, compacted slices, tile
// classes, slice lists, work lists and their order), so no part of the array has to start
// at zero and the contents a previous call left behind are never read.  All calls share the
// array: two calls whose kernels overlap on the GPU (different streams, or different host
// threads on one device) race on it and must be serialised by the caller.
#include <mutex>

#include "../../include/ffa.h"
#include "ffa_internal.h"

namespace ffa {
namespace {

static __device__ __align__(256) uint8_t g_fwd_scratch[FFA_FWD_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device.  The first call on a device
// looks it up (cudaGetSymbolAddress) with that device current; later calls reuse it.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FFA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || p == nullptr) return FFA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FFA_OK;
}

}  // namespace
}  // namespace ffa

using namespace ffa;

extern "C" int ffa_fwd_noalloc(const ffa_shape* s, const void* q, const void* k, const void* v,
                               const int32_t* q_ranges, const int32_t* k_ranges, const int32_t* attn_type_map,
                               int32_t n_ranges, float softmax_scale, float softcap, void* out, float* lse,
                               int32_t* status, void* stream) {
  FwdCall c;
  c.shape = s; c.q = q; c.k = k; c.v = v;
  c.q_ranges = q_ranges; c.k_ranges = k_ranges; c.types = attn_type_map; c.n_ranges = n_ranges;
  c.softmax_scale = softmax_scale; c.softcap = softcap; c.out = out; c.lse = lse;
  c.status = status; c.stream = stream;
  // the same argument checks as ffa_fwd; then the size check against the fixed array
  WsLayout L;
  int rc = fwd_check(c, &L);
  if (rc != FFA_OK) return rc;
  if (L.fwd_total > static_cast<size_t>(FFA_FWD_NOALLOC_SCRATCH_BYTES)) return FFA_ERR_TOO_LARGE;
  if (s->total_q == 0) return FFA_OK;
  void* scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc != FFA_OK) return rc;
  return fwd_launch(c, L, scratch);
}
