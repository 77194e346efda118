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
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "../../include/ffa.h"
#include "ffa_internal.h"

namespace ffa {
namespace {

static __device__ __align__(256) uint8_t g_fwd_scratch[FFA_FWD_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[64] = {};

// Device address of the scratch array for the current device.  The first call on a device
// looks it up (cudaGetSymbolAddress) with that device current; later calls reuse it.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FFA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || p == nullptr) return FFA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FFA_OK;
}

__global__ void fill_minus_inf(float* x, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    x[i] = -INFINITY;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uint64_t wait_limit() {
  const char* e = std::getenv("FFA_WAIT_LIMIT_NS");
  const unsigned long long v = e != nullptr ? std::strtoull(e, nullptr, 10) : 0ull;
  return v > 0 ? v : 4000000000ull;
}

}  // namespace
}  // namespace ffa

using namespace ffa;

extern "C" int ffa_fwd_noalloc(const ffa_shape* s, const void* q, const void* k, const void* v,
                               const int32_t* q_ranges, const int32_t* k_ranges, const int32_t* attn_type_map,
                               int32_t n_ranges, float softmax_scale, float softcap, void* out, float* lse,
                               int32_t* status, void* stream) {
  if (s == nullptr || n_ranges < 0) return FFA_ERR_INVALID_ARG;
  if (s->total_q < 0 || s->total_k < 0 || s->num_heads_q < 1 || s->num_heads_kv < 1 ||
      s->num_heads_q % s->num_heads_kv != 0)
    return FFA_ERR_INVALID_ARG;
  if (s->head_dim != 64 && s->head_dim != 128) return FFA_ERR_UNSUPPORTED;
  if (s->total_q > FFA_MAX_TOKENS || s->total_k > FFA_MAX_TOKENS ||
      static_cast<int64_t>(s->num_heads_q) * s->head_dim > 65536)
    return FFA_ERR_UNSUPPORTED;
  if (std::isnan(softcap) || softcap < 0.0f) return FFA_ERR_INVALID_ARG;
  const int64_t nq = s->total_q, nk = s->total_k;
  if (nq > 0 && (out == nullptr || lse == nullptr || q == nullptr)) return FFA_ERR_INVALID_ARG;
  if (nq > 0 && nk > 0 && (k == nullptr || v == nullptr)) return FFA_ERR_INVALID_ARG;
  if (n_ranges > 0 && (q_ranges == nullptr || k_ranges == nullptr || attn_type_map == nullptr))
    return FFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return FFA_ERR_INVALID_ARG;
  const WsLayout L = make_layout(nq, nk, s->num_heads_q, s->num_heads_kv, s->head_dim, n_ranges);
  if (L.fwd_total > static_cast<size_t>(FFA_FWD_NOALLOC_SCRATCH_BYTES)) return FFA_ERR_TOO_LARGE;
  if (nq == 0) return FFA_OK;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FFA_ERR_CUDA;
  if (major != 10 || minor != 3) return FFA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != FFA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int d = s->head_dim, hq = s->num_heads_q;
  if (nk == 0) {  // no key at all: every row is empty
    if (cudaMemsetAsync(out, 0, static_cast<size_t>(nq) * hq * d * 2, st) != cudaSuccess) return FFA_ERR_CUDA;
    fill_minus_inf<<<256, 256, 0, st>>>(lse, static_cast<size_t>(nq) * hq);
    return cudaGetLastError() == cudaSuccess ? FFA_OK : FFA_ERR_CUDA;
  }
  ProblemDims P;
  P.nq = static_cast<int>(L.nq);
  P.nk = static_cast<int>(L.nk);
  P.hq = L.hq;
  P.hkv = L.hkv;
  P.d = L.d;
  P.nqt = L.nqt;
  P.nkt = L.nkt;
  const PlanView pv = plan_view(L, scratch);
  cudaError_t e = launch_plan_slices(P, q_ranges, k_ranges, attn_type_map, n_ranges, pv, status, st);
  if (e == cudaSuccess) e = launch_plan_rows(P, L, pv, st);
  if (e != cudaSuccess) return FFA_ERR_CUDA;
  FwdArgs a;
  a.P = P;
  a.head_pair = L.head_pair ? 1 : 0;
  a.ngrp = L.ngrp;
  a.slots = L.slots;
  a.n_items = L.ngrp * L.nch_max * L.slots;
  a.split = L.split ? 1 : 0;
  a.scale = (!(softmax_scale > 0.0f) || std::isnan(softmax_scale)) ? 1.0f / std::sqrt(static_cast<float>(d))
                                                                     : softmax_scale;
  a.softcap = softcap;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.plan = pv;
  a.status = status;
  a.wait_limit_ns = wait_limit();
  return launch_fwd(a, st) == cudaSuccess ? FFA_OK : FFA_ERR_CUDA;
}
