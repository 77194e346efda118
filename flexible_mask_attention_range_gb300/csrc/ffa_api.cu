// C-ABI entry points of libffa.so: argument checks, workspace carving, TMA descriptors and
// the stream-ordered launch sequence (planner -> forward, planner -> backward).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/ffa.h"
#include "ffa_internal.h"

namespace ffa {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

__global__ void fill_empty_fwd_kernel(float* lse, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    lse[i] = -INFINITY;
}

uint64_t wait_limit_ns() {
  const char* e = std::getenv("FFA_WAIT_LIMIT_NS");
  if (e != nullptr) {
    const unsigned long long v = std::strtoull(e, nullptr, 10);
    if (v > 0) return v;
  }
  return 4000000000ull;  // 4 s
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FFA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FFA_ERR_CUDA;
  if (major != 10 || minor != 3) return FFA_ERR_UNSUPPORTED;
  return FFA_OK;
}

float resolve_scale(float scale, int d) {
  if (!(scale > 0.0f) || std::isnan(scale)) return 1.0f / std::sqrt(static_cast<float>(d));
  return scale;
}

ProblemDims dims_of(const WsLayout& L) {
  ProblemDims P;
  P.nq = static_cast<int>(L.nq);
  P.nk = static_cast<int>(L.nk);
  P.hq = L.hq;
  P.hkv = L.hkv;
  P.d = L.d;
  P.nqt = L.nqt;
  P.nkt = L.nkt;
  return P;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? FFA_OK : FFA_ERR_CUDA; }

// Failure-detection test hook: FFA_TEST_STALL=1 makes the first wait of every CTA of the
// next attention kernels wait on a barrier that nothing arrives on, so that the bounded wait
// runs out (FFA_WAIT_LIMIT_NS) and the kernel takes its abort path.  Off unless set.
int test_stall() {
  const char* e = std::getenv("FFA_TEST_STALL");
  return (e != nullptr && e[0] == '1' && e[1] == '\0') ? 1 : 0;
}

}  // namespace

KernelEvents g_kernel_events;

bool encode_tile_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                     uint32_t box_rows) {
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tile_map_f32(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                         uint32_t box_rows) {
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int cache[kMaxDevices];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  if (cache[dev] <= 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

int check_shape(const ffa_shape* s, int32_t n_ranges) {
  if (s == nullptr || n_ranges < 0) return FFA_ERR_INVALID_ARG;
  if (s->total_q < 0 || s->total_k < 0 || s->num_heads_q < 1 || s->num_heads_kv < 1) return FFA_ERR_INVALID_ARG;
  if (s->num_heads_q % s->num_heads_kv != 0) return FFA_ERR_INVALID_ARG;
  if (s->head_dim != 64 && s->head_dim != 128) return FFA_ERR_UNSUPPORTED;
  if (s->total_q > FFA_MAX_TOKENS || s->total_k > FFA_MAX_TOKENS) return FFA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(s->num_heads_q) * s->head_dim > 65536) return FFA_ERR_UNSUPPORTED;
  return FFA_OK;
}

int check_options(const ffa_options* o) {
  if (o == nullptr) return FFA_OK;
  for (int i = 0; i < 7; ++i)
    if (o->reserved[i] != 0) return FFA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(o->alibi_slopes) & 3u) != 0) return FFA_ERR_INVALID_ARG;
  return FFA_OK;
}

int fwd_check(const FwdCall& c, WsLayout* out_layout) {
  const ffa_shape* shape = c.shape;
  int rc = check_shape(shape, c.n_ranges);
  if (rc != FFA_OK) return rc;
  rc = check_options(c.options);
  if (rc != FFA_OK) return rc;
  if (c.paged) {
    const int ps = c.page_size;
    if (ps != 16 && ps != 32 && ps != 64 && ps != 128) return FFA_ERR_INVALID_ARG;
    if (c.n_pages < 1 || c.n_pages * static_cast<int64_t>(ps) >= (static_cast<int64_t>(1) << 31))
      return FFA_ERR_INVALID_ARG;
    if (shape->total_k > 0 && c.page_table == nullptr) return FFA_ERR_INVALID_ARG;
  }
  if (std::isnan(c.softcap) || c.softcap < 0.0f) return FFA_ERR_INVALID_ARG;
  const int64_t nq = shape->total_q, nk = shape->total_k;
  if (nq > 0 && (c.out == nullptr || c.lse == nullptr || c.q == nullptr)) return FFA_ERR_INVALID_ARG;
  if (nq > 0 && nk > 0 && (c.k == nullptr || c.v == nullptr)) return FFA_ERR_INVALID_ARG;
  if (c.n_ranges > 0 && (c.q_ranges == nullptr || c.k_ranges == nullptr || c.types == nullptr))
    return FFA_ERR_INVALID_ARG;
  if (!aligned16(c.q) || !aligned16(c.k) || !aligned16(c.v) || !aligned16(c.out) ||
      (reinterpret_cast<uintptr_t>(c.lse) & 3u) != 0)
    return FFA_ERR_INVALID_ARG;
  *out_layout = make_layout(nq, nk, shape->num_heads_q, shape->num_heads_kv, shape->head_dim, c.n_ranges,
                            c.key_split);
  return FFA_OK;
}

int fwd_launch(const FwdCall& c, const WsLayout& L, void* scratch) {
  int rc = check_device();
  if (rc != FFA_OK) return rc;
  const ffa_shape* shape = c.shape;
  const int64_t nq = shape->total_q, nk = shape->total_k;
  cudaStream_t s = static_cast<cudaStream_t>(c.stream);
  const int d = shape->head_dim, hq = shape->num_heads_q;
  if (nk == 0) {  // no key at all: every row is empty (the unpacked layout has the same sizes)
    void* o = c.unpack_out != nullptr ? c.unpack_out : c.out;
    float* l = c.unpack_lse != nullptr ? c.unpack_lse : c.lse;
    if (cudaMemsetAsync(o, 0, static_cast<size_t>(nq) * hq * d * 2, s) != cudaSuccess) return FFA_ERR_CUDA;
    fill_empty_fwd_kernel<<<256, 256, 0, s>>>(l, static_cast<size_t>(nq) * hq);
    return cuda_status(cudaGetLastError());
  }
  const ProblemDims P = dims_of(L);
  const PlanView pv = plan_view(L, scratch);
  cudaError_t e =
      launch_plan_slices(P, c.q_ranges, c.k_ranges, c.types, c.n_ranges, pv, c.status, s, c.after_own_kernel);
  if (e == cudaSuccess) e = launch_plan_rows(P, L, pv, s);
  if (e != cudaSuccess) return FFA_ERR_CUDA;
  FwdArgs a;
  a.P = P;
  a.head_pair = L.head_pair ? 1 : 0;
  a.ngrp = L.ngrp;
  a.slots = L.slots;
  a.n_items = L.ngrp * L.nch_max * L.slots;
  a.split = L.split ? 1 : 0;
  a.key_split = L.key_split ? 1 : 0;
  if (L.key_split) {
    a.unpack_out = c.unpack_out;
    a.unpack_lse = c.unpack_lse;
  }
  a.scale = resolve_scale(c.softmax_scale, d);
  a.softcap = c.softcap;
  a.q = c.q;
  a.k = c.k;
  a.v = c.v;
  a.out = c.out;
  a.lse = c.lse;
  a.alibi = c.options != nullptr ? c.options->alibi_slopes : nullptr;
  a.alibi_pack = c.alibi_pack;
  if (c.paged) {
    a.page_table = c.page_table;
    a.page_size = c.page_size;
    a.n_pages = c.n_pages;
  }
  a.plan = pv;
  a.status = c.status;
  a.wait_limit_ns = wait_limit_ns();
  a.stall_test = test_stall();
  return cuda_status(launch_fwd(a, s));
}

int fwd_with_workspace(const FwdCall& c, void* workspace, size_t workspace_bytes) {
  WsLayout L;
  int rc = fwd_check(c, &L);
  if (rc != FFA_OK) return rc;
  if (c.shape->total_q == 0) return FFA_OK;
  if (workspace == nullptr || workspace_bytes < L.fwd_total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FFA_ERR_WORKSPACE;
  return fwd_launch(c, L, workspace);
}

}  // namespace ffa

using namespace ffa;

extern "C" {

size_t ffa_fwd_workspace_size(const ffa_shape* s, int32_t n_ranges) {
  if (check_shape(s, n_ranges) != FFA_OK) return 0;
  return make_layout(s->total_q, s->total_k, s->num_heads_q, s->num_heads_kv, s->head_dim, n_ranges).fwd_total;
}

size_t ffa_bwd_workspace_size(const ffa_shape* s, int32_t n_ranges) {
  if (check_shape(s, n_ranges) != FFA_OK) return 0;
  return make_layout(s->total_q, s->total_k, s->num_heads_q, s->num_heads_kv, s->head_dim, n_ranges).bwd_total;
}

int ffa_fwd(const ffa_shape* shape, const void* q, const void* k, const void* v, const int32_t* q_ranges,
            const int32_t* k_ranges, const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale,
            float softcap, void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* status,
            void* stream) {
  return ffa_fwd_ex(shape, q, k, v, q_ranges, k_ranges, attn_type_map, n_ranges, softmax_scale, softcap, out, lse,
                    workspace, workspace_bytes, status, stream, nullptr);
}

int ffa_fwd_ex(const ffa_shape* shape, const void* q, const void* k, const void* v, const int32_t* q_ranges,
               const int32_t* k_ranges, const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale,
               float softcap, void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* status,
               void* stream, const ffa_options* options) {
  FwdCall c;
  c.shape = shape; c.q = q; c.k = k; c.v = v;
  c.q_ranges = q_ranges; c.k_ranges = k_ranges; c.types = attn_type_map; c.n_ranges = n_ranges;
  c.softmax_scale = softmax_scale; c.softcap = softcap; c.out = out; c.lse = lse;
  c.status = status; c.stream = stream; c.options = options;
  return fwd_with_workspace(c, workspace, workspace_bytes);
}

int ffa_fwd_paged(const ffa_shape* shape, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* page_table, int32_t page_size, int64_t n_pages, const int32_t* q_ranges,
                  const int32_t* k_ranges, const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale,
                  float softcap, void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* status,
                  void* stream, const ffa_options* options) {
  FwdCall c;
  c.shape = shape; c.q = q; c.k = k_pages; c.v = v_pages;
  c.q_ranges = q_ranges; c.k_ranges = k_ranges; c.types = attn_type_map; c.n_ranges = n_ranges;
  c.softmax_scale = softmax_scale; c.softcap = softcap; c.out = out; c.lse = lse;
  c.status = status; c.stream = stream; c.options = options;
  c.page_table = page_table; c.page_size = page_size; c.n_pages = n_pages;
  c.paged = true;
  return fwd_with_workspace(c, workspace, workspace_bytes);
}

int ffa_bwd(const ffa_shape* shape, const void* q, const void* k, const void* v, const void* out,
            const float* lse, const void* dout, const int32_t* q_ranges, const int32_t* k_ranges,
            const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale, float softcap, void* dq,
            void* dk, void* dv, void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  return ffa_bwd_ex(shape, q, k, v, out, lse, dout, q_ranges, k_ranges, attn_type_map, n_ranges, softmax_scale,
                    softcap, dq, dk, dv, workspace, workspace_bytes, status, stream, nullptr);
}

int ffa_bwd_ex(const ffa_shape* shape, const void* q, const void* k, const void* v, const void* out,
               const float* lse, const void* dout, const int32_t* q_ranges, const int32_t* k_ranges,
               const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale, float softcap, void* dq,
               void* dk, void* dv, void* workspace, size_t workspace_bytes, int32_t* status, void* stream,
               const ffa_options* options) {
  int rc = check_shape(shape, n_ranges);
  if (rc != FFA_OK) return rc;
  rc = check_options(options);
  if (rc != FFA_OK) return rc;
  if (std::isnan(softcap) || softcap < 0.0f) return FFA_ERR_INVALID_ARG;
  const int64_t nq = shape->total_q, nk = shape->total_k;
  if (nq > 0 && (q == nullptr || out == nullptr || lse == nullptr || dout == nullptr || dq == nullptr))
    return FFA_ERR_INVALID_ARG;
  if (nk > 0 && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr)) return FFA_ERR_INVALID_ARG;
  if (n_ranges > 0 && (q_ranges == nullptr || k_ranges == nullptr || attn_type_map == nullptr))
    return FFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return FFA_ERR_INVALID_ARG;
  const WsLayout L = make_layout(nq, nk, shape->num_heads_q, shape->num_heads_kv, shape->head_dim, n_ranges);
  if (nq == 0 && nk == 0) return FFA_OK;
  if (workspace == nullptr || workspace_bytes < L.bwd_total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FFA_ERR_WORKSPACE;
  rc = check_device();
  if (rc != FFA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int d = shape->head_dim;
  if (nq == 0 || nk == 0) {  // nothing visible: all gradients are zero
    if (nq > 0 && cudaMemsetAsync(dq, 0, static_cast<size_t>(nq) * shape->num_heads_q * d * 2, s) != cudaSuccess)
      return FFA_ERR_CUDA;
    if (nk > 0) {
      const size_t b = static_cast<size_t>(nk) * shape->num_heads_kv * d * 2;
      if (cudaMemsetAsync(dk, 0, b, s) != cudaSuccess || cudaMemsetAsync(dv, 0, b, s) != cudaSuccess)
        return FFA_ERR_CUDA;
    }
    return FFA_OK;
  }
  const ProblemDims P = dims_of(L);
  const PlanView pv = plan_view(L, workspace);
  cudaError_t e = launch_plan_slices(P, q_ranges, k_ranges, attn_type_map, n_ranges, pv, status, s);
  if (e == cudaSuccess) e = launch_plan_cols(P, pv, s);
  if (e != cudaSuccess) return FFA_ERR_CUDA;
  BwdArgs a;
  a.P = P;
  a.scale = resolve_scale(softmax_scale, d);
  a.softcap = softcap;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  char* wb = static_cast<char*>(workspace);
  a.rowD = reinterpret_cast<float*>(wb + L.rowD);
  a.lse2 = reinterpret_cast<float*>(wb + L.lse2);
  a.dqacc = reinterpret_cast<float*>(wb + L.dqacc);
  a.alibi = options != nullptr ? options->alibi_slopes : nullptr;
  a.deterministic = (options != nullptr && options->deterministic) ? 1 : 0;
  a.tile_rank = reinterpret_cast<int*>(wb + L.tile_rank);
  a.dq_sem = reinterpret_cast<int*>(wb + L.dq_sem);
  if (a.deterministic) {
    if (launch_plan_ranks(P, pv, a.tile_rank, s) != cudaSuccess) return FFA_ERR_CUDA;
    if (cudaMemsetAsync(a.dq_sem, 0, static_cast<size_t>(P.hq) * P.nqt * sizeof(int), s) != cudaSuccess)
      return FFA_ERR_CUDA;
  }
  a.plan = pv;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns();
  a.stall_test = test_stall();
  return cuda_status(launch_bwd(a, s));
}

int ffa_plan_tiles(const ffa_shape* shape, const int32_t* q_ranges, const int32_t* k_ranges,
                   const int32_t* attn_type_map, int32_t n_ranges, int32_t by_column, uint8_t* tile_class,
                   void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  int rc = check_shape(shape, n_ranges);
  if (rc != FFA_OK) return rc;
  if (n_ranges > 0 && (q_ranges == nullptr || k_ranges == nullptr || attn_type_map == nullptr))
    return FFA_ERR_INVALID_ARG;
  const WsLayout L = make_layout(shape->total_q, shape->total_k, shape->num_heads_q, shape->num_heads_kv,
                                 shape->head_dim, n_ranges);
  if (L.nqt == 0 || L.nkt == 0) return FFA_OK;
  if (tile_class == nullptr) return FFA_ERR_INVALID_ARG;
  const size_t need = by_column ? L.bwd_total : L.fwd_total;
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FFA_ERR_WORKSPACE;
  rc = check_device();
  if (rc != FFA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const ProblemDims P = dims_of(L);
  const PlanView pv = plan_view(L, workspace);
  cudaError_t e = launch_plan_slices(P, q_ranges, k_ranges, attn_type_map, n_ranges, pv, status, s);
  if (e == cudaSuccess) e = by_column ? launch_plan_cols(P, pv, s) : launch_plan_rows(P, L, pv, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(tile_class, pv.cls, static_cast<size_t>(L.nqt) * L.nkt, cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

int ffa_set_kernel_events(void* fwd_start, void* fwd_stop, void* bwd_start, void* bwd_stop) {
  g_kernel_events.fwd_start = static_cast<cudaEvent_t>(fwd_start);
  g_kernel_events.fwd_stop = static_cast<cudaEvent_t>(fwd_stop);
  g_kernel_events.bwd_start = static_cast<cudaEvent_t>(bwd_start);
  g_kernel_events.bwd_stop = static_cast<cudaEvent_t>(bwd_stop);
  return FFA_OK;
}

const char* ffa_status_string(int code) {
  switch (code) {
    case FFA_OK: return "ok";
    case FFA_ERR_INVALID_ARG: return "invalid argument";
    case FFA_ERR_UNSUPPORTED: return "unsupported shape or device (needs sm_103a, head_dim 64 or 128)";
    case FFA_ERR_CUDA: return "CUDA call failed";
    case FFA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FFA_ERR_TOO_LARGE: return "problem needs more scratch than the library's fixed device array holds";
    default: return "unknown status";
  }
}

const char* ffa_build_info(void) {
  return "libffa: sm_103a tcgen05/TMEM/TMA; tile 128x128 (query x key); forward: 2 query tiles per CTA, "
         "K/V ring 2 stages (d=128) / 4 stages (d=64), lazy rescale threshold 2^8; backward: KV-stationary, "
         "one key tile per CTA, dq accumulated in fp32";
}

}  // extern "C"
