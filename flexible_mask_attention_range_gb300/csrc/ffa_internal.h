// Internal structures shared by the host entry points and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <utility>

#include "../../include/ffa.h"

namespace ffa {

constexpr int kTile = 128;         // global tile edge (query rows and key columns)
constexpr int kSliceCap = 64;      // slice ids stored per tile row / tile column for masks
constexpr int kSliceSmem = 512;    // slices staged in shared memory by the planner
constexpr int kMaxTiles = 8192;    // ceil(FFA_MAX_TOKENS / 128)
constexpr int kMaxDevices = 64;    // per-device caches (function attributes, SM counts, scratch)
// Forward work lists are cut into chunks when there are too few work items to fill the GPU:
// the planner then aims at about kSplitTarget chunks (two per SM on a 152-SM part) of at least
// kMinChunk key tiles, and a merge kernel combines the chunks' partial results by LSE.
constexpr int kSplitTarget = 304;
constexpr int kMinChunk = 16;
constexpr int kMinSplitTiles = 32;

// Entry of a work list: key-tile (or query-tile) index in bits 0..23, class of sub-tile a
// in bits 24..25 and of sub-tile b in bits 26..27.
__host__ __device__ inline uint32_t make_entry(int idx, int ca, int cb) {
  return static_cast<uint32_t>(idx) | (static_cast<uint32_t>(ca) << 24) | (static_cast<uint32_t>(cb) << 26);
}
__host__ __device__ inline int entry_idx(uint32_t e) { return static_cast<int>(e & 0xFFFFFFu); }
__host__ __device__ inline int entry_cls(uint32_t e, int sub) { return static_cast<int>((e >> (24 + 2 * sub)) & 3u); }

// Workspace layout.  Every region starts on a 256-byte boundary.
struct WsLayout {
  int64_t nq = 0, nk = 0;
  int hq = 0, hkv = 0, d = 0, R = 0;
  int nqt = 0, nkt = 0;
  bool head_pair = true;  // forward pairs two query heads of one KV group (else two q-tiles)
  // forward key split (decode): an item is one query tile of one head; its two softmax
  // warpgroups take alternate key tiles and write two partial results for the merge
  bool key_split = false;
  int ngrp = 0, slots = 0;
  int split_len = 0;      // key tiles per forward chunk (>= nkt: no row is split)
  int nch_max = 1;        // most chunks one group can have
  bool split = false;
  size_t hdr = 0, slices = 0, stypes = 0, cls = 0;
  size_t row_nsl = 0, row_sl = 0, grp_cnt = 0, grp_ent = 0;
  size_t grp_nch = 0, grp_pslot = 0, chunks = 0, chunk_len = 0, chunk_order = 0, part_o = 0, part_lse = 0;
  size_t col_nsl = 0, col_sl = 0, col_cnt = 0, col_ent = 0, col_order = 0;
  size_t rowD = 0, lse2 = 0, dqacc = 0, tile_rank = 0, dq_sem = 0;
  size_t fwd_total = 0, bwd_total = 0;
};

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Softcap as a polynomial: tanh(y) / y ~ c0 + c1 y^2 + c2 y^4 + c3 y^6 on |y| <= kTanhPolyY.
// The coefficients are the output of fit_tanh_poly.py (next to this package's build script):
// a float64 minimax fit of the relative error (least squares on Chebyshev nodes, reweighted
// by the error until it equioscillates).  Evaluated by Horner's rule in float32, the product
// y * P(y^2) stays within 1.6e-7 of tanh(y), relative, over the whole interval.
constexpr double kTanhPolyY = 0.375;
constexpr double kTanhPoly[4] = {9.999999405e-01, -3.333197486e-01, 1.328450275e-01, -4.827228855e-02};
// Degree 5 (tanh(y) / y ~ c0 + c1 y^2 + c2 y^4 on the same interval, same fit): within 4.5e-6
// of tanh(y), relative.  The bounded-softcap forward kernel (softcap * log2(e) <= 60) uses it:
// there the capped logit's error stays below 4.5e-6 * 60 * tanh(0.375) < 1e-4 in the log2
// domain, a relative error of p below 7e-5, far inside the bf16 rounding of P (2^-9).
constexpr double kTanhPoly5[3] = {9.999957083e-01, -3.327806792e-01, 1.226476579e-01};

// The capped logit in the log2 domain, x(s) = C tanh(a s) with a = scale / softcap and
// C = softcap * log2(e), folded into one odd polynomial of the raw score:
// x(s) = s * sum_i q_i s^{2i}, q_i = C c_i a^{2i+1}, valid for |s| <= *slim.  *slim < 0 (the
// polynomial unused) without softcap or when a folded coefficient would not be a normal float.
inline void fold_cap_poly(float scale, float softcap, float (&q_out)[4], float* slim) {
  *slim = -1.0f;
  for (int i = 0; i < 4; ++i) q_out[i] = 0.0f;
  if (!(softcap > 0.0f) || !(scale > 0.0f)) return;
  const double a = static_cast<double>(scale) / softcap;
  const double C = static_cast<double>(softcap) * 1.4426950408889634;
  float q[4];
  for (int i = 0; i < 4; ++i) {
    q[i] = static_cast<float>(C * kTanhPoly[i] * std::pow(a, 2 * i + 1));
    if (!std::isnormal(q[i])) return;
  }
  const float s = static_cast<float>(kTanhPolyY / a * (1.0 - 1e-6));
  if (!std::isfinite(s) || !std::isfinite(s * s)) return;
  for (int i = 0; i < 4; ++i) q_out[i] = q[i];
  *slim = s;
}

// The degree-5 form of fold_cap_poly (kTanhPoly5), same interval and *slim.
inline void fold_cap_poly5(float scale, float softcap, float (&q_out)[3]) {
  for (int i = 0; i < 3; ++i) q_out[i] = 0.0f;
  if (!(softcap > 0.0f) || !(scale > 0.0f)) return;
  const double a = static_cast<double>(scale) / softcap;
  const double C = static_cast<double>(softcap) * 1.4426950408889634;
  for (int i = 0; i < 3; ++i) q_out[i] = static_cast<float>(C * kTanhPoly5[i] * std::pow(a, 2 * i + 1));
}

inline WsLayout make_layout(int64_t nq, int64_t nk, int hq, int hkv, int d, int R, bool key_split = false) {
  WsLayout L;
  L.nq = nq; L.nk = nk; L.hq = hq; L.hkv = hkv; L.d = d; L.R = R;
  L.nqt = static_cast<int>((nq + kTile - 1) / kTile);
  L.nkt = static_cast<int>((nk + kTile - 1) / kTile);
  const int G = hkv > 0 ? hq / hkv : 1;
  L.key_split = key_split;
  L.head_pair = !key_split && (G % 2 == 0);
  L.ngrp = (L.head_pair || key_split) ? L.nqt : (L.nqt + 1) / 2;
  L.slots = L.head_pair ? hq / 2 : hq;
  {
    const int64_t items = static_cast<int64_t>(L.ngrp) * L.slots;
    L.split_len = L.nkt > 0 ? L.nkt : 1;
    // The key split's items run both warpgroups on one chunk, so half as many chunks fill the
    // GPU; its rows (decoding: every query tile holds its own tokens' sequences) see about
    // nkt / nqt key tiles each, which is what the chunk length is cut from
    const int64_t target = key_split ? kSplitTarget / 2 : kSplitTarget;
    const int64_t row_len = key_split && L.nqt > 0 ? (L.nkt + L.nqt - 1) / L.nqt : L.nkt;
    if (items > 0 && items < target && L.nkt >= kMinSplitTiles) {
      const int64_t splits = (target + items - 1) / items;
      int64_t len = (row_len + splits - 1) / splits;
      if (len < kMinChunk) len = kMinChunk;
      if (len < L.nkt) {
        L.split_len = static_cast<int>(len);
        L.split = true;
      }
    }
    L.nch_max = (L.nkt + L.split_len - 1) / L.split_len;
    if (L.nch_max < 1) L.nch_max = 1;
    if (key_split) L.split = true;  // every item leaves two partial results
  }
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
  const size_t Rn = static_cast<size_t>(R > 0 ? R : 1);
  const size_t nqt = static_cast<size_t>(L.nqt > 0 ? L.nqt : 1), nkt = static_cast<size_t>(L.nkt > 0 ? L.nkt : 1);
  const size_t ngrp = static_cast<size_t>(L.ngrp > 0 ? L.ngrp : 1);
  L.hdr = take(64);
  L.slices = take(Rn * 16);
  L.stypes = take(Rn * 4);
  L.cls = take(nqt * nkt);
  const size_t common = o;
  L.row_nsl = take(nqt * 4);
  L.row_sl = take(nqt * kSliceCap * 4);
  L.grp_cnt = take(ngrp * 4);
  L.grp_ent = take(ngrp * nkt * 4);
  const size_t nch = ngrp * static_cast<size_t>(L.nch_max);
  L.grp_nch = take(ngrp * 4);
  L.grp_pslot = take(ngrp * 4);
  L.chunks = take(nch * 16);
  L.chunk_len = take(nch * 4);
  L.chunk_order = take(nch * 4);
  if (L.split) {  // partial O (fp32) and LSE of every chunk of a split group
    const size_t rows = nch * static_cast<size_t>(L.slots) * 2 * kTile;
    L.part_o = take(rows * static_cast<size_t>(d) * 4);
    L.part_lse = take(rows * 4);
  }
  L.fwd_total = o;
  o = common;
  L.col_nsl = take(nkt * 4);
  L.col_sl = take(nkt * kSliceCap * 4);
  L.col_cnt = take(nkt * 4);
  L.col_ent = take(nkt * nqt * 4);
  L.col_order = take(nkt * 4);
  // per-row statistics padded to whole tiles: [Hq, nqt * 128]
  L.rowD = take(static_cast<size_t>(hq) * nqt * kTile * 4);
  L.lse2 = take(static_cast<size_t>(hq) * nqt * kTile * 4);
  L.dqacc = take(static_cast<size_t>(nq > 0 ? nq : 1) * hq * d * 4);
  L.tile_rank = take(nqt * nkt * 4);                       // deterministic backward only
  L.dq_sem = take(static_cast<size_t>(hq) * nqt * 4);
  L.bwd_total = o;
  return L;
}

// Device-side view of the planner's output.
struct PlanView {
  int* hdr;              // [0] = number of valid slices
  int4* slices;          // (qs, qe, ks, ke) of valid, non-empty slices, input order
  int* stypes;           // type of each
  uint8_t* cls;          // [nqt, nkt]
  int* row_nsl;          // per query tile: number of slices touching it, -1 if > kSliceCap
  int* row_sl;           // [nqt, kSliceCap]
  int* grp_cnt;          // per forward group: number of work-list entries
  uint32_t* grp_ent;     // [ngrp, nkt]
  int* grp_nch;          // chunks of each group
  int* grp_pslot;        // first partial slot of a split group, -1 if not split
  int4* chunks;          // (group, first entry, end entry, partial slot or -1); hdr[1] = count
  int* chunk_len;
  int* chunk_order;      // chunks, longest first
  float* part_o;         // [slot][head slot][sub-tile][row][d] partial outputs of split chunks
  float* part_lse;       // [slot][head slot][sub-tile][row]
  int* col_nsl;          // per key tile: number of slices touching it, -1 if > kSliceCap
  int* col_sl;           // [nkt, kSliceCap]
  int* col_cnt;
  uint32_t* col_ent;     // [nkt, nqt]
  int* col_order;
};

// Programmatic dependent launch.  A kernel launched by launch_pdl may begin while the kernel
// before it in the stream is still running (once every block of that kernel has called
// pdl_launch_dependents or exited), which hides the launch gap between the short planner
// kernels and the attention kernel.  Such a kernel calls pdl_wait() before it touches global
// memory that an earlier kernel of the stream writes or reads: the wait returns once the
// kernel before it has completed and its writes are visible (and that kernel itself waited for
// the one before it, or was launched in plain stream order).  Without the launch attribute
// both calls do nothing.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

inline PlanView plan_view(const WsLayout& L, void* ws) {
  char* b = static_cast<char*>(ws);
  PlanView v;
  v.hdr = reinterpret_cast<int*>(b + L.hdr);
  v.slices = reinterpret_cast<int4*>(b + L.slices);
  v.stypes = reinterpret_cast<int*>(b + L.stypes);
  v.cls = reinterpret_cast<uint8_t*>(b + L.cls);
  v.row_nsl = reinterpret_cast<int*>(b + L.row_nsl);
  v.row_sl = reinterpret_cast<int*>(b + L.row_sl);
  v.grp_cnt = reinterpret_cast<int*>(b + L.grp_cnt);
  v.grp_ent = reinterpret_cast<uint32_t*>(b + L.grp_ent);
  v.grp_nch = reinterpret_cast<int*>(b + L.grp_nch);
  v.grp_pslot = reinterpret_cast<int*>(b + L.grp_pslot);
  v.chunks = reinterpret_cast<int4*>(b + L.chunks);
  v.chunk_len = reinterpret_cast<int*>(b + L.chunk_len);
  v.chunk_order = reinterpret_cast<int*>(b + L.chunk_order);
  v.part_o = L.split ? reinterpret_cast<float*>(b + L.part_o) : nullptr;
  v.part_lse = L.split ? reinterpret_cast<float*>(b + L.part_lse) : nullptr;
  v.col_nsl = reinterpret_cast<int*>(b + L.col_nsl);
  v.col_sl = reinterpret_cast<int*>(b + L.col_sl);
  v.col_cnt = reinterpret_cast<int*>(b + L.col_cnt);
  v.col_ent = reinterpret_cast<uint32_t*>(b + L.col_ent);
  v.col_order = reinterpret_cast<int*>(b + L.col_order);
  return v;
}

struct ProblemDims {
  int nq, nk, hq, hkv, d, nqt, nkt;
};

// Planner launches (ffa_plan.cu).  Each returns a cudaError_t of the launches.
// (dependent: launched as a programmatic dependent of the kernel before it, which must be
// one of this library's)
cudaError_t launch_plan_slices(const ProblemDims& P, const int32_t* q_ranges, const int32_t* k_ranges,
                               const int32_t* types, int R, const PlanView& v, int32_t* status, cudaStream_t s,
                               bool dependent = false);
cudaError_t launch_plan_rows(const ProblemDims& P, const WsLayout& L, const PlanView& v, cudaStream_t s);
cudaError_t launch_plan_cols(const ProblemDims& P, const PlanView& v, cudaStream_t s);
cudaError_t launch_plan_ranks(const ProblemDims& P, const PlanView& v, int* tile_rank, cudaStream_t s);

// Forward (ffa_fwd.cu)
struct FwdArgs {
  ProblemDims P;
  int head_pair, ngrp, slots, n_items;  // n_items: upper bound (chunks x slots) for the grid
  int split;
  int key_split = 0;  // WsLayout::key_split
  // key split only: the LSE merge writes O [nq / alibi_pack, hq * alibi_pack, d] and LSE
  // [hq * alibi_pack, nq / alibi_pack] here (the caller's token-major layout), not out / lse
  void* unpack_out = nullptr;
  float* unpack_lse = nullptr;
  float scale, softcap;
  const void *q, *k, *v;
  void* out;
  float* lse;
  const float* alibi = nullptr;  // per-query-head ALiBi slopes (device) or null
  // alibi_pack > 0 (decode): row r of query head h is token r / alibi_pack of the caller's
  // query head h * alibi_pack + r % alibi_pack; the bias uses that head's slope and that
  // token's position.
  int alibi_pack = 0;
  // Paged K/V (page_size > 0): k and v are physical page pools [n_pages * page_size, Hkv, d];
  // logical page j of the key sequence lives in physical page page_table[j].
  const int32_t* page_table = nullptr;
  int page_size = 0;
  int64_t n_pages = 0;
  PlanView plan;
  int32_t* status;
  uint64_t wait_limit_ns;
  int stall_test = 0;  // failure-detection test hook (FFA_TEST_STALL)
};
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s);

// Backward (ffa_bwd.cu)
struct BwdArgs {
  ProblemDims P;
  float scale, softcap;
  const void *q, *k, *v, *out, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  float* rowD;   // -D_i = -(dO_i . O_i), [Hq, nqt*128], 0 beyond Nq
  float* lse2;   // -LSE_i * log2(e), [Hq, nqt*128], -inf for empty rows and beyond Nq
  float* dqacc;  // float32 [Nq, Hq, d]
  const float* alibi = nullptr;
  int deterministic = 0;
  int* tile_rank = nullptr;  // [nqt, nkt]: position of key tile kt in query tile qt's list
  int* dq_sem = nullptr;     // [Hq, nqt]: dq contributions added so far
  PlanView plan;
  int32_t* status;
  uint64_t wait_limit_ns;
  int stall_test = 0;  // failure-detection test hook (FFA_TEST_STALL)
};
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s);

// The forward entry points' arguments (ffa_api.cu).  ffa_fwd_ex, ffa_fwd_paged, ffa_fwd_decode
// and ffa_fwd_noalloc fill one and share the checks and the launch sequence.
struct FwdCall {
  const ffa_shape* shape = nullptr;
  const void *q = nullptr, *k = nullptr, *v = nullptr;
  const int32_t *q_ranges = nullptr, *k_ranges = nullptr, *types = nullptr;
  int32_t n_ranges = 0;
  float softmax_scale = 0.0f, softcap = 0.0f;
  void* out = nullptr;
  float* lse = nullptr;
  int32_t* status = nullptr;
  void* stream = nullptr;
  const ffa_options* options = nullptr;
  bool paged = false;  // k, v are page pools reached through page_table
  const int32_t* page_table = nullptr;
  int page_size = 0;
  int64_t n_pages = 0;
  int alibi_pack = 0;  // > 0: rows are packed (token, query head) pairs (decode), see FwdArgs
  bool key_split = false;  // WsLayout::key_split (decode)
  void* unpack_out = nullptr;  // FwdArgs::unpack_out
  float* unpack_lse = nullptr;
  // the stream's last operation is a kernel of this library (decode: the packing kernel), so
  // the planner's first kernel may be launched as its programmatic dependent
  bool after_own_kernel = false;
};
// Shape check shared by the entry points (FFA_OK or the error code).
int check_shape(const ffa_shape* s, int32_t n_ranges);
// Options check shared by the entry points: reserved fields zero, slopes 4-byte aligned.
int check_options(const ffa_options* o);
// Host-detectable errors of a forward call (nothing is launched); fills the workspace layout.
int fwd_check(const FwdCall& c, WsLayout* layout);
// Device check, planner and kernels, with the planner's scratch at `scratch` (at least
// layout.fwd_total bytes, 256-byte aligned).  total_q must be > 0.
int fwd_launch(const FwdCall& c, const WsLayout& layout, void* scratch);
// fwd_check, then fwd_launch on a caller workspace.
int fwd_with_workspace(const FwdCall& c, void* workspace, size_t workspace_bytes);

// Optional events recorded around the main kernels (ffa_api.cu)
struct KernelEvents {
  cudaEvent_t fwd_start = nullptr, fwd_stop = nullptr, bwd_start = nullptr, bwd_stop = nullptr;
};
extern KernelEvents g_kernel_events;

// TMA descriptor creation (ffa_api.cu)
bool encode_tile_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                     uint32_t box_rows);
bool encode_tile_map_f32(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                         uint32_t box_rows);
int num_sms();

}  // namespace ffa
