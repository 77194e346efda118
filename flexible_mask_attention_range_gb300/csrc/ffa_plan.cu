// Range-to-tile planner.
//
// Turns the slice list (q_range, k_range, FULL|CAUSAL) into the data the attention kernels
// walk: the class of every tile of the global 128 x 128 grid (EMPTY / PARTIAL / FULL, the
// block classification of the Flex Attention paper, section 4, "Block Sparsity" and "Full
// Block Optimization"), per-row (forward) and per-column (backward) lists of the non-empty
// tiles with their classes (the paper's non-masked block counts and indices), the slices
// that touch each tile row / column (used to rebuild the element mask of PARTIAL tiles),
// and a longest-first order of the lists for load balance.  Zero-area slices (start == end
// in either range) are dropped first and cost nothing afterwards (MagiAttention issue #180,
// maintainer reply: the tile scheduler skips empty ranges).
//
// Visibility of (i, j) under slice [qs,qe) x [ks,ke): qs <= i < qe, ks <= j < ke and, for
// CAUSAL, j <= i + ke - qe (bottom-right alignment).  Several slices combine by OR.
#include "ffa_internal.h"
#include "../../include/ffa.h"

namespace ffa {
namespace {

__device__ int block_exclusive_scan(int v, int* warp_buf, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < nw ? warp_buf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_buf[lane] = s;
  }
  __syncthreads();
  const int excl = x - v + (w > 0 ? warp_buf[w - 1] : 0);
  *total = warp_buf[nw - 1];
  __syncthreads();
  return excl;
}

// ---------------------------------------------------------------- 1. slice filter
// One block: validate, drop zero-area slices, compact the rest in input order.
__global__ void __launch_bounds__(1024) plan_slices_kernel(const int32_t* __restrict__ qr,
                                                           const int32_t* __restrict__ kr,
                                                           const int32_t* __restrict__ ty, int R, int nq, int nk,
                                                           PlanView v, int32_t* status) {
  __shared__ int warp_buf[32];
  pdl_wait();  // (launched as a dependent of the decode packing kernel, which writes the slices)
  pdl_launch_dependents();
  int base = 0, bad = 0;
  for (int c = 0; c < R; c += blockDim.x) {
    const int r = c + threadIdx.x;
    int keep = 0;
    int4 s = make_int4(0, 0, 0, 0);
    int t = 0;
    if (r < R) {
      s = make_int4(qr[2 * r], qr[2 * r + 1], kr[2 * r], kr[2 * r + 1]);
      t = ty[r];
      const bool ok = 0 <= s.x && s.x <= s.y && s.y <= nq && 0 <= s.z && s.z <= s.w && s.w <= nk &&
                      (t == FFA_FULL || t == FFA_CAUSAL);
      if (!ok) bad = 1;
      keep = ok && s.x < s.y && s.z < s.w;
    }
    int total;
    const int pos = block_exclusive_scan(keep, warp_buf, &total);
    if (keep) {
      v.slices[base + pos] = s;
      v.stypes[base + pos] = t;
    }
    base += total;
  }
  if (bad && status != nullptr) atomicOr(status, FFA_STATUS_BAD_RANGE);
  if (threadIdx.x == 0) v.hdr[0] = base;
}

// ---------------------------------------------------------------- tile classification
// Is any pair of rows [r0,r1) x columns [c0,c1) visible under slice s?
__device__ __forceinline__ bool slice_touches(int4 s, int t, int r0, int r1, int c0, int c1) {
  const int a = max(s.x, r0), b = min(s.y, r1);
  if (a >= b) return false;
  const int hi_last = (t == FFA_CAUSAL) ? min(s.w, (b - 1) + s.w - s.y + 1) : s.w;
  return max(s.z, c0) < min(hi_last, c1);
}
// Is every pair of rows [r0,r1) x columns [c0,c1) visible under slice s alone?
__device__ __forceinline__ bool slice_covers(int4 s, int t, int r0, int r1, int c0, int c1) {
  if (s.x > r0 || s.y < r1 || s.z > c0) return false;
  const int hi_first = (t == FFA_CAUSAL) ? min(s.w, r0 + s.w - s.y + 1) : s.w;
  return hi_first >= c1;
}

// Slice list access: either staged in shared memory or read from the global compact list
// (when more slices touch the row/column than fit in shared memory).
struct SliceList {
  const int4* s;
  const int* t;
  int n;
};

// Class of the tile rows [r0,r1) x columns [c0,c1) under the union of the slices in `L`
// (which must contain every slice that touches the tile).
__device__ int classify_tile(const SliceList& L, int r0, int r1, int c0, int c1) {
  int n_touch = 0;
  for (int i = 0; i < L.n; ++i) {
    const int4 s = L.s[i];
    const int t = L.t[i];
    if (!slice_touches(s, t, r0, r1, c0, c1)) continue;
    if (slice_covers(s, t, r0, r1, c0, c1)) return FFA_TILE_FULL;
    ++n_touch;
  }
  if (n_touch == 0) return FFA_TILE_EMPTY;
  if (n_touch == 1) return FFA_TILE_PARTIAL;
  // Several slices touch the tile and none covers it alone: check, row by row, whether the
  // union of their visible intervals covers [c0, c1).
  for (int i = r0; i < r1; ++i) {
    int cur = c0;
    bool progressed = true;
    while (cur < c1 && progressed) {
      progressed = false;
      for (int k = 0; k < L.n; ++k) {
        const int4 s = L.s[k];
        if (i < s.x || i >= s.y) continue;
        const int hi = (L.t[k] == FFA_CAUSAL) ? min(s.w, i + s.w - s.y + 1) : s.w;
        if (s.z <= cur && hi > cur) {
          cur = hi;
          progressed = true;
        }
      }
    }
    if (cur < c1) return FFA_TILE_PARTIAL;
  }
  return FFA_TILE_FULL;
}

// Collect, in input order, the valid slices that touch rows [r0,r1) (by_col = false) or
// columns [c0,c1) (by_col = true) into shared memory (up to kSliceSmem) and into the global
// per-tile list (up to kSliceCap).  Returns the list to classify with.
__device__ SliceList gather_slices(const PlanView& v, int n_valid, bool by_col, int lo, int hi, int4* sm_s,
                                   int* sm_t, int* warp_buf, int* g_nsl, int* g_sl) {
  int count = 0;
  for (int c = 0; c < n_valid; c += blockDim.x) {
    const int r = c + threadIdx.x;
    int keep = 0;
    int4 s = make_int4(0, 0, 0, 0);
    int t = 0;
    if (r < n_valid) {
      s = v.slices[r];
      t = v.stypes[r];
      if (by_col) {
        // at the slice's last row every key of [ks, ke) is visible, for both types
        keep = s.z < hi && s.w > lo;
      } else {
        const int a = max(s.x, lo), b = min(s.y, hi);
        keep = a < b && ((t == FFA_FULL) || (min(s.w, b + s.w - s.y) > s.z));
      }
    }
    int total;
    const int pos = count + block_exclusive_scan(keep, warp_buf, &total);
    if (keep) {
      if (pos < kSliceSmem) {
        sm_s[pos] = s;
        sm_t[pos] = t;
      }
      if (pos < kSliceCap && g_sl != nullptr) g_sl[pos] = r;
    }
    count += total;
  }
  if (threadIdx.x == 0 && g_nsl != nullptr) *g_nsl = count <= kSliceCap ? count : -1;
  __syncthreads();
  SliceList L;
  if (count <= kSliceSmem) {
    L.s = sm_s;
    L.t = sm_t;
    L.n = count;
  } else {  // too many to stage: classify against every valid slice
    L.s = v.slices;
    L.t = v.stypes;
    L.n = n_valid;
  }
  return L;
}

// ---------------------------------------------------------------- 2. forward rows
// Classification: one block per (query tile, range of kPlanSpan key tiles), so that rows with
// many key tiles (decoding batches: one query tile, thousands of key tiles) are classified
// by many blocks.  The block with the first range also stores the tile row's slice list.
constexpr int kPlanSpan = 256;
__global__ void __launch_bounds__(256) plan_row_classes_kernel(ProblemDims P, PlanView v) {
  __shared__ int4 sm_s[kSliceSmem];
  __shared__ int sm_t[kSliceSmem];
  __shared__ int warp_buf[32];
  pdl_wait();
  pdl_launch_dependents();
  const int qt = blockIdx.x;
  const int k0 = blockIdx.y * kPlanSpan, k1 = min(P.nkt, k0 + kPlanSpan);
  const int n_valid = v.hdr[0];
  const int r0 = qt * kTile, r1 = min(r0 + kTile, P.nq);
  const bool first = blockIdx.y == 0;
  SliceList L = gather_slices(v, n_valid, false, r0, r1, sm_s, sm_t, warp_buf, first ? &v.row_nsl[qt] : nullptr,
                              first ? &v.row_sl[static_cast<size_t>(qt) * kSliceCap] : nullptr);
  for (int kt = k0 + threadIdx.x; kt < k1; kt += blockDim.x) {
    const int c0 = kt * kTile, c1 = min(c0 + kTile, P.nk);
    const int c = L.n ? classify_tile(L, r0, r1, c0, c1) : FFA_TILE_EMPTY;
    v.cls[static_cast<size_t>(qt) * P.nkt + kt] = static_cast<uint8_t>(c);
  }
}

// Work lists: one block per forward group.  head_pair: the group is one query tile; otherwise
// it is the query-tile pair (2g, 2g+1) whose work list is the union of both rows.  Entries:
// key tiles non-empty for either sub-tile, ascending, with both sub-tiles' classes.  A thread
// takes kListRun consecutive key tiles per pass, so a row of thousands of key tiles (a
// decoding batch) needs few block-wide scans.
constexpr int kListRun = 16;
__global__ void __launch_bounds__(256) plan_row_lists_kernel(ProblemDims P, int head_pair, PlanView v) {
  __shared__ int warp_buf[32];
  pdl_wait();
  pdl_launch_dependents();
  const int g = blockIdx.x;
  const int qa = head_pair ? g : 2 * g, qb = head_pair ? g : 2 * g + 1;
  const uint8_t* ca_row = v.cls + static_cast<size_t>(qa) * P.nkt;
  const uint8_t* cb_row = qb < P.nqt ? v.cls + static_cast<size_t>(qb) * P.nkt : nullptr;
  int count = 0;
  for (int c = 0; c < P.nkt; c += blockDim.x * kListRun) {
    const int kt0 = c + threadIdx.x * kListRun;
    uint8_t ca[kListRun], cb[kListRun];
    int n_keep = 0;
#pragma unroll
    for (int i = 0; i < kListRun; ++i) {
      const int kt = kt0 + i;
      ca[i] = kt < P.nkt ? ca_row[kt] : static_cast<uint8_t>(FFA_TILE_EMPTY);
      cb[i] = head_pair ? ca[i] : (cb_row != nullptr && kt < P.nkt ? cb_row[kt] : static_cast<uint8_t>(FFA_TILE_EMPTY));
      n_keep += (ca[i] | cb[i]) != 0;
    }
    int total;
    int pos = count + block_exclusive_scan(n_keep, warp_buf, &total);
#pragma unroll
    for (int i = 0; i < kListRun; ++i)
      if ((ca[i] | cb[i]) != 0) v.grp_ent[static_cast<size_t>(g) * P.nkt + pos++] = make_entry(kt0 + i, ca[i], cb[i]);
    count += total;
  }
  if (threadIdx.x == 0) v.grp_cnt[g] = count;
}

// ---------------------------------------------------------------- 2'. backward columns
// One block per key tile: slices touching the column, class of every tile in the column
// (same classification function, so the classes equal the row planner's), the list of
// non-empty query tiles, ascending.
__global__ void __launch_bounds__(256) plan_cols_kernel(ProblemDims P, PlanView v) {
  __shared__ int4 sm_s[kSliceSmem];
  __shared__ int sm_t[kSliceSmem];
  __shared__ int warp_buf[32];
  pdl_wait();
  pdl_launch_dependents();
  const int kt = blockIdx.x;
  const int n_valid = v.hdr[0];
  const int c0 = kt * kTile, c1 = min(c0 + kTile, P.nk);
  SliceList L = gather_slices(v, n_valid, true, c0, c1, sm_s, sm_t, warp_buf, &v.col_nsl[kt],
                              &v.col_sl[static_cast<size_t>(kt) * kSliceCap]);
  int count = 0;
  for (int c = 0; c < P.nqt; c += blockDim.x) {
    const int qt = c + threadIdx.x;
    int cl = 0;
    if (qt < P.nqt) {
      const int r0 = qt * kTile, r1 = min(r0 + kTile, P.nq);
      cl = L.n ? classify_tile(L, r0, r1, c0, c1) : FFA_TILE_EMPTY;
      v.cls[static_cast<size_t>(qt) * P.nkt + kt] = static_cast<uint8_t>(cl);
    }
    const int keep = cl != 0;
    int total;
    const int pos = count + block_exclusive_scan(keep, warp_buf, &total);
    if (keep) v.col_ent[static_cast<size_t>(kt) * P.nqt + pos] = make_entry(qt, cl, cl);
    count += total;
  }
  if (threadIdx.x == 0) v.col_cnt[kt] = count;
}

// ---------------------------------------------------------------- 3. longest-first order
// Counting sort (one block) of `n` lists by length (0..max_len), descending.  `hist` holds
// max_len + 1 ints of shared memory.
__device__ void counting_sort_desc(const int* __restrict__ len, int n, int max_len, int* __restrict__ order,
                                   int* hist, int* warp_buf) {
  for (int i = threadIdx.x; i <= max_len; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) atomicAdd(&hist[min(max(len[i], 0), max_len)], 1);
  __syncthreads();
  // start[c] = number of lists longer than c: exclusive scan over c = max_len .. 0
  const int per = (max_len + 1 + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * per;  // position in the reversed array
  int local = 0;
  for (int q = lo; q < min(lo + per, max_len + 1); ++q) local += hist[max_len - q];
  int total;
  int run = block_exclusive_scan(local, warp_buf, &total);
  for (int q = lo; q < min(lo + per, max_len + 1); ++q) {
    const int c = max_len - q;
    const int h = hist[c];
    hist[c] = run;
    run += h;
  }
  __syncthreads();
  // Placement is stable (equal lengths keep ascending index order), so items of similar
  // length that run at the same time are neighbours: for the backward, CTAs on neighbouring
  // key tiles add into neighbouring query tiles, which keeps the dq accumulator's working set
  // in L2.  Items go in chunks of blockDim.x, the warps of a chunk one after another; inside a
  // warp, lanes with the same length rank by lane order.
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int c = i < n ? min(max(len[i], 0), max_len) : -1;
    // only the warps that hold items of this pass take turns
    const int nw_pass = min(nw, (n - base + 31) >> 5);
    for (int ww = 0; ww < nw_pass; ++ww) {
      if (w == ww) {
        const unsigned peers = __match_any_sync(0xffffffffu, c);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int first = __ffs(peers) - 1;
        int start = 0;
        if (c >= 0) start = hist[c];
        __syncwarp();
        if (c >= 0) {
          order[start + rank] = i;
          if (lane == first) hist[c] = start + __popc(peers);
        }
        __syncwarp();
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(1024) plan_order_kernel(const int* __restrict__ cnt, int n, int max_len,
                                                          int* __restrict__ order) {
  extern __shared__ int hist[];
  __shared__ int warp_buf[32];
  pdl_wait();
  pdl_launch_dependents();
  counting_sort_desc(cnt, n, max_len, order, hist, warp_buf);
}

// ---------------------------------------------------------------- 3'. forward chunks
// One block.  Cuts every group's work list into chunks of at most `split_len` entries (one
// chunk, possibly empty, when the list is short), gives the chunks of split groups (every
// group when `all_split`: the key-split forward) consecutive partial-output slots, and orders
// all chunks longest first.  hdr[1] = chunks.
__global__ void __launch_bounds__(1024) plan_chunks_kernel(int ngrp, int split_len, int all_split, PlanView v) {
  extern __shared__ int hist[];  // split_len + 1
  __shared__ int warp_buf[32];
  pdl_wait();
  pdl_launch_dependents();
  int base = 0, pbase = 0;
  for (int c = 0; c < ngrp; c += blockDim.x) {
    const int g = c + threadIdx.x;
    int cnt = 0, nch = 0;
    if (g < ngrp) {
      cnt = v.grp_cnt[g];
      nch = max(1, (cnt + split_len - 1) / split_len);
    }
    const bool split = nch > 1 || (all_split && g < ngrp);
    int total, ptotal;
    const int pos = base + block_exclusive_scan(nch, warp_buf, &total);
    const int ppos = pbase + block_exclusive_scan(split ? nch : 0, warp_buf, &ptotal);
    if (g < ngrp) {
      v.grp_nch[g] = nch;
      v.grp_pslot[g] = split ? ppos : -1;
      for (int k = 0; k < nch; ++k) {
        const int e0 = k * split_len, e1 = min(cnt, e0 + split_len);
        v.chunks[pos + k] = make_int4(g, e0, e1, split ? ppos + k : -1);
        v.chunk_len[pos + k] = e1 - e0;
      }
    }
    base += total;
    pbase += ptotal;
  }
  if (threadIdx.x == 0) v.hdr[1] = base;
  __syncthreads();
  if (all_split) {  // key split: the chunks are all split_len long but each group's last, so
                    // their own order is already (nearly) longest first
    for (int i = threadIdx.x; i < base; i += blockDim.x) v.chunk_order[i] = i;
    return;
  }
  counting_sort_desc(v.chunk_len, base, split_len, v.chunk_order, hist, warp_buf);
}

// ---------------------------------------------------------------- 4. ranks (deterministic bwd)
// One block per query tile: tile_rank[qt][kt] = number of non-empty tiles (qt, kt' < kt).
__global__ void __launch_bounds__(256) plan_ranks_kernel(ProblemDims P, PlanView v, int* __restrict__ rank) {
  __shared__ int warp_buf[32];
  const int qt = blockIdx.x;
  int base = 0;
  for (int c = 0; c < P.nkt; c += blockDim.x) {
    const int kt = c + threadIdx.x;
    const int ne = (kt < P.nkt && v.cls[static_cast<size_t>(qt) * P.nkt + kt] != 0) ? 1 : 0;
    int total;
    const int pos = base + block_exclusive_scan(ne, warp_buf, &total);
    if (kt < P.nkt) rank[static_cast<size_t>(qt) * P.nkt + kt] = pos;
    base += total;
  }
}

}  // namespace

cudaError_t launch_plan_ranks(const ProblemDims& P, const PlanView& v, int* tile_rank, cudaStream_t s) {
  if (P.nqt == 0) return cudaSuccess;
  plan_ranks_kernel<<<P.nqt, 256, 0, s>>>(P, v, tile_rank);
  return cudaGetLastError();
}

cudaError_t launch_plan_slices(const ProblemDims& P, const int32_t* q_ranges, const int32_t* k_ranges,
                               const int32_t* types, int R, const PlanView& v, int32_t* status, cudaStream_t s,
                               bool dependent) {
  if (dependent)
    return launch_pdl(plan_slices_kernel, dim3(1), dim3(1024), 0, s, q_ranges, k_ranges, types, R,
                      static_cast<int>(P.nq), static_cast<int>(P.nk), v, status);
  plan_slices_kernel<<<1, 1024, 0, s>>>(q_ranges, k_ranges, types, R, P.nq, P.nk, v, status);
  return cudaGetLastError();
}

cudaError_t launch_plan_rows(const ProblemDims& P, const WsLayout& L, const PlanView& v, cudaStream_t s) {
  if (L.ngrp == 0) return cudaSuccess;
  // (each launched as a programmatic dependent of the planner kernel before it)
  cudaError_t e = launch_pdl(plan_row_classes_kernel, dim3(P.nqt, (P.nkt + kPlanSpan - 1) / kPlanSpan), dim3(256),
                             0, s, P, v);
  if (e != cudaSuccess) return e;
  // a key-split group is one query tile, as a head pair's is
  e = launch_pdl(plan_row_lists_kernel, dim3(L.ngrp), dim3(256), 0, s, P, (L.head_pair || L.key_split) ? 1 : 0, v);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(L.split_len + 1) * sizeof(int);
  return launch_pdl(plan_chunks_kernel, dim3(1), dim3(1024), smem, s, L.ngrp, L.split_len, L.key_split ? 1 : 0, v);
}

cudaError_t launch_plan_cols(const ProblemDims& P, const PlanView& v, cudaStream_t s) {
  if (P.nkt == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(plan_cols_kernel, dim3(P.nkt), dim3(256), 0, s, P, v);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(P.nqt + 1) * sizeof(int);
  return launch_pdl(plan_order_kernel, dim3(1), dim3(1024), smem, s, static_cast<const int*>(v.col_cnt), P.nkt, P.nqt,
                    v.col_order);
}

}  // namespace ffa
