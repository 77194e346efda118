// Forward kernel: fused range-masked softmax attention on sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes: for every query row i and head h, over the keys j visible to i under
// the union of the slices, O_i = sum_j softmax_j(x_ij) v_j and LSE_i = log sum_j e^{x_ij},
// with x = scale * q.k, or softcap * tanh(scale * q.k / softcap) when softcap > 0.  The
// interface is flex_flash_attn_func's (MagiAttention issue #180); the mask is applied by
// zeroing P where a pair is not visible, with no padding and no per-sequence descriptor
// edits, because the slice ranges index the flat packed tensors directly ("Questions about
// ex77 blackwell Flash attention", CUTLASS issue #2192: masking P during softmax instead of
// tensormap.replace or front padding).  Fully masked tiles are skipped and fully visible
// tiles skip the element mask (Flex Attention paper, section 4, "Full Block Optimization");
// later K/V tiles are prefetched while the current one is processed (same section, "Data
// Prefetching Pipeline").
//
// CTA = one work item = two 128-row query tiles sharing one K/V stream: either two query
// heads of one GQA group over the same query tile (G even) or two adjacent query tiles of
// one head (G odd).  Persistent grid (one CTA per SM), static longest-first snake schedule.
//
// Warp roles (384 threads):
//   warps 0-3  softmax warpgroup 0: row r of query tile 0 <-> TMEM lane r
//   warps 4-7  softmax warpgroup 1: query tile 1
//   warp 8     TMA producer (lane 0): Q tiles once per item, K/V tiles through a ring
//   warp 9     MMA issuer (lane 0): S_t = Q_t K^T into TMEM, O_t += P_t V with P_t read
//              from TMEM; owns the TMEM allocation
//   warps 10-11 idle: they complete the producer warpgroup, so that each SM sub-partition
//              (warp % 4) holds two softmax warps and one producer warp
// Registers: launched at 168 per thread; the producer warpgroup gives registers back
// (setmaxnreg.dec to kRegsProducer) and the softmax warpgroups take them
// (setmaxnreg.inc to kRegsSoftmax).  A warp's registers come from its own sub-partition's
// file, so the split must balance per sub-partition: 2 * kRegsSoftmax + kRegsProducer =
// 3 * 168, which also equals the block's launch total per warp triple.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).  P_t is
// written as bf16 over the first 64 columns of S_t.
//
// Online softmax in the log2 domain with a lazily updated reference max: the reference m
// of a row moves only when a new tile's max exceeds it by more than kTau (p <= 2^kTau), and
// only then is that row of O rescaled in TMEM.  Rows with no visible key so far use 0 as
// the reference (safe softmax), so fully masked rows end with l = 0: O = 0, LSE = -inf.
#include <cmath>
#include <mutex>
#include <type_traits>

#include "ffa_internal.h"
#include "ffa_ptx.cuh"
#include "../../include/ffa.h"

namespace ffa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kTau = 8.0f;
constexpr int kThreads = 384;
constexpr int kRegsLaunch = 168, kRegsSoftmax = 200, kRegsProducer = 104;
static_assert(2 * kRegsSoftmax + kRegsProducer == 3 * kRegsLaunch, "per sub-partition register split");
static_assert(kThreads * kRegsLaunch <= 65536, "launch register file");
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpDec = 10;  // item decoder: stages the next work items for the softmax warps
constexpr int kStageSl = 4;   // slices of a query tile staged with its item

// One work item as the softmax warpgroups need it, staged in shared memory by the decoder warp
// ahead of use: the item's chunk, the first list entry of each warpgroup, and per warpgroup
// the slices touching its query tile (when at most kStageSl do; else the warpgroup reads the
// planner's list from global memory).  A slot is released when the item's epilogue is done.
struct ItemStage {
  int4 ch;  // the item's chunk (group, first entry, end entry, partial slot)
  uint32_t e_first[2];
  int pad0[2];
  struct Tile {
    int nsl;  // row_nsl of the query tile (0 past the last query tile)
    int type[kStageSl];
    int pad[3];
    int4 s[kStageSl];
  } tile[2];
};
static_assert(sizeof(ItemStage) <= 256, "item staging slot");

template <int D>
struct FwdSmem {
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kTileBytes = kTile * D * 2;  // 128 rows x D bf16
  static constexpr int kBoxBytes = kTile * 128;     // 128 rows x 64 bf16 (one TMA box)
  static constexpr int kQ0 = 0;
  static constexpr int kQ1 = kTileBytes;
  static constexpr int kK = 2 * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  // output staging: one 128-row x 64-column bf16 box per softmax warpgroup
  static constexpr int kOst = kV + kStages * kTileBytes;
  static constexpr int kOstBytes = kTile * 128;
  // two work-item staging slots (ItemStage)
  static constexpr int kIt = kOst + 2 * kOstBytes;
  static constexpr int kItBytes = 256;
  static constexpr int kBar = kIt + 2 * kItBytes;
  // q_full, q_empty, k_full[S+1], v_full[S+1], kv_empty[S+1], s_full[2], p_full[2], o_full[2],
  // drain, stall (never arrived on; the failure-detection test waits on it), it_full[2],
  // it_empty[2].  Slot S exists with the key split only: its K sits in the (then unused)
  // second query tile, its V in the (then unused) output staging boxes.
  static constexpr int kNumBars = 2 + 3 * (kStages + 1) + 12;
  static_assert(kTileBytes <= 2 * kTile * 128, "a V tile fits the two output staging boxes");
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kAlloc = kTotal + 1024;
  static_assert(kAlloc <= 232448, "forward shared memory exceeds the per-block limit");
};

struct FwdParams {
  int nq, nk, hq, hkv, G, nqt, nkt;
  int head_pair, slots;
  float scale_log2;  // softmax_scale * log2(e)
  float cap_c;       // softcap * log2(e)
  float cap_k;       // 2 * softmax_scale * log2(e) / softcap
  // capped logit in the log2 domain as an odd polynomial of the raw score s,
  // x = s * (q0 + q1 s^2 + q2 s^4 + q3 s^6), valid for |s| <= cap_slim (< 0: never used)
  float cap_q[4];
  float cap_slim;
  // softcap bounds every logit to (-cap_c, cap_c) (log2 domain); when 2 * cap_c <= 120 the
  // exponentials of the softcap kernel use the fixed reference cap_c: 2^(x - cap_c) lies in
  // (2^-120, 1], so nothing overflows or flushes to zero and no row max or rescale is needed
  int cap_fixed;
  PlanView plan;
  __nv_bfloat16* out;
  float* lse;
  const float* alibi;  // per-query-head ALiBi slopes, or null
  int alibi_pack;      // > 0: packed decode rows (slope of head h*pack + r%pack, position r/pack)
  const int32_t* page_table;  // paged K/V: physical page of each logical page, else null
  int page_size, n_lpages, n_pages;
  int* status;
  uint64_t wait_limit_ns;
  int stall;  // failure-detection test: the first wait of every CTA never completes
  // key split (decode): an item is one query tile of one head; warpgroup w takes the key
  // tiles w, w + 2, ... of the chunk and writes its own partial result (sub-tile w).  (Last
  // member: placed earlier, it changed the register allocation of the other kernels.)
  int key_split;
  float cap_q5[3];  // cap_q in degree 5 (kTanhPoly5): the bounded-softcap kernel's form
  // Decoding (key split): the merge writes O and LSE straight into the caller's token-major
  // layout, row r of packed head h being token r / upack of query head h * upack + r % upack
  // (out [nq / upack, hq * upack, D], lse [hq * upack, nq / upack]); null: packed layout
  __nv_bfloat16* uout;
  float* ulse;
  int upack;
};

struct Item {
  int g, qt0, qt1, h0, h1, kvh, slot;
  int n;                 // key tiles of this chunk
  int pslot;             // partial-output slot when the group is split, else -1
  const uint32_t* ents;  // the chunk's work-list entries
};

// Work item -> (chunk of a group's work list, head slot).  Chunks are taken longest first.
__device__ __forceinline__ int4 item_chunk(const FwdParams& p, int item) {
  return p.plan.chunks[p.plan.chunk_order[item / p.slots]];
}
template <bool kKS>
__device__ __forceinline__ Item decode_item(const FwdParams& p, int item, int4 ch) {
  Item it;
  const int slot = item - (item / p.slots) * p.slots;
  it.g = ch.x;
  it.n = ch.z - ch.y;
  it.pslot = ch.w;
  it.ents = p.plan.grp_ent + static_cast<size_t>(it.g) * p.nkt + ch.y;
  it.slot = slot;
  if (kKS) {
    it.qt0 = it.qt1 = it.g;
    it.h0 = it.h1 = slot;
  } else if (p.head_pair) {
    it.qt0 = it.qt1 = it.g;
    it.h0 = 2 * slot;
    it.h1 = 2 * slot + 1;
  } else {
    it.qt0 = 2 * it.g;
    it.qt1 = 2 * it.g + 1;
    it.h0 = it.h1 = slot;
  }
  it.kvh = it.h0 / p.G;
  return it;
}
template <bool kKS>
__device__ __forceinline__ Item decode_item(const FwdParams& p, int item) {
  return decode_item<kKS>(p, item, item_chunk(p, item));
}

// Static snake schedule over the longest-first item order.
__device__ __forceinline__ int sched_item(int wave) {
  const int c = blockIdx.x, C = gridDim.x;
  return wave * C + ((wave & 1) ? (C - 1 - c) : c);
}

__device__ __forceinline__ void record_abort(volatile int* abort_flag, int* status) {
  *abort_flag = 1;
  if (status != nullptr) atomicOr(status, FFA_STATUS_TIMEOUT);
}

// bits [lo, hi) of a 128-bit row mask, lo/hi relative to the tile
__device__ __forceinline__ void set_bits(uint32_t (&w)[4], int lo, int hi) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int a = max(lo - 32 * k, 0), b = min(hi - 32 * k, 32);
    if (a < b) w[k] |= (b - a == 32) ? 0xffffffffu : (((1u << (b - a)) - 1u) << a);
  }
}

// Element mask of query row `row` over key tile kt: bit c set iff key kt*128+c is visible.
__device__ __forceinline__ void row_mask(const FwdParams& p, int cls, int row, int kt, int nsl, const int* sl,
                                         uint32_t (&w)[4]) {
  const int c0 = kt * kTile;
  if (cls == FFA_TILE_FULL) {
    w[0] = w[1] = w[2] = w[3] = 0xffffffffu;
  } else {
    w[0] = w[1] = w[2] = w[3] = 0u;
    if (cls == FFA_TILE_PARTIAL) {
      const int n = nsl >= 0 ? nsl : p.plan.hdr[0];
      for (int k = 0; k < n; ++k) {
        const int si = nsl >= 0 ? sl[k] : k;
        const int4 s = p.plan.slices[si];
        if (row < s.x || row >= s.y) continue;
        const int hi = (p.plan.stypes[si] == FFA_CAUSAL) ? min(s.w, row + s.w - s.y + 1) : s.w;
        const int lo_c = max(s.z, c0) - c0, hi_c = min(hi, c0 + kTile) - c0;
        if (lo_c < hi_c) set_bits(w, lo_c, hi_c);
      }
    }
  }
  const int valid = p.nk - c0;  // keys beyond Nk are never visible
  if (valid < kTile) {
    uint32_t t[4] = {0u, 0u, 0u, 0u};
    set_bits(t, 0, valid);
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] &= t[k];
  }
}

// Element mask of query row `row` over key tile kt from the row's visible intervals (when the
// union of its slices has at most two) or from the slice list.
__device__ __forceinline__ void tile_mask(const FwdParams& p, int cls, int row, int kt, const int* nsl_p, int qt,
                                          bool ivl_ok, int ilo0, int ihi0, int ilo1, int ihi1, uint32_t (&w)[4]) {
  if (ivl_ok && cls != FFA_TILE_FULL) {
    const int c0 = kt * kTile;
    w[0] = w[1] = w[2] = w[3] = 0u;
    if (cls == FFA_TILE_PARTIAL) {
      set_bits(w, max(ilo0 - c0, 0), min(ihi0 - c0, kTile));
      set_bits(w, max(ilo1 - c0, 0), min(ihi1 - c0, kTile));
    }
    const int valid = p.nk - c0;
    if (valid < kTile) {
      uint32_t t4[4] = {0u, 0u, 0u, 0u};
      set_bits(t4, 0, valid);
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] &= t4[k];
    }
  } else {
    // (the slice count is read here only: nsl_p points into the item's staging slot)
    const int* sl = p.plan.row_sl + static_cast<size_t>(qt < p.nqt ? qt : 0) * kSliceCap;
    row_mask(p, cls, row, kt, *nsl_p, sl, w);
  }
}

// The keys visible to query row `row` as at most two disjoint intervals (the union of the
// n slices that fetch(k, slice, type) gives, merged).  Returns false when the union needs
// more than two intervals.
template <class F>
__device__ __forceinline__ bool row_intervals_of(int row, int n, F&& fetch, int& lo0, int& hi0, int& lo1,
                                                 int& hi1) {
  lo0 = hi0 = lo1 = hi1 = 0;
  int n_ivl = 0;
  for (int k = 0; k < n; ++k) {
    int4 s;
    int type;
    fetch(k, s, type);
    if (row < s.x || row >= s.y) continue;
    const int lo = s.z;
    const int hi = (type == FFA_CAUSAL) ? min(s.w, row + s.w - s.y + 1) : s.w;
    if (lo >= hi) continue;
    // merge with an existing interval when they overlap or touch
    if (n_ivl > 0 && lo <= hi0 && hi >= lo0) {
      lo0 = min(lo0, lo);
      hi0 = max(hi0, hi);
    } else if (n_ivl > 1 && lo <= hi1 && hi >= lo1) {
      lo1 = min(lo1, lo);
      hi1 = max(hi1, hi);
    } else if (n_ivl == 0) {
      lo0 = lo; hi0 = hi; n_ivl = 1;
    } else if (n_ivl == 1) {
      lo1 = lo; hi1 = hi; n_ivl = 2;
    } else {
      return false;
    }
    if (n_ivl == 2 && lo0 <= hi1 && hi0 >= lo1) {  // the two became one
      lo0 = min(lo0, lo1);
      hi0 = max(hi0, hi1);
      lo1 = hi1 = 0;
      n_ivl = 1;
    }
  }
  return true;
}

// ... of the planner's slice list of the row's query tile (nsl < 0: every valid slice)
__device__ __forceinline__ bool row_intervals(const FwdParams& p, int row, int nsl, const int* sl, int& lo0,
                                              int& hi0, int& lo1, int& hi1) {
  const int n = nsl >= 0 ? nsl : p.plan.hdr[0];
  return row_intervals_of(
      row, n,
      [&](int k, int4& s, int& type) {
        const int si = nsl >= 0 ? sl[k] : k;
        s = p.plan.slices[si];
        type = p.plan.stypes[si];
      },
      lo0, hi0, lo1, hi1);
}

// tanh(y) * C in the log2 domain from one exp2 and one reciprocal:
// tanh(y) = 1 - 2 / (1 + e^{2y}); e^{2y} = 2^{s * cap_k}.
__device__ __forceinline__ float capped_log2(float s, float cap_c, float cap_k) {
  const float e = ex2_approx(s * cap_k);
  return fmaf(-2.0f * cap_c, rcp_approx(1.0f + e), cap_c);
}

template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t sQ, uint32_t sK, uint32_t idesc) {
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    const uint32_t off = (s / 4) * FwdSmem<D>::kBoxBytes + (s % 4) * 32;
    umma_ss(d_tmem, make_sdesc(sQ + off, 16, 1024, kSwizzle128B), make_sdesc(sK + off, 16, 1024, kSwizzle128B),
            idesc, s > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t a_tmem, uint32_t sV, uint32_t idesc,
                                        bool accumulate) {
#pragma unroll
  for (int s = 0; s < kTile / 16; ++s) {
    umma_ts(d_tmem, a_tmem + s * 8, make_sdesc(sV + s * 2048, FwdSmem<D>::kBoxBytes, 1024, kSwizzle128B), idesc,
            (accumulate || s > 0) ? 1u : 0u);
  }
}

// kFixed: bounded softcap (kCap, no bias, 2 * cap_c <= 120): fixed reference max cap_c.
// kKS: the key split (FwdParams::key_split), a separate instance so that the other kernels
// carry none of its bookkeeping
template <int D, bool kCap, bool kBias, bool kFixed, bool kKS>
__global__ void __launch_bounds__(kThreads, 1)
    ffa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const FwdParams p) {
  using SM = FwdSmem<D>;
  constexpr int S = SM::kStages;
  constexpr bool kPre = kCap || kBias;  // logits formed in the log2 domain before the row max
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* sm = smem_raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SM::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* v_full = bars + 2 + (S + 1);
  uint64_t* kv_empty = bars + 2 + 2 * (S + 1);
  uint64_t* s_full = bars + 2 + 3 * (S + 1);
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = s_full + 4;
  uint64_t* drain = s_full + 6;
  uint64_t* stall_bar = s_full + 7;
  uint64_t* it_full = s_full + 8;
  uint64_t* it_empty = s_full + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SM::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + SM::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s <= S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&o_full[t], 1);
    }
    mbar_init(drain, 1);
    mbar_init(stall_bar, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&it_full[t], 32);    // every lane of the decoder warp
      mbar_init(&it_empty[t], 256);  // every softmax thread
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint64_t lim = p.wait_limit_ns;
  pdl_wait();  // the planner's kernels have completed (everything above overlapped their tail)
  const int n_items = p.plan.hdr[1] * p.slots;  // chunks x head slots, written by the planner
  // K/V ring: S slots, one more with the key split (see FwdSmem)
  constexpr uint32_t nst = kKS ? S + 1 : S;
  auto k_slot = [&](uint32_t st) {
    return (kKS && st >= static_cast<uint32_t>(S)) ? static_cast<uint32_t>(SM::kQ1) : SM::kK + st * SM::kTileBytes;
  };
  auto v_slot = [&](uint32_t st) {
    return (kKS && st >= static_cast<uint32_t>(S)) ? static_cast<uint32_t>(SM::kOst) : SM::kV + st * SM::kTileBytes;
  };

  if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    reg_alloc<kRegsSoftmax>();
    const int wg = warp >> 2, q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tbase + lane_base + wg * 128;
    const uint32_t tO = tbase + lane_base + 256 + wg * D;
    uint8_t* ost = sm + SM::kOst + wg * SM::kOstBytes;  // this warpgroup's output staging box
    const bool leader = (q4 == 0 && lane == 0);         // issues the warpgroup's output copies
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    for (int wave = 0; ok; ++wave) {
      const int item = sched_item(wave);
      if (item >= n_items) break;
      // the item and its first entries from the decoder's slot; this row's visible keys from
      // the slices staged there
      const int ib = wave & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&it_full[ib], (wave >> 1) & 1u, abort_flag, lim));
      if (!ok) break;
      const ItemStage* ist = reinterpret_cast<const ItemStage*>(sm + SM::kIt) + ib;
      const Item it = decode_item<kKS>(p, item, ist->ch);
      const int n = it.n;
      const int qt = wg ? it.qt1 : it.qt0;
      const int h = wg ? it.h1 : it.h0;
      const int row = qt * kTile + r;
      const bool in_rows = row < p.nq;
      const int nsl = ist->tile[wg].nsl;
      // this row's visible keys once per item; PARTIAL tiles clip them instead of rereading
      // the slice list (rows whose union needs more than two intervals use the list)
      int ilo0, ihi0, ilo1, ihi1;
      bool ivl_ok;
      if (nsl >= 0 && nsl <= kStageSl) {
        ivl_ok = row_intervals_of(
            row, nsl,
            [&](int k, int4& s4, int& type) {
              s4 = ist->tile[wg].s[k];
              type = ist->tile[wg].type[k];
            },
            ilo0, ihi0, ilo1, ihi1);
      } else {
        const int* sl = p.plan.row_sl + static_cast<size_t>(qt < p.nqt ? qt : 0) * kSliceCap;
        ivl_ok = row_intervals(p, row, nsl, sl, ilo0, ihi0, ilo1, ihi1);
      }
      const uint32_t e_first = ist->e_first[kKS ? wg : 0];
      // this warpgroup's key tiles: entries j0, j0 + step, ... of the chunk (key split: every
      // other one, starting at the warpgroup's index)
      constexpr int step = kKS ? 2 : 1;
      const int j0 = kKS ? wg : 0;
      const int n_w = kKS ? (n + 1 - wg) / 2 : n;
      const int csub = kKS ? 0 : wg;  // which sub-tile's class an entry gives
      if (n_w == 0) {  // nothing visible here: O = 0, LSE = -inf (a partial result of that value)
        if (in_rows) {
          if (!kKS) {  // (a chunk of a split row is never empty)
            uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(row) * p.hq + h) * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[static_cast<size_t>(h) * p.nq + row] = -INFINITY;
          } else {
            const size_t prow = (static_cast<size_t>(it.pslot) * p.slots + it.slot) * 2 * kTile + wg * kTile + r;
            float4* dst = reinterpret_cast<float4*>(p.plan.part_o + prow * D);
#pragma unroll
            for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            p.plan.part_lse[prow] = -INFINITY;
          }
        }
        mbar_arrive(&it_empty[ib]);
        continue;
      }
      const uint32_t* ents = it.ents;
      // ALiBi slope and query position of this row (packed decode rows: the row's own query
      // head and token)
      int a_head = h, a_pos = row;
      if (kBias && p.alibi_pack > 0) {
        a_head = h * p.alibi_pack + row % p.alibi_pack;
        a_pos = row / p.alibi_pack;
      }
      const float slope_log2 = kBias ? p.alibi[a_head] * kLog2e : 0.0f;
      uint32_t e_next = e_first;
      // l_run: sum of the fp32 p (for the LSE); r_run: sum of the bf16-rounded p that the PV
      // MMA actually multiplies (normalising O by it keeps the weights a convex combination,
      // so a dominant key is reproduced exactly even when the reference max is stale).  On
      // tiles without ALiBi and without a mask r_run takes the fp32 sum plus the rounding error
      // of the tile's largest p only: that is the term that matters when one key dominates,
      // at a fraction of the cost of rounding every p back
      // m_run: the reference max of the exponentials (log2 domain); a bounded softcap fixes it
      float m_run = kFixed ? p.cap_c : -INFINITY, l_run = 0.0f, r_run = 0.0f;
      for (int jj = 0; jj < n_w; ++jj) {
        const int j = j0 + jj * step;
        const uint32_t e = e_next;
        if (jj + 1 < n_w) e_next = ents[j + step];  // in flight while this tile is processed
        const int kt = entry_idx(e);
        const int cls = entry_cls(e, csub);
        uint64_t* sb = (p.stall && s_cnt == 0) ? stall_bar : &s_full[wg];
        ok = __all_sync(0xffffffffu, mbar_wait(sb, s_cnt & 1u, abort_flag, lim));
        if (!ok) break;
        ++s_cnt;
        tc_fence_after();
        uint32_t sv[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, sv[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence(sv[c]);
        const bool masked = (cls != FFA_TILE_FULL) || (kt * kTile + kTile > p.nk);
        // element mask of this row over the tile (bit c: key kt * 128 + c visible)
        uint32_t wm[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        if (!kFixed && masked) {  // (the bounded-softcap kernel masks inside its own pass)
          tile_mask(p, cls, row, kt, &ist->tile[wg].nsl, qt, ivl_ok, ilo0, ihi0, ilo1, ihi1, wm);
          // none of the warp's 32 rows sees a key of this tile (a decoding batch's tile
          // belongs to one sequence; rows past the end): P = 0, nothing else changes
          if (__all_sync(0xffffffffu, (wm[0] | wm[1] | wm[2] | wm[3]) == 0u)) {
            const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) tmem_st16(tS + 16 * c4, z);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[wg]);
            continue;
          }
        }
        bool rescale = false;  // the reference max moved: O rows are scaled by alpha
        float alpha = 1.0f;
        if constexpr (kFixed) {
          // Bounded softcap: every capped logit lies in (-cap_c, cap_c), so the exponentials
          // use the fixed reference m_run = cap_c and no row max is taken.  The tanh
          // polynomial forms the logits inside the exponential pass when every raw score of
          // the warp's rows lies where it holds (tanh is odd: a bound on |s|); otherwise the
          // exact transform runs first.  Masked entries are set to -inf after the transform.
          float hi[4], lo[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            hi[u] = -INFINITY;
            lo[u] = INFINITY;
          }
#pragma unroll
          for (int c = 0; c < 128; c += 2) {
            const float a = __uint_as_float(sv[c >> 5][c & 31]), b = __uint_as_float(sv[c >> 5][(c & 31) + 1]);
            hi[(c >> 1) & 3] = fmax3(hi[(c >> 1) & 3], a, b);
            lo[(c >> 1) & 3] = fmin3(lo[(c >> 1) & 3], a, b);
          }
          const float smax = fmaxf(fmaxf(hi[0], hi[1]), fmaxf(hi[2], hi[3]));
          const float smin = fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3]));
          const bool poly_f = __all_sync(0xffffffffu, fmaxf(smax, -smin) <= p.cap_slim);
          if (!poly_f) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              sv[c >> 5][c & 31] =
                  __float_as_uint(capped_log2(__uint_as_float(sv[c >> 5][c & 31]), p.cap_c, p.cap_k));
          }
          uint32_t w[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
          if (masked) tile_mask(p, cls, row, kt, &ist->tile[wg].nsl, qt, ivl_ok, ilo0, ihi0, ilo1, ihi1, w);
          float2 sum2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
          float2 sumr2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
          const float2 nm2 = make_float2(-p.cap_c, -p.cap_c);
          auto exp_fixed = [&](auto poly_tag, auto mask_tag) {
            constexpr bool kP = decltype(poly_tag)::value, kM = decltype(mask_tag)::value;
            // the degree-5 polynomial (four packed instructions per pair of scores)
            const float2 q0 = make_float2(p.cap_q5[0], p.cap_q5[0]), q1 = make_float2(p.cap_q5[1], p.cap_q5[1]);
            const float2 q2 = make_float2(p.cap_q5[2], p.cap_q5[2]);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              uint32_t pk[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const float2 s2 = make_float2(__uint_as_float(sv[c4][2 * k]), __uint_as_float(sv[c4][2 * k + 1]));
                float2 y;
                if constexpr (kP) {
                  const float2 t = mul2(s2, s2);
                  y = fma2(s2, fma2(fma2(q2, t, q1), t, q0), nm2);
                } else {
                  y = add2(s2, nm2);
                }
                if constexpr (kM) {
                  y.x = ((w[c4] >> (2 * k)) & 1u) ? y.x : -INFINITY;
                  y.y = ((w[c4] >> (2 * k + 1)) & 1u) ? y.y : -INFINITY;
                }
                const float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
                sum2[k & 1] = add2(sum2[k & 1], make_float2(p0, p1));
                pk[k] = pack_bf16x2(p0, p1);
                if constexpr (kM)
                  sumr2[k & 1] = add2(sumr2[k & 1], make_float2(__uint_as_float(pk[k] << 16),
                                                                __uint_as_float(pk[k] & 0xffff0000u)));
              }
              tmem_st16(tS + 16 * c4, pk);
            }
          };
          if (poly_f) {
            if (masked) {
              exp_fixed(std::true_type{}, std::true_type{});
            } else {
              exp_fixed(std::true_type{}, std::false_type{});
            }
          } else {
            if (masked) {
              exp_fixed(std::false_type{}, std::true_type{});
            } else {
              exp_fixed(std::false_type{}, std::false_type{});
            }
          }
          const float tile_l = (sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y);
          l_run += tile_l;
          if (masked) {
            r_run += (sumr2[0].x + sumr2[0].y) + (sumr2[1].x + sumr2[1].y);
          } else {
            // the sum of the bf16 values the PV MMA uses, as the fp32 sum plus the rounding
            // error of the tile's largest p (the only one that can dominate a row), recomputed
            // with the exponential pass's exact operations
            const float t = smax * smax;
            const float y_max = poly_f ? fmaf(smax, fmaf(fmaf(p.cap_q5[2], t, p.cap_q5[1]), t, p.cap_q5[0]), -p.cap_c)
                                       : capped_log2(smax, p.cap_c, p.cap_k) + (-p.cap_c);
            const float p_max = ex2_approx(y_max);
            r_run += tile_l + (__uint_as_float(pack_bf16x2(p_max, 0.0f) << 16) - p_max);
          }
        } else {
          // ALiBi in the log2 domain: slope * log2(e) * (key - row) = bbase + slope * log2(e) * c
          const float bbase = kBias ? slope_log2 * static_cast<float>(kt * kTile - a_pos) : 0.0f;
          // Softcap on a fully visible tile: when every raw score of the warp's rows lies where
          // the tanh polynomial holds, the logits are formed inside the exponential pass (FMA
          // pipe only), and the row max is the polynomial at the raw max, the transform being
          // increasing there.  Otherwise (and on masked tiles) the exact transform runs first.
          constexpr bool kPolyCap = kCap && !kBias;
          bool poly = false;
          float mx = -INFINITY, smax_p = -INFINITY;
          if (kPolyCap && !masked) {
            float hi[4], lo[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              hi[u] = -INFINITY;
              lo[u] = INFINITY;
            }
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
              const float a = __uint_as_float(sv[c >> 5][c & 31]), b = __uint_as_float(sv[c >> 5][(c & 31) + 1]);
              hi[(c >> 1) & 3] = fmax3(hi[(c >> 1) & 3], a, b);
              lo[(c >> 1) & 3] = fmin3(lo[(c >> 1) & 3], a, b);
            }
            const float smax = fmaxf(fmaxf(hi[0], hi[1]), fmaxf(hi[2], hi[3]));
            const float smin = fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3]));
            poly = __all_sync(0xffffffffu, fmaxf(smax, -smin) <= p.cap_slim);
            if (poly) {
              const float t = smax * smax;
              mx = smax * fmaf(fmaf(fmaf(p.cap_q[3], t, p.cap_q[2]), t, p.cap_q[1]), t, p.cap_q[0]);
              smax_p = smax;
            }
          }
          // row max: eight independent partial maxima when the logits are formed first (a
          // longer transform per element), one chain otherwise (measured faster there)
          constexpr int kMx = kPre ? 8 : 1;
          float mxs[kMx];
#pragma unroll
          for (int u = 0; u < kMx; ++u) mxs[u] = -INFINITY;
          if (poly) {
            // the maximum is known
          } else if (masked) {
            const uint32_t(&w)[4] = wm;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              float x = __uint_as_float(sv[c >> 5][c & 31]);
              if (kCap) x = capped_log2(x, p.cap_c, p.cap_k);
              if (kBias) x = (kCap ? x : x * p.scale_log2) + fmaf(slope_log2, static_cast<float>(c), bbase);
              x = ((w[c >> 5] >> (c & 31)) & 1u) ? x : -INFINITY;
              sv[c >> 5][c & 31] = __float_as_uint(x);
              mxs[c % kMx] = fmaxf(mxs[c % kMx], x);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              float x = __uint_as_float(sv[c >> 5][c & 31]);
              if (kCap) x = capped_log2(x, p.cap_c, p.cap_k);
              if (kBias) x = (kCap ? x : x * p.scale_log2) + fmaf(slope_log2, static_cast<float>(c), bbase);
              if (kPre) sv[c >> 5][c & 31] = __float_as_uint(x);
              mxs[c % kMx] = fmaxf(mxs[c % kMx], x);
            }
          }
          if (!poly) {
            mx = mxs[0];
#pragma unroll
            for (int u = 1; u < kMx; ++u) mx = fmaxf(mx, mxs[u]);
          }
          const float m_tile = kPre ? mx : mx * p.scale_log2;
          const bool need = m_tile > m_run + kTau;
          rescale = need && (m_run != -INFINITY);
          alpha = rescale ? ex2_approx(m_run - m_tile) : 1.0f;
          if (need) m_run = m_tile;
          if (rescale) {
            l_run *= alpha;
            r_run *= alpha;
          }
          const float neg_m = (m_run == -INFINITY) ? 0.0f : -m_run;
          // exponentials two columns at a time: the argument and both running sums use packed
          // fp32 pair instructions; two accumulator pairs each shorten the addition chains
          float2 sum2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
          float2 sumr2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
          const float sc = kPre ? 1.0f : p.scale_log2;
          const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(neg_m, neg_m);
          auto exp_pass = [&](auto poly_tag) {
            constexpr bool kP = decltype(poly_tag)::value;
            float2 q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = kP ? make_float2(p.cap_q[i], p.cap_q[i]) : make_float2(0.0f, 0.0f);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              uint32_t pk[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const float2 s2 = make_float2(__uint_as_float(sv[c4][2 * k]), __uint_as_float(sv[c4][2 * k + 1]));
                float2 y;
                if constexpr (kP) {
                  const float2 t = mul2(s2, s2);
                  const float2 w = fma2(fma2(fma2(q[3], t, q[2]), t, q[1]), t, q[0]);
                  y = fma2(s2, w, nm2);
                } else {
                  y = fma2(s2, sc2, nm2);
                }
                const float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
                sum2[k & 1] = add2(sum2[k & 1], make_float2(p0, p1));
                pk[k] = pack_bf16x2(p0, p1);
                if constexpr (kBias)
                  sumr2[k & 1] = add2(sumr2[k & 1], make_float2(__uint_as_float(pk[k] << 16),
                                                                __uint_as_float(pk[k] & 0xffff0000u)));
              }
              tmem_st16(tS + 16 * c4, pk);
            }
          };
          if constexpr (kPolyCap) {
            if (poly) {
              exp_pass(std::true_type{});
            } else {
              exp_pass(std::false_type{});
            }
          } else {
            exp_pass(std::false_type{});
          }
          const float tile_l = (sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y);
          l_run += tile_l;
          if constexpr (kBias) {
            r_run += (sumr2[0].x + sumr2[0].y) + (sumr2[1].x + sumr2[1].y);
          } else {
            // the fp32 sum plus the rounding error of the tile's largest p, recomputed with the
            // exponential pass's exact operations (its argument is the largest one)
            float y_max;
            if (poly) {
              const float t = smax_p * smax_p;
              y_max = fmaf(smax_p, fmaf(fmaf(fmaf(p.cap_q[3], t, p.cap_q[2]), t, p.cap_q[1]), t, p.cap_q[0]), neg_m);
            } else {
              y_max = fmaf(mx, sc, neg_m);
            }
            const float p_max = ex2_approx(y_max);
            r_run += tile_l + (__uint_as_float(pack_bf16x2(p_max, 0.0f) << 16) - p_max);
          }
        }
        // Rescale this row of O when its reference max moved.  O is stable here: the S MMA
        // that produced this tile was issued after the previous PV MMA, and the next PV MMA
        // waits for this warpgroup's p_full arrival below.
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st32(tO + 32 * c, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[wg]);
      }
      // epilogue: O / l -> bf16, LSE.  The warpgroup's four warps agree on going on (a warp
      // whose wait ran out still reaches the barrier, after raising the abort flag)
      if (!ok) record_abort(abort_flag, p.status);
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_full[wg], o_cnt & 1u, abort_flag, lim));
      ok = named_bar_and(1 + wg, 128, ok);
      if (!ok) break;
      ++o_cnt;
      tc_fence_after();
      const float inv_l = r_run > 0.0f ? 1.0f / r_run : 0.0f;
      const float lse_row = l_run > 0.0f ? (m_run + lg2_approx(l_run)) * kLn2 : -INFINITY;
      // the item's head and partial slot, decoded again from the staging slot here rather than
      // held in registers through the tile loop
      const Item ie = decode_item<kKS>(p, item, ist->ch);
      const int he = wg ? ie.h1 : ie.h0;
      if (ie.pslot < 0) {
        // O through shared memory: each 64-column box of the tile is written row by row into
        // the staging box (128-byte swizzle: 16-byte chunk k of row r at chunk k ^ (r % 8)) and
        // stored with one TMA copy, which leaves out the rows past the end
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          // the box's 64 columns are read and packed while the previous copy out of the
          // staging box may still be reading it
          uint32_t o[2][32];
          tmem_ld32(tO + 64 * b, o[0]);
          tmem_ld32(tO + 64 * b + 32, o[1]);
          tmem_wait_ld();
          reg_fence(o[0]);
          reg_fence(o[1]);
          uint4 v[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t* ok8 = o[k >> 2] + 8 * (k & 3);
            v[k].x = pack_bf16x2(__uint_as_float(ok8[0]) * inv_l, __uint_as_float(ok8[1]) * inv_l);
            v[k].y = pack_bf16x2(__uint_as_float(ok8[2]) * inv_l, __uint_as_float(ok8[3]) * inv_l);
            v[k].z = pack_bf16x2(__uint_as_float(ok8[4]) * inv_l, __uint_as_float(ok8[5]) * inv_l);
            v[k].w = pack_bf16x2(__uint_as_float(ok8[6]) * inv_l, __uint_as_float(ok8[7]) * inv_l);
          }
          // the previous copy out of the staging box has read it
          if (leader) bulk_wait_group_read<0>();
          named_bar_sync(1 + wg, 128);
#pragma unroll
          for (int k = 0; k < 8; ++k) *reinterpret_cast<uint4*>(ost + r * 128 + ((k ^ (r & 7)) * 16)) = v[k];
          fence_proxy_async_smem();
          named_bar_sync(1 + wg, 128);
          if (leader) {
            tma_store_2d(&tmO, ost, he * D + 64 * b, qt * kTile);
            bulk_commit_group();
          }
        }
        if (in_rows) p.lse[static_cast<size_t>(he) * p.nq + row] = lse_row;
      } else {
        // one chunk of a split row: normalised partial O (fp32) and its LSE for the merge
        // (rows past the end are never merged)
        const size_t prow = (static_cast<size_t>(ie.pslot) * p.slots + ie.slot) * 2 * kTile + wg * kTile + r;
        float4* dst = reinterpret_cast<float4*>(p.plan.part_o + prow * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_wait_ld();
          reg_fence(o);
          if (in_rows) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              dst[8 * c + k] = make_float4(__uint_as_float(o[4 * k]) * inv_l, __uint_as_float(o[4 * k + 1]) * inv_l,
                                           __uint_as_float(o[4 * k + 2]) * inv_l,
                                           __uint_as_float(o[4 * k + 3]) * inv_l);
          }
        }
        if (in_rows) p.plan.part_lse[prow] = lse_row;
      }
      mbar_arrive(&it_empty[ib]);  // the item's staging slot is no longer read
    }
    if (!ok) record_abort(abort_flag, p.status);
    if (leader) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // output copies done
  } else {
  reg_dealloc<kRegsProducer>();
  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it_cnt = 0;
      uint32_t gk = 0;
      bool ok = true;
      int last_use[S + 1];
      for (int s = 0; s <= S; ++s) last_use[s] = -1;
      int last_q = -1;
      for (int wave = 0; ok; ++wave) {
        const int item = sched_item(wave);
        if (item >= n_items) break;
        const Item it = decode_item<kKS>(p, item);
        const int n = it.n;
        if (n == 0) continue;
        if (it_cnt > 0) {
          ok = mbar_wait(q_empty, (it_cnt - 1) & 1u, abort_flag, lim);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(q_full, (kKS ? 1 : 2) * SM::kTileBytes);
        last_q = static_cast<int>(it_cnt);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(sm + SM::kQ0 + b * SM::kBoxBytes, &tmQ, q_full, it.h0 * D + 64 * b, it.qt0 * kTile);
          if (!kKS)  // (key split: both warpgroups' S use the one query tile)
            tma_load_2d(sm + SM::kQ1 + b * SM::kBoxBytes, &tmQ, q_full, it.h1 * D + 64 * b, it.qt1 * kTile);
        }
        const uint32_t* ents = it.ents;
        for (int j = 0; j < n; ++j) {
          const int kt = entry_idx(ents[j]);
          const uint32_t st = gk % nst, u = gk / nst;
          if (u > 0) {
            ok = mbar_wait(&kv_empty[st], (u - 1) & 1u, abort_flag, lim);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(&k_full[st], SM::kTileBytes);
          mbar_arrive_expect_tx(&v_full[st], SM::kTileBytes);
          if (p.page_table == nullptr) {
#pragma unroll
            for (int b = 0; b < D / 64; ++b)
              tma_load_2d(sm + k_slot(st) + b * SM::kBoxBytes, &tmK, &k_full[st],
                          it.kvh * D + 64 * b, kt * kTile);
#pragma unroll
            for (int b = 0; b < D / 64; ++b)
              tma_load_2d(sm + v_slot(st) + b * SM::kBoxBytes, &tmV, &v_full[st],
                          it.kvh * D + 64 * b, kt * kTile);
          } else {
            // Paged K/V (FlexAttention paper, section 5, Paged Attention): the tile's 128
            // logical keys are 128 / page_size pages, each fetched from its physical page into
            // its rows of the tile (row offsets are multiples of 8, so the 128-byte swizzle
            // pattern is the one a whole-tile load gives).  Logical pages past the table,
            // and table entries outside the pool (reported), load zeros: the box starts past
            // the last physical row.
            const int per = kTile / p.page_size;
            for (int pj = 0; pj < per; ++pj) {
              const int lp = kt * per + pj;
              int y = p.n_pages * p.page_size;
              if (lp < p.n_lpages) {
                const int phys = p.page_table[lp];
                if (phys >= 0 && phys < p.n_pages) {
                  y = phys * p.page_size;
                } else if (p.status != nullptr) {
                  atomicOr(p.status, FFA_STATUS_BAD_PAGE);
                }
              }
              const uint32_t roff = static_cast<uint32_t>(pj * p.page_size) * 128u;
#pragma unroll
              for (int b = 0; b < D / 64; ++b) {
                tma_load_2d(sm + k_slot(st) + b * SM::kBoxBytes + roff, &tmK, &k_full[st],
                            it.kvh * D + 64 * b, y);
                tma_load_2d(sm + v_slot(st) + b * SM::kBoxBytes + roff, &tmV, &v_full[st],
                            it.kvh * D + 64 * b, y);
              }
            }
          }
          last_use[st] = static_cast<int>(u);
          ++gk;
        }
        ++it_cnt;
      }
      if (!ok) {
        record_abort(abort_flag, p.status);
        // let the copies already issued land before the CTA's shared memory is released
        const uint64_t short_lim = 100000000ull;
        if (last_q >= 0) mbar_wait(q_full, static_cast<uint32_t>(last_q) & 1u, nullptr, short_lim);
        for (int s = 0; s <= S; ++s) {
          if (last_use[s] < 0) continue;
          mbar_wait(&k_full[s], static_cast<uint32_t>(last_use[s]) & 1u, nullptr, short_lim);
          mbar_wait(&v_full[s], static_cast<uint32_t>(last_use[s]) & 1u, nullptr, short_lim);
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, D, false, true);
      const uint32_t sQ0 = smem_u32(sm + SM::kQ0), sQ1 = smem_u32(sm + SM::kQ1);
      const uint32_t sbase = smem_u32(sm);
      const uint32_t tS0 = tbase, tS1 = tbase + 128, tO0 = tbase + 256, tO1 = tbase + 256 + D;
      uint32_t it_cnt = 0, gk = 0, pc0 = 0, pc1 = 0;
      bool ok = true;
      for (int wave = 0; ok; ++wave) {
        const int item = sched_item(wave);
        if (item >= n_items) break;
        const Item it = decode_item<kKS>(p, item);
        const int n = it.n;
        if (n == 0) continue;
        ok = mbar_wait(q_full, it_cnt & 1u, abort_flag, lim);
        if (!ok) break;
        if constexpr (kKS) {
          // warpgroup 0 takes the chunk's key tiles 0, 2, 4, ..., warpgroup 1 the tiles 1, 3,
          // ...; both multiply the one query tile (Q0).  A tile's K/V slot is released after
          // its own PV.
          const int n1 = n / 2, n0 = n - n1;
          for (int t = 0; t < 2 && t < n; ++t) {  // the first S of each warpgroup
            const uint32_t g = gk + t, st = g % nst;
            ok = mbar_wait(&k_full[st], (g / nst) & 1u, abort_flag, lim);
            if (!ok) break;
            tc_fence_after();
            issue_qk<D>(t ? tS1 : tS0, sQ0, sbase + k_slot(st), idesc_qk);
            umma_commit(&s_full[t]);
            if (t == n - 1) umma_commit(q_empty);
          }
          for (int i = 0; i < n0 && ok; ++i) {
            for (int w = 0; w < 2; ++w) {
              const int jt = 2 * i + w;  // warpgroup w's i-th tile
              if (jt >= n) break;
              const uint32_t g = gk + jt, st = g % nst;
              uint32_t& pc = w ? pc1 : pc0;
              ok = mbar_wait(&v_full[st], (g / nst) & 1u, abort_flag, lim) &&
                   mbar_wait(&p_full[w], pc & 1u, abort_flag, lim);
              if (!ok) break;
              ++pc;
              tc_fence_after();
              issue_pv<D>(w ? tO1 : tO0, w ? tS1 : tS0, sbase + v_slot(st), idesc_pv, i > 0);
              umma_commit(&kv_empty[st]);
              if (i == (w ? n1 : n0) - 1) umma_commit(&o_full[w]);
              const int jn = jt + 2;  // the warpgroup's next tile
              if (jn < n) {
                const uint32_t g2 = gk + jn, st2 = g2 % nst;
                ok = mbar_wait(&k_full[st2], (g2 / nst) & 1u, abort_flag, lim);
                if (!ok) break;
                tc_fence_after();
                issue_qk<D>(w ? tS1 : tS0, sQ0, sbase + k_slot(st2), idesc_qk);
                umma_commit(&s_full[w]);
                if (jn == n - 1) umma_commit(q_empty);
              }
            }
          }
          gk += n;
          ++it_cnt;
          continue;
        }
        {
          const uint32_t st = gk % nst;
          ok = mbar_wait(&k_full[st], (gk / nst) & 1u, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          issue_qk<D>(tS0, sQ0, sbase + k_slot(st), idesc_qk);
          umma_commit(&s_full[0]);
          issue_qk<D>(tS1, sQ1, sbase + k_slot(st), idesc_qk);
          umma_commit(&s_full[1]);
          if (n == 1) umma_commit(q_empty);
        }
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t g = gk + j, st = g % nst;
          ok = mbar_wait(&v_full[st], (g / nst) & 1u, abort_flag, lim) &&
               mbar_wait(&p_full[0], pc0 & 1u, abort_flag, lim);
          if (!ok) break;
          ++pc0;
          tc_fence_after();
          issue_pv<D>(tO0, tS0, sbase + v_slot(st), idesc_pv, j > 0);
          if (j == n - 1) umma_commit(&o_full[0]);
          const uint32_t g1 = g + 1, st1 = g1 % nst;
          if (j + 1 < n) {
            ok = mbar_wait(&k_full[st1], (g1 / nst) & 1u, abort_flag, lim);
            if (!ok) break;
            tc_fence_after();
            issue_qk<D>(tS0, sQ0, sbase + k_slot(st1), idesc_qk);
            umma_commit(&s_full[0]);
          }
          ok = mbar_wait(&p_full[1], pc1 & 1u, abort_flag, lim);
          if (!ok) break;
          ++pc1;
          tc_fence_after();
          issue_pv<D>(tO1, tS1, sbase + v_slot(st), idesc_pv, j > 0);
          umma_commit(&kv_empty[st]);
          if (j == n - 1) umma_commit(&o_full[1]);
          if (j + 1 < n) {
            issue_qk<D>(tS1, sQ1, sbase + k_slot(st1), idesc_qk);
            umma_commit(&s_full[1]);
            if (j + 2 == n) umma_commit(q_empty);
          }
        }
        gk += n;
        ++it_cnt;
      }
      if (!ok) record_abort(abort_flag, p.status);
      // every MMA issued by this thread has completed once `drain` fires
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr, 100000000ull);
    }
    __syncwarp();
  } else if (warp == kWarpDec) {
    // ------------------------------------------------------------ item decoder
    // Stages each item while the softmax warpgroups still work on the one before it, so that
    // the chain of dependent loads behind an item (chunk order, chunk, the query tile's slice
    // list, its slices, the first entry) is off their path at the item boundary.  Lanes 0-7: query tile t = lane / 4,
    // staged slice k = lane % 4; lanes 8-9: first entries; lane 10: the item's chunk.
    bool ok = true;
    for (int wave = 0; ok; ++wave) {
      const int item = sched_item(wave);
      if (item >= n_items) break;
      const int ib = wave & 1;
      if (wave >= 2) {  // the softmax threads have read this slot's previous item
        ok = __all_sync(0xffffffffu, mbar_wait(&it_empty[ib], ((wave >> 1) - 1) & 1u, abort_flag, lim));
        if (!ok) break;
      }
      ItemStage* ist = reinterpret_cast<ItemStage*>(sm + SM::kIt) + ib;
      const int4 ch = item_chunk(p, item);
      const Item it = decode_item<kKS>(p, item, ch);
      const int t = (lane >> 2) & 1, k = lane & 3;
      const int qt = t ? it.qt1 : it.qt0;
      if (lane < 8) {
        int nsl = 0, si = 0;
        if (qt < p.nqt) {
          nsl = p.plan.row_nsl[qt];
          si = p.plan.row_sl[static_cast<size_t>(qt) * kSliceCap + k];
        }
        if (k < nsl) {
          ist->tile[t].s[k] = p.plan.slices[si];
          ist->tile[t].type[k] = p.plan.stypes[si];
        }
        if (k == 0) ist->tile[t].nsl = nsl;
      } else if (lane < 10) {
        const int j = lane - 8;
        ist->e_first[j] = j < it.n ? it.ents[j] : 0u;
      } else if (lane == 10) {
        ist->ch = ch;
      }
      mbar_arrive(&it_full[ib]);
    }
    if (!ok) record_abort(abort_flag, p.status);
    __syncwarp();
  }
  }  // producer warpgroup

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// LSE merge of split rows: for a group whose work list was cut into chunks, every row combines
// its chunks' partial results, L = log sum_c e^{L_c} and O = sum_c e^{L_c - L} O_c (the
// chunks cover disjoint key sets of the row); rows whose chunks all have L_c = -inf get
// O = 0 and L = -inf.  One block per (group, head slot, sub-tile, row) — with the key split,
// per (query tile, head, row), over both warpgroups' partials of every chunk: its sixteen warps
// take every sixteenth partial, a lane holds D / 32 columns (coalesced loads of a partial row),
// and the warps' sums are combined in shared memory.  Rows past the end return at once.
constexpr int kMergeWarps = 16;
template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) ffa_fwd_merge(const FwdParams p) {
  constexpr int kPer = D / 32;  // columns per lane
  __shared__ float sh_acc[kMergeWarps][D];
  __shared__ float sh_w[kMergeWarps];
  __shared__ float sh_max[kMergeWarps];
  pdl_wait();  // the attention kernel's partial results are complete
  int b = blockIdx.x;
  const int r = b % kTile;
  b /= kTile;
  // key split: one block per row, merging both warpgroups' partials of every chunk
  const int sub = p.key_split ? 0 : (b & 1);
  if (!p.key_split) b >>= 1;
  const int g = b / p.slots, slot = b - (b / p.slots) * p.slots;
  const int nch = p.plan.grp_nch[g];
  if (!p.key_split && nch <= 1) return;
  const int nsub = p.key_split ? 2 : 1;
  const int npart = nch * nsub;  // partial results of this row
  int qt, h;
  if (p.key_split) {
    qt = g;
    h = slot;
  } else if (p.head_pair) {
    qt = g;
    h = 2 * slot + sub;
  } else {
    qt = 2 * g + sub;
    h = slot;
  }
  const int row = qt * kTile + r;
  if (row >= p.nq) return;
  const int ps = p.plan.grp_pslot[g];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // partial k: chunk k / nsub, sub-tile (key split: warpgroup) k % nsub
  auto prow = [&](int k) {
    return (static_cast<size_t>(ps + k / nsub) * p.slots + slot) * 2 * kTile + (sub + k % nsub) * kTile + r;
  };
  // the largest partial LSE
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < npart; c += blockDim.x) mx = fmaxf(mx, p.plan.part_lse[prow(c)]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) sh_max[warp] = mx;
  __syncthreads();
  mx = sh_max[0];
#pragma unroll
  for (int w = 1; w < kMergeWarps; ++w) mx = fmaxf(mx, sh_max[w]);
  __nv_bfloat16* out = p.out + (static_cast<size_t>(row) * p.hq + h) * D;
  float* lse_at = p.lse + static_cast<size_t>(h) * p.nq + row;
  if (p.uout != nullptr) {
    const int tok = row / p.upack, hu = h * p.upack + row % p.upack;
    const int ntok = p.nq / p.upack;
    out = p.uout + (static_cast<size_t>(tok) * p.hq * p.upack + hu) * D;
    lse_at = p.ulse + static_cast<size_t>(hu) * ntok + tok;
  }
  if (mx == -INFINITY) {
    if (warp == 0) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) out[lane * kPer + k] = __float2bfloat16(0.0f);
      if (lane == 0) *lse_at = -INFINITY;
    }
    return;
  }
  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.0f;
  float wsum = 0.0f;
#pragma unroll 4
  for (int c = warp; c < npart; c += kMergeWarps) {
    const size_t pr = prow(c);
    const float w = ex2_approx((p.plan.part_lse[pr] - mx) * kLog2e);
    wsum += w;
    const float* src = p.plan.part_o + pr * D + lane * kPer;
    if constexpr (kPer == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]);
      acc[3] = fmaf(w, v.w, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
    }
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) sh_acc[warp][lane * kPer + k] = acc[k];
  if (lane == 0) sh_w[warp] = wsum;
  __syncthreads();
  if (warp == 0) {
    float tw = 0.0f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) tw += sh_w[w];
    const float inv = 1.0f / tw;
#pragma unroll
    for (int k = 0; k < kPer; k += 2) {
      float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
      for (int w = 0; w < kMergeWarps; ++w) {
        a0 += sh_acc[w][lane * kPer + k];
        a1 += sh_acc[w][lane * kPer + k + 1];
      }
      *reinterpret_cast<uint32_t*>(out + lane * kPer + k) = pack_bf16x2(a0 * inv, a1 * inv);
    }
    if (lane == 0) *lse_at = mx + lg2_approx(tw) * kLn2;
  }
}

template <int D, bool kCap, bool kBias, bool kFixed, bool kKS>
cudaError_t launch_impl(const FwdArgs& a, cudaStream_t stream) {
  using SM = FwdSmem<D>;
  auto kern = ffa_fwd_kernel<D, kCap, kBias, kFixed, kKS>;
  // Once per device (the shared-memory attribute applies to the device current when it is
  // set).  The register split (setmaxnreg) is balanced for exactly kRegsLaunch registers per
  // thread at launch; with any other count a softmax warp's increase could never be granted,
  // so such a build is refused here rather than launched.
  static std::once_flag once[kMaxDevices];
  static cudaError_t setup_err[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e == cudaSuccess && fa.numRegs != kRegsLaunch) e = cudaErrorInvalidKernelImage;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kAlloc);
    setup_err[dev] = e;
  });
  if (setup_err[dev] != cudaSuccess) return setup_err[dev];
  CUtensorMap mq, mk, mv, mo;
  const auto& P = a.P;
  // paged: K/V maps cover the physical pool, one page of rows per box
  const bool paged = a.page_table != nullptr;
  const uint64_t kv_rows = paged ? static_cast<uint64_t>(a.n_pages) * a.page_size : static_cast<uint64_t>(P.nk);
  const uint32_t kv_box = paged ? static_cast<uint32_t>(a.page_size) : static_cast<uint32_t>(kTile);
  if (!encode_tile_map(&mq, a.q, static_cast<uint64_t>(P.hq) * D, P.nq, 64, kTile) ||
      !encode_tile_map(&mk, a.k, static_cast<uint64_t>(P.hkv) * D, kv_rows, 64, kv_box) ||
      !encode_tile_map(&mv, a.v, static_cast<uint64_t>(P.hkv) * D, kv_rows, 64, kv_box) ||
      !encode_tile_map(&mo, a.out, static_cast<uint64_t>(P.hq) * D, P.nq, 64, kTile))
    return cudaErrorInvalidValue;
  FwdParams p;
  p.nq = P.nq; p.nk = P.nk; p.hq = P.hq; p.hkv = P.hkv; p.G = P.hq / P.hkv;
  p.nqt = P.nqt; p.nkt = P.nkt;
  p.head_pair = a.head_pair; p.slots = a.slots;
  p.key_split = a.key_split;
  p.scale_log2 = a.scale * kLog2e;
  p.cap_c = a.softcap * kLog2e;
  p.cap_k = a.softcap > 0.0f ? 2.0f * a.scale * kLog2e / a.softcap : 0.0f;
  fold_cap_poly(a.scale, a.softcap, p.cap_q, &p.cap_slim);
  fold_cap_poly5(a.scale, a.softcap, p.cap_q5);
  p.cap_fixed = (a.softcap > 0.0f && 2.0f * p.cap_c <= 120.0f) ? 1 : 0;
  p.plan = a.plan;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.uout = static_cast<__nv_bfloat16*>(a.unpack_out);
  p.ulse = a.unpack_lse;
  p.upack = a.unpack_out != nullptr ? a.alibi_pack : 1;
  p.alibi = a.alibi;
  p.alibi_pack = a.alibi_pack;
  p.page_table = a.page_table;
  p.page_size = paged ? a.page_size : 0;
  p.n_pages = paged ? static_cast<int>(a.n_pages) : 0;
  p.n_lpages = paged ? static_cast<int>((static_cast<int64_t>(P.nk) + a.page_size - 1) / a.page_size) : 0;
  p.status = a.status;
  p.wait_limit_ns = a.wait_limit_ns;
  p.stall = a.stall_test;
  const int grid = a.n_items < num_sms() ? a.n_items : num_sms();
  if (grid <= 0) return cudaSuccess;
  if (g_kernel_events.fwd_start != nullptr) cudaEventRecord(g_kernel_events.fwd_start, stream);
  // a programmatic dependent of the planner's last kernel: the CTAs set up their barriers and
  // TMEM while it finishes (with a timing event recorded in between, plain stream order)
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kThreads), SM::kAlloc, stream, mq, mk, mv, mo, p);
  if (g_kernel_events.fwd_stop != nullptr) cudaEventRecord(g_kernel_events.fwd_stop, stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || !a.split) return e;
  return launch_pdl(ffa_fwd_merge<D>, dim3(a.ngrp * a.slots * (a.key_split ? 1 : 2) * kTile), dim3(32 * kMergeWarps),
                    0, stream, p);
}

template <bool kKS>
cudaError_t launch_variant(const FwdArgs& a, cudaStream_t s) {
  const bool cap = a.softcap > 0.0f, bias = a.alibi != nullptr;
  // a bounded softcap without ALiBi takes the fixed-reference kernel (FwdParams::cap_fixed)
  const bool fixed = cap && !bias && 2.0f * a.softcap * kLog2e <= 120.0f;
  if (a.P.d == 64) {
    if (bias) return cap ? launch_impl<64, true, true, false, kKS>(a, s) : launch_impl<64, false, true, false, kKS>(a, s);
    if (fixed) return launch_impl<64, true, false, true, kKS>(a, s);
    return cap ? launch_impl<64, true, false, false, kKS>(a, s) : launch_impl<64, false, false, false, kKS>(a, s);
  }
  if (bias) return cap ? launch_impl<128, true, true, false, kKS>(a, s) : launch_impl<128, false, true, false, kKS>(a, s);
  if (fixed) return launch_impl<128, true, false, true, kKS>(a, s);
  return cap ? launch_impl<128, true, false, false, kKS>(a, s) : launch_impl<128, false, false, false, kKS>(a, s);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s) {
  return a.key_split ? launch_variant<true>(a, s) : launch_variant<false>(a, s);
}

}  // namespace ffa
