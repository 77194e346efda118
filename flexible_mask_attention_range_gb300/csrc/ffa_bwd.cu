// Backward kernels: gradients of sum(O * dO) for range-masked attention on sm_103a.
//
// For every visible (i, j) with P_ij = exp(x_ij - LSE_i) (recomputed from the forward LSE):
//   dV_j += P_ij dO_i;  dP_ij = dO_i . V_j;  D_i = dO_i . O_i  (= sum_j P_ij dP_ij);
//   dX_ij = P_ij (dP_ij - D_i);  dS = dX * (1 - tanh^2(scale q.k / softcap)) with softcap;
//   dK_j += scale dS_ij Q_i;  dQ_i += scale dS_ij K_j.
// The pages ask for dq/dk/dv through autograd (MagiAttention issue #180, question code:
// out.backward(do)) without fixing the kernel; this follows the usual recomputation scheme.
//
// Three launches after the column planner:
//   1. ffa_bwd_pre: -D_i (fp32) and -LSE_i * log2(e) padded to whole tiles, dq accumulator = 0.
//   2. ffa_bwd_kernel: KV-stationary.  One work item = (key tile, KV head); its CTA walks the
//      query tiles of the key tile's column list and the G query heads of the group.  Five
//      tcgen05 GEMMs per step: S^T = K Q^T and dP^T = V dO^T (keys on TMEM lanes), then
//      dV += P^T dO and dK += dS^T Q with P^T / dS^T read from TMEM, and dQ = dS K with dS
//      staged in shared memory; dQ is added into the fp32 accumulator with TMA bulk
//      reduce-adds (cp.reduce.async.bulk.tensor, add) of 32-column boxes staged in a buffer
//      of their own, so the next step's dS^T may be written as soon as the dQ MMA has run.
//      dK and dV stay in TMEM for the whole item and are written once.
//   3. ffa_bwd_dq_convert: fp32 accumulator -> bf16 dq.
//
// Warp roles (448 threads):
//   warps 0-7  two compute warpgroups: warpgroup h handles query columns [64h, 64h+64) of the
//              tile, key row r <-> TMEM lane r; P^T, dS^T; epilogue (h = 0: dV, h = 1: dK)
//   warps 8-11 dQ warpgroup: query row r <-> TMEM lane r; drains dQ into the accumulator
//   warp 12    TMA producer;  warp 13  MMA issuer (owns TMEM)
// TMEM columns: S^T [0,128) with P^T of half h (bf16) over [64h, 64h+32); dP^T [128,256) with
// dS^T of half h over [128+64h, 128+64h+32), then dQ [128,128+D); dV [256,256+D),
// dK [256+D,256+2D).
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "ffa_internal.h"
#include "ffa_ptx.cuh"
#include "../../include/ffa.h"

namespace ffa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 448;
constexpr int kWarpDq = 8;
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;

template <int D>
struct BwdSmem {
  // Q (with its row statistics) and dO rings; at d = 128 dO has one slot, so that the dQ drain
  // has a staging buffer of its own
  static constexpr int kStagesQ = D == 128 ? 2 : 3;
  static constexpr int kStagesDO = D == 128 ? 1 : 3;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kBoxBytes = kTile * 128;
  static constexpr int kStatBytes = 2 * kTile * 4;  // LSE*log2e and D of one query tile
  static constexpr int kK = 0;
  static constexpr int kV = kTileBytes;
  static constexpr int kQ = 2 * kTileBytes;                        // + s * kTileBytes
  static constexpr int kDO = kQ + kStagesQ * kTileBytes;           // + s * kTileBytes
  static constexpr int kDS = kDO + kStagesDO * kTileBytes;         // 128 keys x 128 queries bf16
  static constexpr int kDQS = kDS + kTile * kTile * 2;             // dQ staging: two 128 x 32 fp32 boxes
  static constexpr int kStat = kDQS + 2 * kTile * 128;             // + s * kStatBytes
  static constexpr int kBar = kStat + kStagesQ * kStatBytes;
  // kv_full, kv_empty, q_full[SQ], q_empty[SQ], do_full[SD], do_empty[SD], s_full, dp_full,
  // p_full, ds_full, dq_full, dq_empty, dkv_full, drain, stall (never arrived on;
  // failure-detection test)
  static constexpr int kNumBars = 2 + 2 * kStagesQ + 2 * kStagesDO + 9;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kMaxDyn = 232448;
  static constexpr int kAlloc = (kTotal + 1024 <= kMaxDyn) ? kTotal + 1024 : kMaxDyn;
  static_assert(kTotal <= kMaxDyn, "backward shared memory exceeds the per-block limit");
};

struct BwdParams {
  int nq, nk, hq, hkv, G, nqt, nkt, n_items, qpad;
  float scale;
  float scale_log2;
  float cap_c, cap_k, inv_cap_c;
  // capped logit as an odd polynomial of the raw score, valid for |s| <= cap_slim (< 0: unused):
  // degree 5 (kTanhPoly5 folded, cap_q[3] unused), within 4.5e-6 of tanh, i.e. within
  // 4.5e-6 * cap_c * tanh(0.375) of the logit in the log2 domain (1e-4 at softcap 41, 1e-3 at
  // softcap 400): a relative error of P of that size times ln 2, far below the gradients'
  // tolerance and the bf16 rounding of P and dS
  float cap_q[4];
  float cap_slim;
  PlanView plan;
  const float* lse2;
  const float* rowD;
  float* dqacc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* alibi;  // per-query-head ALiBi slopes, or null
  int det;              // deterministic dq: ordered additions, items by ascending key tile
  const int* tile_rank;
  int* dq_sem;
  int* status;
  uint64_t wait_limit_ns;
  int stall;  // failure-detection test: the first wait of every CTA never completes
};

__device__ __forceinline__ int sched_item(int wave) {
  const int c = blockIdx.x, C = gridDim.x;
  return wave * C + ((wave & 1) ? (C - 1 - c) : c);
}

__device__ __forceinline__ void record_abort(volatile int* abort_flag, int* status) {
  *abort_flag = 1;
  if (status != nullptr) atomicOr(status, FFA_STATUS_TIMEOUT);
}

__device__ __forceinline__ void set_bits(uint32_t (&w)[4], int lo, int hi) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int a = max(lo - 32 * k, 0), b = min(hi - 32 * k, 32);
    if (a < b) w[k] |= (b - a == 32) ? 0xffffffffu : (((1u << (b - a)) - 1u) << a);
  }
}

// Mask of key row j over query tile qt: bit c set iff query qt*128+c sees key j.
__device__ __forceinline__ void key_mask(const BwdParams& p, int cls, int j, int qt, int nsl, const int* sl,
                                         uint32_t (&w)[4]) {
  const int r0 = qt * kTile;
  if (j >= p.nk) {
    w[0] = w[1] = w[2] = w[3] = 0u;
    return;
  }
  if (cls == FFA_TILE_FULL) {
    w[0] = w[1] = w[2] = w[3] = 0xffffffffu;
  } else {
    w[0] = w[1] = w[2] = w[3] = 0u;
    if (cls == FFA_TILE_PARTIAL) {
      const int n = nsl >= 0 ? nsl : p.plan.hdr[0];
      for (int k = 0; k < n; ++k) {
        const int si = nsl >= 0 ? sl[k] : k;
        const int4 s = p.plan.slices[si];
        if (j < s.z || j >= s.w) continue;
        const int lo = (p.plan.stypes[si] == FFA_CAUSAL) ? max(s.x, j + s.y - s.w) : s.x;
        const int lo_c = max(lo, r0) - r0, hi_c = min(s.y, r0 + kTile) - r0;
        if (lo_c < hi_c) set_bits(w, lo_c, hi_c);
      }
    }
  }
  const int valid = p.nq - r0;
  if (valid < kTile) {
    uint32_t t[4] = {0u, 0u, 0u, 0u};
    set_bits(t, 0, valid);
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] &= t[k];
  }
}

__device__ __forceinline__ float capped_log2(float s, float cap_c, float cap_k) {
  const float e = ex2_approx(s * cap_k);
  return fmaf(-2.0f * cap_c, rcp_approx(1.0f + e), cap_c);
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Waits until *counter reaches `target` (another CTA's release), bounded like mbar_wait.
__device__ bool wait_counter(const int* counter, int target, const volatile int* abort, uint64_t limit_ns) {
  if (ld_acquire_gpu(counter) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i) {
      if (ld_acquire_gpu(counter) >= target) return true;
      __nanosleep(64);
    }
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// A[m][k] K-major x B[n][k] K-major, both 128-row tiles of D columns (2 boxes when D = 128)
template <int D>
__device__ __forceinline__ void issue_kmajor(uint32_t d_tmem, uint32_t sA, uint32_t sB, uint32_t idesc) {
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    const uint32_t off = (s / 4) * BwdSmem<D>::kBoxBytes + (s % 4) * 32;
    umma_ss(d_tmem, make_sdesc(sA + off, 16, 1024, kSwizzle128B), make_sdesc(sB + off, 16, 1024, kSwizzle128B),
            idesc, s > 0 ? 1u : 0u);
  }
}

// D (+)= A[tmem] x B where B is a 128-row (K) tile of N columns stored MN-major.  A (bf16,
// K = 128 queries) sits in two halves: queries [0,64) at columns [0,32) of a_tmem and
// queries [64,128) at columns [64,96).
template <int N>
__device__ __forceinline__ void issue_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t sB, uint32_t idesc,
                                        bool accumulate) {
#pragma unroll
  for (int s = 0; s < kTile / 16; ++s)
    umma_ts(d_tmem, a_tmem + (s / 4) * 64 + (s % 4) * 8, make_sdesc(sB + s * 2048, kTile * 128, 1024, kSwizzle128B),
            idesc, (accumulate || s > 0) ? 1u : 0u);
}

// dQ = dS K: A = dS^T stored [key][query] (MN-major, 2 boxes of 64 queries), B = K tile [key][d]
template <int D>
__device__ __forceinline__ void issue_dq(uint32_t d_tmem, uint32_t sDS, uint32_t sK, uint32_t idesc) {
#pragma unroll
  for (int s = 0; s < kTile / 16; ++s)
    umma_ss(d_tmem, make_sdesc(sDS + s * 2048, kTile * 128, 1024, kSwizzle128B),
            make_sdesc(sK + s * 2048, kTile * 128, 1024, kSwizzle128B), idesc, s > 0 ? 1u : 0u);
}

struct BwdItem {
  int kt, kvh, n_ent, n_steps, rot;
  const uint32_t* ents;
  // the item's e-th entry in processing order: the list rotated so that it starts at the
  // query tile that is a multiple of its length (see decode_item)
  __device__ __forceinline__ uint32_t ent(int e) const {
    const int i = e + rot;
    return ents[i < n_ent ? i : i - n_ent];
  }
};

constexpr int kRotateMax = 64;
__device__ __forceinline__ BwdItem decode_item(const BwdParams& p, int item) {
  BwdItem it;
  const int rank = item / p.hkv;
  it.kvh = item - rank * p.hkv;
  it.kt = p.det ? rank : p.plan.col_order[rank];  // deterministic: ascending key tiles (p.det == kDet)
  it.n_ent = p.plan.col_cnt[it.kt];
  it.n_steps = it.n_ent * p.G;
  it.ents = p.plan.col_ent + static_cast<size_t>(it.kt) * p.nqt;
  // Rotation of short lists (not in deterministic mode, whose additions follow ascending key
  // tiles): a list of n <= kRotateMax consecutive query tiles starts at the one whose index is
  // a multiple of n, so CTAs on neighbouring key tiles with lists of the same length (a
  // sliding window) work on the same query tile at the same time and share its Q, dO and dq
  // accumulator in L2.  Any other short list is only rotated; every entry is still visited
  // once.  Long lists keep the ascending order: neighbouring causal columns then walk the
  // same query tiles one step apart, which shares them already (rotated, the 64K long-causal
  // backward moved 3.7 times the DRAM bytes).
  it.rot = 0;
  if (!p.det && it.n_ent > 1 && it.n_ent <= kRotateMax) {
    const int r = entry_idx(it.ents[0]) % it.n_ent;
    it.rot = r == 0 ? 0 : it.n_ent - r;
  }
  return it;
}

template <int D, bool kCap, bool kBias, bool kDet>
__global__ void __launch_bounds__(kThreads, 1)
    ffa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                   const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using SM = BwdSmem<D>;
  constexpr int SQ = SM::kStagesQ, SD = SM::kStagesDO;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad + SM::kTotal > SM::kAlloc) {  // cannot place the swizzled tiles: report and stop
    if (threadIdx.x == 0 && p.status != nullptr) atomicOr(p.status, FFA_STATUS_SMEM);
    return;
  }
  uint8_t* sm = smem_raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SM::kBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* q_full = bars + 2;
  uint64_t* q_empty = q_full + SQ;
  uint64_t* do_full = q_empty + SQ;
  uint64_t* do_empty = do_full + SD;
  uint64_t* s_full = do_empty + SD;
  uint64_t* dp_full = s_full + 1;
  uint64_t* p_full = s_full + 2;
  uint64_t* ds_full = s_full + 3;
  uint64_t* dq_full = s_full + 4;  // the dQ MMA has run: dQ in TMEM, the dS^T tile free again
  uint64_t* dq_empty = s_full + 5;
  uint64_t* dkv_full = s_full + 6;
  uint64_t* drain = s_full + 7;
  uint64_t* stall_bar = s_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SM::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + SM::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < SQ; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < SD; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 256);
    mbar_init(ds_full, 256);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(dkv_full, 1);
    mbar_init(drain, 1);
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
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
  pdl_wait();  // the preprocess has completed (the setup above overlapped its tail)

  if (warp < 8) {
    // ------------------------------------------------------------ compute warpgroups
    const int hf = warp >> 2, q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int c0 = hf * 64;  // first query column of this warpgroup
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tbase + lane_base + c0, tP = tbase + lane_base + 128 + c0;
    const uint32_t tOut = tbase + lane_base + 256 + hf * D;  // hf 0: dV, hf 1: dK
    uint8_t* sDS = sm + SM::kDS + hf * (kTile * 128);
    uint32_t step_cnt = 0, item_cnt = 0;
    bool ok = true;
    for (int wave = 0; ok; ++wave) {
      const int item = sched_item(wave);
      if (item >= p.n_items) break;
      const BwdItem it = decode_item(p, item);
      const int j = it.kt * kTile + r;  // key row
      const bool in_keys = j < p.nk;
      const size_t orow = (static_cast<size_t>(j) * p.hkv + it.kvh) * D;
      __nv_bfloat16* gout = hf ? p.dk : p.dv;
      if (it.n_steps == 0) {
        if (in_keys) {
          uint4* a = reinterpret_cast<uint4*>(gout + orow);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) a[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const int nsl = p.plan.col_nsl[it.kt];
      const int* sl = p.plan.col_sl + static_cast<size_t>(it.kt) * kSliceCap;
      for (int t = 0; t < it.n_steps && ok; ++t) {
        const uint32_t e = it.ent(t / p.G);
        const int qt = entry_idx(e);
        const int cls = entry_cls(e, 0);
        const uint32_t st = step_cnt % SQ;
        const float* stat = reinterpret_cast<const float*>(sm + SM::kStat + st * SM::kStatBytes);
        // the row statistics arrive with the step's Q (q_full); S^T with s_full
        uint64_t* sb = (p.stall && step_cnt == 0) ? stall_bar : s_full;
        ok = __all_sync(0xffffffffu, mbar_wait(&q_full[st], (step_cnt / SQ) & 1u, abort_flag, lim) &&
                                         mbar_wait(sb, step_cnt & 1u, abort_flag, lim));
        if (!ok) break;
        tc_fence_after();
        uint32_t w[4];
        const bool masked = (cls != FFA_TILE_FULL) || (qt * kTile + kTile > p.nq) || !in_keys;
        if (masked) key_mask(p, cls, j, qt, nsl, sl, w);
        const float slope_log2 = kBias ? p.alibi[it.kvh * p.G + (t % p.G)] * kLog2e : 0.0f;
        const float bbase = kBias ? slope_log2 * static_cast<float>(j - qt * kTile) : 0.0f;
        // phase 1: P^T of this warpgroup's 64 queries from S^T and the row LSEs; keep
        // P' = P (or P (1 - tanh^2) with softcap) packed as bf16 for phase 2
        uint32_t pp[32];
        // kM: this tile may hide elements (mk says whether it does).  The loop exists twice so
        // fully visible tiles carry no per-element mask test.
        auto p1_body = [&](auto mtag, bool mk) {
        constexpr bool kM = decltype(mtag)::value;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sv[32];
          tmem_ld32(tS + 32 * c, sv);
          tmem_wait_ld();
          reg_fence(sv);
          uint32_t pk[16];
          // Softcap without a bias: when every raw score of this chunk over the warp lies where
          // the tanh polynomial holds, the capped logits come from the polynomial (FMA pipe,
          // two columns per packed instruction); otherwise from the exact form.
          auto k4_loop = [&](auto ptag) {
          constexpr bool kPoly = decltype(ptag)::value;
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            const float4 l4 = *reinterpret_cast<const float4*>(stat + c0 + 32 * c + 4 * k4);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
            // the row statistics are stored negated: -LSE * log2(e) (see ffa_bwd_pre)
            float pv[4], pd[4];
            if (kCap && kPoly) {
              const float2 invc2 = make_float2(p.inv_cap_c, p.inv_cap_c), one2 = make_float2(1.0f, 1.0f);
              const float2 q0 = make_float2(p.cap_q[0], p.cap_q[0]), q1 = make_float2(p.cap_q[1], p.cap_q[1]);
              const float2 q2 = make_float2(p.cap_q[2], p.cap_q[2]);
#pragma unroll
              for (int hp = 0; hp < 2; ++hp) {
                const int col0 = c0 + 32 * c + 4 * k4 + 2 * hp;
                const float2 s2 = make_float2(__uint_as_float(sv[4 * k4 + 2 * hp]), __uint_as_float(sv[4 * k4 + 2 * hp + 1]));
                const float2 t = mul2(s2, s2);
                const float2 x = mul2(s2, fma2(fma2(q2, t, q1), t, q0));
                const float2 y = add2(x, make_float2(lv[2 * hp], lv[2 * hp + 1]));
                float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
                const float2 th = mul2(x, invc2);
                const float2 dd = mul2(make_float2(p0, p1), fma2(make_float2(-th.x, -th.y), th, one2));
                float d0 = dd.x, d1 = dd.y;
                if (kM && mk) {
                  if (!((w[col0 >> 5] >> (col0 & 31)) & 1u)) p0 = d0 = 0.0f;
                  if (!((w[(col0 + 1) >> 5] >> ((col0 + 1) & 31)) & 1u)) p1 = d1 = 0.0f;
                }
                pv[2 * hp] = p0;
                pv[2 * hp + 1] = p1;
                pd[2 * hp] = d0;
                pd[2 * hp + 1] = d1;
              }
            } else if (kCap) {
#pragma unroll
              for (int h4 = 0; h4 < 4; ++h4) {
                const int col = c0 + 32 * c + 4 * k4 + h4;
                // ALiBi (log2 domain): slope * log2(e) * (key j - query qt*128+col)
                const float lb = kBias ? fmaf(-slope_log2, static_cast<float>(col), bbase) + lv[h4] : lv[h4];
                const float x = capped_log2(__uint_as_float(sv[4 * k4 + h4]), p.cap_c, p.cap_k);
                float pr = ex2_approx(x + lb);
                const float th = x * p.inv_cap_c;
                pd[h4] = pr * (1.0f - th * th);
                if (kM && mk && !((w[col >> 5] >> (col & 31)) & 1u)) {
                  pr = 0.0f;
                  pd[h4] = 0.0f;
                }
                pv[h4] = pr;
              }
            } else {
              // two columns per packed fp32 pair instruction
              const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
              for (int hp = 0; hp < 2; ++hp) {
                const int col0 = c0 + 32 * c + 4 * k4 + 2 * hp;
                float2 lb2 = make_float2(lv[2 * hp], lv[2 * hp + 1]);
                if (kBias) lb2 = make_float2(fmaf(-slope_log2, static_cast<float>(col0), bbase) + lv[2 * hp],
                                             fmaf(-slope_log2, static_cast<float>(col0 + 1), bbase) + lv[2 * hp + 1]);
                const float2 y = fma2(make_float2(__uint_as_float(sv[4 * k4 + 2 * hp]), __uint_as_float(sv[4 * k4 + 2 * hp + 1])), sc2, lb2);
                float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
                if (kM && mk) {
                  if (!((w[col0 >> 5] >> (col0 & 31)) & 1u)) p0 = 0.0f;
                  if (!((w[(col0 + 1) >> 5] >> ((col0 + 1) & 31)) & 1u)) p1 = 0.0f;
                }
                pv[2 * hp] = p0;
                pv[2 * hp + 1] = p1;
              }
            }
            pk[2 * k4] = pack_bf16x2(pv[0], pv[1]);
            pk[2 * k4 + 1] = pack_bf16x2(pv[2], pv[3]);
            if (kCap) {
              pp[16 * c + 2 * k4] = pack_bf16x2(pd[0], pd[1]);
              pp[16 * c + 2 * k4 + 1] = pack_bf16x2(pd[2], pd[3]);
            } else {
              pp[16 * c + 2 * k4] = pk[2 * k4];
              pp[16 * c + 2 * k4 + 1] = pk[2 * k4 + 1];
            }
          }
          };
          if constexpr (kCap && !kBias) {
            float hi[2] = {-INFINITY, -INFINITY}, lo[2] = {INFINITY, INFINITY};
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float a = __uint_as_float(sv[i]), b = __uint_as_float(sv[i + 1]);
              hi[(i >> 1) & 1] = fmax3(hi[(i >> 1) & 1], a, b);
              lo[(i >> 1) & 1] = fmin3(lo[(i >> 1) & 1], a, b);
            }
            if (__all_sync(0xffffffffu, fmaxf(fmaxf(hi[0], hi[1]), -fminf(lo[0], lo[1])) <= p.cap_slim)) {
              k4_loop(std::true_type{});
            } else {
              k4_loop(std::false_type{});
            }
          } else {
            k4_loop(std::false_type{});
          }
          tmem_st16(tS + 16 * c, pk);
        }
        };
        // One copy per warp: the tensor-memory loads and stores and the polynomial's vote in the
        // pass are warp-collective, so the warp takes the masking copy when any of its key rows
        // needs a mask (a ragged last key tile masks some lanes only), each lane with its own mk.
        if (__any_sync(0xffffffffu, masked)) {
          p1_body(std::true_type{}, masked);
        } else {
          p1_body(std::false_type{}, false);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
        // phase 2: dS^T = P' (dP^T - D) -> TMEM (for dK) and shared memory (for dQ)
        ok = __all_sync(0xffffffffu, mbar_wait(dp_full, step_cnt & 1u, abort_flag, lim));
        if (ok && step_cnt > 0)  // the previous step's dQ MMA (the dS^T tile's reader) has run
          ok = __all_sync(0xffffffffu, mbar_wait(dq_full, (step_cnt - 1) & 1u, abort_flag, lim));
        if (!ok) break;
        tc_fence_after();
        const float* Drow = stat + kTile;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dv[32];
          tmem_ld32(tP + 32 * c, dv);
          tmem_wait_ld();
          reg_fence(dv);
          uint32_t pk[16];
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            const float4 d4 = *reinterpret_cast<const float4*>(Drow + c0 + 32 * c + 4 * k4);
            const uint32_t pa = pp[16 * c + 2 * k4], pb = pp[16 * c + 2 * k4 + 1];
            const float2 e01 = mul2(make_float2(__uint_as_float(pa << 16), __uint_as_float(pa & 0xffff0000u)),
                                    add2(make_float2(__uint_as_float(dv[4 * k4]), __uint_as_float(dv[4 * k4 + 1])),
                                         make_float2(d4.x, d4.y)));
            const float2 e23 = mul2(make_float2(__uint_as_float(pb << 16), __uint_as_float(pb & 0xffff0000u)),
                                    add2(make_float2(__uint_as_float(dv[4 * k4 + 2]), __uint_as_float(dv[4 * k4 + 3])),
                                         make_float2(d4.z, d4.w)));
            pk[2 * k4] = pack_bf16x2(e01.x, e01.y);
            pk[2 * k4 + 1] = pack_bf16x2(e23.x, e23.y);
          }
          tmem_st16(tP + 16 * c, pk);
          // shared-memory copy: row r, this half's queries 32c..32c+31 -> 16-byte chunks
          // c*4 .. c*4+3 of the half's 128-byte row, 128-byte swizzle (chunk ^= row % 8)
          uint8_t* rowp = sDS + r * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = (c * 4 + q) ^ (r & 7);
            *reinterpret_cast<uint4*>(rowp + chunk * 16) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(ds_full);
        ++step_cnt;
      }
      if (!ok) break;
      // epilogue: warpgroup 0 writes dV, warpgroup 1 writes scale * dK of this key tile
      ok = __all_sync(0xffffffffu, mbar_wait(dkv_full, item_cnt & 1u, abort_flag, lim));
      if (!ok) break;
      ++item_cnt;
      tc_fence_after();
      const float f = hf ? p.scale : 1.0f;
      uint4* dst = reinterpret_cast<uint4*>(gout + orow);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tOut + 32 * c, o);
        tmem_wait_ld();
        reg_fence(o);
        if (in_keys) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * f, __uint_as_float(o[8 * k + 1]) * f);
            v.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * f, __uint_as_float(o[8 * k + 3]) * f);
            v.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * f, __uint_as_float(o[8 * k + 5]) * f);
            v.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * f, __uint_as_float(o[8 * k + 7]) * f);
            dst[4 * c + k] = v;
          }
        }
      }
    }
    if (!ok) record_abort(abort_flag, p.status);
  } else if (warp < kWarpTma) {
    // ------------------------------------------------------------ dQ warpgroup
    // Reads its dQ row from TMEM (64 columns at a time; the columns are released once the
    // whole row is in registers), then adds the tile into the fp32 accumulator with TMA bulk
    // reduce-adds of 32-column boxes staged through the two 16 KB halves of its own staging
    // buffer, box after box; a half is rewritten once the reduce issued from it two boxes
    // before has read it, so the drain of one step runs on while the next step computes.
    const int q4 = warp - kWarpDq;
    const int r = q4 * 32 + lane;
    const bool leader = (q4 == 0 && lane == 0);
    const uint32_t tQ = tbase + (static_cast<uint32_t>(q4 * 32) << 16) + 128;
    uint8_t* sDQS = sm + SM::kDQS;  // two 16 KB halves, used alternately box after box
    uint32_t step_cnt = 0;
    bool ok = true;
    for (int wave = 0; ok; ++wave) {
      const int item = sched_item(wave);
      if (item >= p.n_items) break;
      const BwdItem it = decode_item(p, item);
      for (int t = 0; t < it.n_steps; ++t) {
        const int qt = entry_idx(it.ent(t / p.G));
        const int h = it.kvh * p.G + (t % p.G);
        // one decision for the whole warpgroup: it meets again at named barrier 1 below
        ok = named_bar_and(1, 128, mbar_wait(dq_full, step_cnt & 1u, abort_flag, lim));
        if (!ok) break;
        tc_fence_after();
        bool turn = true;  // deterministic mode: this CTA's turn to add into (h, qt) came
#pragma unroll
        for (int half = 0; half < D / 64; ++half) {
          uint32_t o[2][32];
          tmem_ld32(tQ + 64 * half, o[0]);
          tmem_ld32(tQ + 64 * half + 32, o[1]);
          tmem_wait_ld();
          reg_fence(o[0]);
          reg_fence(o[1]);
          if (half == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(dq_empty);
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * half + cc;
            uint8_t* buf = sDQS + (c & 1) * (kTile * 128);
            // the reduce issued from this half two boxes ago (in this step or the previous
            // one) has read it
            if (leader) bulk_wait_group_read<1>();
            named_bar_sync(1, 128);
            uint8_t* rowp = buf + r * 128;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int chunk = k ^ (r & 7);
              *reinterpret_cast<float4*>(rowp + chunk * 16) = make_float4(
                  __uint_as_float(o[cc][4 * k]) * p.scale, __uint_as_float(o[cc][4 * k + 1]) * p.scale,
                  __uint_as_float(o[cc][4 * k + 2]) * p.scale, __uint_as_float(o[cc][4 * k + 3]) * p.scale);
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (leader) {
              if (kDet && c == 0) {  // wait for the key tiles before this one in qt's list
                turn = wait_counter(p.dq_sem + static_cast<size_t>(h) * p.nqt + qt,
                                    p.tile_rank[static_cast<size_t>(qt) * p.nkt + it.kt], abort_flag, lim);
                if (!turn) record_abort(abort_flag, p.status);
                fence_proxy_async_global();
              }
              if (turn) {
                tma_reduce_add_2d(&tmDQ, buf, h * D + 32 * c, qt * kTile);
                bulk_commit_group();
              }
            }
          }
        }
        if (kDet && leader) {  // the additions must have landed before the next key tile may add
          asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
          fence_proxy_async_global();
          if (turn) red_release_gpu_add(p.dq_sem + static_cast<size_t>(h) * p.nqt + qt, 1);
        }
        ++step_cnt;
      }
    }
    if (leader) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (!ok) record_abort(abort_flag, p.status);
  } else if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t item_cnt = 0, gq = 0;
      bool ok = true;
      int last_q[SQ], last_do[SD];  // the last use of each slot whose copies were issued
      for (int s = 0; s < SQ; ++s) last_q[s] = -1;
      for (int s = 0; s < SD; ++s) last_do[s] = -1;
      int last_kv = -1;
      for (int wave = 0; ok; ++wave) {
        const int item = sched_item(wave);
        if (item >= p.n_items) break;
        const BwdItem it = decode_item(p, item);
        if (it.n_steps == 0) continue;
        if (item_cnt > 0) {
          ok = mbar_wait(kv_empty, (item_cnt - 1) & 1u, abort_flag, lim);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(kv_full, 2 * SM::kTileBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(sm + SM::kK + b * SM::kBoxBytes, &tmK, kv_full, it.kvh * D + 64 * b, it.kt * kTile);
          tma_load_2d(sm + SM::kV + b * SM::kBoxBytes, &tmV, kv_full, it.kvh * D + 64 * b, it.kt * kTile);
        }
        last_kv = static_cast<int>(item_cnt);
        for (int t = 0; t < it.n_steps; ++t) {
          const int qt = entry_idx(it.ent(t / p.G));
          const int h = it.kvh * p.G + (t % p.G);
          // Q and its row statistics (released after the step's dK MMA), then dO (released
          // after the step's dV MMA)
          const uint32_t st = gq % SQ, u = gq / SQ;
          if (u > 0) {
            ok = mbar_wait(&q_empty[st], (u - 1) & 1u, abort_flag, lim);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(&q_full[st], SM::kTileBytes + SM::kStatBytes);
#pragma unroll
          for (int b = 0; b < D / 64; ++b)
            tma_load_2d(sm + SM::kQ + st * SM::kTileBytes + b * SM::kBoxBytes, &tmQ, &q_full[st],
                        h * D + 64 * b, qt * kTile);
          const size_t so = static_cast<size_t>(h) * p.qpad + static_cast<size_t>(qt) * kTile;
          uint8_t* sst = sm + SM::kStat + st * SM::kStatBytes;
          bulk_load(sst, p.lse2 + so, kTile * 4, &q_full[st]);
          bulk_load(sst + kTile * 4, p.rowD + so, kTile * 4, &q_full[st]);
          last_q[st] = static_cast<int>(u);
          const uint32_t sd = gq % SD, ud = gq / SD;
          if (ud > 0) {
            ok = mbar_wait(&do_empty[sd], (ud - 1) & 1u, abort_flag, lim);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(&do_full[sd], SM::kTileBytes);
#pragma unroll
          for (int b = 0; b < D / 64; ++b)
            tma_load_2d(sm + SM::kDO + sd * SM::kTileBytes + b * SM::kBoxBytes, &tmDO, &do_full[sd],
                        h * D + 64 * b, qt * kTile);
          last_do[sd] = static_cast<int>(ud);
          ++gq;
        }
        ++item_cnt;
      }
      if (!ok) {
        record_abort(abort_flag, p.status);
        const uint64_t short_lim = 100000000ull;
        if (last_kv >= 0) mbar_wait(kv_full, static_cast<uint32_t>(last_kv) & 1u, nullptr, short_lim);
        for (int s = 0; s < SQ; ++s)
          if (last_q[s] >= 0) mbar_wait(&q_full[s], static_cast<uint32_t>(last_q[s]) & 1u, nullptr, short_lim);
        for (int s = 0; s < SD; ++s)
          if (last_do[s] >= 0) mbar_wait(&do_full[s], static_cast<uint32_t>(last_do[s]) & 1u, nullptr, short_lim);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_st = make_idesc_bf16(128, 128, false, false);  // S^T, dP^T: N = 128 queries
      constexpr uint32_t idesc_acc = make_idesc_bf16(128, D, false, true);    // dV, dK: B MN-major
      constexpr uint32_t idesc_dq = make_idesc_bf16(128, D, true, true);      // dQ: A and B MN-major
      const uint32_t sK = smem_u32(sm + SM::kK), sV = smem_u32(sm + SM::kV);
      const uint32_t sQ = smem_u32(sm + SM::kQ), sDO = smem_u32(sm + SM::kDO), sDS = smem_u32(sm + SM::kDS);
      const uint32_t tS = tbase, tP = tbase + 128, tDV = tbase + 256, tDK = tbase + 256 + D;
      uint32_t item_cnt = 0, gq = 0;
      bool ok = true;
      for (int wave = 0; ok; ++wave) {
        const int item = sched_item(wave);
        if (item >= p.n_items) break;
        const BwdItem it = decode_item(p, item);
        if (it.n_steps == 0) continue;
        ok = mbar_wait(kv_full, item_cnt & 1u, abort_flag, lim);
        if (!ok) break;
        {  // S^T of the item's first step
          const uint32_t st = gq % SQ;
          ok = mbar_wait(&q_full[st], (gq / SQ) & 1u, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          issue_kmajor<D>(tS, sK, sQ + st * SM::kTileBytes, idesc_st);  // S^T = K Q^T
          umma_commit(s_full);
        }
        for (int t = 0; t < it.n_steps; ++t) {
          const uint32_t st = gq % SQ, sd = gq % SD;
          const uint32_t q_s = sQ + st * SM::kTileBytes, do_s = sDO + sd * SM::kTileBytes;
          if (gq > 0) {  // the previous dQ has been drained from the dP^T columns
            ok = mbar_wait(dq_empty, (gq - 1) & 1u, abort_flag, lim);
            if (!ok) break;
          }
          ok = mbar_wait(&do_full[sd], (gq / SD) & 1u, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          issue_kmajor<D>(tP, sV, do_s, idesc_st);  // dP^T = V dO^T
          umma_commit(dp_full);
          ok = mbar_wait(p_full, gq & 1u, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          issue_ts<D>(tDV, tS, do_s, idesc_acc, t > 0);  // dV += P^T dO
          umma_commit(&do_empty[sd]);                     // dO's last reader
          if (t + 1 < it.n_steps) {
            // S^T of the next step now, so P^T of step t+1 is computed while dK and dQ of this
            // step run (P^T of step t has been read by the dV MMA issued just before)
            const uint32_t g1 = gq + 1, st1 = g1 % SQ;
            ok = mbar_wait(&q_full[st1], (g1 / SQ) & 1u, abort_flag, lim);
            if (!ok) break;
            tc_fence_after();
            issue_kmajor<D>(tS, sK, sQ + st1 * SM::kTileBytes, idesc_st);
            umma_commit(s_full);
          }
          ok = mbar_wait(ds_full, gq & 1u, abort_flag, lim);
          if (!ok) break;
          tc_fence_after();
          issue_ts<D>(tDK, tP, q_s, idesc_acc, t > 0);  // dK += dS^T Q
          issue_dq<D>(tP, sDS, sK, idesc_dq);           // dQ = dS K (into the dP^T columns)
          umma_commit(dq_full);
          umma_commit(&q_empty[st]);
          ++gq;
        }
        if (!ok) break;
        umma_commit(kv_empty);
        umma_commit(dkv_full);
        ++item_cnt;
      }
      if (!ok) record_abort(abort_flag, p.status);
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr, 100000000ull);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// -D_i = -(dO_i . O_i) and -LSE_i * log2(e) per (head, row), padded to whole tiles (stored
// negated so the main kernel adds them with packed pair instructions); zero the dq
// accumulator.  D / 8 lanes per (row, head), 16 bytes of O and of dO per lane, and kUnroll
// row groups per warp pass with every load issued before the first use, so that enough
// bytes are in flight to run at the copy bandwidth.
template <int D>
__global__ void __launch_bounds__(256) ffa_bwd_pre(const __nv_bfloat16* __restrict__ out,
                                                   const __nv_bfloat16* __restrict__ dout,
                                                   const float* __restrict__ lse, float* __restrict__ rowD,
                                                   float* __restrict__ lse2, float* __restrict__ dqacc, int nq,
                                                   int hq, int qpad) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int kLanes = D / 8;          // lanes of one (row, head)
  constexpr int kRows = 32 / kLanes;     // (row, head) units per warp and group
  constexpr int kUnroll = 4;
  constexpr int kPass = kRows * kUnroll;  // units per warp pass
  const int lane = threadIdx.x & 31, sub = lane / kLanes, sl = lane % kLanes;
  const size_t nwarps = static_cast<size_t>(gridDim.x) * (blockDim.x >> 5);
  const size_t total = static_cast<size_t>(qpad) * hq;
  for (size_t w0 = (blockIdx.x * static_cast<size_t>(blockDim.x >> 5) + (threadIdx.x >> 5)) * kPass; w0 < total;
       w0 += nwarps * kPass) {
    uint4 a[kUnroll], b[kUnroll];
    size_t base[kUnroll];
    bool live[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const size_t wi = w0 + u * kRows + sub;
      const int h = static_cast<int>(wi / qpad);
      const int i = static_cast<int>(wi - static_cast<size_t>(h) * qpad);
      live[u] = wi < total && i < nq;
      base[u] = live[u] ? (static_cast<size_t>(i) * hq + h) * D + sl * 8 : 0;
      a[u] = live[u] ? *reinterpret_cast<const uint4*>(out + base[u]) : make_uint4(0u, 0u, 0u, 0u);
      b[u] = live[u] ? *reinterpret_cast<const uint4*>(dout + base[u]) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t av[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, bv[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
      float dsum = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        dsum += __uint_as_float(av[e] << 16) * __uint_as_float(bv[e] << 16);
        dsum += __uint_as_float(av[e] & 0xffff0000u) * __uint_as_float(bv[e] & 0xffff0000u);
      }
#pragma unroll
      for (int o = kLanes / 2; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
      const size_t wi = w0 + u * kRows + sub;
      if (live[u]) {
        float4* z = reinterpret_cast<float4*>(dqacc + base[u]);
        z[0] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        z[1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
      if (sl == 0 && wi < total) {
        const int h = static_cast<int>(wi / qpad);
        const int i = static_cast<int>(wi - static_cast<size_t>(h) * qpad);
        float l2 = -INFINITY;
        if (i < nq) {
          const float l = lse[static_cast<size_t>(h) * nq + i];
          l2 = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
        }
        rowD[wi] = i < nq ? -dsum : 0.0f;
        lse2[wi] = l2;
      }
    }
  }
}

__global__ void __launch_bounds__(256) ffa_bwd_dq_convert(const float* __restrict__ acc,
                                                          __nv_bfloat16* __restrict__ dq, size_t n) {
  pdl_wait();
  const size_t n4 = n / 4;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(acc)[i];
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    reinterpret_cast<uint2*>(dq)[i] = o;
  }
}

template <int D, bool kCap, bool kBias, bool kDet>
cudaError_t launch_impl(const BwdArgs& a, cudaStream_t stream) {
  using SM = BwdSmem<D>;
  auto kern = ffa_bwd_kernel<D, kCap, kBias, kDet>;
  // once per device: the shared-memory attribute applies to the device current when it is set
  static std::once_flag once[kMaxDevices];
  static cudaError_t setup_err[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    setup_err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kAlloc);
  });
  if (setup_err[dev] != cudaSuccess) return setup_err[dev];
  const auto& P = a.P;
  const int qpad = P.nqt * kTile;
  const int nsm = num_sms();
  {
    // (row, head) units over warps of D / 8 lanes per unit, four groups per warp pass
    const size_t warps = (static_cast<size_t>(qpad) * P.hq * (D / 8) / 32 + 3) / 4;
    const int blocks = static_cast<int>(std::min<size_t>((warps + 7) / 8, static_cast<size_t>(nsm) * 16));
    // programmatic dependents from here on: each kernel's launch overlaps the tail of the one
    // before it and waits (pdl_wait) before it touches what that one writes
    cudaError_t e = launch_pdl(ffa_bwd_pre<D>, dim3(blocks), dim3(256), 0, stream,
                               static_cast<const __nv_bfloat16*>(a.out), static_cast<const __nv_bfloat16*>(a.dout),
                               static_cast<const float*>(a.lse), a.rowD, a.lse2, a.dqacc, static_cast<int>(P.nq), P.hq,
                               qpad);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mq, mk, mv, mdo, mdq;
  if (!encode_tile_map_f32(&mdq, a.dqacc, static_cast<uint64_t>(P.hq) * D, P.nq, 32, kTile) ||
      !encode_tile_map(&mq, a.q, static_cast<uint64_t>(P.hq) * D, P.nq, 64, kTile) ||
      !encode_tile_map(&mdo, a.dout, static_cast<uint64_t>(P.hq) * D, P.nq, 64, kTile) ||
      !encode_tile_map(&mk, a.k, static_cast<uint64_t>(P.hkv) * D, P.nk, 64, kTile) ||
      !encode_tile_map(&mv, a.v, static_cast<uint64_t>(P.hkv) * D, P.nk, 64, kTile))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.nq = P.nq; p.nk = P.nk; p.hq = P.hq; p.hkv = P.hkv; p.G = P.hq / P.hkv;
  p.nqt = P.nqt; p.nkt = P.nkt;
  p.n_items = P.nkt * P.hkv;
  p.qpad = qpad;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.cap_c = a.softcap * kLog2e;
  p.cap_k = a.softcap > 0.0f ? 2.0f * a.scale * kLog2e / a.softcap : 0.0f;
  p.inv_cap_c = a.softcap > 0.0f ? 1.0f / p.cap_c : 0.0f;
  fold_cap_poly(a.scale, a.softcap, p.cap_q, &p.cap_slim);  // (its interval: cap_slim)
  {
    float q5[3];
    fold_cap_poly5(a.scale, a.softcap, q5);
    for (int i = 0; i < 3; ++i) p.cap_q[i] = q5[i];
    p.cap_q[3] = 0.0f;
  }
  p.plan = a.plan;
  p.lse2 = a.lse2;
  p.rowD = a.rowD;
  p.dqacc = a.dqacc;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.alibi = a.alibi;
  p.det = a.deterministic;
  p.tile_rank = a.tile_rank;
  p.dq_sem = a.dq_sem;
  p.status = a.status;
  p.wait_limit_ns = a.wait_limit_ns;
  p.stall = a.stall_test;
  const int grid = p.n_items < nsm ? p.n_items : nsm;
  if (grid > 0) {
    if (g_kernel_events.bwd_start != nullptr) cudaEventRecord(g_kernel_events.bwd_start, stream);
    if (kDet) {
      // CTAs wait on one another's dq additions: all of them must be resident at once
      void* args[] = {&mq, &mk, &mv, &mdo, &mdq, &p};
      cudaError_t le = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(kThreads),
                                                   args, SM::kAlloc, stream);
      if (le != cudaSuccess) return le;
    } else {
      cudaError_t le = launch_pdl(kern, dim3(grid), dim3(kThreads), SM::kAlloc, stream, mq, mk, mv, mdo, mdq, p);
      if (le != cudaSuccess) return le;
    }
    if (g_kernel_events.bwd_stop != nullptr) cudaEventRecord(g_kernel_events.bwd_stop, stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const size_t n = static_cast<size_t>(P.nq) * P.hq * D;
  const int blocks = static_cast<int>(std::min<size_t>((n / 4 + 255) / 256, static_cast<size_t>(nsm) * 8));
  if (blocks <= 0) return cudaSuccess;
  if (kDet) {  // (after the cooperative launch: plain stream order)
    ffa_bwd_dq_convert<<<blocks, 256, 0, stream>>>(a.dqacc, static_cast<__nv_bfloat16*>(a.dq), n);
    return cudaGetLastError();
  }
  return launch_pdl(ffa_bwd_dq_convert, dim3(blocks), dim3(256), 0, stream, static_cast<const float*>(a.dqacc),
                    static_cast<__nv_bfloat16*>(a.dq), n);
}

}  // namespace

template <int D, bool kCap, bool kBias>
cudaError_t launch_det(const BwdArgs& a, cudaStream_t s) {
  return a.deterministic ? launch_impl<D, kCap, kBias, true>(a, s) : launch_impl<D, kCap, kBias, false>(a, s);
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s) {
  const bool cap = a.softcap > 0.0f, bias = a.alibi != nullptr;
  if (a.P.d == 64) {
    if (bias) return cap ? launch_det<64, true, true>(a, s) : launch_det<64, false, true>(a, s);
    return cap ? launch_det<64, true, false>(a, s) : launch_det<64, false, false>(a, s);
  }
  if (bias) return cap ? launch_det<128, true, true>(a, s) : launch_det<128, false, true>(a, s);
  return cap ? launch_det<128, true, false>(a, s) : launch_det<128, false, false>(a, s);
}

}  // namespace ffa
