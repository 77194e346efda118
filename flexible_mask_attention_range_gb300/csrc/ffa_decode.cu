// ffa_fwd_decode: attention for a few new query tokens per sequence (decoding) with GQA
// head packing, over a dense or paged key/value cache.
//
// A decoding step has one (or a few) query tokens per sequence and a long key sequence.
// The FlexAttention paper (section 4, template-based lowering) has a separate decoding
// template with grouped-query attention support, compared against FlashDecoding in section
// 6; it does not spell out that template.  On the token-major layout the forward kernel's
// 128-row query tiles would mix many sequences and read every key tile once per pair of
// query heads, so this library's decoding path packs P query heads of each token into P
// consecutive rows of a problem with Hq / P heads:
//     packed row (i * P + g), packed head h  <-  token i, query head h * P + g,
// with P = G = Hq / Hkv: one packed head per key/value head.  A packed query tile then holds
// 128 / G tokens, and every key tile is read once per (query tile, key/value head).  The
// forward pass runs in its key-split form: a work item is one packed query tile and a chunk of
// its key tiles, the item's two softmax warpgroups take alternate key tiles, so each key tile
// meets one 128-row MMA pair instead of two, and each warpgroup leaves a partial result.  The
// partials of all chunks are merged by LSE, as split rows of the plain forward pass are.
//
// Slices are rewritten for the packed rows: a FULL slice [qs, qe) x [ks, ke) becomes
// [qs * P, qe * P) x [ks, ke); a CAUSAL slice with m = qe - qs query tokens becomes m FULL
// slices, one per token i, over the keys that token sees under the bottom-right alignment
// used everywhere in this library (j <= i + ke - qe).  max_seqlen_q bounds m, so the
// rewritten list has a fixed length n_ranges * max_seqlen_q (unused entries are empty
// slices).  Packing and rewriting share one small kernel before the forward pass (dense or
// paged); the forward pass's LSE merge writes O and LSE in the caller's layout.  With ALiBi (FlexAttention paper, sections 2 and 3.1; decoding with GQA
// and ALiBi is one of the cases its section 6 measures) a packed row keeps the slope of its
// query head and the position of its token, so the bias is the one of the unpacked problem.
#include <cstdint>

#include "../../include/ffa.h"
#include "ffa_internal.h"

namespace ffa {
namespace {

// q [N, Hq, d] -> qp [N * P, Hq / P, d], in 16-byte units (d / 8 of them per row); block b of
// nb blocks.
__device__ void decode_pack_q(const uint4* __restrict__ q, uint4* __restrict__ qp, int64_t n, int hq, int P, int d,
                              int b, int nb) {
  const int hp = hq / P;
  const int64_t per_row = d / 8;
  const int64_t total = n * hq * per_row;
  for (int64_t idx = b * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(nb) * blockDim.x) {
    const int64_t row = idx / per_row, c = idx - row * per_row;  // packed row = (i * P + g) * hp + h
    const int64_t h = row % hp, ig = row / hp;
    const int64_t g = ig % P, i = ig / P;
    qp[idx] = q[(i * hq + h * P + g) * per_row + c];
  }
}

// Slice s, token slot u -> rewritten slice s * M + u (see the file comment).  Invalid slices
// (bounds, type, or a CAUSAL slice longer than M) are reported with FFA_STATUS_BAD_RANGE and
// dropped, as the planner does for the plain forward pass.  Block b of nb blocks.
__device__ void decode_slices(const int32_t* __restrict__ qr, const int32_t* __restrict__ kr,
                              const int32_t* __restrict__ ty, int R, int M, int P, int64_t nq, int64_t nk,
                              int32_t* __restrict__ qr2, int32_t* __restrict__ kr2, int32_t* __restrict__ ty2,
                              int32_t* status, int b, int nb) {
  const int64_t total = static_cast<int64_t>(R) * M;
  for (int64_t slot = b * static_cast<int64_t>(blockDim.x) + threadIdx.x; slot < total;
       slot += static_cast<int64_t>(nb) * blockDim.x) {
    const int64_t s = slot / M;
    const int u = static_cast<int>(slot - s * M);
    const int64_t qs = qr[2 * s], qe = qr[2 * s + 1], ks = kr[2 * s], ke = kr[2 * s + 1];
    const int t = ty[s];
    int64_t a = 0, b = 0, c = 0, e = 0;  // empty slice unless set below
    const bool valid = qs >= 0 && qs <= qe && qe <= nq && ks >= 0 && ks <= ke && ke <= nk && (t == FFA_FULL || t == FFA_CAUSAL);
    const int64_t m = qe - qs;
    if (!valid || (t == FFA_CAUSAL && m > M)) {
      if (u == 0 && status != nullptr) atomicOr(status, FFA_STATUS_BAD_RANGE);
    } else if (t == FFA_FULL) {
      if (u == 0) {
        a = qs * P; b = qe * P; c = ks; e = ke;
      }
    } else if (u < m) {
      const int64_t i = qs + u;
      const int64_t hi = ke - m + 1 + u < ke ? ke - m + 1 + u : ke;  // keys j < hi, i.e. j <= i + ke - qe
      if (hi > ks) {
        a = i * P; b = (i + 1) * P; c = ks; e = hi;
      }
    }
    qr2[2 * slot] = static_cast<int32_t>(a);
    qr2[2 * slot + 1] = static_cast<int32_t>(b);
    kr2[2 * slot] = static_cast<int32_t>(c);
    kr2[2 * slot + 1] = static_cast<int32_t>(e);
    ty2[slot] = FFA_FULL;
  }
}

// Both preparation steps in one launch: the first pack_blocks blocks pack q, the others
// rewrite the slices.
__global__ void __launch_bounds__(256) decode_prepare(const uint4* __restrict__ q, uint4* __restrict__ qp, int64_t n,
                                                      int hq, int P, int d, int pack_blocks,
                                                      const int32_t* __restrict__ qr, const int32_t* __restrict__ kr,
                                                      const int32_t* __restrict__ ty, int R, int M, int64_t nk,
                                                      int32_t* __restrict__ qr2, int32_t* __restrict__ kr2,
                                                      int32_t* __restrict__ ty2, int32_t* status) {
  pdl_launch_dependents();  // the planner's first kernel may start (it waits for this one)
  if (static_cast<int>(blockIdx.x) < pack_blocks)
    decode_pack_q(q, qp, n, hq, P, d, blockIdx.x, pack_blocks);
  else
    decode_slices(qr, kr, ty, R, M, P, n, nk, qr2, kr2, ty2, status, blockIdx.x - pack_blocks,
                  gridDim.x - pack_blocks);
}

// Query heads per packed row group: all G of a key/value head.
int pack_factor(int G) { return G; }

struct DecodeLayout {
  size_t qp = 0, qr2 = 0, kr2 = 0, ty2 = 0, inner = 0, total = 0;
  int64_t R2 = 0;
  int P = 1;
  ffa_shape inner_shape{};
};

bool decode_layout(const ffa_shape* s, int32_t n_ranges, int32_t max_seqlen_q, DecodeLayout* L) {
  if (s == nullptr || n_ranges < 0 || max_seqlen_q < 1 || s->num_heads_kv < 1 || s->num_heads_q < 1 ||
      s->num_heads_q % s->num_heads_kv != 0 || s->total_q < 0)
    return false;
  const int P = pack_factor(s->num_heads_q / s->num_heads_kv);
  const int64_t R2 = static_cast<int64_t>(n_ranges) * max_seqlen_q;
  if (R2 > (static_cast<int64_t>(1) << 30)) return false;
  L->R2 = R2;
  L->P = P;
  L->inner_shape.total_q = s->total_q * P;
  L->inner_shape.total_k = s->total_k;
  L->inner_shape.num_heads_q = s->num_heads_q / P;
  L->inner_shape.num_heads_kv = s->num_heads_kv;
  L->inner_shape.head_dim = s->head_dim;
  if (check_shape(&L->inner_shape, static_cast<int32_t>(R2)) != FFA_OK) return false;
  const size_t inner = make_layout(L->inner_shape.total_q, L->inner_shape.total_k, L->inner_shape.num_heads_q,
                                   L->inner_shape.num_heads_kv, L->inner_shape.head_dim, static_cast<int32_t>(R2),
                                   /*key_split=*/true)
                           .fwd_total;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
  const size_t rows = static_cast<size_t>(s->total_q) * s->num_heads_q;
  L->qp = take(rows * s->head_dim * 2);
  L->qr2 = take(static_cast<size_t>(R2) * 8);
  L->kr2 = take(static_cast<size_t>(R2) * 8);
  L->ty2 = take(static_cast<size_t>(R2) * 4);
  L->inner = take(inner);
  L->total = o;
  return true;
}

}  // namespace
}  // namespace ffa

using namespace ffa;

extern "C" {

size_t ffa_fwd_decode_workspace_size(const ffa_shape* shape, int32_t n_ranges, int32_t max_seqlen_q) {
  DecodeLayout L;
  if (!decode_layout(shape, n_ranges, max_seqlen_q, &L)) return 0;
  return L.total;
}

int ffa_fwd_decode(const ffa_shape* shape, const void* q, const void* k, const void* v, const int32_t* page_table,
                   int32_t page_size, int64_t n_pages, const int32_t* q_ranges, const int32_t* k_ranges,
                   const int32_t* attn_type_map, int32_t n_ranges, int32_t max_seqlen_q, float softmax_scale,
                   float softcap, void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* status,
                   void* stream, const ffa_options* options) {
  if (shape == nullptr || n_ranges < 0 || max_seqlen_q < 1) return FFA_ERR_INVALID_ARG;
  if (check_options(options) != FFA_OK) return FFA_ERR_INVALID_ARG;
  if (shape->head_dim != 64 && shape->head_dim != 128) return FFA_ERR_UNSUPPORTED;
  if (shape->num_heads_kv < 1 || shape->num_heads_q < 1 || shape->num_heads_q % shape->num_heads_kv != 0)
    return FFA_ERR_INVALID_ARG;
  const int P = pack_factor(shape->num_heads_q / shape->num_heads_kv);
  if (shape->total_q < 0 || shape->total_q * P > FFA_MAX_TOKENS) return FFA_ERR_UNSUPPORTED;
  DecodeLayout L;
  if (!decode_layout(shape, n_ranges, max_seqlen_q, &L)) return FFA_ERR_INVALID_ARG;
  const int64_t nq = shape->total_q;
  if (nq > 0 && (q == nullptr || out == nullptr || lse == nullptr)) return FFA_ERR_INVALID_ARG;
  if (n_ranges > 0 && (q_ranges == nullptr || k_ranges == nullptr || attn_type_map == nullptr))
    return FFA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FFA_ERR_INVALID_ARG;
  if (nq == 0) return FFA_OK;
  if (workspace == nullptr || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FFA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* wb = static_cast<char*>(workspace);
  const int hq = shape->num_heads_q, d = shape->head_dim;
  const int nsm = num_sms();
  const int64_t units = nq * hq * (d / 8);
  const int blocks = static_cast<int>(units / 256 + 1 < static_cast<int64_t>(nsm) * 8 ? units / 256 + 1 : nsm * 8);
  int32_t* qr2 = reinterpret_cast<int32_t*>(wb + L.qr2);
  int32_t* kr2 = reinterpret_cast<int32_t*>(wb + L.kr2);
  int32_t* ty2 = reinterpret_cast<int32_t*>(wb + L.ty2);
  const int sb = L.R2 > 0 ? static_cast<int>(L.R2 / 256 + 1 < static_cast<int64_t>(nsm) * 4 ? L.R2 / 256 + 1 : nsm * 4)
                          : 0;
  decode_prepare<<<blocks + sb, 256, 0, s>>>(static_cast<const uint4*>(q), reinterpret_cast<uint4*>(wb + L.qp), nq, hq,
                                             P, d, blocks, q_ranges, k_ranges, attn_type_map, n_ranges, max_seqlen_q,
                                             shape->total_k, qr2, kr2, ty2, status);
  if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
  // the forward pass over the packed problem; with ALiBi each packed row takes the slope of
  // its query head and the position of its token (FwdArgs::alibi_pack)
  FwdCall c;
  c.shape = &L.inner_shape;
  c.q = wb + L.qp; c.k = k; c.v = v;
  c.q_ranges = qr2; c.k_ranges = kr2; c.types = ty2; c.n_ranges = static_cast<int32_t>(L.R2);
  c.softmax_scale = softmax_scale; c.softcap = softcap;
  // (the packed problem's O and LSE have the caller's sizes; with the key split nothing but
  // the merge writes them, through the unpacking map below)
  c.out = out; c.lse = lse;
  c.status = status; c.stream = stream; c.options = options;
  c.alibi_pack = P;
  c.key_split = true;
  c.after_own_kernel = true;
  // every packed row goes through the LSE merge, which writes the caller's layout directly
  c.unpack_out = out;
  c.unpack_lse = lse;
  if (page_table != nullptr) {
    c.paged = true;
    c.page_table = page_table; c.page_size = page_size; c.n_pages = n_pages;
  }
  return fwd_with_workspace(c, wb + L.inner, workspace_bytes - L.inner);
}

}  // extern "C"
