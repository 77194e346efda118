"""Plain, slow, float64 CPU oracle for range-masked softmax attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the benchmark's
CPU-baseline leg may import or call this module.  It shares no code with the CUDA path
(no kernels, headers, helpers or constants) and it never reads values produced there.

What it computes (the plain definition, no blocking or fusion beyond row blocks that cover
each row's whole key set):

  * Interface and slice semantics -- MagiAttention issue #180, "Using dummy/padded
    attention slices with flex_flash_attn_func for torch.compile static shapes":
    ``flex_flash_attn_func(q, k, v, q_ranges, k_ranges, attn_type_map, softmax_scale,
    softcap) -> (out, lse)`` on packed tokens ``q:[Nq,Hq,d]``, ``k,v:[Nk,Hkv,d]``; the mask
    is a list of (q_range, k_range, type) slices with type 0 = FULL and 1 = CAUSAL
    (question's code comments); a slice whose Q-range or K-range has start == end covers
    no area and is ignored (maintainer's reply, "Mechanism").
  * Composition of several slices -- "Flex Attention: A Programming Model for Generating
    Optimized Attention Kernels", section 3 (Composability): masks combine by logical OR,
    e.g. prefix OR causal gives PrefixLM.  A (query, key) pair is visible once, no matter
    how many slices cover it (union semantics).
  * Softcapping (same paper, section 2, attention variants) keeps every logit inside
    (-softcap, softcap); the reading taken here: x = softcap * tanh(scale * q.k / softcap),
    softcap = 0 disables it.
  * Safe softmax (same paper, section 1): rows with no visible key produce O = 0 and
    LSE = -inf instead of NaN.
  * ALiBi score modification (same paper, sections 2 and 3.1: each score gets a bias that
    grows with the distance between query and key): optional per-query-head slopes; reading taken
    here: x_ij = softcap(scale * q.k) + slope_h * (j - i) with i, j the packed token
    positions (the distance between two tokens of one document equals their in-document
    distance).

  * Paged key/value cache -- same paper, section 5 (Paged Attention): the keys of a
    sequence live in a shared physical cache, reached through a page table; masks and score
    modifications keep seeing logical positions.  Logical key j is row j % page_size of
    physical page page_table[j // page_size] (``gather_pages``); attention is then the plain
    definition over the gathered logical keys.

Readings where the pages are silent (each is listed in the design notes):
  * CAUSAL alignment inside a slice with unequal q and k lengths: bottom-right.  Pair (i, j)
    of slice [qs,qe) x [ks,ke) is visible iff qs <= i < qe, ks <= j < ke and
    j <= i + ke - qe.  Under this reading the issue's 2-slice example ([half,N) x [0,N),
    CAUSAL) is the usual "second half causal over all tokens" mask.
  * softmax_scale None -> 1/sqrt(d); LSE is the natural log, laid out [Hq, Nq].
  * GQA: query head h reads key/value head h // (Hq // Hkv).
  * A slice with a bound outside [0, N], start > end, or an unknown type is invalid: it is
    dropped and counted (the CUDA path reports it through its status word).
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

FULL = 0
CAUSAL = 1
TILE_EMPTY = 0
TILE_PARTIAL = 1
TILE_FULL = 2


# ----------------------------------------------------------------------------------------
# Slices
# ----------------------------------------------------------------------------------------

def normalize_slices(q_ranges, k_ranges, attn_type_map, total_q: int, total_k: int
                     ) -> Tuple[np.ndarray, int]:
    """Validate and keep the slices that cover area.

    Returns (slices, n_invalid): ``slices`` is an int64 array [R', 5] of rows
    (qs, qe, ks, ke, type) in input order; zero-area slices (start == end in either range)
    are dropped silently, malformed ones are dropped and counted.
    """
    qr = np.asarray(q_ranges, dtype=np.int64).reshape(-1, 2)
    kr = np.asarray(k_ranges, dtype=np.int64).reshape(-1, 2)
    ty = np.asarray(attn_type_map, dtype=np.int64).reshape(-1)
    assert qr.shape[0] == kr.shape[0] == ty.shape[0]
    keep: List[Tuple[int, int, int, int, int]] = []
    invalid = 0
    for r in range(ty.shape[0]):
        qs, qe = int(qr[r, 0]), int(qr[r, 1])
        ks, ke = int(kr[r, 0]), int(kr[r, 1])
        t = int(ty[r])
        ok = (0 <= qs <= qe <= total_q) and (0 <= ks <= ke <= total_k) and t in (FULL, CAUSAL)
        if not ok:
            invalid += 1
            continue
        if qs == qe or ks == ke:
            continue
        keep.append((qs, qe, ks, ke, t))
    arr = np.array(keep, dtype=np.int64).reshape(-1, 5)
    return arr, invalid


def _rows_touching(slices: np.ndarray, r0: int, r1: int) -> np.ndarray:
    if slices.shape[0] == 0:
        return slices
    sel = (slices[:, 0] < r1) & (slices[:, 1] > r0)
    return slices[sel]


def row_intervals(slices: np.ndarray, rows: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per (row, slice): the visible key interval [lo, hi); empty when hi <= lo.

    FULL slice: [ks, ke) for qs <= i < qe.  CAUSAL slice (bottom-right aligned):
    [ks, min(ke, i + ke - qe + 1)) for qs <= i < qe.
    """
    rows = np.asarray(rows, dtype=np.int64)
    if slices.shape[0] == 0:
        z = np.zeros((rows.shape[0], 0), dtype=np.int64)
        return z, z
    qs, qe, ks, ke, t = (slices[:, c][None, :] for c in range(5))
    i = rows[:, None]
    inside = (i >= qs) & (i < qe)
    hi_causal = np.minimum(ke, i + ke - qe + 1)
    hi = np.where(t == CAUSAL, hi_causal, ke)
    lo = np.broadcast_to(ks, hi.shape).copy()
    hi = np.where(inside, hi, lo)
    hi = np.maximum(hi, lo)
    return lo, hi


def key_intervals(slices: np.ndarray, keys: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per (key, slice): the interval [lo, hi) of query rows that see key j.

    Same predicate as ``row_intervals`` solved for i: FULL -> [qs, qe);
    CAUSAL -> [max(qs, j - ke + qe), qe); both only when ks <= j < ke.
    """
    keys = np.asarray(keys, dtype=np.int64)
    if slices.shape[0] == 0:
        z = np.zeros((keys.shape[0], 0), dtype=np.int64)
        return z, z
    qs, qe, ks, ke, t = (slices[:, c][None, :] for c in range(5))
    j = keys[:, None]
    inside = (j >= ks) & (j < ke)
    lo = np.where(t == CAUSAL, np.maximum(qs, j - ke + qe), np.broadcast_to(qs, inside.shape))
    hi = np.broadcast_to(qe, inside.shape).copy()
    lo = np.where(inside, lo, hi)
    lo = np.minimum(lo, hi)
    return lo, hi


def mask_block(slices: np.ndarray, rows: np.ndarray, c0: int, c1: int) -> np.ndarray:
    """Boolean visibility of rows x [c0, c1): OR over slices of their visible intervals."""
    lo, hi = row_intervals(slices, rows)
    j = np.arange(c0, c1, dtype=np.int64)[None, :]
    m = np.zeros((len(rows), c1 - c0), dtype=bool)
    for r in range(lo.shape[1]):
        m |= (j >= lo[:, r:r + 1]) & (j < hi[:, r:r + 1])
    return m


def dense_mask(q_ranges, k_ranges, attn_type_map, total_q: int, total_k: int) -> np.ndarray:
    """The full [Nq, Nk] boolean mask (small problems only)."""
    sl, _ = normalize_slices(q_ranges, k_ranges, attn_type_map, total_q, total_k)
    return mask_block(sl, np.arange(total_q), 0, total_k)


def _union_length(lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    """Length of the union of intervals [lo[..., r], hi[..., r]) over the last axis."""
    if lo.shape[-1] == 0:
        return np.zeros(lo.shape[:-1], dtype=np.int64)
    empty = hi <= lo
    big = np.iinfo(np.int64).max // 4
    lo_s = np.where(empty, big, lo)
    hi_s = np.where(empty, big, hi)
    order = np.argsort(lo_s, axis=-1, kind="stable")
    lo_s = np.take_along_axis(lo_s, order, axis=-1)
    hi_s = np.take_along_axis(hi_s, order, axis=-1)
    total = np.zeros(lo.shape[:-1], dtype=np.int64)
    cur = np.full(lo.shape[:-1], -big, dtype=np.int64)
    for r in range(lo.shape[-1]):
        a, b = lo_s[..., r], hi_s[..., r]
        valid = a < big
        start = np.maximum(a, cur)
        total += np.where(valid, np.maximum(0, b - start), 0)
        cur = np.where(valid, np.maximum(cur, b), cur)
    return total


def visible_pairs(q_ranges, k_ranges, attn_type_map, total_q: int, total_k: int,
                  block: int = 4096) -> int:
    """Number of visible (query, key) pairs under union semantics (exact integer)."""
    sl, _ = normalize_slices(q_ranges, k_ranges, attn_type_map, total_q, total_k)
    n = 0
    for r0 in range(0, total_q, block):
        r1 = min(total_q, r0 + block)
        rel = _rows_touching(sl, r0, r1)
        lo, hi = row_intervals(rel, np.arange(r0, r1))
        n += int(_union_length(lo, hi).sum())
    return n


def tile_classes(q_ranges, k_ranges, attn_type_map, total_q: int, total_k: int,
                 tile: int = 128) -> np.ndarray:
    """Class of each tile of the global tile grid: uint8 [ceil(Nq/tile), ceil(Nk/tile)].

    FULL (2) if every in-bounds (i, j) of the tile is visible, EMPTY (0) if none is,
    PARTIAL (1) otherwise (block classification as in the Flex Attention paper, section 4,
    "Block Sparsity" and "Full Block Optimization").
    """
    sl, _ = normalize_slices(q_ranges, k_ranges, attn_type_map, total_q, total_k)
    nqt = -(-total_q // tile)
    nkt = -(-total_k // tile)
    out = np.zeros((nqt, nkt), dtype=np.uint8)
    c0 = np.arange(nkt, dtype=np.int64) * tile
    c1 = np.minimum(c0 + tile, total_k)
    width = c1 - c0
    for qt in range(nqt):
        r0, r1 = qt * tile, min(total_q, qt * tile + tile)
        rel = _rows_touching(sl, r0, r1)
        if rel.shape[0] == 0:
            continue
        lo, hi = row_intervals(rel, np.arange(r0, r1))          # [rows, R]
        lo_c = np.clip(lo[:, None, :], c0[None, :, None], c1[None, :, None])
        hi_c = np.clip(hi[:, None, :], c0[None, :, None], c1[None, :, None])
        cov = _union_length(lo_c, hi_c)                           # [rows, nkt]
        full = np.all(cov == width[None, :], axis=0)
        empty = np.all(cov == 0, axis=0)
        out[qt] = np.where(full, TILE_FULL, np.where(empty, TILE_EMPTY, TILE_PARTIAL))
    return out


# ----------------------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------------------

def resolve_scale(softmax_scale: Optional[float], d: int) -> float:
    if softmax_scale is None or not (softmax_scale > 0):
        return 1.0 / math.sqrt(d)
    return float(softmax_scale)


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _capped(s: np.ndarray, softcap: float) -> np.ndarray:
    if softcap > 0:
        return softcap * np.tanh(s / softcap)
    return s


def _row_block_stats(qb, kk, m, scale, softcap, bias=None):
    """For one head and one row block: S, X, LSE and P per the definition."""
    s = scale * (qb @ kk.T)
    xb = _capped(s, softcap) if bias is None else _capped(s, softcap) + bias
    x = np.where(m, xb, -np.inf)
    has = m.any(axis=1)
    mx = np.where(has, np.max(np.where(m, x, -np.inf), axis=1, initial=-np.inf), 0.0)
    with np.errstate(under="ignore"):
        e = np.where(m, np.exp(x - mx[:, None]), 0.0)
    lse = np.where(has, mx + np.log(np.where(has, e.sum(axis=1), 1.0)), -np.inf)
    with np.errstate(under="ignore", invalid="ignore"):
        p = np.where(m, np.exp(x - np.where(has, lse, 0.0)[:, None]), 0.0)
    return s, p, lse


def _span(lo: np.ndarray, hi: np.ndarray) -> Tuple[int, int]:
    ne = hi > lo
    if not ne.any():
        return 0, 0
    return int(lo[ne].min()), int(hi[ne].max())


def _alibi(slopes, h, rows, c0, c1):
    if slopes is None:
        return None
    return float(slopes[h]) * (np.arange(c0, c1, dtype=np.float64)[None, :] - np.asarray(rows, dtype=np.float64)[:, None])


def forward(q, k, v, q_ranges, k_ranges, attn_type_map, softmax_scale=None,
            softcap: float = 0.0, rows: Optional[Sequence[int]] = None, block: int = 128,
            alibi_slopes: Optional[Sequence[float]] = None):
    """O and LSE.  Returns (out [n, Hq, d] f64, lse [Hq, n] f64) for all rows or ``rows``."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    nq, hq, d = q.shape
    nk, hkv, _ = k.shape
    assert hq % hkv == 0
    g = hq // hkv
    scale = resolve_scale(softmax_scale, d)
    sl, _ = normalize_slices(q_ranges, k_ranges, attn_type_map, nq, nk)
    rows = np.arange(nq) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.shape[0], hq, d))
    lse = np.full((hq, rows.shape[0]), -np.inf)
    for b0 in range(0, rows.shape[0], block):
        rb = rows[b0:b0 + block]
        rel = _rows_touching(sl, int(rb.min()), int(rb.max()) + 1)
        lo, hi = row_intervals(rel, rb)
        c0, c1 = _span(lo, hi)
        if c1 <= c0:
            continue
        m = mask_block(rel, rb, c0, c1)
        for h in range(hq):
            kh = h // g
            _, p, l = _row_block_stats(q[rb, h], k[c0:c1, kh], m, scale, softcap,
                                       _alibi(alibi_slopes, h, rb, c0, c1))
            out[b0:b0 + len(rb), h] = p @ v[c0:c1, kh]
            lse[h, b0:b0 + len(rb)] = l
    return out, lse


def _grad_block(qb, kk, vv, dob, m, scale, softcap, bias=None):
    """Analytic gradients of sum(O * dO) for one head and one row block (the ALiBi bias
    does not depend on q or k, so it enters through P only)."""
    s, p, _ = _row_block_stats(qb, kk, m, scale, softcap, bias)
    dp = dob @ vv.T
    dd = np.sum(p * dp, axis=1, keepdims=True)        # D_i = sum_j P_ij dP_ij
    dx = p * (dp - dd)
    if softcap > 0:
        th = np.tanh(s / softcap)
        ds = dx * (1.0 - th * th)
    else:
        ds = dx
    dq = scale * (ds @ kk)
    dk = scale * (ds.T @ qb)
    dv = p.T @ dob
    return dq, dk, dv


def backward(q, k, v, dout, q_ranges, k_ranges, attn_type_map, softmax_scale=None,
             softcap: float = 0.0, rows: Optional[Sequence[int]] = None,
             keys: Optional[Sequence[int]] = None, block: int = 128,
             alibi_slopes: Optional[Sequence[float]] = None):
    """Gradients of sum(O * dO) w.r.t. q, k, v (analytic, float64).

    With neither ``rows`` nor ``keys``: full (dq [Nq,Hq,d], dk, dv [Nk,Hkv,d]).
    With ``rows``: dq for those rows only (dk, dv None).
    With ``keys``: dk, dv for those key rows only (dq None); every query row that sees one
    of them is processed over its full key set.
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    nq, hq, d = q.shape
    nk, hkv, _ = k.shape
    g = hq // hkv
    scale = resolve_scale(softmax_scale, d)
    sl, _ = normalize_slices(q_ranges, k_ranges, attn_type_map, nq, nk)

    want_dq = keys is None
    want_dkv = rows is None
    if keys is not None:
        keys = np.asarray(keys, dtype=np.int64)
        klo, khi = key_intervals(sl, keys)
        need = np.zeros(nq, dtype=bool)
        for a, b in zip(klo.reshape(-1), khi.reshape(-1)):
            if b > a:
                need[a:b] = True
        proc_rows = np.nonzero(need)[0]
        key_pos = {int(j): n for n, j in enumerate(keys)}
    else:
        proc_rows = np.arange(nq) if rows is None else np.asarray(rows, dtype=np.int64)

    dq = np.zeros((proc_rows.shape[0], hq, d)) if want_dq else None
    if want_dkv:
        nkeys = nk if keys is None else keys.shape[0]
        dk = np.zeros((nkeys, hkv, d))
        dv = np.zeros((nkeys, hkv, d))
    else:
        dk = dv = None

    for b0 in range(0, proc_rows.shape[0], block):
        rb = proc_rows[b0:b0 + block]
        if rb.shape[0] == 0:
            continue
        rel = _rows_touching(sl, int(rb.min()), int(rb.max()) + 1)
        lo, hi = row_intervals(rel, rb)
        c0, c1 = _span(lo, hi)
        if c1 <= c0:
            continue
        m = mask_block(rel, rb, c0, c1)
        if keys is not None:
            cols = np.arange(c0, c1)
            sel = np.array([int(j) in key_pos for j in cols], dtype=bool)
            dst = np.array([key_pos[int(j)] for j in cols[sel]], dtype=np.int64)
        for h in range(hq):
            kh = h // g
            gq, gk, gv = _grad_block(q[rb, h], k[c0:c1, kh], v[c0:c1, kh], do[rb, h], m,
                                     scale, softcap, _alibi(alibi_slopes, h, rb, c0, c1))
            if want_dq:
                dq[b0:b0 + len(rb), h] = gq
            if want_dkv:
                if keys is None:
                    dk[c0:c1, kh] += gk
                    dv[c0:c1, kh] += gv
                elif sel.any():
                    dk[dst, kh] += gk[sel]
                    dv[dst, kh] += gv[sel]
    return dq, dk, dv


def gather_pages(pool, page_table, page_size: int, total_k: int) -> np.ndarray:
    """Logical keys (or values) [total_k, ...] of a paged cache: logical key j is row
    j % page_size of physical page page_table[j // page_size] of ``pool``
    [n_pages, page_size, ...] (Flex Attention paper, section 5, Paged Attention)."""
    pool = np.asarray(pool)
    table = np.asarray(page_table, dtype=np.int64).reshape(-1)
    out = np.empty((total_k,) + pool.shape[2:], dtype=pool.dtype)
    for j in range(total_k):
        out[j] = pool[table[j // page_size], j % page_size]
    return out


def lse_merge(outs: Iterable[np.ndarray], lses: Iterable[np.ndarray]):
    """Combine partial results over disjoint key sets of the same rows.

    L = log sum_c exp(L_c) and O = sum_c exp(L_c - L) O_c; rows whose parts all have
    L_c = -inf get O = 0 and L = -inf.  ``outs[c]``: [n, d]; ``lses[c]``: [n].
    """
    outs = [np.asarray(o, dtype=np.float64) for o in outs]
    lses = [np.asarray(x, dtype=np.float64) for x in lses]
    stack = np.stack(lses, axis=0)
    mx = np.max(stack, axis=0)
    has = np.isfinite(mx)
    mref = np.where(has, mx, 0.0)
    with np.errstate(under="ignore"):
        tot = np.sum(np.exp(stack - mref[None, :]), axis=0)
    lse = np.where(has, mref + np.log(np.where(has, tot, 1.0)), -np.inf)
    out = np.zeros_like(outs[0])
    for o, l in zip(outs, lses):
        with np.errstate(under="ignore", invalid="ignore"):
            w = np.where(has, np.exp(l - np.where(has, lse, 0.0)), 0.0)
        out += w[:, None] * o
    return out, lse
