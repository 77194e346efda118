"""Pins for the float64 oracle: each check ties it to something other than itself --
library routines (torch SDPA in float64), closed forms, hand-computed values, finite
differences and invariants.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape)


def _sdpa(q, k, v, mask=None, is_causal=False, scale=None):
    """torch SDPA in float64 per head: q [N,Hq,d], k/v [Nk,Hkv,d] -> O [N,Hq,d], LSE [Hq,N]."""
    hq, hkv = q.shape[1], k.shape[1]
    g = hq // hkv
    qt = torch.tensor(q).permute(1, 0, 2)
    kt = torch.tensor(k).permute(1, 0, 2).repeat_interleave(g, dim=0)
    vt = torch.tensor(v).permute(1, 0, 2).repeat_interleave(g, dim=0)
    m = None if mask is None else torch.tensor(mask)
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, is_causal=is_causal, scale=scale)
    # LSE via torch.logsumexp over the masked scores (library reduction)
    s = (qt @ kt.transpose(1, 2)) * scale
    if m is not None:
        s = s.masked_fill(~m, float("-inf"))
    if is_causal:
        n, nk = s.shape[1], s.shape[2]
        s = s.masked_fill(~torch.ones(n, nk, dtype=torch.bool).tril(), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.numpy()


@pytest.mark.parametrize("n,hq,hkv,d", [(37, 2, 1, 16), (64, 4, 2, 8), (130, 2, 2, 32)])
def test_single_full_slice_matches_sdpa(n, hq, hkv, d):
    q, k, v = _rand((n, hq, d), 1), _rand((n, hkv, d), 2), _rand((n, hkv, d), 3)
    sc = 1.0 / math.sqrt(d)
    o, l = O.forward(q, k, v, [[0, n]], [[0, n]], [O.FULL])
    ro, rl = _sdpa(q, k, v, scale=sc)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


@pytest.mark.parametrize("n,d", [(1, 8), (50, 8), (129, 16)])
def test_square_causal_is_lower_triangle_and_matches_sdpa(n, d):
    m = O.dense_mask([[0, n]], [[0, n]], [O.CAUSAL], n, n)
    assert np.array_equal(m, np.tril(np.ones((n, n), dtype=bool)))
    q, k, v = _rand((n, 4, d), 4), _rand((n, 2, d), 5), _rand((n, 2, d), 6)
    o, l = O.forward(q, k, v, [[0, n]], [[0, n]], [O.CAUSAL], softmax_scale=0.3)
    ro, rl = _sdpa(q, k, v, is_causal=True, scale=0.3)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(l, rl, atol=1e-12)


def test_issue_example_mask_is_bidirectional_prefix_then_causal():
    """The issue's 2-slice mask (FULL [0,h)x[0,h), CAUSAL [h,N)x[0,N)) under the bottom-right
    reading: rows < h see the first half, rows >= h see keys j <= i."""
    n, h = 24, 12
    m = O.dense_mask([[0, h], [h, n]], [[0, h], [0, n]], [O.FULL, O.CAUSAL], n, n)
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    want = ((i < h) & (j < h)) | ((i >= h) & (j <= i))
    assert np.array_equal(m, want)


def test_causal_alignment_with_unequal_lengths():
    """q [4,10) (6 rows) vs k [0,3) (3 keys): bottom-right alignment -> rows 4..6 see nothing,
    row 7 sees key 0, row 9 sees keys 0..2."""
    m = O.dense_mask([[4, 10]], [[0, 3]], [O.CAUSAL], 10, 3)
    assert not m[:7].any()
    assert m[7].tolist() == [True, False, False]
    assert m[9].tolist() == [True, True, True]


def test_documents_equal_independent_attention():
    lens = [5, 17, 1, 9, 33]
    n = sum(lens)
    q, k, v = _rand((n, 2, 8), 7), _rand((n, 2, 8), 8), _rand((n, 2, 8), 9)
    qr, kr, ty, s = [], [], [], 0
    for L in lens:
        qr.append([s, s + L]); kr.append([s, s + L]); ty.append(O.CAUSAL); s += L
    o, l = O.forward(q, k, v, qr, kr, ty)
    s = 0
    for L in lens:
        ro, rl = _sdpa(q[s:s + L], k[s:s + L], v[s:s + L], is_causal=True, scale=1 / math.sqrt(8))
        np.testing.assert_allclose(o[s:s + L], ro, atol=1e-12)
        np.testing.assert_allclose(l[:, s:s + L], rl, atol=1e-12)
        s += L


def test_arbitrary_mask_matches_sdpa_with_boolean_mask():
    n, nk = 40, 33
    qr, kr, ty = W.random_slices(n, nk, 6, seed=3)
    m = O.dense_mask(qr, kr, ty, n, nk)
    q, k, v = _rand((n, 2, 8), 10), _rand((nk, 1, 8), 11), _rand((nk, 1, 8), 12)
    o, l = O.forward(q, k, v, qr, kr, ty, softmax_scale=0.4)
    rows = m.any(axis=1)
    ro, rl = _sdpa(q[rows], k, v, mask=m[rows], scale=0.4)
    np.testing.assert_allclose(o[rows], ro, atol=1e-12)
    np.testing.assert_allclose(l[:, rows], rl, atol=1e-12)


def _dummy_forms(n):
    return ([[0, 0], [5, 5], [0, n], [n, n], [3, 3]],
            [[0, 0], [0, n], [7, 7], [2, 2], [n, n]],
            [0, 1, 1, 0, 1])


def test_dummy_slices_are_bit_identical_noops():
    n = 48
    q, do = _rand((n, 4, 8), 1), _rand((n, 4, 8), 4)
    k, v = _rand((n, 2, 8), 2), _rand((n, 2, 8), 3)
    qr, kr, ty = [[0, 24], [24, n]], [[0, 24], [0, n]], [0, 1]
    dq_, dk_, dt_ = _dummy_forms(n)
    a = O.forward(q, k, v, qr, kr, ty, softcap=3.0)
    b = O.forward(q, k, v, qr + dq_, kr + dk_, ty + dt_, softcap=3.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    ga = O.backward(q, k, v, do, qr, kr, ty, softcap=3.0)
    gb = O.backward(q, k, v, do, dq_ + qr + dq_, dk_ + kr + dk_, dt_ + ty + dt_, softcap=3.0)
    for x, y in zip(ga, gb):
        assert np.array_equal(x, y)


def test_empty_rows_give_zero_output_and_minus_inf_lse():
    n = 20
    q, k, v, do = _rand((n, 2, 4), 1), _rand((n, 1, 4), 2), _rand((n, 1, 4), 3), _rand((n, 2, 4), 4)
    # rows 0..4 uncovered; CAUSAL with q longer than k: rows 5..9 see nothing
    qr, kr, ty = [[5, 15], [15, 20]], [[0, 5], [0, 20]], [O.CAUSAL, O.FULL]
    o, l = O.forward(q, k, v, qr, kr, ty)
    assert np.all(o[:10] == 0) and np.all(np.isneginf(l[:, :10]))
    assert np.all(np.isfinite(l[:, 10:]))
    dq, dk, dv = O.backward(q, k, v, do, qr, kr, ty)
    assert np.all(dq[:10] == 0)
    # nothing at all visible
    o2, l2 = O.forward(q, k, v, [[3, 3]], [[0, 20]], [0])
    assert np.all(o2 == 0) and np.all(np.isneginf(l2))


def test_uniform_keys_closed_form():
    """K = 0 -> every visible score is 0 -> P uniform over the visible keys:
    LSE_i = log(#visible_i) and O_i = mean of the visible V rows."""
    n = 30
    q, v = _rand((n, 2, 8), 1), _rand((n, 1, 8), 2)
    k = np.zeros((n, 1, 8))
    qr, kr, ty = [[0, 30], [10, 20]], [[0, 12], [20, 30]], [O.CAUSAL, O.FULL]
    o, l = O.forward(q, k, v, qr, kr, ty, softcap=5.0)
    for i in range(n):
        vis = [j for j in range(n) if (j < 12 and j <= i + 12 - 30) or (10 <= i < 20 and 20 <= j < 30)]
        if not vis:
            assert np.isneginf(l[0, i])
            continue
        assert abs(l[0, i] - math.log(len(vis))) < 1e-12
        np.testing.assert_allclose(o[i, 0], v[vis, 0].mean(axis=0), atol=1e-12)


def test_softcap_two_keys_golden():
    g = json.load(open(os.path.join(GOLD, "softcap_two_keys.json")))
    # q = [1], k0 = [4], k1 = [-2] -> q.k = 4, -2
    q = np.array([[[1.0]]]); k = np.array([[[4.0]], [[-2.0]]]); v = np.array([[[1.0]], [[0.0]]])
    o, l = O.forward(q, k, v, [[0, 1]], [[0, 2]], [O.FULL], softmax_scale=g["scale"],
                     softcap=g["softcap"])
    assert abs(l[0, 0] - g["lse"]) < 1e-14
    assert abs(o[0, 0, 0] - g["p0"]) < 1e-14


def _loss(q, k, v, do, qr, kr, ty, sc, cap):
    o, _ = O.forward(q, k, v, qr, kr, ty, softmax_scale=sc, softcap=cap)
    return float(np.sum(o * do))


@pytest.mark.parametrize("cap", [0.0, 1.5])
def test_gradients_match_central_finite_differences(cap):
    n, d = 12, 4
    q, k, v, do = _rand((n, 2, d), 21), _rand((n, 1, d), 22), _rand((n, 1, d), 23), _rand((n, 2, d), 24)
    qr, kr, ty = [[0, 6], [4, 12], [2, 2]], [[0, 7], [1, 12], [0, 5]], [O.FULL, O.CAUSAL, O.FULL]
    sc = 0.7
    dq, dk, dv = O.backward(q, k, v, do, qr, kr, ty, softmax_scale=sc, softcap=cap)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            fp = _loss(q, k, v, do, qr, kr, ty, sc, cap)
            x[idx] = old - eps
            fm = _loss(q, k, v, do, qr, kr, ty, sc, cap)
            x[idx] = old
            num[idx] = (fp - fm) / (2 * eps)
        err = np.abs(num - g).max() / max(1e-12, np.abs(g).max())
        assert err < 1e-6, err


def test_gradients_match_sdpa_autograd():
    n, nk, d = 33, 29, 8
    qr, kr, ty = W.random_slices(n, nk, 5, seed=11, p_dummy=0.0)
    m = O.dense_mask(qr, kr, ty, n, nk)
    rows = m.any(axis=1)
    q, k, v, do = _rand((n, 4, d), 31), _rand((nk, 2, d), 32), _rand((nk, 2, d), 33), _rand((n, 4, d), 34)
    do[~rows] = 0.0
    dq, dk, dv = O.backward(q, k, v, do, qr, kr, ty, softmax_scale=0.5)
    qt = torch.tensor(q[rows]).permute(1, 0, 2).requires_grad_(True)
    kt = torch.tensor(k).permute(1, 0, 2).requires_grad_(True)
    vt = torch.tensor(v).permute(1, 0, 2).requires_grad_(True)
    o = F.scaled_dot_product_attention(qt, kt.repeat_interleave(2, 0), vt.repeat_interleave(2, 0),
                                       attn_mask=torch.tensor(m[rows]), scale=0.5)
    (o * torch.tensor(do[rows]).permute(1, 0, 2)).sum().backward()
    np.testing.assert_allclose(dq[rows], qt.grad.permute(1, 0, 2).numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.permute(1, 0, 2).numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.permute(1, 0, 2).numpy(), atol=1e-11)
    assert np.all(dq[~rows] == 0)


def test_row_and_key_subsets_match_full():
    n = 300
    qr, kr, ty = W.random_slices(n, n, 8, seed=5)
    q, k, v, do = _rand((n, 2, 8), 41), _rand((n, 1, 8), 42), _rand((n, 1, 8), 43), _rand((n, 2, 8), 44)
    o, l = O.forward(q, k, v, qr, kr, ty, softcap=2.0)
    dq, dk, dv = O.backward(q, k, v, do, qr, kr, ty, softcap=2.0)
    rows = np.array([0, 5, 127, 128, 129, 299])
    o2, l2 = O.forward(q, k, v, qr, kr, ty, softcap=2.0, rows=rows)
    np.testing.assert_allclose(o2, o[rows], atol=1e-13)
    np.testing.assert_allclose(l2, l[:, rows], atol=1e-13)
    dq2, _, _ = O.backward(q, k, v, do, qr, kr, ty, softcap=2.0, rows=rows)
    np.testing.assert_allclose(dq2, dq[rows], atol=1e-13)
    keys = np.array([1, 64, 200, 299])
    _, dk2, dv2 = O.backward(q, k, v, do, qr, kr, ty, softcap=2.0, keys=keys)
    np.testing.assert_allclose(dk2, dk[keys], atol=1e-13)
    np.testing.assert_allclose(dv2, dv[keys], atol=1e-13)


def test_lse_merge_identity_over_disjoint_key_parts():
    n = 64
    q, k, v = _rand((n, 2, 8), 51), _rand((n, 1, 8), 52), _rand((n, 1, 8), 53)
    full = O.forward(q, k, v, [[0, n]], [[0, n]], [O.CAUSAL])
    parts = []
    for a, b in ((0, 10), (10, 40), (40, 64)):
        # keys [a,b) seen causally by rows: slice rows [a,n) x keys [a,b) with j <= i is
        # CAUSAL on the square [a,b) plus FULL on rows [b,n)
        qr, kr, ty = [[a, b], [b, n]], [[a, b], [a, b]], [O.CAUSAL, O.FULL]
        if b == n:
            qr, kr, ty = qr[:1], kr[:1], ty[:1]
        parts.append(O.forward(q, k, v, qr, kr, ty))
    for h in range(2):
        mo, ml = O.lse_merge([p[0][:, h] for p in parts], [p[1][h] for p in parts])
        np.testing.assert_allclose(mo, full[0][:, h], atol=1e-12)
        np.testing.assert_allclose(ml, full[1][h], atol=1e-12)
    # all parts -inf -> 0 / -inf
    mo, ml = O.lse_merge([np.ones((3, 2)), np.ones((3, 2))], [np.full(3, -np.inf)] * 2)
    assert np.all(mo == 0) and np.all(np.isneginf(ml))


def test_union_semantics_duplicates_and_prefix_lm():
    n, p = 40, 12
    q, k, v, do = _rand((n, 2, 8), 61), _rand((n, 2, 8), 62), _rand((n, 2, 8), 63), _rand((n, 2, 8), 64)
    qr, kr, ty = [[0, n], [0, p], [0, p]], [[0, n], [0, p], [0, p]], [O.CAUSAL, O.FULL, O.FULL]
    a = O.forward(q, k, v, qr, kr, ty)
    b = O.forward(q, k, v, qr[:2], kr[:2], ty[:2])
    np.testing.assert_array_equal(a[0], b[0])
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    prefix_lm = (j <= i) | ((i < p) & (j < p))
    assert np.array_equal(O.dense_mask(qr, kr, ty, n, n), prefix_lm)
    ro, rl = _sdpa(q, k, v, mask=prefix_lm, scale=1 / math.sqrt(8))
    np.testing.assert_allclose(a[0], ro, atol=1e-12)
    np.testing.assert_allclose(a[1], rl, atol=1e-12)
    ga = O.backward(q, k, v, do, qr, kr, ty)
    gb = O.backward(q, k, v, do, qr[:2], kr[:2], ty[:2])
    for x, y in zip(ga, gb):
        np.testing.assert_allclose(x, y, atol=1e-13)


def test_invalid_slices_dropped_and_counted():
    sl, bad = O.normalize_slices([[0, 4], [5, 3], [0, 99], [2, 2], [1, 2]],
                                 [[0, 4], [0, 1], [0, 1], [0, 1], [0, 1]],
                                 [0, 0, 1, 0, 7], 10, 10)
    assert bad == 3
    assert sl.tolist() == [[0, 4, 0, 4, 0]]


def test_tile_classes_and_pairs_closed_forms():
    g = json.load(open(os.path.join(GOLD, "closed_forms.json")))
    for name in ("tiny_256", "page1_2048_gqa", "sliding_32k_softcap", "long_causal_64k_prefix"):
        w = W.get(name)
        tc = O.tile_classes(w.q_ranges, w.k_ranges, w.types, w.total, w.total)
        e = g[name]
        if "tiles" in e:
            assert tc.tolist() == e["tiles"]
        else:
            assert (int((tc == O.TILE_FULL).sum()), int((tc == O.TILE_PARTIAL).sum()),
                    int((tc == O.TILE_EMPTY).sum())) == (e["full"], e["partial"], e["empty"])
        assert O.visible_pairs(w.q_ranges, w.k_ranges, w.types, w.total, w.total) == e["visible_pairs"]
    w = W.documents()
    assert sum(w.doc_lengths) == w.total
    assert O.visible_pairs(w.q_ranges, w.k_ranges, w.types, w.total, w.total) == \
        sum(L * (L + 1) // 2 for L in w.doc_lengths)


def test_tile_classes_match_dense_mask_brute_force():
    """Tiny grids: classes from the dense mask by direct all/any per tile, with tails."""
    for seed, (nq, nk, t) in enumerate([(37, 29, 8), (64, 64, 16), (50, 70, 16), (9, 33, 4)]):
        qr, kr, ty = W.random_slices(nq, nk, 7, seed=seed)
        m = O.dense_mask(qr, kr, ty, nq, nk)
        tc = O.tile_classes(qr, kr, ty, nq, nk, tile=t)
        for a in range(tc.shape[0]):
            for b in range(tc.shape[1]):
                blk = m[a * t:(a + 1) * t, b * t:(b + 1) * t]
                want = O.TILE_FULL if blk.all() else (O.TILE_EMPTY if not blk.any() else O.TILE_PARTIAL)
                assert tc[a, b] == want
        assert O.visible_pairs(qr, kr, ty, nq, nk) == int(m.sum())


# ------------------------------------------------------------------------------------------
# Planted mistakes: each pin above must catch a plausible error in the oracle.  The mistake
# is planted in the oracle (monkeypatched, CPU only) and the pin is expected to fail.
# ------------------------------------------------------------------------------------------

def test_planted_top_left_causal_is_caught(monkeypatch):
    import oracle.ffa_oracle as M
    orig = M.row_intervals

    def wrong(slices, rows):
        lo, hi = orig(slices, rows)
        if slices.shape[0]:
            qs, qe, ks, ke, t = (slices[:, c][None, :] for c in range(5))
            i = np.asarray(rows)[:, None]
            inside = (i >= qs) & (i < qe)
            tl = np.minimum(ke, ks + (i - qs) + 1)          # top-left alignment
            hi = np.where(inside & (t == O.CAUSAL), np.maximum(tl, lo), hi)
        return lo, hi

    monkeypatch.setattr(M, "row_intervals", wrong)
    with pytest.raises(AssertionError):
        test_issue_example_mask_is_bidirectional_prefix_then_causal()


def test_planted_softcap_order_is_caught(monkeypatch):
    import oracle.ffa_oracle as M
    monkeypatch.setattr(M, "_capped", lambda s, cap: s if cap <= 0 else cap * np.tanh(s / cap) * 1.0001)
    with pytest.raises(AssertionError):
        test_softcap_two_keys_golden()


def test_planted_dropped_gradient_term_is_caught(monkeypatch):
    import oracle.ffa_oracle as M
    orig = M._grad_block

    def wrong(*args, **kwargs):
        dq, dk, dv = orig(*args, **kwargs)
        return dq, dk, dv * 0.999
    monkeypatch.setattr(M, "_grad_block", wrong)
    with pytest.raises(AssertionError):
        test_gradients_match_central_finite_differences(0.0)


def test_planted_transposed_gqa_map_is_caught(monkeypatch):
    import oracle.ffa_oracle as M
    orig = M.forward

    def wrong(q, k, v, *a, **kw):
        k = np.asarray(k)[:, ::-1].copy()                    # kv head order flipped
        v = np.asarray(v)[:, ::-1].copy()
        return orig(q, k, v, *a, **kw)
    monkeypatch.setattr(O, "forward", wrong)
    with pytest.raises(AssertionError):
        test_single_full_slice_matches_sdpa(64, 4, 2, 8)


# ------------------------------------------------------------------------------------------
# ALiBi score modification (Flex Attention paper, sections 2 and 3.1)
# ------------------------------------------------------------------------------------------

def test_alibi_matches_sdpa_with_additive_bias():
    n, nk, d = 45, 38, 8
    qr, kr, ty = W.random_slices(n, nk, 6, seed=9, p_dummy=0.0)
    m = O.dense_mask(qr, kr, ty, n, nk)
    rows = m.any(axis=1)
    q, k, v = _rand((n, 4, d), 71), _rand((nk, 2, d), 72), _rand((nk, 2, d), 73)
    slopes = [0.5, 0.25, 0.125, 0.0625]
    o, l = O.forward(q, k, v, qr, kr, ty, softmax_scale=0.4, alibi_slopes=slopes)
    i, j = np.meshgrid(np.arange(n), np.arange(nk), indexing="ij")
    for h in range(4):
        bias = slopes[h] * (j - i)
        bias = np.where(m, bias, -np.inf)[rows]
        qt = torch.tensor(q[rows][:, h])[None]
        kt = torch.tensor(k[:, h // 2])[None]
        vt = torch.tensor(v[:, h // 2])[None]
        ro = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.tensor(bias)[None], scale=0.4)[0]
        np.testing.assert_allclose(o[rows][:, h], ro.numpy(), atol=1e-12)
        sc = 0.4 * (q[rows][:, h] @ k[:, h // 2].T) + bias
        np.testing.assert_allclose(l[h, rows], torch.logsumexp(torch.tensor(sc), dim=-1).numpy(), atol=1e-12)


def test_alibi_zero_slopes_is_identity_and_gradients_match_finite_differences():
    n, d = 10, 4
    q, k, v, do = _rand((n, 2, d), 81), _rand((n, 1, d), 82), _rand((n, 1, d), 83), _rand((n, 2, d), 84)
    qr, kr, ty = [[0, 10]], [[0, 10]], [O.CAUSAL]
    a = O.forward(q, k, v, qr, kr, ty, softcap=2.0)
    b = O.forward(q, k, v, qr, kr, ty, softcap=2.0, alibi_slopes=[0.0, 0.0])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    slopes = [0.3, -0.2]
    dq, dk, dv = O.backward(q, k, v, do, qr, kr, ty, softcap=2.0, alibi_slopes=slopes)

    def loss():
        o, _ = O.forward(q, k, v, qr, kr, ty, softcap=2.0, alibi_slopes=slopes)
        return float(np.sum(o * do))
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps; fp = loss()
            x[idx] = old - eps; fm = loss()
            x[idx] = old
            num[idx] = (fp - fm) / (2 * eps)
        assert np.abs(num - g).max() / max(1e-12, np.abs(g).max()) < 1e-6


def test_gather_pages_hand_example():
    # pool of 3 physical pages of 2 keys (one head, d = 1) holding 10*page + row; logical
    # pages (2, 0) give keys 20, 21, 0, 1 -- and a 3-key sequence stops after 20, 21, 0
    pool = np.array([[[[0.0]], [[1.0]]], [[[10.0]], [[11.0]]], [[[20.0]], [[21.0]]]])
    got = O.gather_pages(pool, [2, 0], 2, 4)
    assert got.reshape(-1).tolist() == [20.0, 21.0, 0.0, 1.0]
    got3 = O.gather_pages(pool, [2, 0], 2, 3)
    assert got3.reshape(-1).tolist() == [20.0, 21.0, 0.0]


def test_attention_over_scattered_pages_equals_logical_attention():
    # scatter logical K/V into a permuted pool with spare pages; attention over the gathered
    # keys must be the attention over the logical keys (SDPA in float64 as the reference)
    nq, nk, hq, hkv, d, ps = 24, 37, 4, 2, 8, 8
    q, k, v = _rand((nq, hq, d), 41), _rand((nk, hkv, d), 42), _rand((nk, hkv, d), 43)
    n_lp = -(-nk // ps)
    rng = np.random.default_rng(44)
    n_pages = n_lp + 3
    table = rng.permutation(n_pages)[:n_lp]
    kp = _rand((n_pages, ps, hkv, d), 45)
    vp = _rand((n_pages, ps, hkv, d), 46)
    for j in range(n_lp):
        rows = min(ps, nk - j * ps)
        kp[table[j], :rows] = k[j * ps:j * ps + rows]
        vp[table[j], :rows] = v[j * ps:j * ps + rows]
    kg, vg = O.gather_pages(kp, table, ps, nk), O.gather_pages(vp, table, ps, nk)
    assert np.array_equal(kg, k) and np.array_equal(vg, v)
    o, lse = O.forward(q, kg, vg, [[0, nq]], [[0, nk]], [O.FULL])
    o_ref, lse_ref = _sdpa(q, k, v, scale=1.0 / math.sqrt(d))
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-12)
