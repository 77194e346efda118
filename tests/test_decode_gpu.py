"""Decoding (ffa_fwd_decode): a few new query tokens per sequence against long key caches,
dense and paged, checked against ffa_fwd on the same inputs and against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import flexible_mask_attention_range_gb300 as ffa
from _parity import assert_lse_close, assert_out_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib_path):
    yield


def _batch(n_seq, q_len, seed, lo=100, hi=3000):
    """Packed decode batch: sequence s has q_len new tokens at the end of kv_len[s] keys;
    slices (q range of its tokens, k range of its keys, CAUSAL: bottom-right alignment)."""
    g = W.make_generator(seed)
    kv_len = (torch.randint(lo, hi, (n_seq,), generator=g)).tolist()
    qr, kr, ty = [], [], []
    q0 = k0 = 0
    for L in kv_len:
        qr.append([q0, q0 + q_len])
        kr.append([k0, k0 + L])
        ty.append(O.CAUSAL)
        q0 += q_len
        k0 += L
    return qr, kr, ty, q0, k0


CASES = [
    # n_seq, q_len, hq, hkv, d, seed
    (16, 1, 8, 1, 128, 1),
    (40, 1, 16, 4, 128, 2),
    (7, 3, 8, 2, 64, 3),
    (64, 1, 4, 4, 128, 4),
    (3, 4, 32, 4, 128, 5),
]


@pytest.mark.parametrize("n_seq,q_len,hq,hkv,d,seed", CASES)
def test_decode_matches_forward_and_oracle(n_seq, q_len, hq, hkv, d, seed):
    qr, kr, ty, nq, nk = _batch(n_seq, q_len, seed)
    g = W.make_generator(seed + 100)
    q = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_d, l_d = ffa.ffa_fwd_decode(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, max_seqlen_q=q_len, status=status)
    o_f, l_f = ffa.ffa_fwd(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rl = O.forward(q, k, v, qr, kr, ty)
    assert_out_close(to64(o_d), ro)
    assert_lse_close(to64(l_d), rl)
    # same arithmetic per row as the token-major forward pass, up to summation order
    assert (o_d.float() - o_f.float()).abs().max().item() <= 2e-2
    assert (l_d - l_f).abs().max().item() <= 1e-3


def test_decode_paged_cache():
    n_seq, q_len, hq, hkv, d, page = 12, 2, 16, 2, 128, 32
    qr, kr, ty, nq, nk = _batch(n_seq, q_len, 9, 200, 2500)
    g = W.make_generator(109)
    q = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    n_lp = math.ceil(nk / page)
    n_pages = n_lp + 5
    table = W.random_page_table(n_lp, n_pages, 110)
    kp = torch.zeros(n_pages, page, hkv, d, dtype=torch.bfloat16)
    vp = torch.zeros(n_pages, page, hkv, d, dtype=torch.bfloat16)
    for j in range(n_lp):
        rows = min(page, nk - j * page)
        kp[int(table[j]), :rows] = k[j * page:j * page + rows]
        vp[int(table[j]), :rows] = v[j * page:j * page + rows]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_p, l_p = ffa.ffa_fwd_decode(q.cuda(), kp.cuda(), vp.cuda(), qr, kr, ty, max_seqlen_q=q_len,
                                  page_table=table.cuda(), total_k=nk, status=status)
    o_d, l_d = ffa.ffa_fwd_decode(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, max_seqlen_q=q_len)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(o_p, o_d) and torch.equal(l_p, l_d)
    kg = O.gather_pages(kp.float().numpy(), table.numpy(), page, nk)
    vg = O.gather_pages(vp.float().numpy(), table.numpy(), page, nk)
    ro, rl = O.forward(q, kg, vg, qr, kr, ty)
    assert_out_close(to64(o_p), ro)
    assert_lse_close(to64(l_p), rl)


def test_decode_reports_causal_slice_longer_than_max_seqlen_q():
    qr, kr, ty, nq, nk = _batch(4, 3, 11, 200, 400)
    g = W.make_generator(111)
    q = torch.randn(nq, 4, 64, generator=g).to(torch.bfloat16)
    k = torch.randn(nk, 2, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(nk, 2, 64, generator=g).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, l = ffa.ffa_fwd_decode(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, max_seqlen_q=2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & ffa.STATUS_BAD_RANGE
    # every slice was dropped: every row is empty (O = 0, LSE = -inf)
    assert torch.count_nonzero(o).item() == 0 and bool(torch.isinf(l).all())


@pytest.mark.parametrize("hq,hkv,cap", [(12, 4, 30.0), (3, 1, 0.0), (16, 16, 5.0)])
def test_decode_softcap_and_odd_groups(hq, hkv, cap):
    # odd G (3 query heads per key/value head) packs all G heads as rows; G = 1 is plain MHA
    qr, kr, ty, nq, nk = _batch(9, 2, 20 + hq, 150, 1800)
    g = W.make_generator(120 + hq)
    d = 128
    q = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    scale = 0.75 / math.sqrt(d)
    o, l = ffa.ffa_fwd_decode(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, max_seqlen_q=2, softmax_scale=scale,
                              softcap=cap)
    torch.cuda.synchronize()
    ro, rl = O.forward(q, k, v, qr, kr, ty, softmax_scale=scale, softcap=cap)
    assert_out_close(to64(o), ro)
    assert_lse_close(to64(l), rl)


# Decoding with GQA and ALiBi (FlexAttention paper, section 6, "Inference Performance": the
# decoding case it singles out): every query head keeps its own slope and every token its
# own position after the heads are packed as rows.
DECODE_ALIBI = [
    # n_seq, q_len, hq, hkv, d, cap, paged, seed
    (24, 1, 16, 4, 128, 0.0, False, 61),    # G = 4: two packed heads of 2 rows per KV head
    (10, 3, 32, 4, 128, 30.0, False, 62),   # G = 8, several new tokens (CAUSAL rewrite)
    (8, 2, 16, 2, 64, 0.0, True, 63),       # G = 8, paged cache
    (6, 2, 12, 4, 128, 5.0, True, 64),      # G = 3 (odd: all heads packed), paged
]


@pytest.mark.parametrize("n_seq,q_len,hq,hkv,d,cap,paged,seed", DECODE_ALIBI)
def test_decode_alibi(n_seq, q_len, hq, hkv, d, cap, paged, seed):
    qr, kr, ty, nq, nk = _batch(n_seq, q_len, seed, 150, 2500)
    g = W.make_generator(seed + 100)
    q = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    # Positions are packed token indices, so the queries of a decode batch sit far from their
    # keys; only the bias differences between the keys of one sequence (up to 2500 apart)
    # shape a row's softmax.  Slopes 2^-6 .. 2^-12 keep those differences between about 40
    # and 0.6 logits: sharp for some heads, flat for others, so a slope taken from the wrong
    # head shows.
    slopes = [2.0 ** (-6.0 - 6.0 * h / (hq - 1)) for h in range(hq)]
    al = torch.tensor(slopes, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if paged:
        page = 32
        n_lp = math.ceil(nk / page)
        table = W.random_page_table(n_lp, n_lp + 3, seed + 200)
        kp = torch.zeros(n_lp + 3, page, hkv, d, dtype=torch.bfloat16)
        vp = torch.zeros(n_lp + 3, page, hkv, d, dtype=torch.bfloat16)
        for j in range(n_lp):
            rows = min(page, nk - j * page)
            kp[int(table[j]), :rows] = k[j * page:j * page + rows]
            vp[int(table[j]), :rows] = v[j * page:j * page + rows]
        o, l = ffa.ffa_fwd_decode(q.cuda(), kp.cuda(), vp.cuda(), qr, kr, ty, max_seqlen_q=q_len, softcap=cap,
                                  page_table=table.cuda(), total_k=nk, status=status, alibi_slopes=al)
    else:
        o, l = ffa.ffa_fwd_decode(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, max_seqlen_q=q_len, softcap=cap,
                                  status=status, alibi_slopes=al)
    o_f, l_f = ffa.ffa_fwd(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, softcap=cap, alibi_slopes=al)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rl = O.forward(q, k, v, qr, kr, ty, softcap=cap, alibi_slopes=slopes)
    assert_out_close(to64(o), ro)
    assert_lse_close(to64(l), rl)
    # the token-major forward pass with the same slopes agrees up to summation order
    assert (o.float() - o_f.float()).abs().max().item() <= 2e-2
    assert (l - l_f).abs().max().item() <= 1e-3


@pytest.mark.parametrize("kv_len,hq,hkv,cap", [(100, 8, 2, 0.0), (128, 16, 2, 30.0), (129, 12, 4, 0.0)])
def test_decode_one_or_two_key_tiles(kv_len, hq, hkv, cap):
    # one sequence with a cache of one key tile (the key split's second warpgroup has no tile
    # and leaves an empty partial) or just over one tile (one tile each)
    qr, kr, ty = [[0, 1]], [[0, kv_len]], [O.CAUSAL]
    g = W.make_generator(300 + kv_len)
    d = 128
    q = torch.randn(1, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(kv_len, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(kv_len, hkv, d, generator=g).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, l = ffa.ffa_fwd_decode(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, max_seqlen_q=1, softcap=cap,
                              status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ro, rl = O.forward(q, k, v, qr, kr, ty, softcap=cap)
    assert_out_close(to64(o), ro)
    assert_lse_close(to64(l), rl)


def test_decode_without_keys():
    # an empty cache: every row is empty, O = 0 and LSE = -inf in the caller's layout
    hq, hkv, d = 8, 2, 64
    q = torch.randn(3, hq, d).to(torch.bfloat16).cuda()
    k = torch.zeros(0, hkv, d, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(0, hkv, d, dtype=torch.bfloat16, device="cuda")
    qr, kr, ty = [[0, 3]], [[0, 0]], [O.FULL]
    out = torch.full((3, hq, d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(hq, 3, dtype=torch.float32, device="cuda")
    o, l = ffa.ffa_fwd_decode(q, k, v, qr, kr, ty, max_seqlen_q=3, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0 and bool(torch.isinf(l).all()) and bool((l < 0).all())
