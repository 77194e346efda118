"""Paged key/value cache (forward): ffa_fwd_paged against ffa_fwd on the logical keys (bit
for bit: the same tiles reach shared memory) and against the float64 oracle, which gathers
the logical keys from the pool with its own page-table reading."""
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


def _draw(nq, nk, hq, hkv, d, seed):
    g = W.make_generator(seed)
    q = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    return q, k, v


def _pool(k, v, page, n_extra, seed):
    """Scatter logical k/v into a pool with n_extra spare pages; spare rows hold noise."""
    nk, hkv, d = k.shape
    n_lp = math.ceil(nk / page)
    n_pages = n_lp + n_extra
    table = W.random_page_table(n_lp, n_pages, seed)
    g = W.make_generator(seed + 1000)
    kp = torch.randn(n_pages, page, hkv, d, generator=g).to(torch.bfloat16)
    vp = torch.randn(n_pages, page, hkv, d, generator=g).to(torch.bfloat16)
    for j in range(n_lp):
        rows = min(page, nk - j * page)
        kp[int(table[j]), :rows] = k[j * page:j * page + rows]
        vp[int(table[j]), :rows] = v[j * page:j * page + rows]
    return kp, vp, table


PAGED = [
    # nq, nk, hq, hkv, d, page, R, cap, seed
    (300, 1000, 4, 2, 128, 16, 5, 0.0, 11),
    (513, 2049, 8, 2, 64, 32, 9, 0.0, 12),
    (130, 777, 4, 4, 128, 64, 3, 20.0, 13),
    (1000, 1500, 2, 1, 128, 128, 12, 0.0, 14),
    (64, 5000, 8, 1, 128, 16, 2, 0.0, 15),  # few queries over a long paged cache (decode-like)
]


@pytest.mark.parametrize("nq,nk,hq,hkv,d,page,R,cap,seed", PAGED)
def test_paged_matches_unpaged_and_oracle(nq, nk, hq, hkv, d, page, R, cap, seed):
    q, k, v = _draw(nq, nk, hq, hkv, d, seed)
    qr, kr, ty = W.random_slices(nq, nk, R, seed)
    kp, vp, table = _pool(k, v, page, 3, seed)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 0.75 / math.sqrt(d)
    o_p, l_p = ffa.ffa_fwd_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), nk, qr, kr, ty, scale, cap,
                                 status=status)
    o_u, l_u = ffa.ffa_fwd(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, scale, cap)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(o_p, o_u) and torch.equal(l_p, l_u)
    kg = O.gather_pages(kp.float().numpy(), table.numpy(), page, nk)
    vg = O.gather_pages(vp.float().numpy(), table.numpy(), page, nk)
    ro, rl = O.forward(q, kg, vg, qr, kr, ty, softmax_scale=scale, softcap=cap)
    assert_out_close(to64(o_p), ro)
    assert_lse_close(to64(l_p), rl)


def test_paged_shared_physical_page():
    # two logical pages with equal contents may share one physical page
    nq, nk, hq, hkv, d, page = 200, 512, 4, 2, 128, 64
    q, k, v = _draw(nq, nk, hq, hkv, d, 21)
    k[3 * page:4 * page] = k[1 * page:2 * page]
    v[3 * page:4 * page] = v[1 * page:2 * page]
    kp, vp, table = _pool(k, v, page, 2, 22)
    table[3] = table[1]
    qr, kr, ty = [[0, nq]], [[0, nk]], [O.CAUSAL]
    o_p, l_p = ffa.ffa_fwd_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), nk, qr, kr, ty)
    o_u, l_u = ffa.ffa_fwd(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty)
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_u) and torch.equal(l_p, l_u)


def test_paged_entry_outside_pool_is_reported():
    nq, nk, hq, hkv, d, page = 128, 256, 2, 1, 64, 32
    q, k, v = _draw(nq, nk, hq, hkv, d, 31)
    kp, vp, table = _pool(k, v, page, 1, 32)
    table[2] = kp.shape[0] + 7  # outside the pool: its keys read as zeros
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_p, l_p = ffa.ffa_fwd_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), nk, [[0, nq]], [[0, nk]], [O.FULL],
                                 status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & ffa.STATUS_BAD_PAGE
    # the reading: that page's keys and values are zero
    k0, v0 = k.clone(), v.clone()
    k0[2 * page:3 * page] = 0
    v0[2 * page:3 * page] = 0
    ro, rl = O.forward(q, k0, v0, [[0, nq]], [[0, nk]], [O.FULL])
    assert_out_close(to64(o_p), ro)
    assert_lse_close(to64(l_p), rl)


def test_paged_with_alibi():
    nq, nk, hq, hkv, d, page = 400, 1100, 8, 2, 128, 64
    q, k, v = _draw(nq, nk, hq, hkv, d, 41)
    qr, kr, ty = W.random_slices(nq, nk, 6, 41)
    kp, vp, table = _pool(k, v, page, 2, 42)
    slopes = torch.tensor([2.0 ** -(h + 5) for h in range(hq)], dtype=torch.float32)
    o_p, l_p = ffa.ffa_fwd_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), nk, qr, kr, ty,
                                 alibi_slopes=slopes.cuda())
    o_u, l_u = ffa.ffa_fwd(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, alibi_slopes=slopes.cuda())
    torch.cuda.synchronize()
    assert torch.equal(o_p, o_u) and torch.equal(l_p, l_u)
    ro, rl = O.forward(q, k, v, qr, kr, ty, alibi_slopes=slopes.numpy())
    assert_out_close(to64(o_p), ro)
    assert_lse_close(to64(l_p), rl)
