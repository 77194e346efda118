"""Planner parity: the device tile classification equals the oracle's, bit for bit, for the
five workloads and random slice sets (overlapping, unaligned, zero-length, ragged tails)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import flexible_mask_attention_range_gb300 as ffa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib_path):
    yield


@pytest.mark.parametrize("name", W.ORDER)
@pytest.mark.parametrize("by_column", [False, True])
def test_workload_tile_classes(name, by_column):
    w = W.get(name).padded()
    ref = O.tile_classes(w.q_ranges, w.k_ranges, w.types, w.total, w.total)
    got = ffa.ffa_plan_tiles(w.total, w.total, w.q_ranges, w.k_ranges, w.types, by_column=by_column,
                             num_heads_q=w.hq, num_heads_kv=w.hkv, head_dim=w.d).cpu().numpy()
    assert np.array_equal(got, ref)


CASES = [(1, 1, 1), (127, 129, 5), (129, 127, 9), (300, 300, 12), (700, 513, 30), (1000, 1000, 200),
         (2050, 1800, 3), (4096, 4096, 70)]


@pytest.mark.parametrize("nq,nk,R", CASES)
@pytest.mark.parametrize("by_column", [False, True])
def test_random_tile_classes(nq, nk, R, by_column):
    for seed in range(3):
        qr, kr, ty = W.random_slices(nq, nk, R, seed=seed * 101 + R)
        ref = O.tile_classes(qr, kr, ty, nq, nk)
        got = ffa.ffa_plan_tiles(nq, nk, qr, kr, ty, by_column=by_column).cpu().numpy()
        assert np.array_equal(got, ref), (seed, np.argwhere(got != ref)[:5])


def test_many_overlapping_slices_use_the_overflow_path():
    # > 512 slices touching one tile row exercises the global-list path of the planner
    nq = nk = 640
    g = np.random.default_rng(0)
    qr, kr, ty = [], [], []
    for i in range(700):
        a = int(g.integers(0, 100)); b = int(g.integers(a + 1, 129))
        c = int(g.integers(0, nk - 1)); d = int(g.integers(c + 1, nk + 1))
        qr.append((a, b)); kr.append((c, d)); ty.append(int(g.integers(0, 2)))
    for by_column in (False, True):
        ref = O.tile_classes(qr, kr, ty, nq, nk)
        got = ffa.ffa_plan_tiles(nq, nk, qr, kr, ty, by_column=by_column).cpu().numpy()
        assert np.array_equal(got, ref)


def test_invalid_slices_set_status_and_are_dropped():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qr = [(0, 100), (50, 40), (0, 999)]
    kr = [(0, 100), (0, 10), (0, 10)]
    ty = [1, 0, 0]
    got = ffa.ffa_plan_tiles(300, 300, qr, kr, ty, status=st).cpu().numpy()
    ref = O.tile_classes(qr[:1], kr[:1], ty[:1], 300, 300)
    assert np.array_equal(got, ref)
    assert int(st.item()) & ffa.STATUS_BAD_RANGE
    st.zero_()
    ffa.ffa_plan_tiles(300, 300, [(0, 100), (5, 5)], [(0, 100), (0, 0)], [1, 0], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
