"""Forward parity: the CUDA path against the float64 oracle on identical seeded inputs."""
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


def _inputs(nq, nk, hq, hkv, d, seed):
    q, k, v, do = W.draw_qkv(nq, nk, hq, hkv, d, seed) if nq == nk else _draw2(nq, nk, hq, hkv, d, seed)
    return q, k, v, do


def _draw2(nq, nk, hq, hkv, d, seed):
    g = W.make_generator(seed)
    q = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    do = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    return q, k, v, do


def _run(q, k, v, qr, kr, ty, scale=None, cap=0.0, status=None):
    out, lse = ffa.ffa_fwd(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, softmax_scale=scale, softcap=cap,
                           status=status)
    torch.cuda.synchronize()
    return out, lse


def _check_full(q, k, v, qr, kr, ty, scale=None, cap=0.0):
    out, lse = _run(q, k, v, qr, kr, ty, scale, cap)
    ro, rl = O.forward(q, k, v, qr, kr, ty, softmax_scale=scale, softcap=cap)
    assert_out_close(to64(out), ro)
    assert_lse_close(to64(lse), rl)
    return out, lse


@pytest.mark.parametrize("name", ["tiny_256", "page1_2048_gqa"])
def test_small_workloads_padded_and_unpadded(name):
    w = W.get(name)
    q, k, v, _ = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    o1, l1 = _check_full(q, k, v, w.q_ranges, w.k_ranges, w.types, w.softmax_scale, w.softcap)
    wp = w.padded()
    assert len(wp.types) == w.pad_to
    o2, l2 = _run(q, k, v, wp.q_ranges, wp.k_ranges, wp.types, w.softmax_scale, w.softcap)
    # padding with start == end slices leaves the forward bit-identical
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_documents_workload_full():
    w = W.get("docs_16k")
    q, k, v, _ = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed, with_dout=False)
    _check_full(q, k, v, w.q_ranges, w.k_ranges, w.types, w.softmax_scale, w.softcap)


RANDOM = [
    # nq, nk, hq, hkv, d, R, cap, seed
    (1, 1, 1, 1, 64, 1, 0.0, 0),
    (127, 127, 2, 1, 64, 3, 0.0, 1),
    (129, 300, 2, 2, 128, 5, 0.0, 2),
    (300, 129, 4, 2, 64, 7, 5.0, 3),
    (300, 300, 3, 1, 128, 9, 0.0, 4),
    (513, 700, 8, 2, 128, 12, 30.0, 5),
    (700, 513, 6, 3, 64, 20, 0.0, 6),
    (1000, 1000, 8, 8, 128, 40, 2.0, 7),
    (1024, 1024, 16, 2, 64, 6, 0.0, 8),
    (1500, 900, 5, 5, 128, 15, 0.0, 9),
]


@pytest.mark.parametrize("nq,nk,hq,hkv,d,R,cap,seed", RANDOM)
def test_random_slices(nq, nk, hq, hkv, d, R, cap, seed):
    q, k, v, _ = _draw2(nq, nk, hq, hkv, d, seed)
    qr, kr, ty = W.random_slices(nq, nk, R, seed=seed)
    # even seeds take an explicit, sharp scale (logit standard deviation 8 at d = 64 and 3.4
    # at d = 128): rows are dominated by a few keys and the lazily moved reference max is
    # often stale.  O is a convex combination of bf16 values of V, so its bf16 rounding stays
    # far inside the bound however sharp the softmax is.
    scale = None if seed % 2 else (1.0 if d == 64 else 0.3)
    _check_full(q, k, v, qr, kr, ty, scale, cap)


@pytest.mark.parametrize("scale,cap", [(1.0, 1.0), (0.05, 50.0), (0.2, 3.0)])
def test_softcap_polynomial_and_exact_paths(scale, cap):
    """Large logits (|scale*q.k/softcap| beyond the tanh polynomial's range) take the exact
    form, small ones the polynomial; some warps mix both across tiles."""
    q, k, v, _ = _draw2(400, 700, 4, 2, 128, 41)
    qr, kr, ty = [(0, 400), (100, 300)], [(0, 700), (0, 150)], [1, 0]
    _check_full(q, k, v, qr, kr, ty, scale, cap)


def test_run_to_run_bit_identical():
    w = W.get("page1_2048_gqa")
    q, k, v, _ = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    a = _run(q, k, v, w.q_ranges, w.k_ranges, w.types)
    b = _run(q, k, v, w.q_ranges, w.k_ranges, w.types)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_empty_rows_and_no_slices():
    q, k, v, _ = _draw2(260, 200, 4, 2, 64, 11)
    # rows [0,50) uncovered, CAUSAL q longer than k: rows 50..149 see nothing
    qr, kr, ty = [(50, 250), (250, 260)], [(0, 100), (0, 200)], [1, 0]
    out, lse = _check_full(q, k, v, qr, kr, ty)
    assert torch.all(out[:150] == 0)
    assert torch.all(torch.isneginf(lse[:, :150]))
    out, lse = _run(q, k, v, [(3, 3)], [(0, 200)], [0])
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    out, lse = _run(q, k, v, torch.zeros(0, 2, dtype=torch.int32), torch.zeros(0, 2, dtype=torch.int32),
                    torch.zeros(0, dtype=torch.int32))
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_invalid_slice_is_dropped_and_flagged():
    q, k, v, _ = _draw2(200, 200, 2, 1, 64, 12)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qr, kr, ty = [(0, 200), (10, 5), (0, 10)], [(0, 200), (0, 10), (0, 10)], [1, 0, 9]
    out, lse = _run(q, k, v, qr, kr, ty, status=st)
    ro, rl = O.forward(q, k, v, qr[:1], kr[:1], ty[:1])
    assert_out_close(to64(out), ro)
    assert_lse_close(to64(lse), rl)
    assert int(st.item()) == ffa.STATUS_BAD_RANGE


def test_flex_flash_attn_func_matches_ffa_fwd():
    w = W.get("tiny_256")
    q, k, v, _ = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    o1, l1 = ffa.flex_flash_attn_func(q.cuda(), k.cuda(), v.cuda(), w.q_ranges, w.k_ranges, w.types,
                                      max_seqlen_q=w.total, max_seqlen_k=w.total,
                                      softmax_scale=w.softmax_scale)
    o2, l2 = _run(q, k, v, w.q_ranges, w.k_ranges, w.types, w.softmax_scale)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# Few work items and long key ranges: the planner cuts each row's work list into chunks that
# run on different SMs, and the LSE merge combines them.
SPLIT = [
    # nq, nk, hq, hkv, d, cap, seed, slices
    (64, 16384, 2, 1, 128, 0.0, 31, ([(0, 64), (0, 32)], [(0, 16384), (0, 100)], [1, 0])),
    (300, 9000, 3, 1, 64, 0.0, 32, None),
    (129, 20000, 8, 8, 128, 5.0, 33, ([(0, 129), (100, 129), (0, 10)], [(0, 20000), (5000, 5200), (7, 7)],
                                       [1, 0, 0])),
    (1, 40000, 2, 2, 64, 0.0, 34, ([(0, 1)], [(0, 40000)], [1])),
]


@pytest.mark.parametrize("nq,nk,hq,hkv,d,cap,seed,sl", SPLIT)
def test_split_rows_lse_merge(nq, nk, hq, hkv, d, cap, seed, sl):
    q, k, v, _ = _draw2(nq, nk, hq, hkv, d, seed)
    qr, kr, ty = sl if sl is not None else W.random_slices(nq, nk, 14, seed=seed)
    out, lse = _check_full(q, k, v, qr, kr, ty, None, cap)
    again = _run(q, k, v, qr, kr, ty, None, cap)
    assert torch.equal(out, again[0]) and torch.equal(lse, again[1])
    pad = _run(q, k, v, list(qr) + [(0, 0), (3, 3)], list(kr) + [(0, 0), (0, nk)], list(ty) + [0, 1], None, cap)
    assert torch.equal(out, pad[0]) and torch.equal(lse, pad[1])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["sliding_32k_softcap", "long_causal_64k_prefix"])
def test_full_size_sampled_rows(name):
    w = W.get(name)
    q, k, v, _ = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed, with_dout=False)
    out, lse = _run(q, k, v, w.q_ranges, w.k_ranges, w.types, w.softmax_scale, w.softcap)
    g = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 4095, 4096, w.total - 1],
                                     g.integers(0, w.total, 40)]))
    ro, rl = O.forward(q, k, v, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale,
                       softcap=w.softcap, rows=rows)
    assert_out_close(to64(out[rows]), ro)
    assert_lse_close(to64(lse[:, rows]), rl)
    # properties at every row: finite outputs, finite LSE (every row sees at least one key)
    assert torch.isfinite(out.float()).all()
    assert torch.isfinite(lse).all()


ALIBI = [
    # nq, nk, hq, hkv, d, cap, seed
    (300, 300, 4, 2, 64, 0.0, 51),
    (513, 700, 6, 3, 128, 5.0, 52),
    (64, 9000, 2, 1, 128, 0.0, 53),      # split rows + merge
    (1000, 1000, 8, 8, 128, 0.0, 54),
]


@pytest.mark.parametrize("nq,nk,hq,hkv,d,cap,seed", ALIBI)
def test_alibi_score_modification(nq, nk, hq, hkv, d, cap, seed):
    q, k, v, _ = _draw2(nq, nk, hq, hkv, d, seed)
    qr, kr, ty = W.random_slices(nq, nk, 9, seed=seed)
    slopes = [2.0 ** (-(h + 1)) for h in range(hq)]
    out, lse = ffa.ffa_fwd(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, softcap=cap,
                           alibi_slopes=torch.tensor(slopes, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    ro, rl = O.forward(q, k, v, qr, kr, ty, softcap=cap, alibi_slopes=slopes)
    assert_out_close(to64(out), ro)
    assert_lse_close(to64(lse), rl)
