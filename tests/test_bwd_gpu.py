"""Backward parity: dq, dk, dv of the CUDA path against the float64 oracle's analytic
gradients on identical seeded inputs (forward inputs, the GPU forward's out/lse feed the GPU
backward; the oracle recomputes everything from q, k, v, dO)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import flexible_mask_attention_range_gb300 as ffa
from _parity import GRAD_MAX_ABS, assert_grad_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib_path):
    yield


def _draw(nq, nk, hq, hkv, d, seed):
    g = W.make_generator(seed)
    q = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    do = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    return q, k, v, do


def _gpu_grads(q, k, v, do, qr, kr, ty, scale=None, cap=0.0, status=None):
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = ffa.ffa_fwd(qc, kc, vc, qr, kr, ty, softmax_scale=scale, softcap=cap, status=status)
    dq, dk, dv = ffa.ffa_bwd(qc, kc, vc, out, lse, dc, qr, kr, ty, softmax_scale=scale, softcap=cap,
                             status=status)
    torch.cuda.synchronize()
    return dq, dk, dv


def _check_full(q, k, v, do, qr, kr, ty, scale=None, cap=0.0):
    dq, dk, dv = _gpu_grads(q, k, v, do, qr, kr, ty, scale, cap)
    rq, rk, rv = O.backward(q, k, v, do, qr, kr, ty, softmax_scale=scale, softcap=cap)
    assert_grad_close(to64(dq), rq, "dq")
    assert_grad_close(to64(dk), rk, "dk")
    assert_grad_close(to64(dv), rv, "dv")
    return dq, dk, dv


@pytest.mark.parametrize("name", ["tiny_256", "page1_2048_gqa"])
def test_small_workloads_padded_and_unpadded(name):
    w = W.get(name)
    q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    g1 = _check_full(q, k, v, do, w.q_ranges, w.k_ranges, w.types, w.softmax_scale, w.softcap)
    wp = w.padded()
    g2 = _gpu_grads(q, k, v, do, wp.q_ranges, wp.k_ranges, wp.types, w.softmax_scale, w.softcap)
    for a, b in zip(g1, g2):
        # dq is accumulated with atomics: equal up to summation order
        assert float((a.float() - b.float()).abs().max()) < GRAD_MAX_ABS / 4
    # dk, dv are written once per key tile: bit-identical under padding
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])


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
    (64, 9000, 2, 1, 128, 4, 0.0, 8),      # forward rows split across CTAs
]


@pytest.mark.parametrize("nq,nk,hq,hkv,d,R,cap,seed", RANDOM)
def test_random_slices(nq, nk, hq, hkv, d, R, cap, seed):
    q, k, v, do = _draw(nq, nk, hq, hkv, d, seed)
    qr, kr, ty = W.random_slices(nq, nk, R, seed=seed)
    # Explicit scales stay near the workloads' logit regime (about 1/sqrt(d)).  The gradients
    # are stored in bf16: from |g| = 8 up half a bf16 unit in the last place is 0.031, already
    # 60 % of the 5e-2 bound, and a scale several times larger drives |dq| to about 11.  The
    # sharp-softmax forward regime is covered by the forward tests, whose outputs are bounded
    # by |V|.
    scale = None if seed % 2 else 0.75 / d ** 0.5
    _check_full(q, k, v, do, qr, kr, ty, scale, cap)


# (0.02, 400): a softcap far above the bounded-softcap range, where the backward's degree-5
# polynomial has its largest logit error (about 1e-3 in the log2 domain)
@pytest.mark.parametrize("scale,cap", [(1.0, 1.0), (0.05, 50.0), (0.2, 3.0), (0.02, 400.0)])
def test_softcap_polynomial_and_exact_paths(scale, cap):
    q, k, v, do = _draw(400, 700, 4, 2, 128, 41)
    qr, kr, ty = [(0, 400), (100, 300)], [(0, 700), (0, 150)], [1, 0]
    _check_full(q, k, v, do, qr, kr, ty, scale, cap)


def test_empty_rows_and_unseen_keys_have_zero_gradients():
    q, k, v, do = _draw(260, 300, 4, 2, 64, 11)
    qr, kr, ty = [(50, 250), (250, 260)], [(0, 100), (0, 200)], [1, 0]   # keys >= 200 unseen
    dq, dk, dv = _check_full(q, k, v, do, qr, kr, ty)
    assert torch.all(dq[:150] == 0)
    assert torch.all(dk[200:] == 0) and torch.all(dv[200:] == 0)


def test_backward_status_clean():
    w = W.get("page1_2048_gqa")
    q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _gpu_grads(q, k, v, do, w.q_ranges, w.k_ranges, w.types, status=st)
    assert int(st.item()) == 0


def test_autograd_wrapper():
    w = W.get("tiny_256")
    q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    qc, kc, vc = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out, _ = ffa.flex_flash_attn_func(qc, kc, vc, w.q_ranges, w.k_ranges, w.types,
                                      softmax_scale=w.softmax_scale)
    out.backward(do.cuda())
    rq, rk, rv = O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale)
    assert_grad_close(to64(qc.grad), rq, "dq")
    assert_grad_close(to64(kc.grad), rk, "dk")
    assert_grad_close(to64(vc.grad), rv, "dv")


@pytest.mark.slow
def test_sliding_softcap_full_size_sampled():
    w = W.get("sliding_32k_softcap")
    q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    dq, dk, dv = _gpu_grads(q, k, v, do, w.q_ranges, w.k_ranges, w.types, w.softmax_scale, w.softcap)
    g = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 255, 256, 1023, 1024, w.total - 1], g.integers(0, w.total, 24)]))
    rq, _, _ = O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale,
                          softcap=w.softcap, rows=rows)
    assert_grad_close(to64(dq[rows]), rq, "dq rows")
    keys = np.unique(np.concatenate([[0, 127, 128, 30000, w.total - 1], g.integers(0, w.total, 12)]))
    _, rk, rv = O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale,
                           softcap=w.softcap, keys=keys)
    assert_grad_close(to64(dk[keys]), rk, "dk keys")
    assert_grad_close(to64(dv[keys]), rv, "dv keys")
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()


@pytest.mark.slow
def test_documents_full_size_sampled():
    """The document-masked batch at full size (its config is forward-only; the backward is
    checked as well): sampled rows around document boundaries and random keys."""
    w = W.get("docs_16k")
    q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    dq, dk, dv = _gpu_grads(q, k, v, do, w.q_ranges, w.k_ranges, w.types)
    starts = np.cumsum([0] + list(w.doc_lengths))[:-1]
    g = np.random.default_rng(6)
    edges = np.concatenate([starts, starts + 1, starts[1:] - 1, [w.total - 1]])
    rows = np.unique(np.concatenate([edges, g.integers(0, w.total, 16)]))
    rq, _, _ = O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, rows=rows)
    assert_grad_close(to64(dq[rows]), rq, "dq rows")
    keys = np.unique(np.concatenate([starts, starts[1:] - 1, g.integers(0, w.total, 12)]))
    _, rk, rv = O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, keys=keys)
    assert_grad_close(to64(dk[keys]), rk, "dk keys")
    assert_grad_close(to64(dv[keys]), rv, "dv keys")
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()


@pytest.mark.slow
def test_long_causal_full_size_sampled_and_sum_property():
    w = W.get("long_causal_64k_prefix")
    q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    dq, dk, dv = _gpu_grads(q, k, v, do, w.q_ranges, w.k_ranges, w.types)
    g = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, 4095, 4096, w.total - 1], g.integers(0, w.total, 6)]))
    rq, _, _ = O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, rows=rows)
    assert_grad_close(to64(dq[rows]), rq, "dq rows")
    keys = np.array([w.total - 200, w.total - 129, w.total - 128, w.total - 1])
    _, rk, rv = O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, keys=keys)
    assert_grad_close(to64(dk[keys]), rk, "dk keys")
    assert_grad_close(to64(dv[keys]), rv, "dv keys")
    # every row sees at least one key, so sum_j P_ij = 1 and sum_j dV_j = sum_i dO_i (per KV
    # group), and without softcap sum_j dK_j = 0 (sum_j dS_ij = 0 for every row)
    G = w.hq // w.hkv
    dvs = dv.double().sum(0).cpu()
    dos = do.double().reshape(w.total, w.hkv, G, w.d).sum(dim=(0, 2))
    assert float((dvs - dos).abs().max()) <= 1e-2 * float(dos.abs().max()) + 1.0
    dks = dk.double().sum(0).cpu()
    assert float(dks.abs().max()) < 2.0


@pytest.mark.parametrize("nq,nk,hq,hkv,d,cap,seed", [(300, 300, 4, 2, 64, 0.0, 51), (513, 700, 6, 3, 128, 5.0, 52),
                                                      (64, 9000, 2, 1, 128, 0.0, 53)])
def test_alibi_score_modification(nq, nk, hq, hkv, d, cap, seed):
    q, k, v, do = _draw(nq, nk, hq, hkv, d, seed)
    qr, kr, ty = W.random_slices(nq, nk, 9, seed=seed)
    # slopes 2^-5 .. : with the strongest ALiBi slopes (0.5) these masks make one key the
    # nearest visible key of many rows and |dv| reaches ~17, where bf16 storage alone costs
    # 0.06 of the absolute 5e-2 bound; these slopes keep |dv| <= 4
    slopes = [2.0 ** (-(h + 5)) for h in range(hq)]
    al = torch.tensor(slopes, dtype=torch.float32, device="cuda")
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = ffa.ffa_fwd(qc, kc, vc, qr, kr, ty, softcap=cap, alibi_slopes=al)
    dq, dk, dv = ffa.ffa_bwd(qc, kc, vc, out, lse, dc, qr, kr, ty, softcap=cap, alibi_slopes=al)
    torch.cuda.synchronize()
    rq, rk, rv = O.backward(q, k, v, do, qr, kr, ty, softcap=cap, alibi_slopes=slopes)
    assert_grad_close(to64(dq), rq, "dq")
    assert_grad_close(to64(dk), rk, "dk")
    assert_grad_close(to64(dv), rv, "dv")


@pytest.mark.parametrize("name", ["tiny_256", "page1_2048_gqa"])
def test_deterministic_backward_is_bit_reproducible_and_padding_invariant(name):
    w = W.get(name)
    q, k, v, do = (t.cuda() for t in W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed))
    out, lse = ffa.ffa_fwd(q, k, v, w.q_ranges, w.k_ranges, w.types, w.softmax_scale)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = ffa.ffa_bwd(q, k, v, out, lse, do, w.q_ranges, w.k_ranges, w.types, w.softmax_scale, deterministic=True,
                    status=st)
    b = ffa.ffa_bwd(q, k, v, out, lse, do, w.q_ranges, w.k_ranges, w.types, w.softmax_scale, deterministic=True)
    wp = w.padded()
    c = ffa.ffa_bwd(q, k, v, out, lse, do, wp.q_ranges, wp.k_ranges, wp.types, w.softmax_scale, deterministic=True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, y, z in zip(a, b, c):
        assert torch.equal(x, y) and torch.equal(x, z)
    rq, rk, rv = O.backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), w.q_ranges, w.k_ranges, w.types,
                            softmax_scale=w.softmax_scale)
    assert_grad_close(to64(a[0]), rq, "dq")
    assert_grad_close(to64(a[1]), rk, "dk")
    assert_grad_close(to64(a[2]), rv, "dv")


@pytest.mark.parametrize("nq,nk,hq,hkv,d,R,cap,seed", [(700, 513, 6, 3, 64, 20, 0.0, 6),
                                                        (1000, 1000, 8, 8, 128, 40, 2.0, 7)])
def test_deterministic_backward_random(nq, nk, hq, hkv, d, R, cap, seed):
    q, k, v, do = _draw(nq, nk, hq, hkv, d, seed)
    qr, kr, ty = W.random_slices(nq, nk, R, seed=seed)
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = ffa.ffa_fwd(qc, kc, vc, qr, kr, ty, softcap=cap)
    g1 = ffa.ffa_bwd(qc, kc, vc, out, lse, dc, qr, kr, ty, softcap=cap, deterministic=True)
    g2 = ffa.ffa_bwd(qc, kc, vc, out, lse, dc, qr, kr, ty, softcap=cap, deterministic=True)
    torch.cuda.synchronize()
    for x, y in zip(g1, g2):
        assert torch.equal(x, y)
    rq, rk, rv = O.backward(q, k, v, do, qr, kr, ty, softcap=cap)
    assert_grad_close(to64(g1[0]), rq, "dq")
    assert_grad_close(to64(g1[1]), rk, "dk")
    assert_grad_close(to64(g1[2]), rv, "dv")
