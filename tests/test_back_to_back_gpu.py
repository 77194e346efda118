"""Calls enqueued back to back on one stream, sharing one workspace, with no synchronisation
between them.  Inside a call every kernel after the first is launched as a programmatic
dependent of the kernel before it; the first kernel of a call keeps plain stream order, so a
call never starts planning into the workspace while the call before it still reads its plan.
Every result is checked against the float64 oracle."""
import pytest
import torch

import oracle as O
import workloads as W
import flexible_mask_attention_range_gb300 as ffa
from _parity import assert_grad_close, assert_lse_close, assert_out_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib_path):
    yield


def _draw(n, hq, hkv, d, seed):
    g = W.make_generator(seed)
    q = torch.randn(n, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16)
    do = torch.randn(n, hq, d, generator=g).to(torch.bfloat16)
    return q, k, v, do


def test_forward_and_backward_calls_back_to_back_on_one_workspace():
    n, hq, hkv, d = 700, 4, 2, 128
    q, k, v, do = _draw(n, hq, hkv, d, 61)
    # two problems with different plans: a causal mask, then random slices with softcap
    probs = [([(0, n)], [(0, n)], [O.CAUSAL], 0.0)]
    qr, kr, ty = W.random_slices(n, n, 9, seed=62)
    probs.append((qr, kr, ty, 20.0))
    R = max(len(p[2]) for p in probs)
    wsf = torch.empty(ffa.ffa_fwd_workspace_size(n, n, hq, hkv, d, R), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(ffa.ffa_bwd_workspace_size(n, n, hq, hkv, d, R), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    fwd = []
    for rep in range(2):  # A, B, A, B
        for qr_, kr_, ty_, cap in probs:
            fwd.append(ffa.ffa_fwd(qc, kc, vc, qr_, kr_, ty_, softcap=cap, workspace=wsf, status=st))
    bwd = []
    for i, (qr_, kr_, ty_, cap) in enumerate(probs):
        out, lse = fwd[i]
        bwd.append(ffa.ffa_bwd(qc, kc, vc, out, lse, dc, qr_, kr_, ty_, softcap=cap, workspace=wsb, status=st))
    for i, (qr_, kr_, ty_, cap) in enumerate(probs):  # again, in deterministic mode
        out, lse = fwd[i]
        bwd.append(ffa.ffa_bwd(qc, kc, vc, out, lse, dc, qr_, kr_, ty_, softcap=cap, workspace=wsb, status=st,
                               deterministic=True))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for i, (qr_, kr_, ty_, cap) in enumerate(probs):
        ro, rl = O.forward(q, k, v, qr_, kr_, ty_, softcap=cap)
        for out, lse in (fwd[i], fwd[i + 2]):
            assert_out_close(to64(out), ro)
            assert_lse_close(to64(lse), rl)
        assert torch.equal(fwd[i][0], fwd[i + 2][0]) and torch.equal(fwd[i][1], fwd[i + 2][1])
        rq, rk, rv = O.backward(q, k, v, do, qr_, kr_, ty_, softcap=cap)
        for dq, dk, dv in (bwd[i], bwd[i + 2]):
            assert_grad_close(to64(dq), rq, "dq")
            assert_grad_close(to64(dk), rk, "dk")
            assert_grad_close(to64(dv), rv, "dv")


def test_decode_calls_back_to_back_on_one_workspace():
    hq, hkv, d = 16, 4, 128
    batches = []
    for seed, n_seq in ((71, 24), (72, 9)):
        g = W.make_generator(seed)
        kv_len = torch.randint(100, 2600, (n_seq,), generator=g).tolist()
        qr, kr, ty = [], [], []
        k0 = 0
        for i, L in enumerate(kv_len):
            qr.append([i, i + 1])
            kr.append([k0, k0 + L])
            ty.append(O.CAUSAL)
            k0 += L
        q = torch.randn(n_seq, hq, d, generator=g).to(torch.bfloat16)
        k = torch.randn(k0, hkv, d, generator=g).to(torch.bfloat16)
        v = torch.randn(k0, hkv, d, generator=g).to(torch.bfloat16)
        batches.append((q, k, v, qr, kr, ty))
    size = max(ffa.ffa_fwd_decode_workspace_size(q.shape[0], k.shape[0], hq, hkv, d, len(ty), 1)
               for q, k, v, qr, kr, ty in batches)
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = [(q.cuda(), k.cuda(), v.cuda()) for q, k, v, _, _, _ in batches]
    res = []
    for rep in range(2):
        for (qc, kc, vc), (_, _, _, qr, kr, ty) in zip(dev, batches):
            res.append(ffa.ffa_fwd_decode(qc, kc, vc, qr, kr, ty, max_seqlen_q=1, workspace=ws, status=st))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for i, (q, k, v, qr, kr, ty) in enumerate(batches):
        ro, rl = O.forward(q, k, v, qr, kr, ty)
        for out, lse in (res[i], res[i + 2]):
            assert_out_close(to64(out), ro)
            assert_lse_close(to64(lse), rl)
