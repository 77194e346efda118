"""The largest problem the C ABI accepts (FFA_MAX_TOKENS = 2^20 packed tokens, one causal
slice over all of them, one head, d = 64): forward and backward on sampled rows and keys
against the float64 oracle, and the column-sum properties of the gradients."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import flexible_mask_attention_range_gb300 as ffa
from _parity import assert_grad_close, assert_lse_close, assert_out_close, to64

pytestmark = pytest.mark.gpu

N = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def _built(lib_path):
    yield


def test_max_tokens_forward_and_backward():
    q, k, v, do = W.draw_qkv(N, N, 1, 1, 64, 77)
    qr, kr, ty = [[0, N]], [[0, N]], [O.CAUSAL]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = ffa.ffa_fwd(qd, kd, vd, qr, kr, ty, status=status)
    dq, dk, dv = ffa.ffa_bwd(qd, kd, vd, out, lse, dod, qr, kr, ty, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N // 2, N - 129, N - 1], g.integers(0, N, 5)]))
    ro, rl = O.forward(q, k, v, qr, kr, ty, rows=rows)
    assert_out_close(to64(out[rows]), ro)
    assert_lse_close(to64(lse[:, rows]), rl)
    rq, _, _ = O.backward(q, k, v, do, qr, kr, ty, rows=rows)
    assert_grad_close(to64(dq[rows]), rq, "dq rows")
    keys = np.array([N - 300, N - 129, N - 128, N - 1])
    _, rk, rv = O.backward(q, k, v, do, qr, kr, ty, keys=keys)
    assert_grad_close(to64(dk[keys]), rk, "dk keys")
    assert_grad_close(to64(dv[keys]), rv, "dv keys")
    # every row sees a key: sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 (no softcap)
    dvs = dv.double().sum(0).cpu()
    dos = do.double().sum(0)
    assert float((dvs - dos).abs().max()) <= 1e-2 * float(dos.abs().max()) + 1.0
    assert float(dk.double().sum(0).abs().max()) < 4.0
