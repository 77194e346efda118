"""Every element of a long-row workload against the float64 oracle.

The 16K-token long-causal workload (one CAUSAL slice over all 16384 tokens plus two FULL
slices over a 4096-token prefix, Hq 16 / Hkv 4, d 128): its key tile 0 is seen by all 128
query tiles of all four query heads of its group, so the backward kernel accumulates dK/dV
of that tile over 512 steps in TMEM and the forward kernel runs rows of up to 128 key
tiles.  Forward O and LSE and backward dQ, dK and dV are compared element by element,
every row and every key (MagiAttention issue #180: the reproduction script compares out and
the gradients obtained with out.backward(do)); the key tiles 0, 31 and 32 (the prefix
boundary at key 4096) are also checked on their own, so a failure names them.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import flexible_mask_attention_range_gb300 as ffa
from _parity import assert_grad_close, assert_lse_close, assert_out_close, to64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built(lib_path):
    yield


def test_long_causal_16k_every_element():
    w = W.get("long_causal_16k_prefix")
    q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = ffa.ffa_fwd(qc, kc, vc, w.q_ranges, w.k_ranges, w.types, w.softmax_scale, status=st)
    dq, dk, dv = ffa.ffa_bwd(qc, kc, vc, out, lse, dc, w.q_ranges, w.k_ranges, w.types, w.softmax_scale,
                             status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    ro, rl = O.forward(q, k, v, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale)
    assert_out_close(to64(out), ro)
    assert_lse_close(to64(lse), rl)

    rq, rk, rv = O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types, softmax_scale=w.softmax_scale)
    gk, gv = to64(dk), to64(dv)
    for kt in (0, 31, 32):
        sl = slice(kt * 128, kt * 128 + 128)
        assert_grad_close(gk[sl], rk[sl], f"dk key tile {kt}")
        assert_grad_close(gv[sl], rv[sl], f"dv key tile {kt}")
    assert_grad_close(to64(dq), rq, "dq")
    assert_grad_close(gk, rk, "dk")
    assert_grad_close(gv, rv, "dv")
