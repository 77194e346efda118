"""Failure detection on the GPU without a fault: bounded waits that run out.

Every wait inside the attention kernels is bounded (FFA_WAIT_LIMIT_NS, read on every call).
The test switch FFA_TEST_STALL=1 makes the first wait of every CTA of the forward and
backward attention kernels target a barrier that nothing arrives on.  With a 20 ms limit
that wait runs out; the kernel then records FFA_STATUS_TIMEOUT in the status word, the
other warps of the CTA see its abort flag, the producer lets the copies it issued land, the
MMA warp waits for its MMAs, tensor memory is freed and the kernel returns.  Checked here:
the status bit, that each call returned within seconds, and that the context is still
usable: the next calls, with the switch off, match the float64 oracle.
"""
import contextlib
import os
import time

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


@contextlib.contextmanager
def _stalled(limit_ns=20_000_000):
    saved = {k: os.environ.get(k) for k in ("FFA_TEST_STALL", "FFA_WAIT_LIMIT_NS")}
    os.environ["FFA_TEST_STALL"] = "1"
    os.environ["FFA_WAIT_LIMIT_NS"] = str(limit_ns)
    try:
        yield
    finally:
        for k, val in saved.items():
            if val is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = val


def _inputs():
    w = W.get("page1_2048_gqa")
    q, k, v, do = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
    return w, q, k, v, do


# softcap 30 takes the bounded-softcap kernel instance (fixed reference, no row max), 0 the
# general one
@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_forward_wait_runs_out_then_next_call_is_correct(softcap):
    w, q, k, v, _ = _inputs()
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with _stalled():
        t0 = time.perf_counter()
        ffa.ffa_fwd(qc, kc, vc, w.q_ranges, w.k_ranges, w.types, softcap=softcap, status=st)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    assert int(st.item()) & ffa.STATUS_TIMEOUT
    assert dt < 10.0
    st.zero_()
    out, lse = ffa.ffa_fwd(qc, kc, vc, w.q_ranges, w.k_ranges, w.types, softcap=softcap, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rl = O.forward(q, k, v, w.q_ranges, w.k_ranges, w.types, softcap=softcap)
    assert_out_close(to64(out), ro)
    assert_lse_close(to64(lse), rl)


@pytest.mark.parametrize("deterministic", [False, True])
def test_backward_wait_runs_out_then_next_call_is_correct(deterministic):
    w, q, k, v, do = _inputs()
    qc, kc, vc, dc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = ffa.ffa_fwd(qc, kc, vc, w.q_ranges, w.k_ranges, w.types)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with _stalled():
        t0 = time.perf_counter()
        ffa.ffa_bwd(qc, kc, vc, out, lse, dc, w.q_ranges, w.k_ranges, w.types, status=st,
                    deterministic=deterministic)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    assert int(st.item()) & ffa.STATUS_TIMEOUT
    assert dt < 10.0
    st.zero_()
    dq, dk, dv = ffa.ffa_bwd(qc, kc, vc, out, lse, dc, w.q_ranges, w.k_ranges, w.types, status=st,
                             deterministic=deterministic)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rq, rk, rv = O.backward(q, k, v, do, w.q_ranges, w.k_ranges, w.types)
    assert_grad_close(to64(dq), rq, "dq")
    assert_grad_close(to64(dk), rk, "dk")
    assert_grad_close(to64(dv), rv, "dv")
