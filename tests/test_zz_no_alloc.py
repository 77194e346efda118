"""ffa_fwd_noalloc: the forward pass for callers that cannot allocate device memory at call
time (runtimes that reserve all device memory up front and forbid later cudaMalloc, or
latency-bound paths that cannot take the device synchronisation an allocation may cause).
It takes its scratch from a fixed device array owned by the library instead of a caller
workspace.

Checked through the C ABI: three calls in a row (two different problems, then the first
again, so leftovers of an earlier call in the shared array cannot leak into a later one)
agree with ffa_fwd with a caller workspace within the parity tolerances, and a problem too
large for the fixed array is rejected before anything is launched.  Collected last so a run
that stops at the first failure has already run every other test."""
import ctypes

import pytest
import torch

import workloads as W
import flexible_mask_attention_range_gb300 as ffa
from _parity import assert_lse_close, assert_out_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(lib_path):
    yield


def _problem(kind):
    if kind == "page1":
        w = W.get("page1_2048_gqa").padded()
        q, k, v, _ = W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, w.seed)
        return q, k, v, w.q_ranges, w.k_ranges, w.types, None, 0.0
    nq, nk, hq, hkv, d = 700, 513, 6, 3, 128
    g = W.make_generator(21)
    q = torch.randn(nq, hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(nk, hkv, d, generator=g).to(torch.bfloat16)
    qr, kr, ty = W.random_slices(nq, nk, 17, seed=21)
    return q, k, v, qr, kr, ty, 0.07, 5.0


def _noalloc_via_abi(q, k, v, qr, kr, ty, scale, cap):
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    qr_d = torch.tensor(qr, dtype=torch.int32, device=dev).reshape(-1, 2).contiguous()
    kr_d = torch.tensor(kr, dtype=torch.int32, device=dev).reshape(-1, 2).contiguous()
    ty_d = torch.tensor(ty, dtype=torch.int32, device=dev).contiguous()
    nq, hq, d = q.shape
    out = torch.empty_like(q)
    lse = torch.empty(hq, nq, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    shp = ffa.FfaShape(nq, k.shape[0], hq, k.shape[1], d)
    rc = ffa.lib().ffa_fwd_noalloc(ctypes.byref(shp), q.data_ptr(), k.data_ptr(), v.data_ptr(), qr_d.data_ptr(),
                                   kr_d.data_ptr(), ty_d.data_ptr(), qr_d.shape[0],
                                   -1.0 if scale is None else float(scale), float(cap), out.data_ptr(),
                                   lse.data_ptr(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, ffa.ffa_status_string(rc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out, lse


def test_noalloc_matches_workspace_forward_on_consecutive_calls():
    for kind in ("page1", "ragged", "page1"):
        q, k, v, qr, kr, ty, scale, cap = _problem(kind)
        out_n, lse_n = _noalloc_via_abi(q, k, v, qr, kr, ty, scale, cap)
        out_w, lse_w = ffa.ffa_fwd(q.cuda(), k.cuda(), v.cuda(), qr, kr, ty, softmax_scale=scale, softcap=cap)
        torch.cuda.synchronize()
        assert_out_close(to64(out_n), to64(out_w))
        assert_lse_close(to64(lse_n), to64(lse_w))


def test_noalloc_rejects_problems_larger_than_its_scratch():
    n = 300000
    shp = ffa.FfaShape(n, n, 2, 1, 64)
    assert ffa.ffa_fwd_workspace_size(n, n, 2, 1, 64, 1) > ffa.FWD_NOALLOC_SCRATCH_BYTES
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    rc = ffa.lib().ffa_fwd_noalloc(ctypes.byref(shp), p, p, p, p, p, p, 1, -1.0, 0.0, p, p, None,
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == ffa.ERR_TOO_LARGE
    assert "scratch" in ffa.ffa_status_string(rc)
