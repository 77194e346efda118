"""torch.library operators ffa::fwd / ffa::bwd: fake implementations (shape inference without
running kernels), autograd registration, and torch.compile over padded slice lists (static
shapes, no recompilation when the real slices change)."""
import pytest
import torch

import workloads as W
import flexible_mask_attention_range_gb300 as ffa
from flexible_mask_attention_range_gb300 import torch_ops


def test_fake_impl_shapes_on_meta_tensors():
    q = torch.empty(300, 8, 64, dtype=torch.bfloat16, device="meta")
    k = torch.empty(500, 2, 64, dtype=torch.bfloat16, device="meta")
    qr = torch.empty(4, 2, dtype=torch.int32, device="meta")
    ty = torch.empty(4, dtype=torch.int32, device="meta")
    out, lse = torch.ops.ffa.fwd(q, k, k, qr, qr, ty, -1.0, 0.0)
    assert out.shape == (300, 8, 64) and out.dtype == torch.bfloat16
    assert lse.shape == (8, 300) and lse.dtype == torch.float32
    dq, dk, dv = torch.ops.ffa.bwd(out, q, k, k, out, lse, qr, qr, ty, -1.0, 0.0)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == k.shape


def _padded(qr, kr, ty, n):
    extra = n - len(ty)
    return (torch.tensor(list(qr) + [(0, 0)] * extra, dtype=torch.int32, device="cuda"),
            torch.tensor(list(kr) + [(0, 0)] * extra, dtype=torch.int32, device="cuda"),
            torch.tensor(list(ty) + [0] * extra, dtype=torch.int32, device="cuda"))


@pytest.mark.gpu
def test_opcheck(lib_path):
    w = W.get("tiny_256").padded()
    q, k, v, _ = (t.cuda() if t is not None else None for t in W.draw_qkv(w.total, w.total, w.hq, w.hkv, w.d, 0))
    qr, kr, ty = _padded(w.q_ranges, w.k_ranges, w.types, 4)
    q.requires_grad_(True)
    torch.library.opcheck(torch.ops.ffa.fwd, (q, k, v, qr, kr, ty, 0.125, 0.0),
                          test_utils=("test_schema", "test_autograd_registration", "test_faketensor"))


@pytest.mark.gpu
def test_compiled_padded_slices_match_eager_without_recompiling(lib_path):
    torch._dynamo.reset()
    n, hq, hkv, d = 1024, 4, 2, 64
    q0, k0, v0, do = (t.cuda() for t in W.draw_qkv(n, n, hq, hkv, d, 5))

    def step(q, k, v, qr, kr, ty):
        out, _ = torch_ops.flex_flash_attn(q, k, v, qr, kr, ty)
        return (out.float() * do.float()).sum()

    compiled = torch.compile(step, backend="aot_eager", fullgraph=True)
    slice_sets = [([(0, 512), (512, 1024)], [(0, 512), (0, 1024)], [0, 1]),
                  ([(0, 1024)], [(0, 1024)], [1]),
                  ([(0, 300), (300, 1024), (100, 200)], [(0, 300), (0, 1024), (500, 900)], [1, 1, 0])]
    with torch._dynamo.config.patch(error_on_recompile=True):
        for qr_l, kr_l, ty_l in slice_sets:
            qr, kr, ty = _padded(qr_l, kr_l, ty_l, 8)
            qa, ka, va = (t.clone().requires_grad_(True) for t in (q0, k0, v0))
            compiled(qa, ka, va, qr, kr, ty).backward()
            out, lse = ffa.ffa_fwd(q0, k0, v0, qr, kr, ty)
            dq, dk, dv = ffa.ffa_bwd(q0, k0, v0, out, lse, do, qr, kr, ty)
            torch.cuda.synchronize()
            assert torch.equal(ka.grad, dk) and torch.equal(va.grad, dv)
            assert float((qa.grad.float() - dq.float()).abs().max()) < 1e-2   # dq: atomic order
