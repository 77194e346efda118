"""Shared helpers for the GPU parity tests: tolerances and comparisons against the oracle."""
import numpy as np
import torch

# Tolerances (float32/bf16 path vs float64 oracle)
O_MAX_ABS = 2e-2
O_MEAN_REL = 1e-2
LSE_MAX_ABS = 1e-3
GRAD_MAX_ABS = 5e-2


def to64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_out_close(got, ref, what="out", max_abs=O_MAX_ABS, mean_rel=O_MEAN_REL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    diff = np.abs(got - ref)
    ma = float(diff.max()) if diff.size else 0.0
    denom = float(np.abs(ref).mean()) if ref.size else 0.0
    mr = float(diff.mean()) / denom if denom > 0 else float(diff.mean())
    assert ma <= max_abs, f"{what}: max-abs {ma:.3e} > {max_abs}"
    assert mr <= mean_rel, f"{what}: mean-rel {mr:.3e} > {mean_rel}"
    return ma, mr


def assert_lse_close(got, ref, what="lse", tol=LSE_MAX_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    ninf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf_ref), f"{what}: -inf rows differ"
    fin = ~ninf_ref
    if fin.any():
        assert np.all(np.isfinite(got[fin])), f"{what}: non-finite where the oracle is finite"
        ma = float(np.abs(got[fin] - ref[fin]).max())
        assert ma <= tol, f"{what}: max-abs {ma:.3e} > {tol}"
        return ma
    return 0.0


def assert_grad_close(got, ref, what, tol=GRAD_MAX_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    ma = float(np.abs(got - ref).max()) if got.size else 0.0
    assert ma <= tol, f"{what}: max-abs {ma:.3e} > {tol}"
    return ma


def cuda(*ts):
    return [None if t is None else t.cuda() for t in ts]
