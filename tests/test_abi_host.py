"""The C-ABI library builds, loads and exports every symbol include/ffa.h declares; host-side
argument checks return error codes before anything touches a GPU.  CPU only."""
import ctypes
import os
import re

import pytest

import flexible_mask_attention_range_gb300 as ffa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "ffa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ffa_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(lib_path):
    h = ctypes.CDLL(lib_path)
    names = _declared_functions()
    assert "ffa_fwd" in names and "ffa_bwd" in names
    for n in names:
        assert hasattr(h, n), f"missing export {n}"
    assert set(names) <= set(ffa.SIGNATURES), "binding lacks a signature for a declared symbol"


def test_build_info_and_status_strings(lib_path):
    assert "sm_103a" in ffa.ffa_build_info()
    for code in range(0, 6):
        assert isinstance(ffa.ffa_status_string(code), str)


def test_workspace_sizes(lib_path):
    a = ffa.ffa_fwd_workspace_size(2048, 2048, 8, 2, 64, 20)
    b = ffa.ffa_fwd_workspace_size(65536, 65536, 16, 4, 128, 3)
    c = ffa.ffa_bwd_workspace_size(65536, 65536, 16, 4, 128, 3)
    assert 0 < a < b < c
    # the backward workspace holds the fp32 dq accumulator
    assert c >= 65536 * 16 * 128 * 4
    assert ffa.ffa_fwd_workspace_size(100, 100, 3, 2, 64, 1) == 0          # Hq % Hkv != 0
    assert ffa.ffa_fwd_workspace_size(100, 100, 2, 1, 96, 1) == 0          # head_dim
    assert ffa.ffa_fwd_workspace_size(100, 100, 2, 1, 64, -1) == 0         # n_ranges < 0
    assert ffa.ffa_fwd_workspace_size((1 << 20) + 1, 8, 2, 1, 64, 1) == 0  # too many tokens


def _call_fwd(shape, R=1, softcap=0.0, ptr=16, ws=None, ws_bytes=0):
    L = ffa.lib()
    p = ctypes.c_void_p(ptr)
    return L.ffa_fwd(ctypes.byref(shape) if shape is not None else None, p, p, p, p, p, p, R, -1.0, softcap,
                     p, p, ws, ws_bytes, None, None)


def test_host_argument_checks_return_before_launch(lib_path):
    s = ffa.FfaShape(256, 256, 2, 1, 64)
    assert _call_fwd(None) == 1
    assert _call_fwd(ffa.FfaShape(256, 256, 3, 2, 64)) == 1      # Hq % Hkv
    assert _call_fwd(ffa.FfaShape(256, 256, 2, 1, 80)) == 2      # unsupported head_dim
    assert _call_fwd(s, R=-1) == 1
    assert _call_fwd(s, softcap=-1.0) == 1
    assert _call_fwd(s, softcap=float("nan")) == 1
    assert _call_fwd(s, ptr=18) == 1                              # misaligned pointers
    assert _call_fwd(s, ws=None, ws_bytes=0) == 4                 # no workspace
    assert _call_fwd(s, ws=ctypes.c_void_p(4096), ws_bytes=16) == 4  # too small
    assert _call_fwd(ffa.FfaShape(0, 0, 2, 1, 64)) == 0            # empty problem: nothing to do
    L = ffa.lib()
    p = ctypes.c_void_p(16)
    assert L.ffa_bwd(ctypes.byref(ffa.FfaShape(256, 256, 4, 3, 64)), p, p, p, p, p, p, p, p, p, 1, -1.0,
                     0.0, p, p, p, None, 0, None, None) == 1
    assert L.ffa_plan_tiles(ctypes.byref(s), None, None, None, 2, 0, p, None, 0, None, None) == 1


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    import flexible_mask_attention_range_gb300.build as b
    monkeypatch.setattr(b, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ffa, "_LIB", None)
    with pytest.raises(ffa.FfaError):
        ffa.lib()


def test_paged_forward_argument_checks(lib_path):
    L = ffa.lib()
    p = ctypes.c_void_p(16)
    s = ffa.FfaShape(256, 256, 2, 1, 64)

    def call(page_size=32, n_pages=8, table=p, shape=s):
        return L.ffa_fwd_paged(ctypes.byref(shape), p, p, p, table, page_size, n_pages, p, p, p, 1, -1.0, 0.0, p, p,
                               None, 0, None, None, None)

    for bad in (0, 8, 48, 256):
        assert call(page_size=bad) == 1                 # page sizes 16, 32, 64, 128 only
    assert call(n_pages=0) == 1
    assert call(page_size=128, n_pages=1 << 24) == 1    # pool rows must stay below 2^31
    assert call(table=None) == 1                        # keys present, no page table
    assert call() == 4                                  # valid paging arguments: then no workspace


def test_decode_argument_checks(lib_path):
    L = ffa.lib()
    p = ctypes.c_void_p(16)
    s = ffa.FfaShape(16, 4096, 8, 2, 128)
    assert L.ffa_fwd_decode_workspace_size(ctypes.byref(s), 16, 1) > 0
    assert L.ffa_fwd_decode_workspace_size(ctypes.byref(s), 16, 0) == 0      # max_seqlen_q >= 1
    assert L.ffa_fwd_decode_workspace_size(ctypes.byref(ffa.FfaShape(16, 16, 6, 4, 64)), 1, 1) == 0

    def call(shape=s, max_q=1, opts=None):
        return L.ffa_fwd_decode(ctypes.byref(shape), p, p, p, None, 0, 0, p, p, p, 16, max_q, -1.0, 0.0, p, p,
                                None, 0, None, None, opts)

    assert call(max_q=0) == 1
    assert call(shape=ffa.FfaShape(16, 4096, 8, 2, 96)) == 2                # head_dim
    assert call(opts=ctypes.byref(ffa.FfaOptions(18))) == 1                 # misaligned slopes
    assert call(opts=ctypes.byref(ffa.FfaOptions(16, 0, (ctypes.c_int32 * 7)(1)))) == 1   # reserved
    assert call(opts=ctypes.byref(ffa.FfaOptions(16))) == 4                 # ALiBi accepted
    assert call() == 4                                                      # then: no workspace


def test_build_refuses_forward_kernels_with_another_register_count():
    import flexible_mask_attention_range_gb300.build as b
    ok_log = ("ptxas info    : Compiling entry function '_ZN3ffa14ffa_fwd_kernelILi128ELb0ELb0EEEvv' for 'sm_103a'\n"
              "ptxas info    : Used 168 registers, used 1 barriers\n"
              "ptxas info    : Compiling entry function '_ZN3ffa14ffa_fwd_mergeILi128EEEvv' for 'sm_103a'\n"
              "ptxas info    : Used 40 registers\n")
    b.check_forward_registers(ok_log)
    with pytest.raises(RuntimeError):
        b.check_forward_registers(ok_log.replace("Used 168", "Used 160"))
    with pytest.raises(RuntimeError):
        b.check_forward_registers("no report at all\n")


def test_options_argument_checks(lib_path):
    """ffa_fwd_ex / ffa_bwd_ex: reserved option fields must be zero and the ALiBi slope array
    4-byte aligned; valid options (or none) pass on to the workspace check."""
    L = ffa.lib()
    p = ctypes.c_void_p(16)
    s = ffa.FfaShape(256, 256, 2, 1, 64)

    def fwd(opts):
        return L.ffa_fwd_ex(ctypes.byref(s), p, p, p, p, p, p, 1, -1.0, 0.0, p, p, None, 0, None, None, opts)

    def bwd(opts):
        return L.ffa_bwd_ex(ctypes.byref(s), p, p, p, p, p, p, p, p, p, 1, -1.0, 0.0, p, p, p, None, 0, None, None,
                            opts)

    for call in (fwd, bwd):
        assert call(None) == 4
        assert call(ctypes.byref(ffa.FfaOptions())) == 4
        det = ffa.FfaOptions()
        det.deterministic = 1
        assert call(ctypes.byref(det)) == 4
        for i in range(7):
            bad = ffa.FfaOptions()
            bad.reserved[i] = 1
            assert call(ctypes.byref(bad)) == 1
        mis = ffa.FfaOptions()
        mis.alibi_slopes = 18
        assert call(ctypes.byref(mis)) == 1


def test_noalloc_host_checks(lib_path):
    """ffa_fwd_noalloc refuses, before any launch, shapes whose forward workspace exceeds its
    fixed scratch (FFA_ERR_TOO_LARGE) and the usual invalid arguments."""
    L = ffa.lib()
    p = ctypes.c_void_p(16)

    def call(shape, ptr=p, softcap=0.0, R=1):
        return L.ffa_fwd_noalloc(ctypes.byref(shape), ptr, ptr, ptr, ptr, ptr, ptr, R, -1.0, softcap, ptr, ptr,
                                 None, None)

    n = 300000
    assert ffa.ffa_fwd_workspace_size(n, n, 2, 1, 64, 1) > ffa.FWD_NOALLOC_SCRATCH_BYTES
    rc = call(ffa.FfaShape(n, n, 2, 1, 64))
    assert rc == ffa.ERR_TOO_LARGE
    assert "scratch" in ffa.ffa_status_string(rc)
    s = ffa.FfaShape(256, 256, 2, 1, 64)
    assert call(ffa.FfaShape(256, 256, 3, 2, 64)) == 1       # Hq % Hkv
    assert call(ffa.FfaShape(256, 256, 2, 1, 96)) == 2       # head_dim
    assert call(s, softcap=-1.0) == 1
    assert call(s, ptr=ctypes.c_void_p(18)) == 1              # misaligned
    assert call(s, R=-1) == 1


def test_binding_refuses_cpu_tensors(lib_path):
    """The kernels take device pointers: every entry point rejects host tensors up front."""
    import torch
    q = torch.randn(256, 2, 64).to(torch.bfloat16)
    k = torch.randn(256, 1, 64).to(torch.bfloat16)
    lse = torch.zeros(2, 256)
    sl = ([(0, 256)], [(0, 256)], [1])
    pool = torch.zeros(2, 128, 1, 64, dtype=torch.bfloat16)
    table = torch.zeros(2, dtype=torch.int32)
    calls = [
        lambda: ffa.ffa_fwd(q, k, k, *sl),
        lambda: ffa.ffa_bwd(q, k, k, q, lse, q, *sl),
        lambda: ffa.ffa_fwd_noalloc(q, k, k, *sl),
        lambda: ffa.ffa_fwd_paged(q, pool, pool, table, 256, *sl),
        lambda: ffa.ffa_fwd_decode(q, k, k, *sl, max_seqlen_q=256),
        lambda: ffa.flex_flash_attn_func(q, k, k, *sl),
        lambda: ffa.ffa_plan_tiles(256, 256, *sl, device="cpu"),
    ]
    for c in calls:
        with pytest.raises(ValueError, match="CUDA"):
            c()
