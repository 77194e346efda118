"""GB300 (sm_103a) range-masked flash attention: thin Python binding over libffa.so.

Every function here only marshals arguments: it checks tensor properties, allocates outputs
and the workspace with torch, and passes raw device pointers and the current CUDA stream to
the C ABI declared in include/ffa.h.  All computation runs in the library's CUDA kernels;
there is no fallback.  If libffa.so has not been built, importing works but every call
raises.

Interface after flex_flash_attn_func (MagiAttention issue #180): packed q [Nq, Hq, d],
k/v [Nk, Hkv, d] in bf16, slices q_ranges/k_ranges int32 [R, 2] and attn_type_map int32 [R]
(0 = FULL, 1 = CAUSAL); slices with start == end are no-ops.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import build as _build

FULL = 0
CAUSAL = 1
TILE_EMPTY, TILE_PARTIAL, TILE_FULL = 0, 1, 2
STATUS_BAD_RANGE = 1
STATUS_TIMEOUT = 2
STATUS_SMEM = 4
STATUS_BAD_PAGE = 8
FWD_NOALLOC_SCRATCH_BYTES = 8 << 20
ERR_TOO_LARGE = 5
TILE = 128


class FfaShape(ctypes.Structure):
    _fields_ = [("total_q", ctypes.c_int64), ("total_k", ctypes.c_int64),
                ("num_heads_q", ctypes.c_int32), ("num_heads_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


class FfaOptions(ctypes.Structure):
    _fields_ = [("alibi_slopes", ctypes.c_void_p), ("deterministic", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 7)]


class FfaError(RuntimeError):
    pass


_LIB = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# exported symbol -> (restype, argtypes), mirroring include/ffa.h
SIGNATURES = {
    "ffa_fwd_workspace_size": (_SZ, [ctypes.POINTER(FfaShape), _I32]),
    "ffa_bwd_workspace_size": (_SZ, [ctypes.POINTER(FfaShape), _I32]),
    "ffa_fwd": (ctypes.c_int, [ctypes.POINTER(FfaShape), _P, _P, _P, _P, _P, _P, _I32, _F, _F, _P, _P, _P,
                               _SZ, _P, _P]),
    "ffa_bwd": (ctypes.c_int, [ctypes.POINTER(FfaShape), _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _F, _F,
                               _P, _P, _P, _P, _SZ, _P, _P]),
    "ffa_fwd_ex": (ctypes.c_int, [ctypes.POINTER(FfaShape), _P, _P, _P, _P, _P, _P, _I32, _F, _F, _P, _P, _P,
                                  _SZ, _P, _P, ctypes.POINTER(FfaOptions)]),
    "ffa_bwd_ex": (ctypes.c_int, [ctypes.POINTER(FfaShape), _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _F, _F,
                                  _P, _P, _P, _P, _SZ, _P, _P, ctypes.POINTER(FfaOptions)]),
    "ffa_plan_tiles": (ctypes.c_int, [ctypes.POINTER(FfaShape), _P, _P, _P, _I32, _I32, _P, _P, _SZ, _P,
                                      _P]),
    "ffa_fwd_paged": (ctypes.c_int, [ctypes.POINTER(FfaShape), _P, _P, _P, _P, _I32, ctypes.c_int64, _P, _P, _P,
                                     _I32, _F, _F, _P, _P, _P, _SZ, _P, _P, ctypes.POINTER(FfaOptions)]),
    "ffa_fwd_decode_workspace_size": (_SZ, [ctypes.POINTER(FfaShape), _I32, _I32]),
    "ffa_fwd_decode": (ctypes.c_int, [ctypes.POINTER(FfaShape), _P, _P, _P, _P, _I32, ctypes.c_int64, _P, _P, _P,
                                      _I32, _I32, _F, _F, _P, _P, _P, _SZ, _P, _P, ctypes.POINTER(FfaOptions)]),
    "ffa_fwd_noalloc": (ctypes.c_int, [ctypes.POINTER(FfaShape), _P, _P, _P, _P, _P, _P, _I32, _F, _F, _P, _P,
                                       _P, _P]),
    "ffa_set_kernel_events": (ctypes.c_int, [_P, _P, _P, _P]),
    "ffa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ffa_build_info": (ctypes.c_char_p, []),
}


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libffa.so.  Raises if it has not been built (no fallback exists)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise FfaError(f"{path} is not built; run flexible_mask_attention_range_gb300.build.build() "
                           "(nvcc, sm_103a) first")
        h = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _LIB = h
    return _LIB


def _on(dev: torch.device, fn, *args):
    """Call a library entry point with ``dev`` current: the library resolves the device (SM
    count, function attributes, the no-alloc scratch address) through the current device."""
    with torch.cuda.device(dev):
        return fn(*args)


def _check(rc: int, what: str):
    if rc != 0:
        msg = lib().ffa_status_string(rc).decode()
        raise FfaError(f"{what} failed: {msg} (code {rc})")


def _shape(total_q, total_k, hq, hkv, d) -> FfaShape:
    return FfaShape(int(total_q), int(total_k), int(hq), int(hkv), int(d))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _cuda_device(t, name: str = "q") -> torch.device:
    """The device of the call: a CUDA device, else an error (the kernels take device pointers;
    there is no CPU path)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device}); there is no CPU path")
    return t.device


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, device: torch.device, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _ranges(q_ranges, k_ranges, attn_type_map, device):
    def conv(x, last):
        if not isinstance(x, torch.Tensor):
            x = torch.tensor(x, dtype=torch.int32)
        x = x.to(device=device, dtype=torch.int32).contiguous()
        return x.reshape(-1, 2) if last else x.reshape(-1)
    qr, kr, ty = conv(q_ranges, True), conv(k_ranges, True), conv(attn_type_map, False)
    if not (qr.shape[0] == kr.shape[0] == ty.shape[0]):
        raise ValueError("q_ranges, k_ranges and attn_type_map must have the same number of slices")
    return qr, kr, ty


def ffa_fwd_workspace_size(total_q, total_k, num_heads_q, num_heads_kv, head_dim, n_ranges) -> int:
    s = _shape(total_q, total_k, num_heads_q, num_heads_kv, head_dim)
    return int(lib().ffa_fwd_workspace_size(ctypes.byref(s), int(n_ranges)))


def ffa_bwd_workspace_size(total_q, total_k, num_heads_q, num_heads_kv, head_dim, n_ranges) -> int:
    s = _shape(total_q, total_k, num_heads_q, num_heads_kv, head_dim)
    return int(lib().ffa_bwd_workspace_size(ctypes.byref(s), int(n_ranges)))


def ffa_fwd_decode_workspace_size(total_q, total_k, num_heads_q, num_heads_kv, head_dim, n_ranges,
                                  max_seqlen_q) -> int:
    s = _shape(total_q, total_k, num_heads_q, num_heads_kv, head_dim)
    return int(lib().ffa_fwd_decode_workspace_size(ctypes.byref(s), int(n_ranges), int(max_seqlen_q)))


def ffa_status_string(code: int) -> str:
    return lib().ffa_status_string(int(code)).decode()


def ffa_set_kernel_events(fwd_start=None, fwd_stop=None, bwd_start=None, bwd_stop=None) -> None:
    """Record torch.cuda.Event objects around the main forward / backward kernels (or stop)."""
    h = [None if e is None else e.cuda_event for e in (fwd_start, fwd_stop, bwd_start, bwd_stop)]
    _check(lib().ffa_set_kernel_events(*h), "ffa_set_kernel_events")


def ffa_build_info() -> str:
    return lib().ffa_build_info().decode()


def ffa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_ranges, k_ranges, attn_type_map,
            softmax_scale: Optional[float] = None, softcap: float = 0.0,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
            alibi_slopes: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """out [Nq,Hq,d] bf16 and lse [Hq,Nq] float32 (natural log); see include/ffa.h.
    ``alibi_slopes`` (float32 [Hq]) adds slope_h * (key - query position) to the scores."""
    dev = _cuda_device(q)
    nq, hq, d = q.shape
    nk, hkv = k.shape[0], k.shape[1]
    _need(q, "q", torch.bfloat16, dev)
    _need(k, "k", torch.bfloat16, dev, (nk, hkv, d))
    _need(v, "v", torch.bfloat16, dev, (nk, hkv, d))
    qr, kr, ty = _ranges(q_ranges, k_ranges, attn_type_map, dev)
    if out is None:
        out = torch.empty(nq, hq, d, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(hq, nq, dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev, (nq, hq, d))
    _need(lse, "lse", torch.float32, dev, (hq, nq))
    R = qr.shape[0]
    shp = _shape(nq, nk, hq, hkv, d)
    ws_bytes = int(lib().ffa_fwd_workspace_size(ctypes.byref(shp), R))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    if alibi_slopes is None:
        rc = _on(dev, lib().ffa_fwd, ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(qr), _ptr(kr), _ptr(ty), R,
                           scale, float(softcap), _ptr(out), _ptr(lse), _ptr(workspace),
                           workspace.numel(), _ptr(status), _stream(dev))
    else:
        _need(alibi_slopes, "alibi_slopes", torch.float32, dev, (hq,))
        opts = FfaOptions(alibi_slopes.data_ptr())
        rc = _on(dev, lib().ffa_fwd_ex, ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(qr), _ptr(kr), _ptr(ty), R,
                              scale, float(softcap), _ptr(out), _ptr(lse), _ptr(workspace),
                              workspace.numel(), _ptr(status), _stream(dev), ctypes.byref(opts))
    _check(rc, "ffa_fwd")
    return out, lse


def ffa_fwd_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, page_table: torch.Tensor,
                  total_k: int, q_ranges, k_ranges, attn_type_map, softmax_scale: Optional[float] = None,
                  softcap: float = 0.0, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                  alibi_slopes: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """ffa_fwd over a paged key/value cache: ``k_pages``/``v_pages`` are bf16
    [n_pages, page_size, Hkv, d] pools and ``page_table`` (int32 [ceil(total_k / page_size)])
    maps each logical page of the ``total_k`` keys to a physical page; ranges, masks and
    results use logical positions (see include/ffa.h)."""
    dev = _cuda_device(q)
    nq, hq, d = q.shape
    n_pages, page_size, hkv = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    _need(q, "q", torch.bfloat16, dev)
    _need(k_pages, "k_pages", torch.bfloat16, dev, (n_pages, page_size, hkv, d))
    _need(v_pages, "v_pages", torch.bfloat16, dev, (n_pages, page_size, hkv, d))
    n_lp = (int(total_k) + page_size - 1) // page_size
    _need(page_table, "page_table", torch.int32, dev, (n_lp,))
    qr, kr, ty = _ranges(q_ranges, k_ranges, attn_type_map, dev)
    if out is None:
        out = torch.empty(nq, hq, d, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(hq, nq, dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev, (nq, hq, d))
    _need(lse, "lse", torch.float32, dev, (hq, nq))
    R = qr.shape[0]
    shp = _shape(nq, int(total_k), hq, hkv, d)
    ws_bytes = int(lib().ffa_fwd_workspace_size(ctypes.byref(shp), R))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    opts = None
    if alibi_slopes is not None:
        _need(alibi_slopes, "alibi_slopes", torch.float32, dev, (hq,))
        opts = FfaOptions(alibi_slopes.data_ptr())
    rc = _on(dev, lib().ffa_fwd_paged, ctypes.byref(shp), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                             int(page_size), int(n_pages), _ptr(qr), _ptr(kr), _ptr(ty), R, scale, float(softcap),
                             _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev),
                             ctypes.byref(opts) if opts is not None else None)
    _check(rc, "ffa_fwd_paged")
    return out, lse


def ffa_fwd_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_ranges, k_ranges, attn_type_map,
                   max_seqlen_q: int, softmax_scale: Optional[float] = None, softcap: float = 0.0,
                   page_table: Optional[torch.Tensor] = None, total_k: Optional[int] = None,
                   out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None,
                   alibi_slopes: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Decoding form of ffa_fwd (see include/ffa.h): the query heads of a key/value head are
    processed as rows of one problem.  Dense cache: k, v [Nk, Hkv, d].  Paged cache: k, v are
    [n_pages, page_size, Hkv, d] pools, ``page_table`` int32 and ``total_k`` the logical key
    count.  ``max_seqlen_q`` bounds the query tokens of any CAUSAL slice.  ``alibi_slopes``
    (float32 [Hq]) adds slope_h * (key - query position) as in ffa_fwd."""
    dev = _cuda_device(q)
    nq, hq, d = q.shape
    _need(q, "q", torch.bfloat16, dev)
    if page_table is None:
        nk, hkv = k.shape[0], k.shape[1]
        _need(k, "k", torch.bfloat16, dev, (nk, hkv, d))
        _need(v, "v", torch.bfloat16, dev, (nk, hkv, d))
        page_size, n_pages = 0, 0
    else:
        n_pages, page_size, hkv = k.shape[0], k.shape[1], k.shape[2]
        _need(k, "k", torch.bfloat16, dev, (n_pages, page_size, hkv, d))
        _need(v, "v", torch.bfloat16, dev, (n_pages, page_size, hkv, d))
        if total_k is None:
            raise ValueError("total_k is required with a page table")
        nk = int(total_k)
        _need(page_table, "page_table", torch.int32, dev, ((nk + page_size - 1) // page_size,))
    qr, kr, ty = _ranges(q_ranges, k_ranges, attn_type_map, dev)
    if out is None:
        out = torch.empty(nq, hq, d, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(hq, nq, dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev, (nq, hq, d))
    _need(lse, "lse", torch.float32, dev, (hq, nq))
    R = qr.shape[0]
    shp = _shape(nq, nk, hq, hkv, d)
    ws_bytes = int(lib().ffa_fwd_decode_workspace_size(ctypes.byref(shp), R, int(max_seqlen_q)))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    opts = None
    if alibi_slopes is not None:
        _need(alibi_slopes, "alibi_slopes", torch.float32, dev, (hq,))
        opts = FfaOptions(alibi_slopes.data_ptr())
    rc = _on(dev, lib().ffa_fwd_decode, ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(page_table),
             int(page_size), int(n_pages), _ptr(qr), _ptr(kr), _ptr(ty), R, int(max_seqlen_q), scale,
             float(softcap), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev),
             ctypes.byref(opts) if opts is not None else None)
    _check(rc, "ffa_fwd_decode")
    return out, lse


def ffa_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_ranges, k_ranges, attn_type_map,
                    softmax_scale: Optional[float] = None, softcap: float = 0.0,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """ffa_fwd without a workspace, for callers that cannot allocate device memory at call
    time: the library's fixed device scratch array is used instead (see include/ffa.h).
    Pass preallocated ``out``/``lse`` (and device-resident ranges) to keep the call itself
    free of allocations."""
    dev = _cuda_device(q)
    nq, hq, d = q.shape
    nk, hkv = k.shape[0], k.shape[1]
    _need(q, "q", torch.bfloat16, dev)
    _need(k, "k", torch.bfloat16, dev, (nk, hkv, d))
    _need(v, "v", torch.bfloat16, dev, (nk, hkv, d))
    qr, kr, ty = _ranges(q_ranges, k_ranges, attn_type_map, dev)
    if out is None:
        out = torch.empty(nq, hq, d, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(hq, nq, dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev, (nq, hq, d))
    _need(lse, "lse", torch.float32, dev, (hq, nq))
    if status is not None:
        _need(status, "status", torch.int32, dev)
    shp = _shape(nq, nk, hq, hkv, d)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    rc = _on(dev, lib().ffa_fwd_noalloc, ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(qr), _ptr(kr), _ptr(ty),
                               qr.shape[0], scale, float(softcap), _ptr(out), _ptr(lse), _ptr(status),
                               _stream(dev))
    _check(rc, "ffa_fwd_noalloc")
    return out, lse


def ffa_bwd(q, k, v, out, lse, dout, q_ranges, k_ranges, attn_type_map,
            softmax_scale: Optional[float] = None, softcap: float = 0.0,
            dq=None, dk=None, dv=None, workspace=None, status=None, alibi_slopes=None,
            deterministic: bool = False):
    """Gradients (dq, dk, dv) of sum(out * dout); see include/ffa.h.  ``deterministic``
    orders the dq additions so the results are bit-reproducible."""
    dev = _cuda_device(q)
    nq, hq, d = q.shape
    nk, hkv = k.shape[0], k.shape[1]
    _need(q, "q", torch.bfloat16, dev)
    _need(k, "k", torch.bfloat16, dev, (nk, hkv, d))
    _need(v, "v", torch.bfloat16, dev, (nk, hkv, d))
    _need(out, "out", torch.bfloat16, dev, (nq, hq, d))
    _need(dout, "dout", torch.bfloat16, dev, (nq, hq, d))
    _need(lse, "lse", torch.float32, dev, (hq, nq))
    qr, kr, ty = _ranges(q_ranges, k_ranges, attn_type_map, dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need(dq, "dq", torch.bfloat16, dev, q.shape)
    _need(dk, "dk", torch.bfloat16, dev, k.shape)
    _need(dv, "dv", torch.bfloat16, dev, v.shape)
    R = qr.shape[0]
    shp = _shape(nq, nk, hq, hkv, d)
    ws_bytes = int(lib().ffa_bwd_workspace_size(ctypes.byref(shp), R))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    if status is not None:
        _need(status, "status", torch.int32, dev)
    scale = -1.0 if softmax_scale is None else float(softmax_scale)
    if alibi_slopes is None and not deterministic:
        rc = _on(dev, lib().ffa_bwd, ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                           _ptr(qr), _ptr(kr), _ptr(ty), R, scale, float(softcap), _ptr(dq), _ptr(dk),
                           _ptr(dv), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev))
    else:
        if alibi_slopes is not None:
            _need(alibi_slopes, "alibi_slopes", torch.float32, dev, (hq,))
        opts = FfaOptions(_ptr(alibi_slopes), 1 if deterministic else 0)
        rc = _on(dev, lib().ffa_bwd_ex, ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                              _ptr(qr), _ptr(kr), _ptr(ty), R, scale, float(softcap), _ptr(dq), _ptr(dk),
                              _ptr(dv), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev),
                              ctypes.byref(opts))
    _check(rc, "ffa_bwd")
    return dq, dk, dv


def ffa_plan_tiles(total_q: int, total_k: int, q_ranges, k_ranges, attn_type_map, device="cuda",
                   by_column: bool = False, num_heads_q: int = 1, num_heads_kv: int = 1,
                   head_dim: int = 64, status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Tile classes uint8 [ceil(Nq/128), ceil(Nk/128)] computed by the device planner."""
    dev = torch.device(device)
    if dev.type != "cuda":
        raise ValueError(f"device must be a CUDA device (got {dev}); there is no CPU path")
    qr, kr, ty = _ranges(q_ranges, k_ranges, attn_type_map, dev)
    R = qr.shape[0]
    shp = _shape(total_q, total_k, num_heads_q, num_heads_kv, head_dim)
    nqt, nkt = -(-int(total_q) // TILE), -(-int(total_k) // TILE)
    tc = torch.empty(max(nqt, 0), max(nkt, 0), dtype=torch.uint8, device=dev)
    f = lib().ffa_bwd_workspace_size if by_column else lib().ffa_fwd_workspace_size
    ws = torch.empty(max(int(f(ctypes.byref(shp), R)), 256), dtype=torch.uint8, device=dev)
    rc = _on(dev, lib().ffa_plan_tiles, ctypes.byref(shp), _ptr(qr), _ptr(kr), _ptr(ty), R, 1 if by_column else 0,
                              _ptr(tc), _ptr(ws), ws.numel(), _ptr(status), _stream(dev))
    _check(rc, "ffa_plan_tiles")
    return tc


class _FlexFlashAttn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, q_ranges, k_ranges, attn_type_map, softmax_scale, softcap):
        out, lse = ffa_fwd(q, k, v, q_ranges, k_ranges, attn_type_map, softmax_scale, softcap)
        ctx.save_for_backward(q, k, v, out, lse, q_ranges, k_ranges, attn_type_map)
        ctx.softmax_scale, ctx.softcap = softmax_scale, softcap
        return out, lse

    @staticmethod
    def backward(ctx, dout, dlse):
        q, k, v, out, lse, qr, kr, ty = ctx.saved_tensors
        dq, dk, dv = ffa_bwd(q, k, v, out, lse, dout.contiguous(), qr, kr, ty, ctx.softmax_scale,
                             ctx.softcap)
        return dq, dk, dv, None, None, None, None, None


def flex_flash_attn_func(q, k, v, q_ranges, k_ranges, attn_type_map, max_seqlen_q=None,
                         max_seqlen_k=None, softmax_scale=None, softcap=0.0):
    """(out, lse) with autograd; max_seqlen_q/k are accepted and not needed (global tiling).

    The gradient flows through `out` only (the lse output is treated as non-differentiable).
    """
    dev = _cuda_device(q)
    qr, kr, ty = _ranges(q_ranges, k_ranges, attn_type_map, dev)
    return _FlexFlashAttn.apply(q, k, v, qr, kr, ty, softmax_scale, softcap)
