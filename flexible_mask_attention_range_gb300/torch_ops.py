"""torch.library registration of the attention so torch.compile can trace it.

The operators only forward to the C ABI through this package's binding (no computation
here).  They follow the integration pattern of "Add torch.compile support to flash attention
3" (flash-attention pull request #1769): custom operators with fake (shape-only)
implementations, so the compiler can trace through them without running kernels, plus an
autograd registration that routes the backward pass to the backward kernel.  With the slice
list padded to a fixed length by start == end slices (MagiAttention issue #180), a compiled
function keeps static shapes while the real slices change from call to call.

    ffa::fwd(q, k, v, q_ranges, k_ranges, attn_type_map, softmax_scale, softcap) -> (out, lse)
    ffa::bwd(dout, q, k, v, out, lse, q_ranges, k_ranges, attn_type_map, softmax_scale,
             softcap) -> (dq, dk, dv)

softmax_scale <= 0 selects 1/sqrt(d).
"""
from __future__ import annotations

from typing import Tuple

import torch
from torch import Tensor

from . import ffa_bwd as _ffa_bwd
from . import ffa_fwd as _ffa_fwd


@torch.library.custom_op("ffa::fwd", mutates_args=())
def fwd(q: Tensor, k: Tensor, v: Tensor, q_ranges: Tensor, k_ranges: Tensor, attn_type_map: Tensor,
        softmax_scale: float, softcap: float) -> Tuple[Tensor, Tensor]:
    scale = None if softmax_scale <= 0 else softmax_scale
    return _ffa_fwd(q, k, v, q_ranges, k_ranges, attn_type_map, scale, softcap)


@fwd.register_fake
def _fwd_fake(q, k, v, q_ranges, k_ranges, attn_type_map, softmax_scale, softcap):
    nq, hq, d = q.shape
    return q.new_empty(nq, hq, d), q.new_empty(hq, nq, dtype=torch.float32)


@torch.library.custom_op("ffa::bwd", mutates_args=())
def bwd(dout: Tensor, q: Tensor, k: Tensor, v: Tensor, out: Tensor, lse: Tensor, q_ranges: Tensor,
        k_ranges: Tensor, attn_type_map: Tensor, softmax_scale: float,
        softcap: float) -> Tuple[Tensor, Tensor, Tensor]:
    scale = None if softmax_scale <= 0 else softmax_scale
    return _ffa_bwd(q, k, v, out, lse, dout.contiguous(), q_ranges, k_ranges, attn_type_map, scale, softcap)


@bwd.register_fake
def _bwd_fake(dout, q, k, v, out, lse, q_ranges, k_ranges, attn_type_map, softmax_scale, softcap):
    return torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)


def _setup_context(ctx, inputs, output):
    q, k, v, q_ranges, k_ranges, attn_type_map, softmax_scale, softcap = inputs
    out, lse = output
    ctx.save_for_backward(q, k, v, out, lse, q_ranges, k_ranges, attn_type_map)
    ctx.softmax_scale = softmax_scale
    ctx.softcap = softcap


def _backward(ctx, dout, dlse):
    q, k, v, out, lse, q_ranges, k_ranges, attn_type_map = ctx.saved_tensors
    dq, dk, dv = bwd(dout, q, k, v, out, lse, q_ranges, k_ranges, attn_type_map, ctx.softmax_scale, ctx.softcap)
    return dq, dk, dv, None, None, None, None, None


fwd.register_autograd(_backward, setup_context=_setup_context)


def flex_flash_attn(q: Tensor, k: Tensor, v: Tensor, q_ranges: Tensor, k_ranges: Tensor, attn_type_map: Tensor,
                    softmax_scale: float | None = None, softcap: float = 0.0) -> Tuple[Tensor, Tensor]:
    """(out, lse) through the registered operator (traceable by torch.compile; gradients
    flow through `out`).  Ranges must already be int32 tensors on q's device."""
    return fwd(q, k, v, q_ranges, k_ranges, attn_type_map, -1.0 if softmax_scale is None else float(softmax_scale),
               float(softcap))
