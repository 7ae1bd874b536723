"""torch.autograd functions whose reverse pass is deterministic.

Warp user guide "Deterministic Execution", "Tape and Backward Passes": a
forward gather has no atomic, but its adjoint accumulates the output gradient
into the gradient of the gathered array -- a scatter-add, and with repeated
indices a nondeterministic one.  Here the forward runs ``det_gather_rows`` and
the adjoint runs ``det_scatter_add`` (1-D values) or ``det_scatter_add_rows``
(row tables) of the library, so the gradient bits are the same on every run
and at every launch shape.  Indices outside the source get zero outputs and
send no gradient.  Argument marshalling only: every step runs in the
library's CUDA kernels (the gradient buffer is zero-filled by torch).
"""
from __future__ import annotations

import torch

from . import det


class _Gather(torch.autograd.Function):
    @staticmethod
    def forward(ctx, src: torch.Tensor, idx: torch.Tensor, row_offset: int):
        ctx.save_for_backward(idx)
        ctx.src_shape = src.shape
        ctx.row_offset = row_offset
        return det.det_gather_rows(src.contiguous(), idx, row_offset=row_offset)

    @staticmethod
    def backward(ctx, grad_out: torch.Tensor):
        (idx,) = ctx.saved_tensors
        grad_src = None
        if ctx.needs_input_grad[0]:
            g = grad_out.contiguous()
            grad_src = torch.zeros(ctx.src_shape, dtype=g.dtype, device=g.device)
            if len(ctx.src_shape) == 1 and ctx.row_offset == 0:
                det.det_scatter_add(grad_src, idx, g)
            elif len(ctx.src_shape) == 1:   # same bits as det_scatter_add: rows of one element
                det.det_scatter_add_rows(grad_src.view(-1, 1), idx, g.view(-1, 1), row_offset=ctx.row_offset)
            else:
                det.det_scatter_add_rows(grad_src, idx, g, row_offset=ctx.row_offset)
        return grad_src, None, None


def gather(src: torch.Tensor, idx: torch.Tensor, row_offset: int = 0) -> torch.Tensor:
    """``src[idx + row_offset]`` (rows for a 2-D ``src``) with a deterministic backward.

    ``src`` is float32 or float64 on CUDA, ``idx`` int32 on the same device."""
    return _Gather.apply(src, idx, int(row_offset))
