"""Autograd binding of the fused Q+K rotation.

"How Unsloth Optimizes RoPE Embedding Computations in Triton Kernels",
Autograd Function Wrappers and Frequently Asked Questions: the rotation sits
in a ``torch.autograd.Function`` whose forward keeps the constants it needs
and whose backward runs the same kernel with the backward flag.  The
rotation is orthogonal, so the gradient of y = R(t) x is R(-t) applied to
dy; the pass-through tail and unrotated tokens pass their gradient through.

Here the forward is out of place (autograd keeps the inputs intact) and the
backward writes fresh gradient tensors; both are single launches of the
CUDA library.
"""
from __future__ import annotations

import torch

from . import rotate_qk


class RotaryQK(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, cos, sin, pos_idx, rotary_dim, layout, seq_before_head):
        q_out, k_out = rotate_qk(q.contiguous(), None if k is None else k.contiguous(), cos, sin,
                                 pos_idx, rotary_dim, layout, seq_before_head, backward=False)
        ctx.save_for_backward(cos, sin, pos_idx)
        ctx.cfg = (rotary_dim, layout, seq_before_head, k is not None)
        return q_out, k_out

    @staticmethod
    def backward(ctx, grad_q, grad_k):
        cos, sin, pos_idx = ctx.saved_tensors
        rotary_dim, layout, seq_before_head, has_k = ctx.cfg
        # an output that took no part in the loss arrives as None: rotate only the given ones
        gq = grad_q.contiguous() if grad_q is not None else None
        gk = grad_k.contiguous() if (has_k and grad_k is not None) else None
        dq = dk = None
        if gq is not None and gk is not None:
            dq, dk = rotate_qk(gq, gk, cos, sin, pos_idx, rotary_dim, layout, seq_before_head,
                               backward=True)
        elif gq is not None:
            dq, _ = rotate_qk(gq, None, cos, sin, pos_idx, rotary_dim, layout, seq_before_head,
                              backward=True)
        elif gk is not None:
            dk, _ = rotate_qk(gk, None, cos, sin, pos_idx, rotary_dim, layout, seq_before_head,
                              backward=True)
        return dq, dk, None, None, None, None, None, None


def rotary_qk(q: torch.Tensor, k: torch.Tensor | None, cos: torch.Tensor, sin: torch.Tensor,
              pos_idx: torch.Tensor | None = None, rotary_dim: int | None = None,
              layout: str = "split_half", seq_before_head: bool = False):
    """Differentiable fused rotation of q and k (k may be None): returns (q_rot, k_rot)."""
    rd = 2 * cos.shape[1] if rotary_dim is None else rotary_dim
    return RotaryQK.apply(q, k, cos, sin, pos_idx, rd, layout, seq_before_head)
