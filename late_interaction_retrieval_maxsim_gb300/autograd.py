"""``torch.autograd`` entry point over the C ABI.

"FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Retrieval"
(arXiv 2605.29517) §4.2.2 derives the inverse-grid map during the training
step itself: the forward saves its argmax, and the backward turns it into dQ
and dD without materialising the similarity tensor.  ``maxsim`` wraps exactly
that: ``maxsim_forward`` keeps its argmax for ``maxsim_backward``, which sorts
each document's sources by token in shared memory and reduces them
destination by destination.  Every step runs in the library's CUDA kernels;
this module only routes tensors.

Gradients are computed in FP32 by the kernels and returned in the inputs'
dtype (autograd requires a gradient of its input's dtype); callers that need
the FP32 gradients call ``maxsim_backward`` directly.
"""
from __future__ import annotations

import torch

from . import maxsim_backward, maxsim_forward


class MaxSimFunction(torch.autograd.Function):
    """scores[q, b] = sum_i max_t <Q[q, i], D[cu[b] + t]> with its closed-form
    backward (Eqs. (2)-(3) of §4.2.1)."""

    @staticmethod
    def forward(ctx, Q, D, q_lens, cu_seqlens):
        scores, argmax, _ = maxsim_forward(Q, q_lens, D, cu_seqlens)
        ctx.save_for_backward(Q, D, q_lens, cu_seqlens, argmax)
        return scores

    @staticmethod
    def backward(ctx, grad_scores):
        Q, D, q_lens, cu_seqlens, argmax = ctx.saved_tensors
        dQ, dD = maxsim_backward(grad_scores.float().contiguous(), argmax, Q, q_lens, D, cu_seqlens)
        return (dQ.to(Q.dtype) if ctx.needs_input_grad[0] else None,
                dD.to(D.dtype) if ctx.needs_input_grad[1] else None, None, None)


def maxsim(Q: torch.Tensor, D: torch.Tensor, q_lens: torch.Tensor, cu_seqlens: torch.Tensor) -> torch.Tensor:
    """Differentiable fused MaxSim.

    Q [n_q, lq_max, 128] and D [total, 128] (FP16/BF16, CUDA, contiguous);
    q_lens [n_q] and cu_seqlens [n_docs + 1] int32 on the same device.
    Returns FP32 scores [n_q, n_docs]."""
    return MaxSimFunction.apply(Q, D, q_lens, cu_seqlens)
