"""torch.autograd binding of context-parallel causal attention.

The multimodal context-parallel page (§4.2, gradient path; §5.2, the image
prefix) has every CP rank differentiate its own text queries against the
replicated image prefix, then sums those per-rank prefix gradients with an
AllReduce hooked onto the image embeddings' gradient.  Here every rank lives
in one GPU's memory: ``cp_attn_bwd`` sums the per-rank prefix terms in a fixed
order (ranks 0..P-1, then the prefix queries' own term) before it returns, so
the gradients that reach autograd are already the reduced ones.

``prefix_hook`` gives a caller the quantity the page's hook reduces.  It is
called during the backward with the per-rank terms ``[2, P+1, n*N, H_kv, d]``
(dK, dV; slot P is the prefix queries' own term), before autograd receives
the summed gradients.

Every step runs in the library's CUDA kernels; this module only marshals
tensors through :mod:`torch.autograd`.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence

import torch

from . import cp_attn_bwd, cp_attn_fwd


class CPAttention(torch.autograd.Function):
    """``(out, lse) = CPAttention.apply(q, k, v, cu_seqlens, P, prefix_len,
    softmax_scale, prefix_hook)``.  lse is not differentiable."""

    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens, P, prefix_len, softmax_scale, prefix_hook):
        cu = tuple(int(x) for x in cu_seqlens)
        if q.dtype == torch.bfloat16:
            # the bf16 remainder of the output keeps D = dO.O exact in the backward
            out, lse, out_lo = cp_attn_fwd(q, k, v, cu, P, prefix_len, softmax_scale,
                                           residual=True)
        else:
            out, lse = cp_attn_fwd(q, k, v, cu, P, prefix_len, softmax_scale)
            out_lo = None
        ctx.save_for_backward(q, k, v, out, lse, out_lo)
        ctx.meta = (cu, int(P), int(prefix_len), float(softmax_scale), prefix_hook)
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, out, lse, out_lo = ctx.saved_tensors
        cu, P, N, scale, hook = ctx.meta
        if dout is None:
            dout = torch.zeros_like(out)
        dout = dout.to(q.dtype).contiguous()
        want_pre = hook is not None and N > 0
        res = cp_attn_bwd(q, k, v, out, lse, dout, cu, P, N, scale,
                          per_rank_prefix=want_pre, out_lo=out_lo)
        dq, dk, dv = res[:3]
        if want_pre:
            hook(res[3])
        grads = []
        for g, x, need in zip((dq, dk, dv), (q, k, v), ctx.needs_input_grad[:3]):
            grads.append(g.to(x.dtype) if need else None)
        return (*grads, None, None, None, None, None)


def cp_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                 cu_seqlens: Sequence[int], P: int, prefix_len: int = 0,
                 softmax_scale: Optional[float] = None,
                 prefix_hook: Optional[Callable[[torch.Tensor], None]] = None):
    """Differentiable zigzag context-parallel causal attention over packed
    samples ``[prefix_i ++ text_i]`` (THD layout ``[T, H, d]``, bf16 or fp32,
    on a CUDA device).  Returns ``(out, lse)``; gradients flow to q, k and v.
    ``k`` / ``v`` may hold fewer heads than ``q`` (grouped-query attention:
    query head h reads KV head h // (H / H_kv)).  ``softmax_scale`` defaults
    to ``1/sqrt(d)``."""
    if softmax_scale is None:
        softmax_scale = q.shape[-1] ** -0.5
    return CPAttention.apply(q, k, v, cu_seqlens, P, prefix_len, softmax_scale, prefix_hook)
