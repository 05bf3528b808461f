"""Differentiable entry point: the forward pass through ``gdr_chunk_fwd`` and
its gradient through ``gdr_chunk_bwd``, both on the CUDA library.

The call follows the public shape of the chunked gated-delta-rule operator
(q, k, v, g, beta, scale, initial state, whether to return the final state,
packed-sequence offsets), so code written against that interface can call
this one.  Layouts are those of ``include/gdr.h``: q, k [B, T, H, K];
v [B, T, H, V]; g (per-token log gate) and beta [B, T, H] float32; states
[N, H, K, V] float32 (h = S^T).  ``beta=None`` selects the beta-free mode.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import api


class _ChunkGatedDeltaRule(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, scale, initial_state, output_final_state, cu_seqlens):
        o, ht = api.gdr_chunk_fwd(q, k, v, g, beta, cu_seqlens=cu_seqlens, h0=initial_state,
                                  output_final_state=output_final_state, scale=scale)
        ctx.save_for_backward(q, k, v, g, beta, initial_state, cu_seqlens)
        ctx.scale = scale
        return o, ht

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, g, beta, h0, cu = ctx.saved_tensors
        want_dh0 = h0 is not None and ctx.needs_input_grad[6]
        dq, dk, dv, dg, dbeta, dh0 = api.gdr_chunk_bwd(
            q, k, v, g, beta, do.contiguous(), cu_seqlens=cu, h0=h0,
            dht=None if dht is None else dht.contiguous(), scale=ctx.scale, want_dh0=want_dh0)
        return dq, dk, dv, dg, dbeta, None, dh0, None, None


def chunk_gated_delta_rule(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                           beta: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                           initial_state: Optional[torch.Tensor] = None,
                           output_final_state: bool = False,
                           cu_seqlens: Optional[torch.Tensor] = None
                           ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """o, final_state of the chunked gated delta rule, differentiable with
    respect to q, k, v, g, beta and initial_state.  ``scale`` defaults to
    1/sqrt(K).  ``final_state`` is None unless ``output_final_state``.  q, k
    and v may be views with token and head strides (e.g. slices of one fused
    projection); the library reads them in place."""
    return _ChunkGatedDeltaRule.apply(q, k, v, g.contiguous(),
                                      None if beta is None else beta.contiguous(),
                                      0.0 if scale is None else float(scale),
                                      None if initial_state is None else initial_state.contiguous(),
                                      bool(output_final_state), cu_seqlens)
