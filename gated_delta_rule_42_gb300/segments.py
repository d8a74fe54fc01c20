"""Long sequences on one GPU: every sequence split into S segments that run at once.

The state chain of the chunked op is sequential per (sequence, value head), so
a batch with few long sequences keeps few SMs busy (a 65,536-token sequence
with 16 heads runs 16 chains of 1,024 chunks).  Here each sequence of a dense
batch is presented to the library as S consecutive segments of one packed
batch, so S times as many chains run side by side.  The segments' true start
states come from the state relay of the context-parallel path (``cp.py``):
each segment maps the state it starts from affinely, S_end = M S_start + c,
so a local pass (c, with segment 0 started from the real initial state), a
transition pass (M, the same records) and a scan of ``kda_state_compose``
calls give every segment its start state, from which the final pass runs.
The backward mirrors it: the start-state gradients from zero end gradients
(the reverse scan alone), a reverse relay with M^T, and the full backward.

The three forward passes share q, k, g and beta, so the per-chunk records are
computed once and reused through one forward context, which the backward then
reads.  All arithmetic runs in libkda; this module sequences the calls.
Results equal the unsplit op's up to rounding (the relay reorders the sums).
"""
from __future__ import annotations

from typing import NamedTuple, Optional

import torch

from . import cp
from .ops import chunk_kda_bwd_ctx, chunk_kda_bwd_state, chunk_kda_fwd_ctx, chunk_kda_fwd_reuse

__all__ = ["SegmentedContext", "segment_offsets", "chunk_kda_fwd_segmented", "chunk_kda_bwd_segmented"]


class SegmentedContext(NamedTuple):
    """What the segmented forward keeps for its backward."""
    cu: torch.Tensor            # int32 [B * S + 1] segment offsets over the flattened tokens
    h_start: torch.Tensor       # [B * S, HV, K, V] fp32: every segment's true start state
    M: torch.Tensor             # [B * S, HV, K, K] fp32: every segment's transition
    kctx: torch.Tensor          # the forward context of the final pass
    B: int
    S: int


def segment_offsets(B: int, T: int, S: int, device) -> torch.Tensor:
    """Offsets of S equal segments of each of B sequences of T tokens, as one
    packed batch (T must split into S whole 64-token chunks)."""
    if S < 1 or T % S != 0 or (T // S) % 64 != 0:
        raise ValueError(f"T={T} must split into S={S} segments of whole 64-token chunks")
    return torch.arange(0, B * T + 1, T // S, dtype=torch.int32, device=device)


def _flat(x: torch.Tensor) -> torch.Tensor:
    return x.reshape(1, x.shape[0] * x.shape[1], *x.shape[2:])


def chunk_kda_fwd_segmented(q, k, v, g, beta, initial_state=None, segments: int = 8,
                            output_final_state: bool = False, use_qk_l2norm: bool = False):
    """Forward of a dense batch [B, T, ...] with every sequence split into
    ``segments`` parts.  Returns (o [B, T, HV, V], final_state or None,
    SegmentedContext)."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    S = segments
    dev = q.device
    cu = segment_offsets(B, T, S, dev)
    q1, k1, v1, g1, b1 = (_flat(x) for x in (q, k, v, g, beta))
    kw = dict(use_qk_l2norm=use_qk_l2norm)
    # local pass: segment 0 of each sequence from its real initial state, the others from zero
    h_local = torch.zeros((B * S, HV, K, V), dtype=torch.float32, device=dev)
    if initial_state is not None:
        h_local[::S] = initial_state
    _, c, kctx = chunk_kda_fwd_ctx(q1, k1, v1, g1, b1, h_local, cu, True, need_output=False, **kw)
    # transitions, on the same records
    v0 = torch.zeros((1, B * T, HV, K), dtype=q.dtype, device=dev)
    eye = torch.eye(K, dtype=torch.float32, device=dev).expand(B * S, HV, K, K).contiguous()
    _, M = chunk_kda_fwd_reuse(q1, k1, v0, g1, b1, eye, cu, kctx, True, need_output=False, **kw)
    # relay: h_1 = c_0 (segment 0 started from the real state), h_{s+1} = M_s h_s + c_s
    h = h_local.clone()
    for b in range(B):
        if S > 1:
            h[b * S + 1] = c[b * S]
        for s in range(1, S - 1):
            i = b * S + s
            h[i + 1] = cp.compose(M[i:i + 1], h[i:i + 1], c[i:i + 1])[0]
    o, hT = chunk_kda_fwd_reuse(q1, k1, v1, g1, b1, h, cu, kctx, True, **kw)
    final = hT[S - 1::S].contiguous() if output_final_state else None
    return o.view(B, T, HV, V), final, SegmentedContext(cu, h, M, kctx, B, S)


def chunk_kda_bwd_segmented(q, k, v, g, beta, ctx: SegmentedContext, do, dht: Optional[torch.Tensor] = None,
                            need_dh0: bool = True, use_qk_l2norm: bool = False):
    """Backward on what :func:`chunk_kda_fwd_segmented` kept.  Returns dq, dk,
    dv, dg, dbeta (shaped like the inputs) and dh0 (or None)."""
    B, T = q.shape[0], q.shape[1]
    S = ctx.S
    q1, k1, v1, g1, b1, do1 = (_flat(x) for x in (q, k, v, g, beta, do))
    kw = dict(use_qk_l2norm=use_qk_l2norm)
    # start-state gradients: the last segment of each sequence from the real final-state
    # gradient, the others from zero
    end_local = torch.zeros_like(ctx.h_start)
    if dht is not None:
        end_local[S - 1::S] = dht
    d = chunk_kda_bwd_state(q1, k1, v1, g1, b1, ctx.h_start, ctx.cu, do1, end_local, ctx.kctx, **kw)
    # reverse relay: end_{S-2} = d_{S-1}, end_{s-1} = M_s^T end_s + d_s
    ends = end_local.clone()
    for b in range(B):
        if S > 1:
            ends[b * S + S - 2] = d[b * S + S - 1]
        for s in range(S - 2, 0, -1):
            i = b * S + s
            ends[i - 1] = cp.compose(ctx.M[i:i + 1], ends[i:i + 1], d[i:i + 1], True)[0]
    dq, dk, dv, dg, db, dh0 = chunk_kda_bwd_ctx(q1, k1, v1, g1, b1, ctx.h_start, ctx.cu, ctx.kctx, do1, ends,
                                                need_dh0=need_dh0, **kw)
    shape = lambda x, like: x.view(like.shape)  # noqa: E731
    return (shape(dq, q), shape(dk, k), shape(dv, v), shape(dg, g), shape(db, beta),
            dh0[::S].contiguous() if need_dh0 else None)
