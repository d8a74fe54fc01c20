"""Context parallelism: one sequence split across ranks, with a state relay.

Rank r holds tokens [T_r, T_{r+1}) of every sequence of a dense batch (the same
B on every rank).  Its segment maps the state it starts from affinely,
S_end = M_r S_start + c_r, where c_r is its final state from a zero start and
M_r (K x K) the segment's transition: ``kda_chunk_fwd`` on the segment with
v = 0, V = K and h0 = the identity returns M_r as its final state.  The forward
exchanges (c_r, M_r) once (all-gather) and runs the exclusive scan
h_{r+1} = M_r h_r + c_r locally, so every rank gets its true start state and
reruns its segment from it.  The backward is the mirror image: the gradient of a
segment's start state is dh_start = M_r^T dh_end + d_r, with d_r the gradient
from a zero end gradient, so one exchange of (d_r, M_r) and the reverse scan
dh_end(r) = M_{r+1}^T dh_end(r+1) + d_{r+1} give every rank its end-state
gradient.  This is the synchronous context parallelism of "[KDA] Add Paddle
training compatibility" (PFCCLab/flash-linear-attention PR #2, summary and
test plan: two-GPU context-parallel forward/backward checks).

The arithmetic runs in libkda (the chunked kernels and ``kda_state_compose``);
this module only moves states between ranks (``torch.distributed``) and
sequences the calls.  The exchange and scan are separated from the per-rank
compute (``relay_start_state``, ``relay_end_grad``) so that the host logic can
be checked with CPU ranks.
"""
from __future__ import annotations

import ctypes
from typing import Callable, List, NamedTuple, Optional, Union

import torch

from . import _lib
from .ops import (chunk_kda_bwd, chunk_kda_bwd_ctx, chunk_kda_bwd_state, chunk_kda_fwd, chunk_kda_fwd_ctx,
                  chunk_kda_fwd_reuse)


def compose(M: torch.Tensor, h: torch.Tensor, c: Optional[torch.Tensor], transpose: bool = False) -> torch.Tensor:
    """op(M) h + c per (sequence, value head) on the GPU (``kda_state_compose``).
    M [N, HV, K, K], h and c [N, HV, K, V] fp32."""
    lib = _lib.load()
    N, HV, K, V = h.shape
    out = torch.empty_like(h)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    _lib.check(lib, lib.kda_state_compose(p(M.contiguous()), p(h.contiguous()),
                                          p(None if c is None else c.contiguous()), p(out), N * HV, K, V,
                                          1 if transpose else 0,
                                          ctypes.c_void_p(torch.cuda.current_stream(h.device).cuda_stream)))
    return out


def relay_start_state(c: torch.Tensor, M: torch.Tensor, h0: Optional[torch.Tensor], rank: int,
                      gather: Callable[[torch.Tensor], List[torch.Tensor]],
                      compose_fn: Callable = compose) -> torch.Tensor:
    """The state this rank's segment starts from: exclusive scan of the
    segments' affine maps over the ranks before it, starting from rank 0's h0
    (the sequences' initial state; None = zeros; other ranks' h0 is ignored)."""
    cs, Ms = gather(c), gather(M)
    h = gather(torch.zeros_like(c) if h0 is None else h0)[0]
    for r in range(rank):
        h = compose_fn(Ms[r], h, cs[r], False)
    return h


def relay_end_grad(d: torch.Tensor, M: torch.Tensor, dhT: Optional[torch.Tensor], rank: int, world: int,
                   gather: Callable[[torch.Tensor], List[torch.Tensor]],
                   compose_fn: Callable = compose) -> torch.Tensor:
    """The gradient of this rank's segment-end state: reverse exclusive scan of
    dh_start = M^T dh_end + d over the ranks after it, starting from the last
    rank's dhT (the final-state gradient; None = zeros; other ranks' dhT is
    ignored)."""
    ds, Ms = gather(d), gather(M)
    g = gather(torch.zeros_like(d) if dhT is None else dhT)[world - 1]
    for r in range(world - 1, rank, -1):
        g = compose_fn(Ms[r], g, ds[r], True)
    return g


def all_gather_fn(group=None) -> Callable[[torch.Tensor], List[torch.Tensor]]:
    import torch.distributed as dist

    def gather(x):
        out = [torch.empty_like(x) for _ in range(dist.get_world_size(group))]
        dist.all_gather(out, x.contiguous(), group=group)
        return out

    return gather


def segment_transition(q, k, g, beta, kctx=None, **kw) -> torch.Tensor:
    """M [B, HV, K, K] of this segment: the forward with v = 0, V = K and
    h0 = the identity, whose final state is M (the state evolves linearly);
    the final state alone, no output.  kctx: a forward context of this segment
    (same q, k, g, beta) whose records it reuses (the context then holds this
    pass's chunk-start states)."""
    B, T, H, K = q.shape
    HV = beta.shape[2]
    v0 = torch.zeros((B, T, HV, K), dtype=q.dtype, device=q.device)
    eye = torch.eye(K, dtype=torch.float32, device=q.device).expand(B, HV, K, K).contiguous()
    if kctx is not None:
        return chunk_kda_fwd_reuse(q, k, v0, g, beta, eye, None, kctx, True, need_output=False, **kw)[1]
    return chunk_kda_fwd(q, k, v0, g, beta, eye, None, True, need_output=False, **kw)[1]


class SegmentContext(NamedTuple):
    """What a rank's forward keeps for its backward: the segment's true start
    state, its transition M, and the forward context of the final pass (the
    per-chunk records and chunk-start states; None when not kept)."""
    h_start: torch.Tensor
    M: torch.Tensor
    kctx: Optional[torch.Tensor]


def cp_forward(q, k, v, g, beta, h0, rank: int, gather, compose_fn: Callable = compose,
               keep_context: bool = True, **kw):
    """Forward of this rank's segment.  h0: the sequences' initial state (read
    from rank 0; may be None).  Returns (o, hT, SegmentContext): hT of the last
    rank is the sequences' final state.  keep_context: the final pass keeps its
    forward context, so the two backward passes do not recompute it."""
    if keep_context:  # one record pass: the transition and the final pass reuse the context's records
        _, c, kctx = chunk_kda_fwd_ctx(q, k, v, g, beta, None, None, True, need_output=False, **kw)
        M = segment_transition(q, k, g, beta, kctx, **kw)
        hs = relay_start_state(c, M, h0, rank, gather, compose_fn)
        o, hT = chunk_kda_fwd_reuse(q, k, v, g, beta, hs, None, kctx, True, **kw)
    else:
        _, c = chunk_kda_fwd(q, k, v, g, beta, None, None, True, need_output=False, **kw)
        M = segment_transition(q, k, g, beta, **kw)
        hs = relay_start_state(c, M, h0, rank, gather, compose_fn)
        (o, hT), kctx = chunk_kda_fwd(q, k, v, g, beta, hs, None, True, **kw), None
    return o, hT, SegmentContext(hs, M, kctx)


def cp_backward(q, k, v, g, beta, seg: Union[SegmentContext, torch.Tensor], do, dhT, rank: int, world: int,
                gather, compose_fn: Callable = compose, **kw):
    """Backward of this rank's segment given what :func:`cp_forward` kept (or
    just the start state, in which case M and the forward context are
    recomputed) and dhT (the final-state gradient, read from the last rank; may
    be None).  Returns dq, dk, dv, dg, dbeta and the start-state gradient (rank 0:
    the gradient of the sequences' initial state)."""
    if not isinstance(seg, SegmentContext):
        seg = SegmentContext(seg, segment_transition(q, k, g, beta, **kw), None)

    def bwd(dh_end):
        if seg.kctx is not None:
            return chunk_kda_bwd_ctx(q, k, v, g, beta, seg.h_start, None, seg.kctx, do, dh_end, **kw)
        return chunk_kda_bwd(q, k, v, g, beta, seg.h_start, None, do, dh_end, **kw)

    # d: the start-state gradient from a zero end gradient (the reverse scan alone)
    d = chunk_kda_bwd_state(q, k, v, g, beta, seg.h_start, None, do, None, seg.kctx, **kw)
    dh_end = relay_end_grad(d, seg.M, dhT, rank, world, gather, compose_fn)
    return bwd(dh_end)
