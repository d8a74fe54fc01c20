"""PyTorch-facing entry points: ``chunk_kda`` (autograd) and ``recurrent_kda``.

The signatures follow the KDA contract of "kda in torchtitan (training)"
(pytorch/torchtitan PR #4164, agent note on ``recurrent_kda``):
``(q, k, v, gate, beta, initial_state=None, *, cu_seqlens=None,
output_final_state=False) -> (output, final_state)`` where ``gate`` is the
per-token log2 decay, queries are scaled by 1/sqrt(K) internally,
``cu_seqlens`` is a device int32 offset array (repeated offsets are empty
slots) and states are fp32 with one entry per logical sequence.

PyTorch provides device memory and the current stream; every step of the
computation runs in libkda's CUDA kernels.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib

__all__ = ["chunk_kda", "recurrent_kda", "chunk_kda_fwd", "chunk_kda_bwd", "chunk_kda_fwd_ctx",
           "chunk_kda_bwd_ctx", "chunk_kda_bwd_state", "chunk_kda_fwd_reuse", "make_inputs_struct", "KdaGateParams"]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tensor(name, t, dtype, device, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


class KdaGateParams:
    """The KDA gate inside the op (KDA_GATE_IN_KERNEL): ``g`` then holds the raw
    gate pre-activations a and the op makes the per-token log2 decay itself,
    g = -exp(A_log) softplus(a + bias) (unbounded, ``lower_bound`` None) or
    g = lower_bound sigmoid(exp(A_log) (a + bias)) (bounded, lower_bound < 0).
    A_log [HV] and bias [HV, K] are fp32 device tensors or None (an omitted
    A_log is a unit scale, the same as zeros)."""

    def __init__(self, A_log=None, bias=None, lower_bound=None):
        self.A_log, self.bias = A_log, bias
        self.lower_bound = 0.0 if lower_bound is None else float(lower_bound)


def make_inputs_struct(q, k, v, g, beta, initial_state=None, cu_seqlens=None, use_qk_l2norm=False,
                       gate: Optional[KdaGateParams] = None, dA_log=None, dbias=None):
    """Validate the tensors and build the C ``kda_inputs`` struct.  With
    use_qk_l2norm the library L2-normalises every q and k row itself; a gate of
    shape [B, T, HV] (instead of [B, T, HV, K]) is the scalar-gate variant;
    ``gate`` (:class:`KdaGateParams`) makes the op apply the KDA gate to the raw
    gate in ``g``, and a backward writes its parameter gradients into dA_log,
    dbias when they are given."""
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, K]")
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("KDA kernels run on CUDA tensors only")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("q, k, v must be bfloat16 or float32")
    _check_tensor("q", q, q.dtype, dev)
    _check_tensor("k", k, q.dtype, dev, (B, T, H, K))
    _check_tensor("v", v, q.dtype, dev, (B, T, HV, V))
    scalar_gate = g.dim() == 3  # [B, T, HV]: one decay per (token, value head), the GDN variant
    _check_tensor("g", g, torch.float32, dev, (B, T, HV) if scalar_gate else (B, T, HV, K))
    _check_tensor("beta", beta, torch.float32, dev, (B, T, HV))
    if cu_seqlens is not None:
        _check_tensor("cu_seqlens", cu_seqlens, torch.int32, dev)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    if initial_state is not None:
        _check_tensor("initial_state", initial_state, torch.float32, dev, (N, HV, K, V))
    s = _lib.KdaInputs()
    s.B, s.T, s.H, s.HV, s.K, s.V, s.N = B, T, H, HV, K, V, N
    s.dtype = _lib.KDA_BF16 if q.dtype == torch.bfloat16 else _lib.KDA_F32
    s.q, s.k, s.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    s.g, s.beta = g.data_ptr(), beta.data_ptr()
    s.h0 = None if initial_state is None else initial_state.data_ptr()
    s.cu_seqlens = None if cu_seqlens is None else cu_seqlens.data_ptr()
    s.flags = (_lib.KDA_QK_L2NORM if use_qk_l2norm else 0) | (_lib.KDA_SCALAR_GATE if scalar_gate else 0)
    if gate is not None:
        if scalar_gate:
            raise ValueError("the KDA gate takes a per-channel raw gate [B, T, HV, K]")
        if gate.A_log is not None:
            _check_tensor("A_log", gate.A_log, torch.float32, dev, (HV,))
        if gate.bias is not None:
            _check_tensor("gate bias", gate.bias, torch.float32, dev, (HV, K))
        for name, t, shape in (("dA_log", dA_log, (HV,)), ("dbias", dbias, (HV, K))):
            if t is not None:
                _check_tensor(name, t, torch.float32, dev, shape)
        gs = _lib.KdaGate()
        gs.A_log = None if gate.A_log is None else gate.A_log.data_ptr()
        gs.bias = None if gate.bias is None else gate.bias.data_ptr()
        gs.lower_bound = gate.lower_bound
        gs.dA_log = None if dA_log is None else dA_log.data_ptr()
        gs.dbias = None if dbias is None else dbias.data_ptr()
        s.gate = ctypes.pointer(gs)
        s._gate_ref = gs  # keeps the struct alive with s
        s.flags |= _lib.KDA_GATE_IN_KERNEL
    return s


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _workspace(nbytes: int, device) -> torch.Tensor:
    ws = torch.empty(max(nbytes, 256) + 256, dtype=torch.uint8, device=device)
    return ws


def _aligned(ws: torch.Tensor):
    p = ws.data_ptr()
    return ctypes.c_void_p((p + 255) & ~255), ws.numel() - (((p + 255) & ~255) - p)


def _output(v, need_output, output_final_state):
    if not need_output and not output_final_state:
        raise ValueError("need_output=False computes the final state alone: it needs output_final_state=True")
    return torch.empty_like(v) if need_output else None


def chunk_kda_fwd(q, k, v, g, beta, initial_state=None, cu_seqlens=None, output_final_state=False,
                  workspace: Optional[torch.Tensor] = None, use_qk_l2norm: bool = False,
                  need_output: bool = True,
                  gate: Optional[KdaGateParams] = None) -> Tuple[Optional[torch.Tensor], Optional[torch.Tensor]]:
    """Chunked forward (no autograd).  need_output=False: the final state alone
    (o is None), without the output work."""
    lib = _lib.load()
    s = make_inputs_struct(q, k, v, g, beta, initial_state, cu_seqlens, use_qk_l2norm, gate)
    o = _output(v, need_output, output_final_state)
    hT = (torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device=q.device)
          if output_final_state else None)
    need = lib.kda_chunk_fwd_workspace_size(ctypes.byref(s))
    if workspace is None or workspace.numel() < need + 256:
        workspace = _workspace(need, q.device)
    wp, wb = _aligned(workspace)
    _lib.check(lib, lib.kda_chunk_fwd(ctypes.byref(s), _ptr(o), _ptr(hT), wp, wb, _stream(q.device)))
    return o, hT


def chunk_kda_bwd(q, k, v, g, beta, initial_state, cu_seqlens, do, dht,
                  workspace: Optional[torch.Tensor] = None, need_dh0: bool = True,
                  use_qk_l2norm: bool = False, gate: Optional[KdaGateParams] = None):
    """Chunked backward with recompute.  Returns (dq, dk, dv, dg, dbeta, dh0) and,
    with ``gate``, also (dA_log or None, dbias or None)."""
    lib = _lib.load()
    dA, dbias = _gate_grads(gate, v)
    s = make_inputs_struct(q, k, v, g, beta, initial_state, cu_seqlens, use_qk_l2norm, gate, dA, dbias)
    _check_tensor("do", do, q.dtype, q.device, tuple(v.shape))
    if dht is not None:
        _check_tensor("dht", dht, torch.float32, q.device, (s.N, s.HV, s.K, s.V))
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dg = torch.empty_like(g)
    db = torch.empty_like(beta)
    dh0 = (torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device=q.device)
           if need_dh0 else None)
    need = lib.kda_chunk_bwd_workspace_size(ctypes.byref(s))
    if workspace is None or workspace.numel() < need + 256:
        workspace = _workspace(need, q.device)
    wp, wb = _aligned(workspace)
    _lib.check(lib, lib.kda_chunk_bwd(ctypes.byref(s), _ptr(do), _ptr(dht), _ptr(dq), _ptr(dk),
                                      _ptr(dv), _ptr(dg), _ptr(db), _ptr(dh0), wp, wb,
                                      _stream(q.device)))
    return (dq, dk, dv, dg, db, dh0) + (() if gate is None else (dA, dbias))


def _gate_grads(gate, v):
    """Output tensors for the gate's parameter gradients (None for an omitted parameter)."""
    if gate is None:
        return None, None
    dA = None if gate.A_log is None else torch.empty_like(gate.A_log)  # [HV]
    dbias = None if gate.bias is None else torch.empty_like(gate.bias)
    return dA, dbias


def chunk_kda_fwd_ctx(q, k, v, g, beta, initial_state=None, cu_seqlens=None, output_final_state=False,
                      use_qk_l2norm: bool = False, need_output: bool = True, gate: Optional[KdaGateParams] = None):
    """Forward that also returns the forward context (a uint8 device tensor,
    empty on the general path) for :func:`chunk_kda_bwd_ctx`: the per-chunk
    records, chunk-start states and X^T, D^T tiles the backward would otherwise
    recompute.  need_output=False computes the final state alone and keeps the
    records only (a backward then needs :func:`chunk_kda_fwd_reuse` with output
    first).  Returns (o or None, final_state or None, context)."""
    lib = _lib.load()
    s = make_inputs_struct(q, k, v, g, beta, initial_state, cu_seqlens, use_qk_l2norm, gate)
    o = _output(v, need_output, output_final_state)
    hT = (torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device=q.device)
          if output_final_state else None)
    nctx = lib.kda_chunk_ctx_size(ctypes.byref(s))
    kctx = _workspace(nctx, q.device) if nctx else torch.empty(0, dtype=torch.uint8, device=q.device)
    cp, cb = _aligned(kctx) if nctx else (None, 0)
    workspace = _workspace(lib.kda_chunk_fwd_ctx_workspace_size(ctypes.byref(s)), q.device)
    wp, wb = _aligned(workspace)
    _lib.check(lib, lib.kda_chunk_fwd_ctx(ctypes.byref(s), _ptr(o), _ptr(hT), cp, cb, wp, wb,
                                          _stream(q.device)))
    return o, hT, kctx


def chunk_kda_fwd_reuse(q, k, v, g, beta, initial_state, cu_seqlens, kctx, output_final_state=False,
                        use_qk_l2norm: bool = False, need_output: bool = True):
    """:func:`chunk_kda_fwd_ctx` for inputs that share q, k, g, beta and
    cu_seqlens with the ones ``kctx`` was last filled from (v and the initial
    state may differ): the per-chunk records are read from the context, not
    recomputed.  With output, the context is rewritten to serve these inputs'
    backward; need_output=False computes the final state alone and leaves the
    context as it was.  Returns (o or None, final_state or None)."""
    lib = _lib.load()
    s = make_inputs_struct(q, k, v, g, beta, initial_state, cu_seqlens, use_qk_l2norm)
    o = _output(v, need_output, output_final_state)
    hT = (torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device=q.device)
          if output_final_state else None)
    _check_tensor("context", kctx, torch.uint8, q.device)
    cp, cb = _aligned(kctx) if kctx.numel() else (None, 0)
    workspace = _workspace(lib.kda_chunk_fwd_ctx_workspace_size(ctypes.byref(s)), q.device)
    wp, wb = _aligned(workspace)
    _lib.check(lib, lib.kda_chunk_fwd_reuse(ctypes.byref(s), _ptr(o), _ptr(hT), cp, cb, wp, wb, _stream(q.device)))
    return o, hT


def chunk_kda_bwd_ctx(q, k, v, g, beta, initial_state, cu_seqlens, kctx, do, dht, need_dh0: bool = True,
                      use_qk_l2norm: bool = False, gate: Optional[KdaGateParams] = None):
    """Backward on the context :func:`chunk_kda_fwd_ctx` returned for the same
    inputs (it is only read).  Same results as :func:`chunk_kda_bwd`."""
    lib = _lib.load()
    dA, dbias = _gate_grads(gate, v)
    s = make_inputs_struct(q, k, v, g, beta, initial_state, cu_seqlens, use_qk_l2norm, gate, dA, dbias)
    _check_tensor("do", do, q.dtype, q.device, tuple(v.shape))
    if dht is not None:
        _check_tensor("dht", dht, torch.float32, q.device, (s.N, s.HV, s.K, s.V))
    _check_tensor("context", kctx, torch.uint8, q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dg = torch.empty_like(g)
    db = torch.empty_like(beta)
    dh0 = (torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device=q.device)
           if need_dh0 else None)
    cp, cb = _aligned(kctx) if kctx.numel() else (None, 0)
    workspace = _workspace(lib.kda_chunk_bwd_ctx_workspace_size(ctypes.byref(s)), q.device)
    wp, wb = _aligned(workspace)
    _lib.check(lib, lib.kda_chunk_bwd_ctx(ctypes.byref(s), cp, cb, _ptr(do), _ptr(dht), _ptr(dq), _ptr(dk),
                                          _ptr(dv), _ptr(dg), _ptr(db), _ptr(dh0), wp, wb,
                                          _stream(q.device)))
    return (dq, dk, dv, dg, db, dh0) + (() if gate is None else (dA, dbias))


def chunk_kda_bwd_state(q, k, v, g, beta, initial_state, cu_seqlens, do, dht, kctx=None,
                        use_qk_l2norm: bool = False) -> torch.Tensor:
    """Gradient of the initial state alone, dh0 [N, HV, K, V] fp32: the reverse
    state scan without the per-token gradient work (the C ABI's backward with
    dq .. dbeta NULL).  kctx: a forward context of the same inputs
    (:func:`chunk_kda_fwd_ctx`), or None to recompute from the inputs."""
    lib = _lib.load()
    s = make_inputs_struct(q, k, v, g, beta, initial_state, cu_seqlens, use_qk_l2norm)
    _check_tensor("do", do, q.dtype, q.device, tuple(v.shape))
    if dht is not None:
        _check_tensor("dht", dht, torch.float32, q.device, (s.N, s.HV, s.K, s.V))
    dh0 = torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device=q.device)
    sp = _stream(q.device)
    if kctx is not None:
        _check_tensor("context", kctx, torch.uint8, q.device)
        cp, cb = _aligned(kctx) if kctx.numel() else (None, 0)
        workspace = _workspace(lib.kda_chunk_bwd_ctx_workspace_size(ctypes.byref(s)), q.device)
        wp, wb = _aligned(workspace)
        _lib.check(lib, lib.kda_chunk_bwd_ctx(ctypes.byref(s), cp, cb, _ptr(do), _ptr(dht), None, None, None, None,
                                              None, _ptr(dh0), wp, wb, sp))
    else:
        workspace = _workspace(lib.kda_chunk_bwd_workspace_size(ctypes.byref(s)), q.device)
        wp, wb = _aligned(workspace)
        _lib.check(lib, lib.kda_chunk_bwd(ctypes.byref(s), _ptr(do), _ptr(dht), None, None, None, None, None,
                                          _ptr(dh0), wp, wb, sp))
    return dh0


class ChunkKDAFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, initial_state, cu_seqlens, output_final_state, use_qk_l2norm,
                keep_context, use_gate, A_log, g_bias, lower_bound):
        gate = KdaGateParams(A_log, g_bias, lower_bound) if use_gate else None
        if keep_context:
            o, hT, ctx.kctx = chunk_kda_fwd_ctx(q, k, v, g, beta, initial_state, cu_seqlens, output_final_state,
                                                use_qk_l2norm=use_qk_l2norm, gate=gate)
        else:
            o, hT = chunk_kda_fwd(q, k, v, g, beta, initial_state, cu_seqlens, output_final_state,
                                  use_qk_l2norm=use_qk_l2norm, gate=gate)
            ctx.kctx = None
        ctx.save_for_backward(q, k, v, g, beta, initial_state, cu_seqlens, A_log, g_bias)
        ctx.has_h0 = initial_state is not None
        ctx.l2 = use_qk_l2norm
        ctx.use_gate, ctx.lower_bound = use_gate, lower_bound
        return o, hT

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, g, beta, h0, cu, A_log, g_bias = ctx.saved_tensors
        do = do.contiguous()
        dht = None if dht is None else dht.contiguous()
        gate = KdaGateParams(A_log, g_bias, ctx.lower_bound) if ctx.use_gate else None
        if ctx.kctx is not None:
            out = chunk_kda_bwd_ctx(q, k, v, g, beta, h0, cu, ctx.kctx, do, dht, need_dh0=ctx.has_h0,
                                    use_qk_l2norm=ctx.l2, gate=gate)
            ctx.kctx = None  # the context's memory goes back as soon as the backward is enqueued
        else:
            out = chunk_kda_bwd(q, k, v, g, beta, h0, cu, do, dht, need_dh0=ctx.has_h0, use_qk_l2norm=ctx.l2,
                                gate=gate)
        dq, dk, dv, dg, db, dh0 = out[:6]
        dA, dbias = out[6:] if gate is not None else (None, None)
        return dq, dk, dv, dg, db, dh0, None, None, None, None, None, dA, dbias, None


class SegmentedChunkKDAFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, initial_state, output_final_state, use_qk_l2norm, segments):
        from .segments import chunk_kda_fwd_segmented
        o, hT, ctx.seg = chunk_kda_fwd_segmented(q, k, v, g, beta, initial_state, segments, output_final_state,
                                                 use_qk_l2norm=use_qk_l2norm)
        ctx.save_for_backward(q, k, v, g, beta)
        ctx.has_h0 = initial_state is not None
        ctx.l2 = use_qk_l2norm
        return o, hT

    @staticmethod
    def backward(ctx, do, dht):
        from .segments import chunk_kda_bwd_segmented
        q, k, v, g, beta = ctx.saved_tensors
        dht = None if dht is None else dht.contiguous()
        dq, dk, dv, dg, db, dh0 = chunk_kda_bwd_segmented(q, k, v, g, beta, ctx.seg, do.contiguous(), dht,
                                                          need_dh0=ctx.has_h0, use_qk_l2norm=ctx.l2)
        ctx.seg = None
        return dq, dk, dv, dg, db, dh0, None, None, None


def chunk_kda(q, k, v, g, beta, initial_state=None, *, cu_seqlens=None, output_final_state=False,
              use_qk_l2norm=False, keep_context=True, segments=1, use_gate_in_kernel=False, A_log=None,
              g_bias=None, lower_bound=None):
    """Chunked KDA forward (with autograd).  Returns (o, final_state or None).
    use_qk_l2norm: L2-normalise every q and k row inside the op (its backward
    included).  keep_context: the forward keeps its per-chunk intermediates
    (about 2 KB per token and value head on the bf16 K = V = 128 path) so that
    the backward does not recompute them; False trades that memory for the
    recompute.  The gradients are the same either way.  segments > 1 (dense
    batches only): every sequence runs as that many segments at once, joined by
    the state relay -- for a few long sequences, whose chunk chains alone would
    leave most SMs idle (see :mod:`.segments`).  use_gate_in_kernel: ``g`` holds
    the raw gate and the op applies the KDA gate with A_log [HV], g_bias [HV, K]
    and lower_bound (:class:`KdaGateParams`); gradients reach a, A_log and g_bias."""
    if segments > 1:
        if cu_seqlens is not None:
            raise ValueError("segments > 1 splits dense batches only")
        if use_gate_in_kernel:
            raise ValueError("segments > 1 takes the per-token decay (use_gate_in_kernel=False)")
        return SegmentedChunkKDAFunction.apply(q, k, v, g, beta, initial_state, output_final_state, use_qk_l2norm,
                                               segments)
    return ChunkKDAFunction.apply(q, k, v, g, beta, initial_state, cu_seqlens, output_final_state,
                                  use_qk_l2norm, keep_context, use_gate_in_kernel, A_log, g_bias, lower_bound)


def recurrent_kda(q, k, v, gate, beta, initial_state=None, *, cu_seqlens=None,
                  output_final_state=False, use_qk_l2norm=False, use_gate_in_kernel=False, A_log=None,
                  g_bias=None, lower_bound=None):
    """Token-by-token KDA forward for inference (fp32 arithmetic).  Rejects
    inputs that require grad: train through :func:`chunk_kda`."""
    if any(t is not None and t.requires_grad for t in (q, k, v, gate, beta, initial_state, A_log, g_bias)):
        raise RuntimeError("recurrent_kda is inference-only; use chunk_kda for training")
    lib = _lib.load()
    gp = KdaGateParams(A_log, g_bias, lower_bound) if use_gate_in_kernel else None
    s = make_inputs_struct(q, k, v, gate, beta, initial_state, cu_seqlens, use_qk_l2norm, gp)
    o = torch.empty_like(v)
    hT = (torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device=q.device)
          if output_final_state else None)
    _lib.check(lib, lib.kda_recurrent_fwd(ctypes.byref(s), _ptr(o), _ptr(hT), _stream(q.device)))
    return o, hT
