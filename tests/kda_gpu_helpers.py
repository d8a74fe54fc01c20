"""Helpers for the GPU parity tests: call libkda through its C ABI with
NaN-poisoned outputs and workspace, run the oracle on the same inputs (whole
problem, or sampled (sequence, q/k head) units of a large one), compare."""
from __future__ import annotations

import ctypes

import numpy as np
import torch

import oracle
from gated_delta_rule_42_gb300 import _lib
from gated_delta_rule_42_gb300.ops import make_inputs_struct

# tolerances (relative RMS): fp32 inputs 1e-5 everywhere; bf16 inputs 5e-3 on
# o / final state, 1e-2 on every gradient
TOL = {torch.float32: dict(fwd=1e-5, bwd=1e-5), torch.bfloat16: dict(fwd=5e-3, bwd=1e-2)}


def _nan_like(shape, dtype, dev):
    return torch.full(shape, float("nan"), dtype=dtype, device=dev)


def _poisoned_ws(nbytes, dev):
    ws = torch.full((nbytes + 512,), 255, dtype=torch.uint8, device=dev)
    p = ws.data_ptr()
    a = (p + 255) & ~255
    return ws, ctypes.c_void_p(a), nbytes + 512 - (a - p)


def status_words(lib, s, ws, wp):
    """The seven int32 status words a call left in its workspace (after a sync)."""
    off = lib.kda_status_offset(ctypes.byref(s))
    base = wp.value - ws.data_ptr() + off
    return ws[base:base + 28].cpu().numpy().view(np.int32).tolist()


def gate_params(d):
    """The KDA gate's parameters of inputs ``d`` (on the device), or None."""
    from gated_delta_rule_42_gb300.ops import KdaGateParams
    return KdaGateParams(d.A_log, d.g_bias, d.lower_bound) if d.meta.get("raw_gate") else None


def gpu_fwd(inp, dev="cuda", lib=None, l2=False, status=None):
    """kda_chunk_fwd on the inputs (moved to dev); returns CPU o, hT.  l2: the
    q/k L2-norm prologue flag.  A ``status`` list receives the call's status words."""
    lib = lib or _lib.load()
    d = inp.to(dev)
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, l2, gate_params(d))
    o = _nan_like(d.v.shape, d.dtype, dev)
    hT = _nan_like((s.N, s.HV, s.K, s.V), torch.float32, dev) if inp.output_final_state else None
    need = lib.kda_chunk_fwd_workspace_size(ctypes.byref(s))
    ws, wp, wb = _poisoned_ws(need, dev)
    st = lib.kda_chunk_fwd(ctypes.byref(s), ctypes.c_void_p(o.data_ptr()),
                           None if hT is None else ctypes.c_void_p(hT.data_ptr()), wp, wb,
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _lib.check(lib, st)
    torch.cuda.synchronize()
    if status is not None:
        status[:] = status_words(lib, s, ws, wp)
    return o.cpu(), (None if hT is None else hT.cpu())


def gpu_bwd(inp, dev="cuda", lib=None, want_dh0=True, l2=False, status=None):
    """kda_chunk_bwd; with the KDA gate the dict also holds dA_log and dbias."""
    lib = lib or _lib.load()
    d = inp.to(dev)
    gp = gate_params(d)
    dA = None if gp is None or d.A_log is None else _nan_like(d.A_log.shape, torch.float32, dev)
    dbias = None if gp is None or d.g_bias is None else _nan_like(d.g_bias.shape, torch.float32, dev)
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, l2, gp, dA, dbias)
    out = dict(dq=_nan_like(d.q.shape, d.dtype, dev), dk=_nan_like(d.k.shape, d.dtype, dev),
               dv=_nan_like(d.v.shape, d.dtype, dev), dg=_nan_like(d.g.shape, torch.float32, dev),
               dbeta=_nan_like(d.beta.shape, torch.float32, dev))
    if gp is not None:
        out["dA_log"], out["dbias"] = dA, dbias
    out["dh0"] = _nan_like((s.N, s.HV, s.K, s.V), torch.float32, dev) if want_dh0 else None
    need = lib.kda_chunk_bwd_workspace_size(ctypes.byref(s))
    ws, wp, wb = _poisoned_ws(need, dev)

    def p(t):
        return None if t is None else ctypes.c_void_p(t.data_ptr())

    st = lib.kda_chunk_bwd(ctypes.byref(s), p(d.do), p(d.dhT), p(out["dq"]), p(out["dk"]),
                           p(out["dv"]), p(out["dg"]), p(out["dbeta"]), p(out["dh0"]), wp, wb,
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _lib.check(lib, st)
    torch.cuda.synchronize()
    if status is not None:
        status[:] = status_words(lib, s, ws, wp)
    return {k: (None if v is None else v.cpu()) for k, v in out.items()}


def gpu_recurrent(inp, dev="cuda", lib=None, l2=False):
    lib = lib or _lib.load()
    d = inp.to(dev)
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, l2, gate_params(d))
    o = _nan_like(d.v.shape, d.dtype, dev)
    hT = _nan_like((s.N, s.HV, s.K, s.V), torch.float32, dev) if inp.output_final_state else None
    st = lib.kda_recurrent_fwd(ctypes.byref(s), ctypes.c_void_p(o.data_ptr()),
                               None if hT is None else ctypes.c_void_p(hT.data_ptr()),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _lib.check(lib, st)
    torch.cuda.synchronize()
    return o.cpu(), (None if hT is None else hT.cpu())


def oracle_fwd(inp, l2=False):
    f = inp.f64()
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
    return oracle.kda_fwd(f["q"], f["k"], f["v"], f["g"], f["beta"], f["h0"], cu, True, qk_l2norm=l2,
                          scalar_gate=f["g"].ndim == 3, gate=inp.gate)


def oracle_bwd(inp, l2=False):
    f = inp.f64()
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
    return oracle.kda_bwd(f["q"], f["k"], f["v"], f["g"], f["beta"], f["h0"], f["do"], f["dhT"], cu,
                          qk_l2norm=l2, scalar_gate=f["g"].ndim == 3, gate=inp.gate)


def valid_mask(inp):
    """Boolean [B*T] of tokens inside the contract."""
    m = np.zeros(inp.B * inp.T, dtype=bool)
    off = inp.offsets()
    for n in range(len(off) - 1):
        m[off[n]:off[n + 1]] = True
    return m


def tok(x, inp):
    """[B,T,...] -> [B*T,...] as fp64 numpy."""
    x = x.detach().cpu()
    if x.dtype != torch.float64:
        x = x.to(torch.float64)
    return x.numpy().reshape(inp.B * inp.T, *x.shape[2:])


def assert_rel(name, got, ref, tol):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values (unwritten or overflow)"
    err = oracle.rel_rms(got, ref)
    assert err <= tol, f"{name}: rel-RMS {err:.3e} > {tol:.1e}"
    return err


def check_fwd(inp, o, hT, ref_o, ref_hT, tol):
    m = valid_mask(inp)
    errs = {"o": assert_rel("o", tok(o, inp)[m], ref_o.reshape(inp.B * inp.T, -1, inp.V)[m], tol)}
    if (~m).any():  # outside the contract: never written
        assert torch.isnan(o.reshape(inp.B * inp.T, -1)[torch.from_numpy(~m)]).all(), "tail written"
    if hT is not None:
        errs["hT"] = assert_rel("hT", hT.numpy(), ref_hT, tol)
        for n in empty_slots(inp):
            want = inp.h0[n] if inp.h0 is not None else torch.zeros_like(hT[n])
            assert torch.equal(hT[n], want), f"empty slot {n} state not passed through bitwise"
    return errs


def check_bwd(inp, gr, ref, tol):
    m = valid_mask(inp)
    errs = {}
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        g = tok(gr[key], inp)
        errs[key] = assert_rel(key, g[m], ref[key].reshape(g.shape)[m], tol)
        if (~m).any():
            assert torch.isnan(gr[key].reshape(inp.B * inp.T, -1)[torch.from_numpy(~m)]).all(), \
                f"{key}: tail written"
    for key in ("dA_log", "dbias"):  # the KDA gate's parameter gradients
        if gr.get(key) is not None:
            errs[key] = assert_rel(key, gr[key].numpy(), ref[key], tol)
    if gr.get("dh0") is not None:
        errs["dh0"] = assert_rel("dh0", gr["dh0"].numpy(), ref["dh0"], tol)
        for n in empty_slots(inp):
            want = inp.dhT[n] if inp.dhT is not None else torch.zeros_like(gr["dh0"][n])
            assert torch.equal(gr["dh0"][n], want), f"empty slot {n} dh0 not passed through bitwise"
    return errs


def empty_slots(inp):
    off = inp.offsets()
    return [n for n in range(len(off) - 1) if off[n] == off[n + 1]]


def sample_units(inp, units):
    """Oracle on sampled (sequence n, q/k head hq) units of a large problem
    (all HV/H value heads of the group, so dq and dk are complete).
    Returns a list of (n, hq, js, t0, t1, (o, hT), bwd dict)."""
    B, T, H, HV = inp.B, inp.T, inp.H, inp.HV
    r = HV // H
    off = inp.offsets()

    def sl(x, t0, t1, cols):
        if x is None:
            return None
        y = x.reshape(B * T, *x.shape[2:])[t0:t1][:, cols]
        return y.to(torch.float64).numpy()[None]

    out = []
    for n, hq in units:
        t0, t1 = int(off[n]), int(off[n + 1])
        js = list(range(hq * r, (hq + 1) * r))
        q, k = sl(inp.q, t0, t1, [hq]), sl(inp.k, t0, t1, [hq])
        v, g, beta, do = (sl(x, t0, t1, js) for x in (inp.v, inp.g, inp.beta, inp.do))
        h0 = None if inp.h0 is None else inp.h0[n:n + 1][:, js].to(torch.float64).numpy()
        dhT = None if inp.dhT is None else inp.dhT[n:n + 1][:, js].to(torch.float64).numpy()
        o, hT = oracle.kda_fwd(q, k, v, g, beta, h0, None, True)
        gr = oracle.kda_bwd(q, k, v, g, beta, h0, do, dhT)
        out.append((n, hq, js, t0, t1, (o, hT), gr))
    return out


def gpu_fwd_bwd_ctx(inp, dev="cuda", lib=None, want_dh0=True, l2=False, backwards=1):
    """kda_chunk_fwd_ctx, then kda_chunk_bwd_ctx ``backwards`` times on the
    context it kept (NaN-poisoned outputs, 0xFF-poisoned context and
    workspaces).  Returns the DEVICE results: o, hT and a list of gradient
    dicts, one per backward call."""
    lib = lib or _lib.load()
    d = inp.to(dev)
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, l2)
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def p(t):
        return None if t is None else ctypes.c_void_p(t.data_ptr())

    o = _nan_like(d.v.shape, d.dtype, dev)
    hT = _nan_like((s.N, s.HV, s.K, s.V), torch.float32, dev) if inp.output_final_state else None
    nctx = lib.kda_chunk_ctx_size(ctypes.byref(s))
    cbuf, cp, cb = _poisoned_ws(nctx, dev) if nctx else (None, None, 0)
    ws, wp, wb = _poisoned_ws(lib.kda_chunk_fwd_ctx_workspace_size(ctypes.byref(s)), dev)
    _lib.check(lib, lib.kda_chunk_fwd_ctx(ctypes.byref(s), p(o), p(hT), cp, cb, wp, wb, sp))
    grads = []
    for _ in range(backwards):
        out = dict(dq=_nan_like(d.q.shape, d.dtype, dev), dk=_nan_like(d.k.shape, d.dtype, dev),
                   dv=_nan_like(d.v.shape, d.dtype, dev), dg=_nan_like(d.g.shape, torch.float32, dev),
                   dbeta=_nan_like(d.beta.shape, torch.float32, dev))
        out["dh0"] = _nan_like((s.N, s.HV, s.K, s.V), torch.float32, dev) if want_dh0 else None
        ws, wp, wb = _poisoned_ws(lib.kda_chunk_bwd_ctx_workspace_size(ctypes.byref(s)), dev)
        _lib.check(lib, lib.kda_chunk_bwd_ctx(ctypes.byref(s), cp, cb, p(d.do), p(d.dhT), p(out["dq"]),
                                              p(out["dk"]), p(out["dv"]), p(out["dg"]), p(out["dbeta"]),
                                              p(out["dh0"]), wp, wb, sp))
        grads.append(out)
    torch.cuda.synchronize()
    return o, hT, grads, nctx
