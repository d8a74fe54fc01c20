"""fp64 CPU oracle for KDA (Kimi Delta Attention) -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / reference leg may import this package.  It shares no code
with the CUDA path (no kernels, headers, helpers or constants), and the CUDA
path never imports it.

Two independent formulations of the same result:

* :func:`kda_fwd` / :func:`kda_bwd` -- the plain token-by-token recurrence and
  its hand-derived backward, in C (``kda_oracle.c``), threaded over
  (sequence, value head).  This is *the* oracle.
* :mod:`oracle.chunked` -- the chunk-wise WY/UT form (chunk-local gate
  cumsum, decayed beta*K*K^T block, (I+L)^-1, w/u, inter-chunk state scan,
  output, and the reverse state-gradient scan with the intra-chunk backward),
  written in numpy fp64 with the pairwise decays formed directly.  It is used to
  pin the token loop and to give per-chunk intermediates.

Array layout (numpy float64): q,k [B,T,H,K]; v,dO [B,T,HV,V]; g [B,T,HV,K];
beta [B,T,HV]; h0,dhT [N,HV,K,V].  ``cu_seqlens`` (int [N+1]) requires B == 1.
Parity unpinned by the pages: they print no worked example, so every pin is
mathematical (closed forms, invariants, finite differences, brute force,
autograd of a naive loop); see ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libkda_oracle.so")
_SRC = os.path.join(_HERE, "kda_oracle.c")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            i64, i32 = ctypes.c_int64, ctypes.c_int
            lib.kda_oracle_fwd.argtypes = [i64, i32, i32, i32, i32, i32, ip] + [dp] * 8 + [i32]
            lib.kda_oracle_fwd.restype = i32
            lib.kda_oracle_bwd.argtypes = [i64, i32, i32, i32, i32, i32, ip] + [dp] * 16 + [i32]
            lib.kda_oracle_bwd.restype = i32
            _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _c64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _offsets(B, T, cu_seqlens):
    if cu_seqlens is None:
        return np.ascontiguousarray(np.arange(B + 1, dtype=np.int32) * T)
    assert B == 1, "packed batches use B == 1"
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))


# The q/k L2-norm prologue.  The KDA layer of "kda in torchtitan (training)"
# (pytorch/torchtitan PR #4164) imports an attention-gym `l2norm` next to
# `recurrent_kda`; the pages print neither its formula nor its epsilon.  Reading:
# each (token, head) row of q and of k is divided by sqrt(sum of its squares +
# eps) over the head dimension, with eps = 1e-6, before the 1/sqrt(K) query
# scale; gradients are taken w.r.t. the raw rows.
L2NORM_EPS = 1e-6


def l2norm_rows(x, eps=L2NORM_EPS):
    """y = x / sqrt(sum_c x_c^2 + eps) over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def l2norm_rows_bwd(x, dy, eps=L2NORM_EPS):
    """Gradient of :func:`l2norm_rows` w.r.t. x given dy: with r = (sum x^2 +
    eps)^(-1/2) and y = x r, dx = r (dy - y (y . dy))."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    y = x * r
    return r * (dy - y * np.sum(y * dy, axis=-1, keepdims=True))


# The scalar-gate (GDN) variant: one log2 decay per (token, value head), shared
# by every key channel -- the gated delta rule that the GDN pipeline of
# "[Fix] Use unit KDA gate scale when A_log is omitted" (fla-org/flash-linear-
# attention PR #1294) and the triton-ascend GDN port of its commit log (PR #1011)
# run, of which KDA is the per-channel generalisation.  g is [B,T,HV]; the
# recurrence is KDA's with that gate repeated over K, and dg sums the
# per-channel gradients over K.
def gate_per_channel(g, K):
    """[B,T,HV] scalar gates -> [B,T,HV,K] (the same decay on every channel)."""
    g = np.asarray(g, dtype=np.float64)
    return np.ascontiguousarray(np.repeat(g[..., None], K, axis=-1))


def gate_grad_reduce(dg):
    """[B,T,HV,K] per-channel gate gradients -> [B,T,HV] (sum over K)."""
    return np.sum(np.asarray(dg, dtype=np.float64), axis=-1)


# The KDA gate inside the op ("[Fix] Use unit KDA gate scale when A_log is
# omitted", fla-org/flash-linear-attention PR #1294, Summary and Breaking
# changes; its commit log's "[Fix] Reduce GDN/KDA gate bias gradients before
# downcasting").  The pages name the pieces -- a decay scale exp(A_log) per
# value head, unit when A_log is omitted (the same as an explicit zero A_log;
# an explicit ones tensor reproduces the former exp(1) scale), a gate bias
# whose gradient is reduced over tokens in fp32, bounded and unbounded gate
# formulas -- but print no formula.  Reading: with x = a + bias (the raw
# pre-activation plus a per (value head, channel) bias) and s = exp(A_log),
#   unbounded: g = -s softplus(x)            (g <= 0)
#   bounded:   g = lower_bound sigmoid(s x)  (lower_bound < g < 0)
# and g is the per-token log2 decay the recurrence takes ("kda in torchtitan
# (training)" calls the output of its bounded gate the per-token log2 decay).
def _softplus(x):
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def _sigmoid(x):
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def _gate_parts(a, A_log, bias, HV):
    a = np.asarray(a, dtype=np.float64)
    s = np.ones(HV) if A_log is None else np.exp(np.asarray(A_log, dtype=np.float64))
    x = a if bias is None else a + np.asarray(bias, dtype=np.float64)  # bias [HV, K] broadcasts over tokens
    return x, s[:, None]


def kda_gate(a, A_log=None, bias=None, lower_bound=None):
    """Raw gate pre-activations a [B,T,HV,K] -> per-token log2 decay g."""
    x, s = _gate_parts(a, A_log, bias, np.shape(a)[2])
    if lower_bound is None:
        return -s * _softplus(x)
    return lower_bound * _sigmoid(s * x)


def kda_gate_bwd(a, dg, A_log=None, bias=None, lower_bound=None):
    """Gradients of the gate given dg = dL/dg: (da [B,T,HV,K], dA_log [HV],
    dbias [HV,K]); the parameter gradients are sums over every token."""
    x, s = _gate_parts(a, A_log, bias, np.shape(a)[2])
    dg = np.asarray(dg, dtype=np.float64)
    if lower_bound is None:
        dx = -s * _sigmoid(x)          # d/dx of -s softplus(x)
        ds = -s * _softplus(x)         # d/dA_log of -exp(A_log) softplus(x)
    else:
        sg = _sigmoid(s * x)
        dx = lower_bound * sg * (1.0 - sg) * s
        ds = lower_bound * sg * (1.0 - sg) * s * x
    da = dg * dx
    return da, np.sum(dg * ds, axis=(0, 1, 3)), np.sum(da, axis=(0, 1))


def kda_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, output_final_state=True, nthreads=0,
            qk_l2norm=False, scalar_gate=False, gate=None):
    """Token-by-token KDA forward.  Returns (o [B,T,HV,V], hT [N,HV,K,V] or None).
    With qk_l2norm, q and k rows are normalised first (:func:`l2norm_rows`);
    with scalar_gate, g is [B,T,HV] (:func:`gate_per_channel`); with gate (a
    dict of :func:`kda_gate`'s A_log, bias, lower_bound), g holds the raw
    pre-activations and the gate makes the decay first."""
    if gate is not None:
        g = kda_gate(g, **gate)
    if qk_l2norm:
        q, k = l2norm_rows(q), l2norm_rows(k)
    if scalar_gate:
        g = gate_per_channel(g, np.shape(q)[-1])
    lib = _load()
    q, k, v, g, beta, h0 = map(_c64, (q, k, v, g, beta, h0))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    cu = _offsets(B, T, cu_seqlens)
    N = len(cu) - 1
    o = np.zeros((B, T, HV, V))
    hT = np.zeros((N, HV, K, V)) if output_final_state else None
    st = lib.kda_oracle_fwd(B * T, N, H, HV, K, V, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                            _p(q), _p(k), _p(v), _p(g), _p(beta), _p(h0), _p(o), _p(hT), nthreads)
    if st != 0:
        raise RuntimeError(f"kda_oracle_fwd failed ({st})")
    return o, hT


def kda_bwd(q, k, v, g, beta, h0, do, dhT, cu_seqlens=None, nthreads=0, qk_l2norm=False,
            scalar_gate=False, gate=None):
    """Token-by-token KDA backward.  Returns dict dq, dk, dv, dg, dbeta, dh0.
    With qk_l2norm, the gradients of the normalised rows are carried back
    through :func:`l2norm_rows` to the raw q and k; with scalar_gate, g and dg
    are [B,T,HV] (:func:`gate_grad_reduce`); with gate, dg is the gradient of
    the raw pre-activations, and dA_log, dbias are added (:func:`kda_gate_bwd`)."""
    if gate is not None:
        out = kda_bwd(q, k, v, kda_gate(g, **gate), beta, h0, do, dhT, cu_seqlens, nthreads, qk_l2norm,
                      scalar_gate)
        out["dg"], out["dA_log"], out["dbias"] = kda_gate_bwd(g, out["dg"], **gate)
        return out
    if scalar_gate:
        out = kda_bwd(q, k, v, gate_per_channel(g, np.shape(q)[-1]), beta, h0, do, dhT, cu_seqlens, nthreads,
                      qk_l2norm)
        out["dg"] = gate_grad_reduce(out["dg"])
        return out
    if qk_l2norm:
        out = kda_bwd(l2norm_rows(q), l2norm_rows(k), v, g, beta, h0, do, dhT, cu_seqlens, nthreads)
        out["dq"] = l2norm_rows_bwd(q, out["dq"])
        out["dk"] = l2norm_rows_bwd(k, out["dk"])
        return out
    lib = _load()
    q, k, v, g, beta, h0, do, dhT = map(_c64, (q, k, v, g, beta, h0, do, dhT))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    cu = _offsets(B, T, cu_seqlens)
    N = len(cu) - 1
    out = dict(dq=np.zeros((B, T, H, K)), dk=np.zeros((B, T, H, K)), dv=np.zeros((B, T, HV, V)),
               dg=np.zeros((B, T, HV, K)), dbeta=np.zeros((B, T, HV)), dh0=np.zeros((N, HV, K, V)))
    dqp = np.zeros((B * T, HV, K))
    dkp = np.zeros((B * T, HV, K))
    st = lib.kda_oracle_bwd(B * T, N, H, HV, K, V, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                            _p(q), _p(k), _p(v), _p(g), _p(beta), _p(h0), _p(do), _p(dhT),
                            _p(out["dq"]), _p(out["dk"]), _p(out["dv"]), _p(out["dg"]),
                            _p(out["dbeta"]), _p(out["dh0"]), _p(dqp), _p(dkp), nthreads)
    if st != 0:
        raise RuntimeError(f"kda_oracle_bwd failed ({st})")
    return out


def rel_rms(x, ref) -> float:
    """Relative RMS error ||x - ref||_2 / ||ref||_2 (the relative-RMS check style
    of FLA's KDA tests).  A zero reference requires x == 0 exactly."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.sqrt(np.sum(ref * ref)))
    num = float(np.sqrt(np.sum((x - ref) ** 2)))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den
