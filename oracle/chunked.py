"""Chunk-wise (WY/UT) fp64 formulation of KDA -- TEST INFRASTRUCTURE.

An independent restatement of the token recurrence in :mod:`oracle` as the
chunked algorithm the FLA KDA/GDN pipeline is built from (chunk-local gate
cumsum, scaled-dot KK^T block, unit-lower-triangular solve, w/u recompute,
inter-chunk state scan ``fwd_h``, output ``fwd_o``; and for the backward the
reverse state-gradient scan ``bwd_dhu`` plus the intra-chunk gradients) -- the
sub-kernel list in the commit log of "[Fix] Use unit KDA gate scale when
A_log is omitted" (fla-org/flash-linear-attention PR #1294, the GDN
per-kernel-baselines commit).  In exact arithmetic it equals the token loop.

Everything is plain numpy fp64.  Pairwise decays 2^(G_r - G_i) are formed
directly (fp64 has the range), so there is no blocking or reference-point
trick here.

Per chunk (rows r, i of C_c <= C tokens; G = inclusive cumsum of g in the
chunk; q~ = q / sqrt(K)):
  L   = strictly-lower [beta_r sum_c k_rc k_ic 2^(G_rc - G_ic)]
  Aqk = lower          [sum_c q~_rc k_ic 2^(G_rc - G_ic)]
  A   = (I + L)^-1 ;  w = A (beta k 2^G) ;  u = A (beta v)
  D   = u - w h                  (h = state at chunk start; D = the deltas)
  O   = (q~ 2^G) h + Aqk D
  h'  = diag(2^G_last) h + (k 2^(G_last - G))^T D
"""
from __future__ import annotations

import math

import numpy as np

LN2 = math.log(2.0)


def _offsets(B, T, cu):
    if cu is None:
        return np.arange(B + 1, dtype=np.int64) * T
    return np.asarray(cu, dtype=np.int64)


def _chunk_forward(q, k, v, g, beta, h):
    """One chunk.  q,k,g [C,K]; v [C,V]; beta [C]; h [K,V].  Returns a dict of
    every intermediate and the next state."""
    C, K = k.shape
    qs = q / math.sqrt(K)
    G = np.cumsum(g, axis=0)
    D = np.exp2(G[:, None, :] - G[None, :, :])            # [r, i, c]
    kk = np.einsum("rc,ic,ric->ri", k, k, D)
    qk = np.einsum("rc,ic,ric->ri", qs, k, D)
    strict = np.tril(np.ones((C, C)), -1)
    lower = np.tril(np.ones((C, C)), 0)
    L = beta[:, None] * kk * strict
    Aqk = qk * lower
    A = np.linalg.inv(np.eye(C) + L)
    Gam = np.exp2(G)
    Bk = beta[:, None] * k * Gam
    Bv = beta[:, None] * v
    w = A @ Bk
    u = A @ Bv
    Dl = u - w @ h
    Qg = qs * Gam
    Khat = k * np.exp2(G[-1][None, :] - G)
    Glast = np.exp2(G[-1])
    O = Qg @ h + Aqk @ Dl
    h_next = Glast[:, None] * h + Khat.T @ Dl
    return dict(G=G, D=D, kk=kk, L=L, Aqk=Aqk, A=A, Gam=Gam, Bk=Bk, Bv=Bv, w=w, u=u,
                delta=Dl, Qg=Qg, Khat=Khat, Glast=Glast, O=O, h=h, h_next=h_next,
                strict=strict, lower=lower, qs=qs)


def _chunk_backward(f, q, k, v, beta, dO, dh_end):
    """Backward of one chunk given its forward dict ``f``, the output
    gradient dO [C,V] and the gradient of the chunk-end state dh_end [K,V].
    Returns (grads dict for the chunk's tokens, gradient of the chunk-start
    state, d_delta)."""
    C, K = k.shape
    h, A, Aqk, w = f["h"], f["A"], f["Aqk"], f["w"]
    Dl, Qg, Khat, Gam, Glast, D = f["delta"], f["Qg"], f["Khat"], f["Gam"], f["Glast"], f["D"]
    qs = f["qs"]
    # reverse state-gradient scan step
    dDl = Aqk.T @ dO + Khat @ dh_end
    dh_start = Glast[:, None] * dh_end + Qg.T @ dO - w.T @ dDl
    # output / state terms
    dQg = dO @ h.T
    dAqk = (dO @ Dl.T) * f["lower"]
    dKhat = Dl @ dh_end.T
    dGlast_vec = np.sum(dh_end * h, axis=1)
    dqs = dQg * Gam
    dG = LN2 * dQg * Qg
    dk = dKhat * np.exp2(f["G"][-1][None, :] - f["G"])
    dG -= LN2 * dKhat * Khat
    dG_last = LN2 * np.sum(dKhat * Khat, axis=0) + LN2 * Glast * dGlast_vec
    # WY part: w = A Bk, u = A Bv, D = u - w h
    du = dDl
    dw = -dDl @ h.T
    dA = du @ f["Bv"].T + dw @ f["Bk"].T
    dBv = A.T @ du
    dBk = A.T @ dw
    dL = -(A.T @ dA @ A.T) * f["strict"]
    dv = beta[:, None] * dBv
    dbeta = np.sum(dBv * v, axis=1)
    Kd = k * Gam
    dk += beta[:, None] * Gam * dBk
    dbeta += np.sum(dBk * Kd, axis=1)
    dG += LN2 * beta[:, None] * dBk * Kd
    # L = beta * kk (strict lower)
    dbeta += np.sum(dL * f["kk"], axis=1)
    dLb = beta[:, None] * dL
    # kk_ri = sum_c k_rc k_ic D_ric ;  Aqk_ri = sum_c qs_rc k_ic D_ric
    Xr = np.einsum("ri,ic,ric->rc", dLb, k, D)        # row-side sums
    Xi = np.einsum("ri,rc,ric->ic", dLb, k, D)        # column-side sums
    dk += Xr + Xi
    dG += LN2 * (k * Xr - k * Xi)
    Yr = np.einsum("ri,ic,ric->rc", dAqk, k, D)
    Yi = np.einsum("ri,rc,ric->ic", dAqk, qs, D)
    dqs += Yr
    dk += Yi
    dG += LN2 * (qs * Yr - k * Yi)
    dG[-1] += dG_last
    dg = np.flip(np.cumsum(np.flip(dG, 0), axis=0), 0)
    dq = dqs / math.sqrt(K)
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dG=dG), dh_start, dDl


def kda_chunked_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, chunk=64, keep=False):
    """Chunked forward.  Same layout and results as :func:`oracle.kda_fwd`
    (hT always returned).  With ``keep`` also returns the per-chunk dicts
    keyed by (n, j, chunk index)."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    r = HV // H
    off = _offsets(B, T, cu_seqlens)
    N = len(off) - 1
    qf, kf = q.reshape(B * T, H, K), k.reshape(B * T, H, K)
    vf, gf, bf = v.reshape(B * T, HV, V), g.reshape(B * T, HV, K), beta.reshape(B * T, HV)
    o = np.zeros((B * T, HV, V))
    hT = np.zeros((N, HV, K, V))
    store = {}
    for n in range(N):
        for j in range(HV):
            hh = j // r
            S = np.zeros((K, V)) if h0 is None else np.array(h0[n, j], dtype=np.float64)
            for ci, t0 in enumerate(range(off[n], off[n + 1], chunk)):
                t1 = min(t0 + chunk, off[n + 1])
                f = _chunk_forward(qf[t0:t1, hh], kf[t0:t1, hh], vf[t0:t1, j], gf[t0:t1, j],
                                   bf[t0:t1, j], S)
                o[t0:t1, j] = f["O"]
                if keep:
                    store[(n, j, ci)] = f
                S = f["h_next"]
            hT[n, j] = S
    o = o.reshape(B, T, HV, V)
    return (o, hT, store) if keep else (o, hT)


def kda_chunked_bwd(q, k, v, g, beta, h0, do, dhT, cu_seqlens=None, chunk=64):
    """Chunked backward (state recompute, reverse dh scan, intra-chunk
    gradients).  Returns the same dict as :func:`oracle.kda_bwd`."""
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    r = HV // H
    off = _offsets(B, T, cu_seqlens)
    N = len(off) - 1
    _, _, store = kda_chunked_fwd(q, k, v, g, beta, h0, cu_seqlens, chunk, keep=True)
    vf, bf = v.reshape(B * T, HV, V), beta.reshape(B * T, HV)
    qf, kf = q.reshape(B * T, H, K), k.reshape(B * T, H, K)
    dof = do.reshape(B * T, HV, V)
    out = dict(dq=np.zeros((B * T, H, K)), dk=np.zeros((B * T, H, K)), dv=np.zeros((B * T, HV, V)),
               dg=np.zeros((B * T, HV, K)), dbeta=np.zeros((B * T, HV)),
               dh0=np.zeros((N, HV, K, V)))
    for n in range(N):
        for j in range(HV):
            hh = j // r
            dS = np.zeros((K, V)) if dhT is None else np.array(dhT[n, j], dtype=np.float64)
            starts = list(range(off[n], off[n + 1], chunk))
            for ci in reversed(range(len(starts))):
                t0 = starts[ci]
                t1 = min(t0 + chunk, off[n + 1])
                f = store[(n, j, ci)]
                gr, dS, _ = _chunk_backward(f, qf[t0:t1, hh], kf[t0:t1, hh], vf[t0:t1, j],
                                            bf[t0:t1, j], dof[t0:t1, j], dS)
                out["dq"][t0:t1, hh] += gr["dq"]
                out["dk"][t0:t1, hh] += gr["dk"]
                out["dv"][t0:t1, j] = gr["dv"]
                out["dg"][t0:t1, j] = gr["dg"]
                out["dbeta"][t0:t1, j] = gr["dbeta"]
            out["dh0"][n, j] = dS
    for key, shp in (("dq", (B, T, H, K)), ("dk", (B, T, H, K)), ("dv", (B, T, HV, V)),
                     ("dg", (B, T, HV, K)), ("dbeta", (B, T, HV))):
        out[key] = out[key].reshape(shp)
    return out
