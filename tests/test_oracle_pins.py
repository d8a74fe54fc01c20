"""Pins for the fp64 oracle: checks against facts fixed by the mathematics,
not by the oracle itself (closed forms, invariants, finite differences,
library autograd of a naive loop, an independent chunked formulation, and a
hand-derived worked example).  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_problem(rng, B=1, T=7, H=1, HV=1, K=3, V=2, h0=True, gscale=1.0):
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, HV, V))
    g = -gscale * np.log1p(np.exp(rng.standard_normal((B, T, HV, K))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, HV))))
    return q, k, v, g, beta


def test_handcalc_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "kda_handcalc_T3_K2_V1.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                name, *xs = line.split()
                vals[name] = np.array([float(x) for x in xs])
    K, V = int(vals["K"][0]), int(vals["V"][0])
    T = 3
    q = vals["q"].reshape(1, T, 1, K)
    k = vals["k"].reshape(1, T, 1, K)
    v = vals["v"].reshape(1, T, 1, V)
    g = vals["g"].reshape(1, T, 1, K)
    beta = vals["beta"].reshape(1, T, 1)
    h0 = vals["h0"].reshape(1, 1, K, V)
    o, hT = oracle.kda_fwd(q, k, v, g, beta, h0)
    np.testing.assert_allclose(o.reshape(-1) * math.sqrt(K), vals["o_times_sqrtK"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(hT.reshape(-1), vals["hT"], rtol=0, atol=1e-13)


def test_no_gate_no_beta_state_unchanged_and_closed_form_grads():
    """g = 0, beta = 0: S never changes, o_t = h0^T q_t / sqrt(K); the
    gradients have closed forms."""
    rng = np.random.default_rng(1)
    B, T, H, HV, K, V = 1, 9, 1, 1, 4, 3
    q, k, v, _, _ = rand_problem(rng, B, T, H, HV, K, V)
    g = np.zeros((B, T, HV, K))
    beta = np.zeros((B, T, HV))
    h0 = rng.standard_normal((1, HV, K, V))
    do = rng.standard_normal((B, T, HV, V))
    dhT = rng.standard_normal((1, HV, K, V))
    o, hT = oracle.kda_fwd(q, k, v, g, beta, h0)
    assert np.array_equal(hT, h0)
    qs = q[0, :, 0] / math.sqrt(K)
    np.testing.assert_allclose(o[0, :, 0], qs @ h0[0, 0], rtol=1e-14, atol=1e-14)
    gr = oracle.kda_bwd(q, k, v, g, beta, h0, do, dhT)
    assert np.all(gr["dv"] == 0)
    np.testing.assert_allclose(gr["dq"][0, :, 0], do[0, :, 0] @ h0[0, 0].T / math.sqrt(K), atol=1e-13)
    np.testing.assert_allclose(gr["dh0"][0, 0], dhT[0, 0] + qs.T @ do[0, :, 0], atol=1e-13)
    # dbeta_t = (v_t - h0^T k_t) . (dS_t^T k_t), dS_t = dhT + sum_{s>=t} q~_s dO_s^T
    for t in range(T):
        dS = dhT[0, 0] + qs[t:].T @ do[0, t:, 0]
        kt = k[0, t, 0]
        want = (v[0, t, 0] - h0[0, 0].T @ kt) @ (dS.T @ kt)
        assert abs(gr["dbeta"][0, t, 0] - want) < 1e-12


def test_beta_zero_pure_decay_closed_form():
    """beta = 0: S_t = diag(2^(g_1+..+g_t)) h0."""
    rng = np.random.default_rng(2)
    B, T, H, HV, K, V = 1, 6, 1, 1, 5, 2
    q, k, v, g, _ = rand_problem(rng, B, T, H, HV, K, V)
    beta = np.zeros((B, T, HV))
    h0 = rng.standard_normal((1, HV, K, V))
    o, hT = oracle.kda_fwd(q, k, v, g, beta, h0)
    G = np.cumsum(g[0, :, 0], axis=0)
    for t in range(T):
        S = np.exp2(G[t])[:, None] * h0[0, 0]
        np.testing.assert_allclose(o[0, t, 0], S.T @ q[0, t, 0] / math.sqrt(K), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(hT[0, 0], np.exp2(G[-1])[:, None] * h0[0, 0], rtol=1e-13)


def test_orthonormal_keys_write_exactly():
    """g = 0, beta = 1, orthonormal keys, h0 = 0: the delta rule stores v_t
    exactly (S^T k_t = v_t), so S = sum_s k_s v_s^T and o is causal linear
    attention over the written pairs."""
    rng = np.random.default_rng(3)
    K, V, T = 6, 4, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm[:, :T].T.reshape(1, T, 1, K)
    q = rng.standard_normal((1, T, 1, K))
    v = rng.standard_normal((1, T, 1, V))
    g = np.zeros((1, T, 1, K))
    beta = np.ones((1, T, 1))
    o, hT = oracle.kda_fwd(q, k, v, g, beta, None)
    S = hT[0, 0]
    for t in range(T):
        np.testing.assert_allclose(S.T @ k[0, t, 0], v[0, t, 0], atol=1e-13)
        want = sum((q[0, t, 0] @ k[0, s, 0]) * v[0, s, 0] for s in range(t + 1)) / math.sqrt(K)
        np.testing.assert_allclose(o[0, t, 0], want, atol=1e-13)


def test_scalar_case_closed_form():
    """K = V = 1: s_t = a_t s + beta k (v - a_t s k) = alpha_t s + b_t with
    alpha_t = a_t (1 - beta k^2), b_t = beta k v; a first-order linear
    recurrence with the textbook solution s_T = (prod alpha) s_0 + sum_t b_t prod_{u>t} alpha_u."""
    rng = np.random.default_rng(4)
    T = 11
    q = rng.standard_normal((1, T, 1, 1))
    k = rng.standard_normal((1, T, 1, 1))
    v = rng.standard_normal((1, T, 1, 1))
    g = -np.abs(rng.standard_normal((1, T, 1, 1)))
    beta = rng.uniform(0, 1, (1, T, 1))
    h0 = rng.standard_normal((1, 1, 1, 1))
    o, hT = oracle.kda_fwd(q, k, v, g, beta, h0)
    a = np.exp2(g.reshape(T))
    kk, vv, bb = k.reshape(T), v.reshape(T), beta.reshape(T)
    alpha = a * (1 - bb * kk * kk)
    b = bb * kk * vv
    for t in range(T):
        s = np.prod(alpha[: t + 1]) * h0.item() + sum(b[u] * np.prod(alpha[u + 1: t + 1]) for u in range(t + 1))
        assert abs(o[0, t, 0, 0] - s * q[0, t, 0, 0]) < 1e-13
    assert abs(hT.item() - (np.prod(alpha) * h0.item() + sum(b[u] * np.prod(alpha[u + 1:]) for u in range(T)))) < 1e-13


def test_empty_slots_pass_state_bitwise_and_split_invariance():
    rng = np.random.default_rng(5)
    T, H, HV, K, V = 40, 1, 2, 4, 3
    q, k, v, g, beta = rand_problem(rng, 1, T, H, HV, K, V)
    cu = [0, 0, 17, 17, 40, 40]
    N = len(cu) - 1
    h0 = rng.standard_normal((N, HV, K, V))
    do = rng.standard_normal((1, T, HV, V))
    dhT = rng.standard_normal((N, HV, K, V))
    o, hT = oracle.kda_fwd(q, k, v, g, beta, h0, cu)
    gr = oracle.kda_bwd(q, k, v, g, beta, h0, do, dhT, cu)
    for n in (0, 2, 4):  # empty slots
        assert np.array_equal(hT[n], h0[n])
        assert np.array_equal(gr["dh0"][n], dhT[n])
    # split sequence [17, 40) at 29: run [17, 29), feed its final state as the
    # initial state of [29, 40); must equal the unsplit run of [17, 40)
    o_u, hT_u = oracle.kda_fwd(q, k, v, g, beta, np.stack([h0[1], h0[3]]), [0, 17, 40])
    o_a, hT_a = oracle.kda_fwd(q, k, v, g, beta, np.stack([h0[1], h0[3]]), [0, 17, 29])
    o_b, hT_b = oracle.kda_fwd(q, k, v, g, beta, np.stack([h0[1], hT_a[1]]), [0, 29, 40])
    # the same operations on the same numbers: bitwise equal
    assert np.array_equal(o_a[0, 17:29], o_u[0, 17:29])
    assert np.array_equal(o_b[0, 29:40], o_u[0, 29:40])
    assert np.array_equal(hT_b[1], hT_u[1])
    # and the split changes nothing in the backward either
    gu = oracle.kda_bwd(q, k, v, g, beta, np.stack([h0[1], h0[3]]), do, np.stack([dhT[1], dhT[3]]),
                        [0, 17, 40])
    gb = oracle.kda_bwd(q, k, v, g, beta, np.stack([h0[1], hT_a[1]]), do, np.stack([dhT[1], dhT[3]]),
                        [0, 29, 40])
    ga = oracle.kda_bwd(q, k, v, g, beta, np.stack([h0[1], h0[3]]), do, np.stack([dhT[1], gb["dh0"][1]]),
                        [0, 17, 29])
    for key in ("dv", "dg", "dbeta", "dq", "dk"):
        np.testing.assert_allclose(gb[key][0, 29:40], gu[key][0, 29:40], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(ga[key][0, 17:29], gu[key][0, 17:29], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ga["dh0"][1], gu["dh0"][1], rtol=1e-12, atol=1e-13)


def test_gva_head_map_contiguous_groups():
    """HV = 2H: value head j reads q/k head j // 2 (contiguous groups)."""
    rng = np.random.default_rng(6)
    T, H, HV, K, V = 12, 2, 4, 3, 2
    q, k, v, g, beta = rand_problem(rng, 1, T, H, HV, K, V)
    h0 = rng.standard_normal((1, HV, K, V))
    o, hT = oracle.kda_fwd(q, k, v, g, beta, h0)
    for j in range(HV):
        h = j // 2
        oj, hTj = oracle.kda_fwd(q[:, :, h:h + 1], k[:, :, h:h + 1], v[:, :, j:j + 1],
                                 g[:, :, j:j + 1], beta[:, :, j:j + 1], h0[:, j:j + 1])
        assert np.array_equal(oj[:, :, 0], o[:, :, j])
        assert np.array_equal(hTj[:, 0], hT[:, j])


@pytest.mark.parametrize("chunk", [1, 16, 64])
def test_chunked_formulation_agrees(chunk):
    rng = np.random.default_rng(7)
    T, H, HV, K, V = 150, 1, 2, 8, 6
    q, k, v, g, beta = rand_problem(rng, 1, T, H, HV, K, V, gscale=2.0)
    cu = [0, 5, 5, 70, 150]
    N = len(cu) - 1
    h0 = rng.standard_normal((N, HV, K, V))
    do = rng.standard_normal((1, T, HV, V))
    dhT = rng.standard_normal((N, HV, K, V))
    o, hT = oracle.kda_fwd(q, k, v, g, beta, h0, cu)
    o2, hT2 = chunked.kda_chunked_fwd(q, k, v, g, beta, h0, cu, chunk=chunk)
    assert oracle.rel_rms(o2, o) < 1e-12 and oracle.rel_rms(hT2, hT) < 1e-12
    gr = oracle.kda_bwd(q, k, v, g, beta, h0, do, dhT, cu)
    gr2 = chunked.kda_chunked_bwd(q, k, v, g, beta, h0, do, dhT, cu, chunk=chunk)
    for key in gr:
        assert oracle.rel_rms(gr2[key], gr[key]) < 1e-11, key


def test_finite_differences_every_gradient():
    """Central differences (fp64) of L = <o, W> + <hT, Wh> against the
    hand-derived backward, for every input element, GVA + an empty slot."""
    rng = np.random.default_rng(8)
    T, H, HV, K, V = 6, 1, 2, 3, 2
    q, k, v, g, beta = rand_problem(rng, 1, T, H, HV, K, V)
    cu = [0, 2, 2, 6]
    N = 3
    h0 = rng.standard_normal((N, HV, K, V))
    W = rng.standard_normal((1, T, HV, V))
    Wh = rng.standard_normal((N, HV, K, V))

    def loss(q, k, v, g, beta, h0):
        o, hT = oracle.kda_fwd(q, k, v, g, beta, h0, cu, nthreads=1)
        return float(np.sum(o * W) + np.sum(hT * Wh))

    gr = oracle.kda_bwd(q, k, v, g, beta, h0, W, Wh, cu, nthreads=1)
    args = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    eps = 1e-6
    for name, arr in args.items():
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss(**args)
            arr[idx] = old - eps
            lm = loss(**args)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.max(np.abs(fd - gr[names[name]])) / max(1.0, np.max(np.abs(fd)))
        assert err < 1e-7, (name, err)


def test_backward_matches_torch_autograd_of_naive_loop():
    """torch.autograd (a library routine) differentiates a naive fp64 loop;
    the oracle's hand-derived backward must agree."""
    rng = np.random.default_rng(9)
    T, H, HV, K, V = 20, 2, 4, 5, 3
    q, k, v, g, beta = rand_problem(rng, 1, T, H, HV, K, V)
    h0 = rng.standard_normal((1, HV, K, V))
    do = rng.standard_normal((1, T, HV, V))
    dhT = rng.standard_normal((1, HV, K, V))
    tq, tk, tv, tg, tb, th = (torch.tensor(x, requires_grad=True) for x in (q, k, v, g, beta, h0))
    outs = []
    finals = []
    for j in range(HV):
        hh = j // (HV // H)
        S = th[0, j]
        oj = []
        for t in range(T):
            S = torch.exp2(tg[0, t, j])[:, None] * S
            e = S.T @ tk[0, t, hh]
            d = tb[0, t, j] * (tv[0, t, j] - e)
            S = S + torch.outer(tk[0, t, hh], d)
            oj.append(S.T @ tq[0, t, hh] / math.sqrt(K))
        outs.append(torch.stack(oj))
        finals.append(S)
    o = torch.stack(outs, dim=1)[None]
    hT = torch.stack(finals)[None]
    L = (o * torch.tensor(do)).sum() + (hT * torch.tensor(dhT)).sum()
    L.backward()
    gr = oracle.kda_bwd(q, k, v, g, beta, h0, do, dhT)
    for t_, key in ((tq, "dq"), (tk, "dk"), (tv, "dv"), (tg, "dg"), (tb, "dbeta"), (th, "dh0")):
        np.testing.assert_allclose(gr[key], t_.grad.numpy(), rtol=1e-11, atol=1e-12, err_msg=key)


def test_rel_rms_definition():
    assert oracle.rel_rms([3.0, 4.0], [3.0, 4.0]) == 0.0
    assert abs(oracle.rel_rms([3.0, 5.0], [3.0, 4.0]) - 0.2) < 1e-15
    assert oracle.rel_rms([0.0], [0.0]) == 0.0
    assert oracle.rel_rms([1e-30], [0.0]) == float("inf")


# ---- the q/k L2-norm prologue ----

def test_l2norm_rows_unit_norm_scale_invariance_and_eps():
    """Rows come out with norm sqrt(s / (s + eps)) (s = the row's sum of
    squares): exactly 1 at eps = 0, where positive row scales drop out."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((2, 5, 3, 7))
    y0 = oracle.l2norm_rows(x, eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.sum(y0 * y0, axis=-1)), 1.0, rtol=0, atol=1e-15)
    c = np.exp(rng.standard_normal((2, 5, 3, 1)))
    np.testing.assert_allclose(oracle.l2norm_rows(c * x, eps=0.0), y0, rtol=1e-14, atol=1e-15)
    s = np.sum(x * x, axis=-1)
    y = oracle.l2norm_rows(x)
    np.testing.assert_allclose(np.sum(y * y, axis=-1), s / (s + oracle.L2NORM_EPS), rtol=1e-14)
    assert np.all(oracle.l2norm_rows(np.zeros((1, 4))) == 0.0)  # zero rows stay zero


def test_l2norm_backward_finite_differences_and_orthogonality():
    """Central differences of <W, l2norm_rows(x)>; and x . dx = r (x . dy) eps / (s + eps):
    at eps = 0 the gradient is orthogonal to its row."""
    rng = np.random.default_rng(22)
    x = rng.standard_normal((3, 6))
    W = rng.standard_normal((3, 6))
    gr = oracle.l2norm_rows_bwd(x, W)
    fd = np.zeros_like(x)
    h = 1e-6
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (np.sum(W * oracle.l2norm_rows(xp)) - np.sum(W * oracle.l2norm_rows(xm))) / (2 * h)
    assert np.max(np.abs(fd - gr)) < 1e-8
    g0 = oracle.l2norm_rows_bwd(x, W, eps=0.0)
    np.testing.assert_allclose(np.sum(x * g0, axis=-1), 0.0, atol=1e-14)
    s = np.sum(x * x, axis=-1)
    r = 1.0 / np.sqrt(s + oracle.L2NORM_EPS)
    np.testing.assert_allclose(np.sum(x * gr, axis=-1),
                               r * np.sum(x * W, axis=-1) * oracle.L2NORM_EPS / (s + oracle.L2NORM_EPS),
                               rtol=0, atol=1e-14)


def test_qk_l2norm_kda_scale_invariance_and_finite_differences():
    """With the prologue, positive per-row scales of q and k leave o and hT
    unchanged (up to the eps effect); dq, dk match central differences of the
    whole layer, GVA with an empty slot."""
    rng = np.random.default_rng(23)
    T, H, HV, K, V = 6, 1, 2, 3, 2
    q, k, v, g, beta = rand_problem(rng, 1, T, H, HV, K, V)
    k = k * np.exp(rng.standard_normal((1, T, H, 1)))  # rows of any norm
    cu = [0, 2, 2, 6]
    N = 3
    h0 = rng.standard_normal((N, HV, K, V))
    o1, h1 = oracle.kda_fwd(q, k, v, g, beta, h0, cu, nthreads=1, qk_l2norm=True)
    cq = np.exp(rng.standard_normal((1, T, H, 1)))
    ck = np.exp(rng.standard_normal((1, T, H, 1)))
    o2, h2 = oracle.kda_fwd(cq * q, ck * k, v, g, beta, h0, cu, nthreads=1, qk_l2norm=True)
    assert oracle.rel_rms(o2, o1) < 1e-5 and oracle.rel_rms(h2, h1) < 1e-5
    W = rng.standard_normal((1, T, HV, V))
    Wh = rng.standard_normal((N, HV, K, V))

    def loss(q, k):
        o, hT = oracle.kda_fwd(q, k, v, g, beta, h0, cu, nthreads=1, qk_l2norm=True)
        return float(np.sum(o * W) + np.sum(hT * Wh))

    gr = oracle.kda_bwd(q, k, v, g, beta, h0, W, Wh, cu, nthreads=1, qk_l2norm=True)
    args = dict(q=q, k=k)
    h = 1e-6
    for name in ("q", "k"):
        arr = args[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = loss(**args)
            arr[idx] = old - h
            lm = loss(**args)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - gr["d" + name])) / max(1.0, np.max(np.abs(fd)))
        assert err < 1e-7, (name, err)


# ---- the scalar-gate (GDN) variant ----

def test_scalar_gate_pure_decay_closed_form():
    """beta = 0: the state only decays, by one scalar factor per token, so
    o_t = 2^(G_t) h0^T q~_t and hT = 2^(G_T) h0 with G_t = sum_{s<=t} g_s, and
    dL/dg_s = ln 2 (sum_{t>=s} <o_t, W_t> + <hT, Wh>)."""
    rng = np.random.default_rng(31)
    T, H, HV, K, V = 5, 1, 2, 3, 2
    q, k, v, _, beta = rand_problem(rng, 1, T, H, HV, K, V)
    beta = np.zeros_like(beta)
    g = -np.log1p(np.exp(rng.standard_normal((1, T, HV))))
    h0 = rng.standard_normal((1, HV, K, V))
    W = rng.standard_normal((1, T, HV, V))
    Wh = rng.standard_normal((1, HV, K, V))
    o, hT = oracle.kda_fwd(q, k, v, g, beta, h0, scalar_gate=True)
    gr = oracle.kda_bwd(q, k, v, g, beta, h0, W, Wh, scalar_gate=True)
    assert gr["dg"].shape == g.shape
    for j in range(HV):
        G = np.cumsum(g[0, :, j])
        ref_o = np.stack([2.0 ** G[t] * (h0[0, j].T @ q[0, t, 0]) / math.sqrt(K) for t in range(T)])
        np.testing.assert_allclose(o[0, :, j], ref_o, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(hT[0, j], 2.0 ** G[-1] * h0[0, j], rtol=1e-13)
        contrib = np.array([np.dot(ref_o[t], W[0, t, j]) for t in range(T)])
        final = np.sum(2.0 ** G[-1] * h0[0, j] * Wh[0, j])
        ref_dg = math.log(2.0) * (np.cumsum(contrib[::-1])[::-1] + final)
        np.testing.assert_allclose(gr["dg"][0, :, j], ref_dg, rtol=1e-12, atol=1e-13)


def test_scalar_gate_finite_differences():
    """Central differences of every input with a scalar gate, GVA + an empty slot."""
    rng = np.random.default_rng(32)
    T, H, HV, K, V = 6, 1, 2, 3, 2
    q, k, v, _, beta = rand_problem(rng, 1, T, H, HV, K, V)
    g = -np.log1p(np.exp(rng.standard_normal((1, T, HV))))
    cu = [0, 2, 2, 6]
    N = 3
    h0 = rng.standard_normal((N, HV, K, V))
    W = rng.standard_normal((1, T, HV, V))
    Wh = rng.standard_normal((N, HV, K, V))

    def loss(q, k, v, g, beta, h0):
        o, hT = oracle.kda_fwd(q, k, v, g, beta, h0, cu, nthreads=1, scalar_gate=True)
        return float(np.sum(o * W) + np.sum(hT * Wh))

    gr = oracle.kda_bwd(q, k, v, g, beta, h0, W, Wh, cu, nthreads=1, scalar_gate=True)
    args = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)
    h = 1e-6
    for name, arr in args.items():
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = loss(**args)
            arr[idx] = old - h
            lm = loss(**args)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        key = "dbeta" if name == "beta" else "dh0" if name == "h0" else "d" + name
        err = np.max(np.abs(fd - gr[key])) / max(1.0, np.max(np.abs(fd)))
        assert err < 1e-7, (name, err)


# ---- the KDA gate inside the op (oracle.kda_gate / kda_gate_bwd) ----

def _gate_inputs(rng, T=5, HV=2, K=3):
    a = 2.0 * rng.standard_normal((1, T, HV, K))
    A_log = 0.5 * rng.standard_normal(HV)
    bias = rng.standard_normal((HV, K))
    return a, A_log, bias


@pytest.mark.parametrize("lower_bound", [None, -5.0], ids=["unbounded", "bounded"])
def test_gate_omitted_A_log_is_zero_A_log_bitwise(lower_bound):
    """[Fix] Use unit KDA gate scale when A_log is omitted: omitting A_log is the
    same as passing an explicit zero A_log, for the gate and for the whole layer."""
    rng = np.random.default_rng(41)
    a, _, bias = _gate_inputs(rng)
    z = np.zeros(a.shape[2])
    assert np.array_equal(oracle.kda_gate(a, None, bias, lower_bound), oracle.kda_gate(a, z, bias, lower_bound))
    q, k, v, _, beta = rand_problem(rng, 1, a.shape[1], 1, a.shape[2], a.shape[3], 2)
    h0 = rng.standard_normal((1, a.shape[2], a.shape[3], 2))
    W, Wh = rng.standard_normal(v.shape), rng.standard_normal(h0.shape)
    g1 = dict(bias=bias, lower_bound=lower_bound)
    g2 = dict(A_log=z, bias=bias, lower_bound=lower_bound)
    o1, h1 = oracle.kda_fwd(q, k, v, a, beta, h0, gate=g1)
    o2, h2 = oracle.kda_fwd(q, k, v, a, beta, h0, gate=g2)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)
    r1 = oracle.kda_bwd(q, k, v, a, beta, h0, W, Wh, gate=g1)
    r2 = oracle.kda_bwd(q, k, v, a, beta, h0, W, Wh, gate=g2)
    for key in r1:
        assert np.array_equal(r1[key], r2[key]), key


def test_gate_closed_forms():
    """Values the formulas fix: softplus(0) = ln 2 and sigmoid(0) = 1/2; an
    explicit ones A_log gives the scale e (the former default); far from 0 the
    unbounded gate tends to -s x and to 0, the bounded one to its bound and to 0;
    the bias only shifts the argument; the unbounded gate scales with exp(A_log)."""
    HV, K = 2, 3
    zero = np.zeros((1, 1, HV, K))
    ln2 = math.log(2.0)
    np.testing.assert_allclose(oracle.kda_gate(zero), -ln2, rtol=1e-15)
    np.testing.assert_allclose(oracle.kda_gate(zero, np.ones(HV)), -math.e * ln2, rtol=1e-15)
    np.testing.assert_allclose(oracle.kda_gate(zero, lower_bound=-5.0), -2.5, rtol=1e-15)
    np.testing.assert_allclose(oracle.kda_gate(zero, np.array([0.3, -1.0]), lower_bound=-5.0), -2.5, rtol=1e-15)
    big = np.full((1, 1, HV, K), 40.0)
    A = np.array([0.2, -0.4])
    per_head = lambda x: np.broadcast_to(np.asarray(x)[:, None], big.shape)  # noqa: E731
    np.testing.assert_allclose(oracle.kda_gate(big, A), per_head(-np.exp(A) * 40.0), rtol=1e-15)
    np.testing.assert_allclose(oracle.kda_gate(big, A, lower_bound=-3.0), -3.0, rtol=1e-10)  # within e^(-40 s)
    np.testing.assert_allclose(oracle.kda_gate(-big, A), per_head(-np.exp(A) * math.exp(-40.0)), rtol=1e-12)
    np.testing.assert_allclose(oracle.kda_gate(-big, A, lower_bound=-3.0),
                               per_head(-3.0 * np.exp(-40.0 * np.exp(A))), rtol=1e-10)  # to e^(-40 s)
    rng = np.random.default_rng(42)
    a, A_log, bias = _gate_inputs(rng, 4, HV, K)
    np.testing.assert_allclose(oracle.kda_gate(a, A_log, bias), oracle.kda_gate(a + bias, A_log), rtol=0, atol=0)
    np.testing.assert_allclose(oracle.kda_gate(a, A_log), np.exp(A_log)[:, None] * oracle.kda_gate(a), rtol=1e-14)


def test_gate_ranges():
    rng = np.random.default_rng(43)
    a, A_log, bias = _gate_inputs(rng, 50, 2, 4)
    a *= 5.0
    gu = oracle.kda_gate(a, A_log, bias)
    gb = oracle.kda_gate(a, A_log, bias, lower_bound=-4.0)
    assert np.all(gu < 0) and np.all(gb < 0) and np.all(gb > -4.0)


@pytest.mark.parametrize("lower_bound", [None, -5.0], ids=["unbounded", "bounded"])
def test_gate_finite_differences(lower_bound):
    """Central differences of L = sum(g W) w.r.t. a, A_log and bias."""
    rng = np.random.default_rng(44)
    a, A_log, bias = _gate_inputs(rng)
    W = rng.standard_normal(a.shape)
    da, dA, db = oracle.kda_gate_bwd(a, W, A_log, bias, lower_bound)
    h = 1e-6
    for arr, ref in ((a, da), (A_log, dA), (bias, db)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = np.sum(oracle.kda_gate(a, A_log, bias, lower_bound) * W)
            arr[idx] = old - h
            lm = np.sum(oracle.kda_gate(a, A_log, bias, lower_bound) * W)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        assert np.max(np.abs(fd - ref)) / max(1.0, np.max(np.abs(fd))) < 1e-8


@pytest.mark.parametrize("lower_bound", [None, -3.0], ids=["unbounded", "bounded"])
def test_gate_layer_finite_differences(lower_bound):
    """The layer with the gate inside: central differences of the raw gate, A_log
    and the bias through the whole recurrence (GVA, an empty slot), so the core's
    dg reaches the gate and the parameter gradients sum over the valid tokens."""
    rng = np.random.default_rng(45)
    T, H, HV, K, V = 6, 1, 2, 3, 2
    q, k, v, _, beta = rand_problem(rng, 1, T, H, HV, K, V)
    a, A_log, bias = _gate_inputs(rng, T, HV, K)
    cu = [0, 2, 2, 5]  # an empty slot and a capacity tail (token 5)
    h0 = rng.standard_normal((3, HV, K, V))
    W = rng.standard_normal((1, T, HV, V))
    Wh = rng.standard_normal((3, HV, K, V))

    def loss():
        gate = dict(A_log=A_log, bias=bias, lower_bound=lower_bound)
        o, hT = oracle.kda_fwd(q, k, v, a, beta, h0, cu, nthreads=1, gate=gate)
        return float(np.sum(o[:, :5] * W[:, :5]) + np.sum(hT * Wh))

    gr = oracle.kda_bwd(q, k, v, a, beta, h0, W * (np.arange(T) < 5)[None, :, None, None], Wh, cu, nthreads=1,
                        gate=dict(A_log=A_log, bias=bias, lower_bound=lower_bound))
    h = 1e-6
    for arr, ref in ((a, gr["dg"]), (A_log, gr["dA_log"]), (bias, gr["dbias"])):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = loss()
            arr[idx] = old - h
            lm = loss()
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        assert np.max(np.abs(fd - ref)) / max(1.0, np.max(np.abs(fd))) < 1e-7


@pytest.mark.parametrize("lower_bound", [None, -5.0], ids=["unbounded", "bounded"])
def test_gate_matches_torch_autograd(lower_bound):
    """torch.nn.functional's softplus / sigmoid with autograd, in fp64."""
    rng = np.random.default_rng(46)
    a, A_log, bias = _gate_inputs(rng)
    W = rng.standard_normal(a.shape)
    ta, tA, tb = (torch.tensor(x, requires_grad=True) for x in (a, A_log, bias))
    s = torch.exp(tA)[:, None]
    x = ta + tb
    g = -s * torch.nn.functional.softplus(x) if lower_bound is None else lower_bound * torch.sigmoid(s * x)
    (g * torch.tensor(W)).sum().backward()
    np.testing.assert_allclose(oracle.kda_gate(a, A_log, bias, lower_bound), g.detach().numpy(), rtol=1e-14)
    da, dA, db = oracle.kda_gate_bwd(a, W, A_log, bias, lower_bound)
    np.testing.assert_allclose(da, ta.grad.numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dA, tA.grad.numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(db, tb.grad.numpy(), rtol=1e-12, atol=1e-15)
