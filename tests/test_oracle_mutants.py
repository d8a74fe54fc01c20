"""The oracle's pins must catch plausible mistakes.  Each case plants one
mistake in a copy of the C oracle (on the CPU) and loads it in place of the
real one, or, for the numpy q/k L2-norm prologue, the scalar gate and the KDA
gate, replaces one of the oracle's functions; then it runs the pins, and at
least one pin must fail."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (name, text to find, replacement) -- each is a one-token slip
MUTANTS = [
    ("output_reads_pre_update_state",
     "token_step(K, V, S, kt, gt, J->beta[(size_t)t * HV + j], vt, e, delta);\n    double *ot",
     "double *ot"),
    ("delta_sign", "delta[x] = bt * (vt[x] - e[x]);", "delta[x] = bt * (e[x] - vt[x]);"),
    ("no_query_scale", "const double qc = qt[c] * scale;", "const double qc = qt[c];"),
    ("decay_after_write_missing", "double a = exp2(gt[c]);\n    double *row = S + (size_t)c * V;\n    for (int x = 0; x < V; ++x) row[x] *= a;",
     "double a = exp2(gt[c]);\n    double *row = S + (size_t)c * V;\n    for (int x = 0; x < V; ++x) row[x] *= a * a;"),
    ("gva_head_modulo", "const int K = J->K, V = J->V, HV = J->HV, r = J->HV / J->H, h = j / r;\n  const double scale = 1.0 / sqrt((double)K);\n  double *S",
     "const int K = J->K, V = J->V, HV = J->HV, r = J->HV / J->H, h = j % J->H;\n  const double scale = 1.0 / sqrt((double)K);\n  double *S"),
    ("bwd_drop_P_de_term", "dkp[c] += acc;", "dkp[c] += 0.0 * acc;"),
    ("bwd_dg_missing_ln2", "dgt[c] = ln2 * a * acc;", "dgt[c] = a * acc;"),
    ("bwd_state_grad_not_decayed", "dsrow[x] = a * dprow[x];", "dsrow[x] = dprow[x];"),
    ("bwd_dq_missing_scale", "dqp[c] = acc * scale;", "dqp[c] = acc;"),
    ("bwd_dbeta_sign", "db += ddel[x] * (vt[x] - e[x]);", "db += ddel[x] * (e[x] - vt[x]);"),
    ("bwd_de_sign", "de[x] = -bt * ddel[x];", "de[x] = bt * ddel[x];"),
    ("bwd_dk_transposed_term", "acc += drow[x] * delta[x];", "acc += drow[x] * dot[x];"),
]

PINS = [
    pins.test_handcalc_golden,
    pins.test_no_gate_no_beta_state_unchanged_and_closed_form_grads,
    pins.test_beta_zero_pure_decay_closed_form,
    pins.test_orthonormal_keys_write_exactly,
    pins.test_scalar_case_closed_form,
    pins.test_finite_differences_every_gradient,
    pins.test_backward_matches_torch_autograd_of_naive_loop,
    pins.test_gva_head_map_contiguous_groups,
]


def _compile(src_text, tmpdir):
    c = os.path.join(tmpdir, "m.c")
    so = os.path.join(tmpdir, "m.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", so, c, "-lm", "-lpthread"])
    return so


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, find, repl, monkeypatch):
    text = open(SRC).read()
    assert text.count(find) == 1, f"mutation anchor not unique/found: {name}"
    with tempfile.TemporaryDirectory() as d:
        so = _compile(text.replace(find, repl), d)
        real = oracle._load()
        lib = ctypes.CDLL(so)
        lib.kda_oracle_fwd.argtypes = real.kda_oracle_fwd.argtypes
        lib.kda_oracle_fwd.restype = real.kda_oracle_fwd.restype
        lib.kda_oracle_bwd.argtypes = real.kda_oracle_bwd.argtypes
        lib.kda_oracle_bwd.restype = real.kda_oracle_bwd.restype
        monkeypatch.setattr(oracle, "_lib", lib)
        caught = []
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin.__name__)
        assert caught, f"no pin caught mutant {name}"


# The q/k L2-norm prologue lives in numpy: its planted mistakes replace the
# oracle's functions in place, and the prologue pins must catch each one.
def _bwd_no_projection(x, dy, eps=oracle.L2NORM_EPS):
    x, dy = np.asarray(x, np.float64), np.asarray(dy, np.float64)
    return dy / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def _bwd_projection_sign(x, dy, eps=oracle.L2NORM_EPS):
    x, dy = np.asarray(x, np.float64), np.asarray(dy, np.float64)
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    y = x * r
    return r * (dy + y * np.sum(y * dy, axis=-1, keepdims=True))


def _fwd_wrong_axis(x, eps=oracle.L2NORM_EPS):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=0, keepdims=True) + eps)


def _fwd_no_sqrt(x, eps=oracle.L2NORM_EPS):
    x = np.asarray(x, np.float64)
    return x / (np.sum(x * x, axis=-1, keepdims=True) + eps)


L2_MUTANTS = [("l2norm_rows_bwd", _bwd_no_projection), ("l2norm_rows_bwd", _bwd_projection_sign),
              ("l2norm_rows", _fwd_wrong_axis), ("l2norm_rows", _fwd_no_sqrt)]
L2_PINS = [pins.test_l2norm_rows_unit_norm_scale_invariance_and_eps,
           pins.test_l2norm_backward_finite_differences_and_orthogonality,
           pins.test_qk_l2norm_kda_scale_invariance_and_finite_differences]


@pytest.mark.parametrize("attr,fn", L2_MUTANTS, ids=[m[1].__name__ for m in L2_MUTANTS])
def test_l2norm_pins_catch_planted_mistake(attr, fn, monkeypatch):
    monkeypatch.setattr(oracle, attr, fn)
    caught = []
    for pin in L2_PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught {fn.__name__}"


def _reduce_mean(dg):
    return np.mean(np.asarray(dg, np.float64), axis=-1)


def _broadcast_scaled(g, K):
    g = np.asarray(g, np.float64)
    return np.ascontiguousarray(np.repeat(g[..., None] / K, K, axis=-1))


def _reduce_first_channel(dg):
    return np.asarray(dg, np.float64)[..., 0]


GATE_MUTANTS = [("gate_grad_reduce", _reduce_mean), ("gate_per_channel", _broadcast_scaled),
                ("gate_grad_reduce", _reduce_first_channel)]
GATE_PINS = [pins.test_scalar_gate_pure_decay_closed_form, pins.test_scalar_gate_finite_differences]


@pytest.mark.parametrize("attr,fn", GATE_MUTANTS, ids=[m[1].__name__ for m in GATE_MUTANTS])
def test_scalar_gate_pins_catch_planted_mistake(attr, fn, monkeypatch):
    monkeypatch.setattr(oracle, attr, fn)
    caught = []
    for pin in GATE_PINS:
        try:
            pin()
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught {fn.__name__}"


# The KDA gate lives in numpy too: planted mistakes in its forward and backward.
def _gate_omitted_scale_e(a, A_log=None, bias=None, lower_bound=None):  # the behaviour the page's fix removed
    return _REAL_GATE(a, np.ones(np.shape(a)[2]) if A_log is None else A_log, bias, lower_bound)


def _gate_bounded_scale_outside(a, A_log=None, bias=None, lower_bound=None):
    if lower_bound is None:
        return _REAL_GATE(a, A_log, bias, None)
    s = 1.0 if A_log is None else np.exp(np.asarray(A_log))[:, None]
    x = a if bias is None else a + bias
    return s * lower_bound / (1.0 + np.exp(-x))


def _gate_bwd_no_scale(a, dg, A_log=None, bias=None, lower_bound=None):
    da, dA, db = _REAL_GATE_BWD(a, dg, A_log, bias, lower_bound)
    s = np.ones((np.shape(a)[2], 1)) if A_log is None else np.exp(np.asarray(A_log))[:, None]
    return da / s, dA, db / s


def _gate_bwd_bias_summed_over_channels(a, dg, A_log=None, bias=None, lower_bound=None):
    da, dA, db = _REAL_GATE_BWD(a, dg, A_log, bias, lower_bound)
    return da, dA, np.broadcast_to(np.sum(da, axis=(0, 1, 3))[:, None], db.shape).copy()


def _gate_bwd_dA_sign(a, dg, A_log=None, bias=None, lower_bound=None):
    da, dA, db = _REAL_GATE_BWD(a, dg, A_log, bias, lower_bound)
    return da, -dA, db


_REAL_GATE, _REAL_GATE_BWD = oracle.kda_gate, oracle.kda_gate_bwd
KDA_GATE_MUTANTS = [("kda_gate", _gate_omitted_scale_e), ("kda_gate", _gate_bounded_scale_outside),
                    ("kda_gate_bwd", _gate_bwd_no_scale), ("kda_gate_bwd", _gate_bwd_bias_summed_over_channels),
                    ("kda_gate_bwd", _gate_bwd_dA_sign)]


def _kda_gate_pins():
    return [lambda: pins.test_gate_omitted_A_log_is_zero_A_log_bitwise(None), pins.test_gate_closed_forms,
            lambda: pins.test_gate_finite_differences(None),
            lambda: pins.test_gate_finite_differences(-5.0), lambda: pins.test_gate_layer_finite_differences(-3.0)]


@pytest.mark.parametrize("attr,fn", KDA_GATE_MUTANTS, ids=[m[1].__name__ for m in KDA_GATE_MUTANTS])
def test_kda_gate_pins_catch_planted_mistake(attr, fn, monkeypatch):
    monkeypatch.setattr(oracle, attr, fn)
    caught = 0
    for pin in _kda_gate_pins():
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught, f"no pin caught {fn.__name__}"
