"""The oracle's pins must catch plausible mistakes.  Each case plants one
mistake in a copy of the C oracle (on the CPU), loads it in place of the real
one and runs the pins; at least one pin must fail."""
import ctypes
import os
import subprocess
import tempfile

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
