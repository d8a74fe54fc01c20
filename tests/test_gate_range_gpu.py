"""GPU parity for strong decays: the tensor-core kernels split each pairwise
decay 2^(G_r - G_i) into factors at references inside the chunk, and these
cases drive those factors to the edges of their range.  A chunk whose decay
span (per channel, G at its first row minus G at its last) is at most 192
(log2) runs on one middle reference per chunk; a wider one goes to the
16-token block-reference kernels (status words 6 for the records, 5 for the
gradients); a 16-token block wider than 192 goes on to the exact path (words 3
and 4).  Gates far below the workloads' clip at -5 (log2) reach every path.
Every case is checked against the fp64 oracle at the bf16 tolerances, and the
status words tell which paths ran."""
import zlib

import numpy as np
import pytest
import torch

from gated_delta_rule_42_gb300 import inputs
from tests import kda_gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_42_gb300 import build
    build.build()
    assert torch.cuda.is_available()


VARLEN_GVA = dict(B=1, T=700, H=2, HV=4, K=128, V=128, cu_seqlens=[0, 0, 3, 260, 260, 700])

# name, gate (mean, std, clip) of clip(-softplus(N(mean, std)), clip, 0), problem, exact path expected
CASES = [
    ("softplus_N2_2_clip30", (2.0, 2.0, -30.0), VARLEN_GVA, False),
    ("strong_N6_3_clip40", (6.0, 3.0, -40.0), VARLEN_GVA, False),  # block spans up to ~140: block references
    ("wide_N16_4_clip60", (16.0, 4.0, -60.0), VARLEN_GVA, True),   # block spans ~240: the exact path
    ("wide_dense_hv_eq_h", (16.0, 4.0, -60.0), dict(B=2, T=200, H=2, HV=2, K=128, V=128), True),
]


def _check(inp, l2=False, expect_exact=None, expect_block=None):
    tol = H.TOL[inp.dtype]
    sf, sb = [], []
    o, hT = H.gpu_fwd(inp, l2=l2, status=sf)
    ro, rhT = H.oracle_fwd(inp, l2=l2)
    H.check_fwd(inp, o, hT, ro, rhT if inp.output_final_state else None, tol["fwd"])
    gr = H.gpu_bwd(inp, want_dh0=inp.h0 is not None, l2=l2, status=sb)
    H.check_bwd(inp, gr, H.oracle_bwd(inp, l2=l2), tol["bwd"])
    if expect_exact is not None:
        # forward: the record kernel (word 3); recompute backward: the record kernel again and the
        # gradient kernel (word 4)
        assert (sf[3] > 0) == expect_exact and (sb[3] > 0) == expect_exact and (sb[4] > 0) == expect_exact, (sf, sb)
    # the gradients run the chunk-reference kernel first except with a scalar gate or the
    # fused L2-norm backward (HV = H), where the block-reference kernel takes every slot
    chunk_grad = not (inp.g.dim() == 3 or (l2 and inp.HV == inp.H))  # (a scalar gate is [B, T, HV])
    if expect_block is not None:  # the block-reference kernels: records (word 6), gradients (word 5)
        assert (sf[6] > 0) == expect_block and (sb[6] > 0) == expect_block, (sf, sb)
        assert not chunk_grad or (sb[5] > 0) == expect_block, (sf, sb)
    if expect_exact:  # a slot on the exact path went through the block-reference kernel first
        assert sf[6] >= sf[3] and sb[6] >= sb[3] and (not chunk_grad or sb[5] >= sb[4]), (sf, sb)
    return sf, sb


@pytest.mark.parametrize("name,gate,kw,exact", CASES, ids=[c[0] for c in CASES])
def test_strong_decays(name, gate, kw, exact):
    mu, sd, lo = gate
    inp = inputs.make_inputs(dtype=torch.bfloat16, seed=zlib.crc32(name.encode()) % 1000, name=name,
                             g_mean=mu, g_std=sd, g_lo=lo, **kw)
    _check(inp, expect_exact=exact, expect_block=None if name.startswith("softplus") else True)


def test_chunk_wide_block_narrow_takes_the_block_reference_path_only():
    """Per-token gates near -4 (log2): every chunk spans ~250 (> 192) while every
    16-token block spans ~60, so each slot goes to the block-reference kernels and
    none to the exact path."""
    inp = inputs.make_inputs(dtype=torch.bfloat16, seed=67, name="chunk_wide", g_mean=4.0, g_std=0.3, g_lo=-8.0,
                             **VARLEN_GVA)
    _check(inp, expect_exact=False, expect_block=True)


def _unnormalised(inp, seed):
    rng = np.random.default_rng(seed)
    for name in ("q", "k"):
        x = getattr(inp, name)
        f = torch.from_numpy(np.exp(rng.normal(0.0, 0.7, size=x.shape[:-1] + (1,))))
        setattr(inp, name, (x.to(torch.float64) * f).to(inp.dtype))
    return inp


@pytest.mark.parametrize("hv", [2, 4], ids=["fused_norm_bwd", "gva_partials"])
def test_wide_decays_with_l2norm_prologue(hv):
    """The exact path reads the raw rows and applies the prologue's norms itself."""
    inp = inputs.make_inputs(B=1, T=300, H=2, HV=hv, K=128, V=128, dtype=torch.bfloat16, seed=61 + hv,
                             cu_seqlens=[0, 0, 130, 300], g_mean=16.0, g_std=4.0, g_lo=-60.0, name="wide_l2")
    _check(_unnormalised(inp, seed=62), l2=True, expect_exact=True)


def test_wide_scalar_gate():
    inp = inputs.make_inputs(B=1, T=300, H=2, HV=4, K=128, V=128, dtype=torch.bfloat16, seed=63,
                             cu_seqlens=[0, 100, 100, 300], g_mean=16.0, g_std=4.0, g_lo=-60.0,
                             scalar_gate=True, name="wide_sg")
    _check(inp, expect_exact=True)


def test_hard_resets_in_a_few_channels():
    """Ordinary gates with a sparse set of (token, value head, channel) entries at
    -250 (a decay of 2^-250: a reset of that channel).  A slot holding one is on
    the exact path for every channel, ordinary ones included."""
    inp = inputs.make_inputs(dtype=torch.bfloat16, seed=64, name="resets", **VARLEN_GVA)
    rng = np.random.default_rng(65)
    mask = rng.random(inp.g.shape) < 0.002
    inp.g = torch.where(torch.from_numpy(mask), torch.tensor(-250.0), inp.g)
    _check(inp, expect_exact=True)


def test_ordinary_gates_stay_on_the_chunk_references():
    sf, sb = [], []
    inp = inputs.make_config(1)
    H.gpu_fwd(inp, status=sf)
    H.gpu_bwd(inp, status=sb)
    assert sf[3:] == [0, 0, 0, 0] and sb[3:] == [0, 0, 0, 0], (sf, sb)


def test_wide_decays_dense_training_shape_sampled():
    """The dense training layer's shape (B=8, T=4096, H=HV=32) with gates on the
    exact path everywhere; the oracle checks sampled (sequence, head) units."""
    inp = inputs.make_inputs(B=8, T=4096, H=32, HV=32, K=128, V=128, dtype=torch.bfloat16, seed=66,
                             h0=False, final_state=False, g_mean=16.0, g_std=4.0, g_lo=-60.0, name="wide_train")
    tol = H.TOL[inp.dtype]
    sf, sb = [], []
    o, _ = H.gpu_fwd(inp, status=sf)
    gr = H.gpu_bwd(inp, want_dh0=False, status=sb)
    assert sf[3] > 0 and sb[3] > 0 and sb[4] > 0
    flat = lambda x: x.reshape(inp.B * inp.T, *x.shape[2:])  # noqa: E731
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.isfinite(gr[key]).all(), key
    for n, hq, js, t0, t1, (ro, _), rg in H.sample_units(inp, [(0, 0), (5, 17)]):
        H.assert_rel(f"o[{n},{hq}]", flat(o)[t0:t1][:, js].double().numpy(), ro[0], tol["fwd"])
        H.assert_rel(f"dq[{n},{hq}]", flat(gr["dq"])[t0:t1, hq:hq + 1].double().numpy(), rg["dq"][0], tol["bwd"])
        H.assert_rel(f"dk[{n},{hq}]", flat(gr["dk"])[t0:t1, hq:hq + 1].double().numpy(), rg["dk"][0], tol["bwd"])
        H.assert_rel(f"dv[{n},{hq}]", flat(gr["dv"])[t0:t1][:, js].double().numpy(), rg["dv"][0], tol["bwd"])
        H.assert_rel(f"dg[{n},{hq}]", flat(gr["dg"])[t0:t1][:, js].double().numpy(), rg["dg"][0], tol["bwd"])
        H.assert_rel(f"dbeta[{n},{hq}]", flat(gr["dbeta"])[t0:t1][:, js].double().numpy(), rg["dbeta"][0],
                     tol["bwd"])
