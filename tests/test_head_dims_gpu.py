"""GPU parity of the tensor-core kernels at head dims 64 (K and V each 64 or
128): the kernels run a 64-wide head zero-padded in their 128-wide tiles (TMA
fills the channels past the head with zeros), with the 1/sqrt(K) scale and
every global load and store at the real head dims.  Includes the pages'
benchmark shape (B=1, T=73, H=1, HV=2, K=V=64 with cu_seqlens [0, 3, 73]) and
the dense training layer's shape at K=V=64 with sampled oracle units."""
import ctypes
import zlib

import pytest
import torch

from gated_delta_rule_42_gb300 import _lib, inputs
from gated_delta_rule_42_gb300.ops import make_inputs_struct
from tests import kda_gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_42_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _on_tensor_cores(inp):
    d = inp.to("cuda")
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens)
    return _lib.load().kda_uses_tensor_cores(ctypes.byref(s)) == 1


def _full(inp, l2=False):
    assert _on_tensor_cores(inp)
    tol = H.TOL[inp.dtype]
    o, hT = H.gpu_fwd(inp, l2=l2)
    ro, rhT = H.oracle_fwd(inp, l2=l2)
    H.check_fwd(inp, o, hT, ro, rhT if inp.output_final_state else None, tol["fwd"])
    gr = H.gpu_bwd(inp, want_dh0=inp.h0 is not None, l2=l2)
    H.check_bwd(inp, gr, H.oracle_bwd(inp, l2=l2), tol["bwd"])


CASES = [
    ("pages_benchmark_shape", dict(B=1, T=73, H=1, HV=2, K=64, V=64, cu_seqlens=[0, 3, 73])),
    ("dense_K64", dict(B=2, T=200, H=2, HV=2, K=64, V=64)),
    ("varlen_gva_K64", dict(B=1, T=400, H=2, HV=4, K=64, V=64, cu_seqlens=[0, 0, 3, 190, 190, 333])),
    ("K64_V128", dict(B=1, T=300, H=2, HV=4, K=64, V=128, cu_seqlens=[0, 100, 100, 300])),
    ("K128_V64", dict(B=1, T=300, H=2, HV=2, K=128, V=64, cu_seqlens=[0, 130, 300])),
    ("no_state_K64", dict(B=2, T=130, H=1, HV=1, K=64, V=64, h0=False, final_state=False)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_head_dims_against_the_oracle(name, kw):
    _full(inputs.make_inputs(dtype=torch.bfloat16, seed=zlib.crc32(name.encode()) % 1000, name=name, **kw))


def _unnormalised(inp, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    for name in ("q", "k"):
        x = getattr(inp, name)
        f = torch.from_numpy(np.exp(rng.normal(0.0, 0.7, size=x.shape[:-1] + (1,))))
        setattr(inp, name, (x.to(torch.float64) * f).to(inp.dtype))
    return inp


@pytest.mark.parametrize("hv", [2, 4], ids=["fused_norm_bwd", "gva_partials"])
def test_head_dim_64_with_l2norm_prologue(hv):
    inp = inputs.make_inputs(B=1, T=300, H=2, HV=hv, K=64, V=64, dtype=torch.bfloat16, seed=91 + hv,
                             cu_seqlens=[0, 0, 130, 300], name="k64_l2")
    _full(_unnormalised(inp, 92), l2=True)


def test_head_dim_64_scalar_gate_and_kda_gate():
    _full(inputs.make_inputs(B=1, T=300, H=2, HV=4, K=64, V=64, dtype=torch.bfloat16, seed=93,
                             cu_seqlens=[0, 120, 120, 300], scalar_gate=True, name="k64_sg"))
    _full(inputs.make_inputs(B=1, T=300, H=2, HV=4, K=64, V=64, dtype=torch.bfloat16, seed=94,
                             cu_seqlens=[0, 120, 120, 300], raw_gate=True, lower_bound=-5.0, name="k64_gate"))


def test_head_dim_64_wide_decays_exact_path():
    inp = inputs.make_inputs(B=1, T=300, H=2, HV=4, K=64, V=64, dtype=torch.bfloat16, seed=95,
                             cu_seqlens=[0, 120, 120, 300], g_mean=16.0, g_std=4.0, g_lo=-60.0, name="k64_wide")
    sf, sb = [], []
    tol = H.TOL[inp.dtype]
    o, hT = H.gpu_fwd(inp, status=sf)
    ro, rhT = H.oracle_fwd(inp)
    H.check_fwd(inp, o, hT, ro, rhT, tol["fwd"])
    gr = H.gpu_bwd(inp, status=sb)
    H.check_bwd(inp, gr, H.oracle_bwd(inp), tol["bwd"])
    assert sf[3] > 0 and sb[4] > 0


def test_head_dim_64_context_pair_is_bitwise_the_recompute_pair():
    inp = inputs.make_inputs(B=1, T=300, H=2, HV=4, K=64, V=64, dtype=torch.bfloat16, seed=96,
                             cu_seqlens=[0, 0, 130, 300], name="k64_ctx")
    o, hT, grads, nctx = H.gpu_fwd_bwd_ctx(inp)
    assert nctx > 0
    o2, h2 = H.gpu_fwd(inp)
    g2 = H.gpu_bwd(inp)
    assert torch.equal(o.cpu(), o2) and torch.equal(hT.cpu(), h2)
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert torch.equal(grads[0][key].cpu(), g2[key]), key


def test_dense_training_shape_at_head_dim_64_sampled():
    inp = inputs.make_inputs(B=8, T=4096, H=32, HV=32, K=64, V=64, dtype=torch.bfloat16, seed=97, h0=False,
                             final_state=False, name="dense_train_K64")
    assert _on_tensor_cores(inp)
    tol = H.TOL[inp.dtype]
    o, _ = H.gpu_fwd(inp)
    gr = H.gpu_bwd(inp, want_dh0=False)
    flat = lambda x: x.reshape(inp.B * inp.T, *x.shape[2:])  # noqa: E731
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.isfinite(gr[key]).all(), key
    for n, hq, js, t0, t1, (ro, _), rg in H.sample_units(inp, [(0, 0), (7, 21)]):
        H.assert_rel(f"o[{n},{hq}]", flat(o)[t0:t1][:, js].double().numpy(), ro[0], tol["fwd"])
        for key in ("dq", "dk"):
            H.assert_rel(f"{key}[{n},{hq}]", flat(gr[key])[t0:t1, hq:hq + 1].double().numpy(), rg[key][0], tol["bwd"])
        for key in ("dv", "dg", "dbeta"):
            H.assert_rel(f"{key}[{n},{hq}]", flat(gr[key])[t0:t1][:, js].double().numpy(), rg[key][0], tol["bwd"])
