"""GPU parity of the KDA gate inside the op (KDA_GATE_IN_KERNEL): g holds the raw
gate pre-activations and the op makes the per-token log2 decay itself,
unbounded (-exp(A_log) softplus(a + bias)) or bounded (lower_bound
sigmoid(exp(A_log) (a + bias))); the backward returns the gradient of the raw
gate and the fp32 sums dA_log, dbias.  Checked against the fp64 oracle
(oracle.kda_gate composed with the recurrence) at the usual tolerances, with the
omitted-A_log contract of "[Fix] Use unit KDA gate scale when A_log is omitted"
checked bitwise."""
import zlib

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


VARLEN_GVA = dict(B=1, T=400, H=2, HV=4, K=128, V=128, cu_seqlens=[0, 0, 3, 190, 190, 400])

CASES = [
    ("tc_unbounded", VARLEN_GVA, torch.bfloat16, None, {}),
    ("tc_bounded", VARLEN_GVA, torch.bfloat16, -5.0, {}),
    ("tc_no_A_log_no_bias", dict(B=2, T=150, H=2, HV=2, K=128, V=128), torch.bfloat16, None,
     dict(A_log=False, g_bias=False)),
    ("tc_bounded_no_bias", dict(B=2, T=150, H=2, HV=2, K=128, V=128), torch.bfloat16, -3.0, dict(g_bias=False)),
    ("fp32_unbounded", dict(B=1, T=130, H=1, HV=2, K=64, V=48, cu_seqlens=[0, 50, 50, 130]), torch.float32,
     None, {}),
    ("fp32_bounded", dict(B=2, T=70, H=1, HV=1, K=32, V=32), torch.float32, -4.0, {}),
]


def _inp(name, kw, dtype, lb, extra, seed=None, **more):
    return inputs.make_inputs(dtype=dtype, seed=zlib.crc32(name.encode()) % 1000 if seed is None else seed,
                              name=name, raw_gate=True, lower_bound=lb, **kw, **extra, **more)


def _param_sum_scales(inp):
    """Sum over the terms of dA_log (per value head) and of dbias (per value head
    and channel) of |dL/dg * dg/dparameter|: what an fp32 error in each per-token
    gradient can add up to in these sums over every token.  The derivatives of
    the gate are central differences of oracle.kda_gate, dL/dg the oracle's
    gradient w.r.t. the decay."""
    import numpy as np
    import oracle
    gate = inp.gate
    f = inp.f64()
    a = f["g"]
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
    geff = oracle.kda_gate(a, **gate)
    dg = oracle.kda_bwd(f["q"], f["k"], f["v"], geff, f["beta"], f["h0"], f["do"], f["dhT"], cu)["dg"]
    h = 1e-6
    ddx = (oracle.kda_gate(a + h, **gate) - oracle.kda_gate(a - h, **gate)) / (2 * h)
    A = np.zeros(inp.HV) if gate["A_log"] is None else gate["A_log"]
    dA = (oracle.kda_gate(a, **dict(gate, A_log=A + h)) - oracle.kda_gate(a, **dict(gate, A_log=A - h))) / (2 * h)
    return np.sum(np.abs(dg * dA), axis=(0, 1, 3)), np.sum(np.abs(dg * ddx), axis=(0, 1))


@pytest.mark.parametrize("name,kw,dtype,lb,extra", CASES, ids=[c[0] for c in CASES])
def test_kda_gate_against_the_oracle(name, kw, dtype, lb, extra):
    """Every output at the usual tolerances.  On the fp32 path, dA_log and dbias
    (sums over every valid token, whose terms can cancel) are held to 1e-5 of the
    sum of their terms' magnitudes instead: the bound that fp32 per-token
    gradients give such a sum."""
    import numpy as np
    inp = _inp(name, kw, dtype, lb, extra)
    tol = H.TOL[dtype]
    o, hT = H.gpu_fwd(inp)
    ro, rhT = H.oracle_fwd(inp)
    H.check_fwd(inp, o, hT, ro, rhT if inp.output_final_state else None, tol["fwd"])
    gr = H.gpu_bwd(inp, want_dh0=inp.h0 is not None)
    assert (gr["dA_log"] is None) == (inp.A_log is None) and (gr["dbias"] is None) == (inp.g_bias is None)
    ref = H.oracle_bwd(inp)
    if dtype == torch.float32:
        sA, sb = _param_sum_scales(inp)
        for key, scale in (("dA_log", sA), ("dbias", sb)):
            if gr[key] is not None:
                err = np.abs(gr.pop(key).double().numpy() - ref[key])
                assert np.all(err <= tol["bwd"] * scale), (key, float(np.max(err / scale)))
    H.check_bwd(inp, gr, ref, tol["bwd"])


@pytest.mark.parametrize("lb", [None, -5.0], ids=["unbounded", "bounded"])
def test_omitted_A_log_equals_zero_A_log_bitwise(lb):
    """An omitted A_log is the same unit scale as an explicit zero A_log, bit for bit."""
    a = _inp("omitted", VARLEN_GVA, torch.bfloat16, lb, dict(A_log=False), seed=81)
    z = _inp("omitted", VARLEN_GVA, torch.bfloat16, lb, dict(A_log=False), seed=81)
    z.A_log = torch.zeros(z.HV, dtype=torch.float32)
    oa, ha = H.gpu_fwd(a)
    oz, hz = H.gpu_fwd(z)
    assert torch.equal(oa, oz) and torch.equal(ha, hz)
    ga, gz = H.gpu_bwd(a), H.gpu_bwd(z)
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dh0", "dbias"):
        assert torch.equal(ga[key], gz[key]), key


def test_kda_gate_recompute_and_context_pairs_agree_bitwise():
    inp = _inp("pairs", VARLEN_GVA, torch.bfloat16, None, {}, seed=82)
    d = inp.to("cuda")
    from gated_delta_rule_42_gb300.ops import chunk_kda_bwd, chunk_kda_bwd_ctx, chunk_kda_fwd_ctx
    gp = H.gate_params(d)
    o, hT, kctx = chunk_kda_fwd_ctx(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, True, gate=gp)
    a = chunk_kda_bwd_ctx(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, kctx, d.do, d.dhT, gate=gp)
    b = chunk_kda_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, d.do, d.dhT, gate=gp)
    m = torch.from_numpy(H.valid_mask(inp)).cuda()
    for i, (x, y) in enumerate(zip(a, b)):
        if x.dim() >= 3 and x.shape[1] == inp.T:  # per-token gradients: the valid tokens
            x, y = x.reshape(inp.B * inp.T, -1)[m], y.reshape(inp.B * inp.T, -1)[m]
        assert torch.equal(x, y), i


@pytest.mark.parametrize("lb", [None, -5.0], ids=["unbounded", "bounded"])
def test_kda_gate_recurrent(lb):
    inp = _inp("recurrent", dict(B=1, T=200, H=2, HV=4, K=128, V=128, cu_seqlens=[0, 0, 80, 80, 200]),
               torch.float32, lb, {}, seed=83)
    o, hT = H.gpu_recurrent(inp)
    ro, rhT = H.oracle_fwd(inp)
    H.check_fwd(inp, o, hT, ro, rhT, H.TOL[torch.float32]["fwd"])


def test_kda_gate_strong_scale_takes_the_exact_path():
    """A large A_log makes the decays strong enough for the exact-path fix-up
    launches (status words 3 and 4), which apply the gate as well."""
    inp = _inp("strong", VARLEN_GVA, torch.bfloat16, None, {}, seed=84, g_mean=2.0)
    inp.A_log = torch.full((inp.HV,), 2.7, dtype=torch.float32)  # scale ~15: spans of ~200
    sf, sb = [], []
    tol = H.TOL[inp.dtype]
    o, hT = H.gpu_fwd(inp, status=sf)
    ro, rhT = H.oracle_fwd(inp)
    H.check_fwd(inp, o, hT, ro, rhT, tol["fwd"])
    gr = H.gpu_bwd(inp, status=sb)
    H.check_bwd(inp, gr, H.oracle_bwd(inp), tol["bwd"])
    assert sf[3] > 0 and sb[4] > 0, (sf, sb)


def test_chunk_kda_autograd_reaches_the_gate_parameters():
    """chunk_kda(use_gate_in_kernel=True) returns the same gradients as the C ABI,
    including those of A_log and the bias."""
    from gated_delta_rule_42_gb300 import chunk_kda
    inp = _inp("autograd", VARLEN_GVA, torch.bfloat16, -5.0, {}, seed=85)
    d = inp.to("cuda")
    leaves = [t.clone().requires_grad_(True) for t in (d.q, d.k, d.v, d.g, d.beta, d.h0, d.A_log, d.g_bias)]
    q, k, v, g, beta, h0, A_log, bias = leaves
    o, hT = chunk_kda(q, k, v, g, beta, h0, cu_seqlens=d.cu_seqlens, output_final_state=True,
                      use_gate_in_kernel=True, A_log=A_log, g_bias=bias, lower_bound=-5.0)
    torch.autograd.backward([o, hT], [d.do, d.dhT])
    gr = H.gpu_bwd(inp)
    m = torch.from_numpy(H.valid_mask(inp))
    for t, key in zip(leaves, ("dq", "dk", "dv", "dg", "dbeta", "dh0", "dA_log", "dbias")):
        got, want = t.grad.cpu(), gr[key]
        if key in ("dq", "dk", "dv", "dg", "dbeta"):
            got, want = got.reshape(inp.T, -1)[m], want.reshape(inp.T, -1)[m]
        assert torch.equal(got, want), key


@pytest.mark.parametrize("hv,lb", [(2, None), (4, -5.0)], ids=["fused_norm_bwd_unbounded", "gva_partials_bounded"])
def test_kda_gate_with_l2norm_prologue(hv, lb):
    """The KDA gate and the q/k L2-norm prologue together, on raw (unnormalised)
    q, k rows: with HV = H the norm's backward is fused into the gradient kernel,
    with HV > H it runs on the per-value-head partials afterwards."""
    import numpy as np
    inp = _inp("gate_l2", dict(B=1, T=300, H=2, HV=hv, K=128, V=128, cu_seqlens=[0, 0, 130, 300]), torch.bfloat16,
               lb, {}, seed=86 + hv)
    rng = np.random.default_rng(87)
    for name in ("q", "k"):  # rows of norm e^N(0, 0.7): the prologue has something to undo
        x = getattr(inp, name)
        f = torch.from_numpy(np.exp(rng.normal(0.0, 0.7, size=x.shape[:-1] + (1,))))
        setattr(inp, name, (x.to(torch.float64) * f).to(inp.dtype))
    tol = H.TOL[inp.dtype]
    o, hT = H.gpu_fwd(inp, l2=True)
    ro, rhT = H.oracle_fwd(inp, l2=True)
    H.check_fwd(inp, o, hT, ro, rhT, tol["fwd"])
    gr = H.gpu_bwd(inp, l2=True)
    H.check_bwd(inp, gr, H.oracle_bwd(inp, l2=True), tol["bwd"])
