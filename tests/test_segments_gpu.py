"""GPU: long sequences split into segments that run at once (segments.py).
The segmented forward and backward match the fp64 oracle on the unsplit
sequences at the usual tolerances (the relay reorders sums, so the match is
to rounding, not bitwise)."""
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


@pytest.mark.parametrize("name,kw,S,l2", [
    ("tc_two_seqs", dict(B=2, T=1024, H=2, HV=4, K=128, V=128, dtype=torch.bfloat16), 4, False),
    ("tc_l2norm", dict(B=1, T=768, H=2, HV=2, K=128, V=128, dtype=torch.bfloat16), 3, True),
    ("fp32_general", dict(B=1, T=512, H=1, HV=2, K=64, V=48, dtype=torch.float32), 2, False),
], ids=["tc_two_seqs", "tc_l2norm", "fp32_general"])
def test_segmented_matches_the_oracle(name, kw, S, l2):
    from gated_delta_rule_42_gb300.segments import chunk_kda_bwd_segmented, chunk_kda_fwd_segmented
    inp = inputs.make_inputs(seed=71, name=name, **kw)
    d = inp.to("cuda")
    o, hT, ctx = chunk_kda_fwd_segmented(d.q, d.k, d.v, d.g, d.beta, d.h0, S, True, use_qk_l2norm=l2)
    dq, dk, dv, dg, db, dh0 = chunk_kda_bwd_segmented(d.q, d.k, d.v, d.g, d.beta, ctx, d.do, d.dhT,
                                                      use_qk_l2norm=l2)
    torch.cuda.synchronize()
    tol = H.TOL[inp.dtype]
    ro, rhT = H.oracle_fwd(inp, l2=l2)
    H.check_fwd(inp, o.cpu(), hT.cpu(), ro, rhT, tol["fwd"])
    gr = dict(dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu(), dg=dg.cpu(), dbeta=db.cpu(), dh0=dh0.cpu())
    H.check_bwd(inp, gr, H.oracle_bwd(inp, l2=l2), tol["bwd"])


def test_chunk_kda_autograd_with_segments():
    """chunk_kda(segments=S) trains through the segmented path: its gradients
    match the unsplit autograd path to rounding."""
    from gated_delta_rule_42_gb300 import chunk_kda
    inp = inputs.make_inputs(B=1, T=512, H=2, HV=2, K=128, V=128, dtype=torch.bfloat16, seed=72, name="seg_autograd")
    d = inp.to("cuda")
    outs = []
    for S in (1, 4):
        leaves = [t.clone().requires_grad_(True) for t in (d.q, d.k, d.v, d.g, d.beta, d.h0)]
        o, hT = chunk_kda(*leaves, output_final_state=True, segments=S)
        torch.autograd.backward([o, hT], [d.do, d.dhT])
        outs.append([o.detach().float()] + [t.grad.float() for t in leaves])
    for name, a, b in zip(("o", "dq", "dk", "dv", "dg", "dbeta", "dh0"), outs[0], outs[1]):
        rel = ((a - b).norm() / b.norm()).item()
        assert rel < 1e-2, (name, rel)


def test_long_context_sixteen_segments_sampled():
    """The long-context workload (T = 65,536, H = HV = 16, near-1 decays) split
    into 16 segments: 15 state compositions in each direction, with the
    transitions on the bf16 tensor-core path.  The oracle checks sampled value
    heads of the unsplit sequence, at the bf16 tolerances, for o, hT and every
    gradient."""
    from gated_delta_rule_42_gb300.segments import chunk_kda_bwd_segmented, chunk_kda_fwd_segmented
    inp = inputs.make_config(3)
    d = inp.to("cuda")
    o, hT, ctx = chunk_kda_fwd_segmented(d.q, d.k, d.v, d.g, d.beta, d.h0, 16, True)
    dq, dk, dv, dg, db, dh0 = chunk_kda_bwd_segmented(d.q, d.k, d.v, d.g, d.beta, ctx, d.do, d.dhT)
    torch.cuda.synchronize()
    tol = H.TOL[inp.dtype]
    flat = lambda x: x.reshape(inp.B * inp.T, *x.shape[2:]).cpu()  # noqa: E731
    for n, hq, js, t0, t1, (ro, rhT), rg in H.sample_units(inp, [(0, 5), (0, 12)]):
        H.assert_rel(f"o[{hq}]", flat(o)[t0:t1][:, js].double().numpy(), ro[0], tol["fwd"])
        H.assert_rel(f"hT[{hq}]", hT[n][js].cpu().double().numpy(), rhT[0], tol["fwd"])
        for key, x in (("dq", dq), ("dk", dk)):
            H.assert_rel(f"{key}[{hq}]", flat(x)[t0:t1, hq:hq + 1].double().numpy(), rg[key][0], tol["bwd"])
        for key, x in (("dv", dv), ("dg", dg), ("dbeta", db)):
            H.assert_rel(f"{key}[{hq}]", flat(x)[t0:t1][:, js].double().numpy(), rg[key][0], tol["bwd"])
        H.assert_rel(f"dh0[{hq}]", dh0[n][js].cpu().double().numpy(), rg["dh0"][0], tol["bwd"])
