"""Context parallelism on one GPU: two ranks emulated by two host threads (each
enqueues its own kernels; no kernel waits on another, the exchange is a host
barrier), the sequences split between them.  The relayed forward and backward
must match the oracle on the unsplit sequences."""
import threading

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_42_gb300 import cp, inputs
from tests import kda_gpu_helpers as Hh

pytestmark = pytest.mark.gpu


class ThreadGather:
    """all-gather between host threads (one per emulated rank)."""

    def __init__(self, world):
        self.world = world
        self.slots = [None] * world
        self.bar = threading.Barrier(world)

    def for_rank(self, rank):
        def gather(x):
            torch.cuda.synchronize()
            self.slots[rank] = x
            self.bar.wait()
            out = list(self.slots)
            self.bar.wait()
            return out
        return gather


@pytest.mark.parametrize("name,kw,dtype,split", [
    ("bf16_tc", dict(B=2, T=300, H=2, HV=4, K=128, V=128), torch.bfloat16, 130),
    ("fp32_small", dict(B=1, T=150, H=1, HV=2, K=64, V=48), torch.float32, 64),
], ids=["bf16_tc", "fp32_small"])
@pytest.mark.parametrize("keep", [True, False], ids=["kept_context", "recompute"])
def test_state_relay_two_emulated_ranks(name, kw, dtype, split, keep):
    inp = inputs.make_inputs(dtype=dtype, seed=77, name=name, **kw)
    d = inp.to("cuda")
    world = 2
    segs = [slice(0, split), slice(split, inp.T)]
    tg = ThreadGather(world)
    res = [None] * world
    errors = []

    def rank_fn(rank):
        try:
            s = segs[rank]
            q, k, v, g, beta, do = (x[:, s].contiguous() for x in (d.q, d.k, d.v, d.g, d.beta, d.do))
            gather = tg.for_rank(rank)
            o, hT, seg = cp.cp_forward(q, k, v, g, beta, d.h0 if rank == 0 else None, rank, gather,
                                       keep_context=keep)
            # kept: the backward reuses M and the forward context; else it gets the start state alone
            grads = cp.cp_backward(q, k, v, g, beta, seg if keep else seg.h_start, do,
                                   d.dhT if rank == world - 1 else None, rank, world, gather)
            torch.cuda.synchronize()
            res[rank] = (o.cpu(), hT.cpu(), [t.cpu() for t in grads])
        except Exception as e:  # surfaced after the join
            errors.append(e)
            tg.bar.abort()

    ths = [threading.Thread(target=rank_fn, args=(r,)) for r in range(world)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    assert not errors, errors
    ro, rhT = Hh.oracle_fwd(inp)
    rg = Hh.oracle_bwd(inp)
    tol = Hh.TOL[dtype]
    o = torch.cat([res[0][0], res[1][0]], dim=1)
    Hh.assert_rel("o", o.to(torch.float64).numpy(), ro, tol["fwd"])
    Hh.assert_rel("hT", res[1][1].numpy(), rhT, tol["fwd"])
    for idx, key in enumerate(("dq", "dk", "dv", "dg", "dbeta")):
        got = torch.cat([res[0][2][idx], res[1][2][idx]], dim=1)
        Hh.assert_rel(key, got.to(torch.float64).numpy(), rg[key], tol["bwd"])
    Hh.assert_rel("dh0", res[0][2][5].numpy(), rg["dh0"], tol["bwd"])


def _run_ranks(d, inp, segs, keep=True):
    world = len(segs)
    tg = ThreadGather(world)
    res = [None] * world
    errors = []

    def rank_fn(rank):
        try:
            s = segs[rank]
            q, k, v, g, beta, do = (x[:, s].contiguous() for x in (d.q, d.k, d.v, d.g, d.beta, d.do))
            gather = tg.for_rank(rank)
            o, hT, seg = cp.cp_forward(q, k, v, g, beta, d.h0 if rank == 0 else None, rank, gather,
                                       keep_context=keep)
            grads = cp.cp_backward(q, k, v, g, beta, seg if keep else seg.h_start, do,
                                   d.dhT if rank == world - 1 else None, rank, world, gather)
            torch.cuda.synchronize()
            res[rank] = (o.cpu(), hT.cpu(), [t.cpu() for t in grads])
        except Exception as e:  # surfaced after the join
            errors.append(e)
            tg.bar.abort()

    ths = [threading.Thread(target=rank_fn, args=(r,)) for r in range(world)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    assert not errors, errors
    return res


def test_state_relay_two_ranks_long_context_sampled():
    """The long-context workload (T = 65,536, H = HV = 16, near-1 decays) split
    between two emulated ranks; the oracle checks sampled value heads of the
    unsplit sequence at the bf16 tolerances."""
    inp = inputs.make_config(3)
    d = inp.to("cuda")
    half = inp.T // 2
    res = _run_ranks(d, inp, [slice(0, half), slice(half, inp.T)])
    tol = Hh.TOL[inp.dtype]
    for n, hq, js, t0, t1, (ro, rhT), rg in Hh.sample_units(inp, [(0, 3)]):
        o = torch.cat([res[0][0], res[1][0]], dim=1)[0]
        Hh.assert_rel("o", o[t0:t1][:, js].double().numpy(), ro[0], tol["fwd"])
        Hh.assert_rel("hT", res[1][1][n][js].double().numpy(), rhT[0], tol["fwd"])
        for idx, key in enumerate(("dq", "dk", "dv", "dg", "dbeta")):
            got = torch.cat([res[0][2][idx], res[1][2][idx]], dim=1)[0]
            got = got[t0:t1, hq:hq + 1] if key in ("dq", "dk") else got[t0:t1][:, js]
            Hh.assert_rel(key, got.double().numpy(), rg[key][0], tol["bwd"])
        Hh.assert_rel("dh0", res[0][2][5][n][js].double().numpy(), rg["dh0"][0], tol["bwd"])


@pytest.mark.parametrize("K,V", [(128, 128), (64, 48), (3, 5)])
@pytest.mark.parametrize("transpose", [False, True])
def test_state_compose_matches_fp64(K, V, transpose):
    rng = np.random.default_rng(K * 1000 + V + transpose)
    M = rng.standard_normal((3, 2, K, K))
    h = rng.standard_normal((3, 2, K, V))
    c = rng.standard_normal((3, 2, K, V))
    dev = lambda x: torch.from_numpy(x).float().cuda()  # noqa: E731
    out = cp.compose(dev(M), dev(h), dev(c), transpose).cpu().double().numpy()
    Mf, hf, cf = (torch.from_numpy(x).float().double().numpy() for x in (M, h, c))
    ref = (np.swapaxes(Mf, -1, -2) if transpose else Mf) @ hf + cf
    assert oracle.rel_rms(out, ref) < 1e-6
    out0 = cp.compose(dev(M), dev(h), None, transpose).cpu().double().numpy()
    assert oracle.rel_rms(out0, ref - cf) < 1e-6
