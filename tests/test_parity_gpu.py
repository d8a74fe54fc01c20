"""GPU parity: libkda (through its C ABI) against the fp64 oracle on the same
seeded inputs.  Tolerances (relative RMS per output tensor over valid tokens):
fp32 inputs 1e-5; bf16 inputs 5e-3 on o / final state and 1e-2 on gradients.
Empty-slot passthrough and the untouched capacity tail are checked bitwise."""
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


def _full_check(inp):
    tol = H.TOL[inp.dtype]
    o, hT = H.gpu_fwd(inp)
    ro, rhT = H.oracle_fwd(inp)
    ef = H.check_fwd(inp, o, hT, ro, rhT if inp.output_final_state else None, tol["fwd"])
    gr = H.gpu_bwd(inp, want_dh0=inp.h0 is not None)
    ref = H.oracle_bwd(inp)
    eb = H.check_bwd(inp, gr, ref, tol["bwd"])
    return ef, eb


def test_tiny_dense_fp32_config():
    _full_check(inputs.make_config(0))


def test_varlen_gva_bf16_config():
    inp = inputs.make_config(1)
    ef, eb = _full_check(inp)
    print("varlen+GVA bf16", ef, eb)


EDGE = [
    # name, kwargs
    # single-token sequences; several of them, so that the bf16 tensor-core path's relative RMS is
    # over more than one dbeta (one token's dbeta is a sum over V that can cancel, and its bf16
    # intermediates then bound it to about 2^-9 times that sum's condition number)
    ("T1", dict(B=3, T=1, H=1, HV=2, K=64, V=64)),
    ("B2_T65_ragged", dict(B=2, T=65, H=2, HV=2, K=64, V=64)),
    ("gva3_odd_dims", dict(B=1, T=129, H=1, HV=3, K=32, V=48)),
    ("varlen_empty_slots", dict(B=1, T=200, H=2, HV=4, K=64, V=64,
                                cu_seqlens=[0, 0, 63, 63, 64, 200, 200])),
    ("capacity_tail", dict(B=1, T=100, H=1, HV=2, K=64, V=64, cu_seqlens=[0, 5, 70])),
    ("K128_V128", dict(B=1, T=130, H=1, HV=1, K=128, V=128)),
    ("no_state", dict(B=2, T=70, H=1, HV=1, K=64, V=64, h0=False, final_state=False)),
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("name,kw", EDGE, ids=[e[0] for e in EDGE])
def test_edge_cases(name, kw, dtype):
    inp = inputs.make_inputs(dtype=dtype, seed=zlib.crc32(name.encode()) % 1000, name=name, **kw)
    _full_check(inp)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_recurrent_against_oracle(dtype):
    inp = inputs.make_inputs(B=1, T=300, H=2, HV=4, K=128, V=128, dtype=dtype, seed=11,
                             cu_seqlens=[0, 0, 100, 100, 300])
    o, hT = H.gpu_recurrent(inp)
    ro, rhT = H.oracle_fwd(inp)
    H.check_fwd(inp, o, hT, ro, rhT, H.TOL[dtype]["fwd"])


def test_recurrent_matches_chunked_fp32():
    inp = inputs.make_inputs(B=2, T=150, H=1, HV=2, K=64, V=64, dtype=torch.float32, seed=12)
    o1, h1 = H.gpu_recurrent(inp)
    o2, h2 = H.gpu_fwd(inp)
    assert H.oracle.rel_rms(o1.double().numpy(), o2.double().numpy()) < 1e-5
    assert H.oracle.rel_rms(h1.double().numpy(), h2.double().numpy()) < 1e-5


@pytest.mark.parametrize("cfg,units", [
    (2, [(0, 0), (7, 31)]),
    (3, [(0, 5)]),
    (4, [(1, 3), (66, 15)]),
], ids=["dense_train", "long_ctx", "packed_varlen"])
def test_full_size_sampled(cfg, units):
    """Full-size configs: the GPU computes everything; the oracle checks
    sampled (sequence, q/k head) units, and every output must be finite."""
    inp = inputs.make_config(cfg)
    tol = H.TOL[inp.dtype]
    o, hT = H.gpu_fwd(inp)
    gr = H.gpu_bwd(inp, want_dh0=inp.h0 is not None)
    m = H.valid_mask(inp)
    assert torch.isfinite(o.reshape(inp.B * inp.T, -1)[torch.from_numpy(m)]).all()
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.isfinite(gr[key].reshape(inp.B * inp.T, -1)[torch.from_numpy(m)]).all(), key
    for n in H.empty_slots(inp):
        assert torch.equal(hT[n], inp.h0[n]) and torch.equal(gr["dh0"][n], inp.dhT[n])
    flat = lambda x: x.reshape(inp.B * inp.T, *x.shape[2:])
    for n, hq, js, t0, t1, (ro, rhT), rg in H.sample_units(inp, units):
        H.assert_rel(f"o[{n},{hq}]", flat(o)[t0:t1][:, js].double().numpy(), ro[0], tol["fwd"])
        if hT is not None:
            H.assert_rel(f"hT[{n},{hq}]", hT[n][js].double().numpy(), rhT[0], tol["fwd"])
        H.assert_rel(f"dq[{n},{hq}]", flat(gr["dq"])[t0:t1, hq:hq + 1].double().numpy(), rg["dq"][0], tol["bwd"])
        H.assert_rel(f"dk[{n},{hq}]", flat(gr["dk"])[t0:t1, hq:hq + 1].double().numpy(), rg["dk"][0], tol["bwd"])
        H.assert_rel(f"dv[{n},{hq}]", flat(gr["dv"])[t0:t1][:, js].double().numpy(), rg["dv"][0], tol["bwd"])
        H.assert_rel(f"dg[{n},{hq}]", flat(gr["dg"])[t0:t1][:, js].double().numpy(), rg["dg"][0], tol["bwd"])
        H.assert_rel(f"dbeta[{n},{hq}]", flat(gr["dbeta"])[t0:t1][:, js].double().numpy(), rg["dbeta"][0], tol["bwd"])
        if gr["dh0"] is not None:
            H.assert_rel(f"dh0[{n},{hq}]", gr["dh0"][n][js].double().numpy(), rg["dh0"][0], tol["bwd"])


def test_autograd_wrapper_matches_c_abi():
    """chunk_kda (torch.autograd.Function over the same C ABI) returns exactly
    what the direct C-ABI calls return."""
    from gated_delta_rule_42_gb300 import chunk_kda
    inp = inputs.make_inputs(B=1, T=200, H=2, HV=4, K=64, V=64, dtype=torch.bfloat16, seed=5,
                             cu_seqlens=[0, 50, 50, 200])
    d = inp.to("cuda")
    leaves = [t.clone().requires_grad_(True) for t in (d.q, d.k, d.v, d.g, d.beta, d.h0)]
    o, hT = chunk_kda(*leaves, cu_seqlens=d.cu_seqlens, output_final_state=True)
    torch.autograd.backward([o, hT], [d.do, d.dhT])
    o2, hT2 = H.gpu_fwd(inp)
    assert torch.equal(o.detach().cpu(), o2) and torch.equal(hT.detach().cpu(), hT2)
    gr = H.gpu_bwd(inp)
    for t, key in zip(leaves, ("dq", "dk", "dv", "dg", "dbeta", "dh0")):
        assert torch.equal(t.grad.cpu(), gr[key]), key


def test_cuda_graph_replay_with_mutated_offsets():
    """The chunk map runs on the device, so a captured forward replays
    correctly after the offsets buffer is overwritten in place."""
    from gated_delta_rule_42_gb300.ops import chunk_kda_fwd
    inp = inputs.make_inputs(B=1, T=256, H=1, HV=2, K=64, V=64, dtype=torch.bfloat16, seed=21,
                             cu_seqlens=[0, 100, 256])
    d = inp.to("cuda")
    ws = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")
    chunk_kda_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, True, workspace=ws)  # warm-up
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            o, hT = chunk_kda_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, True, workspace=ws)
    for cu in ([0, 100, 256], [0, 3, 256], [0, 256, 256]):
        d.cu_seqlens.copy_(torch.tensor(cu, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        ref_inp = inputs.make_inputs(B=1, T=256, H=1, HV=2, K=64, V=64, dtype=torch.bfloat16,
                                     seed=21, cu_seqlens=[0, 100, 256])
        ref_inp.cu_seqlens = torch.tensor(cu, dtype=torch.int32)
        ro, rhT = H.oracle_fwd(ref_inp)
        H.check_fwd(ref_inp, o.cpu(), hT.cpu(), ro, rhT, H.TOL[torch.bfloat16]["fwd"])


def test_backward_is_bitwise_deterministic():
    inp = inputs.make_inputs(B=1, T=300, H=2, HV=4, K=128, V=128, dtype=torch.bfloat16, seed=9,
                             cu_seqlens=[0, 130, 130, 300])
    a = H.gpu_bwd(inp)
    b = H.gpu_bwd(inp)
    for key in a:
        assert torch.equal(a[key], b[key]), key


# ---- the q/k L2-norm prologue (KDA_QK_L2NORM) ----

def _unnormalised(inp, seed):
    """q and k rows rescaled by seeded positive factors (the generator's rows
    are unit-norm, which would hide the prologue)."""
    rng = np.random.default_rng(seed)
    for name in ("q", "k"):
        x = getattr(inp, name)
        f = torch.from_numpy(np.exp(rng.normal(0.0, 0.7, size=x.shape[:-1] + (1,))))
        setattr(inp, name, (x.to(torch.float64) * f).to(inp.dtype))
    return inp


L2 = [
    ("tc_dense", dict(B=2, T=130, H=2, HV=2, K=128, V=128), torch.bfloat16),
    ("tc_varlen_gva", dict(B=1, T=300, H=2, HV=4, K=128, V=128, cu_seqlens=[0, 0, 100, 100, 300]),
     torch.bfloat16),
    ("tc_varlen_fused", dict(B=1, T=300, H=2, HV=2, K=128, V=128, cu_seqlens=[0, 0, 100, 100, 300]),
     torch.bfloat16),  # HV = H: the norm's backward inside the gradient kernel
    ("fp32_gva_odd", dict(B=1, T=129, H=1, HV=3, K=32, V=48), torch.float32),
    ("bf16_small_dims", dict(B=2, T=70, H=2, HV=2, K=64, V=64), torch.bfloat16),
    ("fp32_k128", dict(B=1, T=90, H=1, HV=2, K=128, V=64), torch.float32),
]


@pytest.mark.parametrize("name,kw,dtype", L2, ids=[e[0] for e in L2])
def test_qk_l2norm_prologue(name, kw, dtype):
    inp = _unnormalised(inputs.make_inputs(dtype=dtype, seed=zlib.crc32(name.encode()) % 1000, name=name, **kw),
                        seed=zlib.crc32(name.encode()) % 997)
    tol = H.TOL[dtype]
    o, hT = H.gpu_fwd(inp, l2=True)
    ro, rhT = H.oracle_fwd(inp, l2=True)
    H.check_fwd(inp, o, hT, ro, rhT if inp.output_final_state else None, tol["fwd"])
    gr = H.gpu_bwd(inp, want_dh0=inp.h0 is not None, l2=True)
    H.check_bwd(inp, gr, H.oracle_bwd(inp, l2=True), tol["bwd"])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_qk_l2norm_recurrent(dtype):
    inp = _unnormalised(inputs.make_inputs(B=1, T=200, H=2, HV=4, K=128, V=128, dtype=dtype, seed=13,
                                           cu_seqlens=[0, 0, 80, 80, 200]), seed=14)
    o, hT = H.gpu_recurrent(inp, l2=True)
    ro, rhT = H.oracle_fwd(inp, l2=True)
    H.check_fwd(inp, o, hT, ro, rhT, H.TOL[dtype]["fwd"])


# ---- the scalar-gate (GDN) variant (KDA_SCALAR_GATE: g, dg [B, T, HV]) ----

SG = [
    ("tc_dense", dict(B=2, T=130, H=2, HV=2, K=128, V=128), torch.bfloat16, False),
    ("tc_varlen_gva_l2norm", dict(B=1, T=300, H=2, HV=4, K=128, V=128, cu_seqlens=[0, 0, 100, 100, 250]),
     torch.bfloat16, True),
    ("tc_dense_l2norm", dict(B=1, T=200, H=2, HV=2, K=128, V=128), torch.bfloat16, True),  # fused norm backward
    ("fp32_gva_odd", dict(B=1, T=129, H=1, HV=3, K=32, V=48), torch.float32, False),
]


@pytest.mark.parametrize("name,kw,dtype,l2", SG, ids=[e[0] for e in SG])
def test_scalar_gate(name, kw, dtype, l2):
    inp = inputs.make_inputs(dtype=dtype, seed=zlib.crc32(name.encode()) % 1000, name="sg_" + name,
                             scalar_gate=True, **kw)
    if l2:
        inp = _unnormalised(inp, seed=5)
    assert inp.g.dim() == 3
    tol = H.TOL[dtype]
    o, hT = H.gpu_fwd(inp, l2=l2)
    ro, rhT = H.oracle_fwd(inp, l2=l2)
    H.check_fwd(inp, o, hT, ro, rhT if inp.output_final_state else None, tol["fwd"])
    gr = H.gpu_bwd(inp, want_dh0=inp.h0 is not None, l2=l2)
    H.check_bwd(inp, gr, H.oracle_bwd(inp, l2=l2), tol["bwd"])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_scalar_gate_recurrent(dtype):
    inp = inputs.make_inputs(B=1, T=200, H=2, HV=4, K=128, V=128, dtype=dtype, seed=15,
                             cu_seqlens=[0, 0, 80, 80, 200], scalar_gate=True)
    o, hT = H.gpu_recurrent(inp)
    ro, rhT = H.oracle_fwd(inp)
    H.check_fwd(inp, o, hT, ro, rhT, H.TOL[dtype]["fwd"])


def _misaligned(t):
    """A device copy of t whose data starts one element past a 256-byte boundary."""
    buf = torch.empty(t.numel() + 16, dtype=t.dtype, device="cuda")
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def test_misaligned_bf16_inputs_run_the_general_kernels():
    """bf16 K = V = 128 inputs that are not 16-byte aligned cannot use the TMA
    kernels: the general kernels run instead, with the same results."""
    import ctypes
    from gated_delta_rule_42_gb300 import _lib
    from gated_delta_rule_42_gb300.ops import make_inputs_struct
    inp = inputs.make_inputs(B=1, T=150, H=1, HV=2, K=128, V=128, dtype=torch.bfloat16, seed=23, name="misaligned")
    lib = _lib.load()
    q, k, v, g = (_misaligned(x) for x in (inp.q, inp.k, inp.v, inp.g))
    beta, h0 = inp.beta.cuda(), inp.h0.cuda()
    assert (q.data_ptr() & 15) != 0
    s = make_inputs_struct(q, k, v, g, beta, h0, None)
    o = torch.full(v.shape, float("nan"), dtype=v.dtype, device="cuda")
    hT = torch.empty((s.N, s.HV, 128, 128), dtype=torch.float32, device="cuda")
    need = lib.kda_chunk_fwd_workspace_size(ctypes.byref(s))
    ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    wp = ctypes.c_void_p((ws.data_ptr() + 255) & ~255)
    _lib.check(lib, lib.kda_chunk_fwd(ctypes.byref(s), ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(hT.data_ptr()),
                                      wp, need, None))
    torch.cuda.synchronize()
    ro, rhT = H.oracle_fwd(inp)
    H.check_fwd(inp, o.cpu(), hT.cpu(), ro, rhT, H.TOL[torch.bfloat16]["fwd"])
