"""GPU: the forward-context pair (kda_chunk_fwd_ctx + kda_chunk_bwd_ctx, the
backward reading the intermediates the forward kept) returns, bit for bit,
what the recompute pair (kda_chunk_fwd + kda_chunk_bwd) returns -- the same
kernels compute the kept tiles either way -- and so inherits its oracle parity;
one case is also checked against the oracle directly.  The context is only
read: a second backward on it gives the same bits."""
import zlib

import pytest
import torch

from gated_delta_rule_42_gb300 import inputs
from tests import kda_gpu_helpers as H

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_42_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _same(name, a, b):
    if a is None or b is None:
        assert a is None and b is None, name
        return
    a, b = a.cpu(), b.cpu()
    assert torch.equal(a.isnan(), b.isnan()), name  # the untouched capacity tail stays poisoned in both
    assert torch.equal(torch.nan_to_num(a), torch.nan_to_num(b)), name


CASES = [
    ("tc_dense_states", dict(B=2, T=130, H=2, HV=2, K=128, V=128), False, True),
    ("tc_varlen_gva_empty", dict(B=1, T=300, H=2, HV=4, K=128, V=128, cu_seqlens=[0, 0, 100, 100, 300]),
     False, True),
    ("tc_l2norm", dict(B=1, T=200, H=1, HV=2, K=128, V=128), True, False),
    ("tc_l2norm_fused", dict(B=1, T=200, H=2, HV=2, K=128, V=128), True, True),
    ("tc_scalar_gate", dict(B=1, T=190, H=2, HV=4, K=128, V=128, scalar_gate=True), False, True),
    ("tc_bf16_k64", dict(B=1, T=150, H=1, HV=2, K=64, V=64), False, True),
    ("general_bf16_k96", dict(B=1, T=150, H=1, HV=2, K=96, V=96), False, True),
    ("general_fp32", dict(B=1, T=100, H=1, HV=2, K=128, V=128, dtype=torch.float32), False, True),
]


@pytest.mark.parametrize("name,kw,l2,states", CASES, ids=[c[0] for c in CASES])
def test_context_pair_matches_recompute_bitwise(name, kw, l2, states):
    kw = dict(kw)
    dtype = kw.pop("dtype", torch.bfloat16)
    extra = {} if states else dict(h0=False, final_state=False)
    inp = inputs.make_inputs(dtype=dtype, seed=zlib.crc32(name.encode()) % 1000, name=name, **kw, **extra)
    want_dh0 = inp.h0 is not None
    o, hT, grads, nctx = H.gpu_fwd_bwd_ctx(inp, l2=l2, want_dh0=want_dh0, backwards=2)
    tc = dtype == torch.bfloat16 and kw["K"] in (64, 128) and kw["V"] in (64, 128)
    assert (nctx > 0) == tc
    o2, hT2 = H.gpu_fwd(inp, l2=l2)
    _same("o", o, o2)
    _same("hT", hT, hT2)
    ref = H.gpu_bwd(inp, want_dh0=want_dh0, l2=l2)
    for key in GRADS:
        _same(key, grads[0][key], ref[key])
        _same(key + " (second backward on the context)", grads[1][key], ref[key])


def test_context_pair_against_oracle():
    inp = inputs.make_inputs(B=1, T=260, H=2, HV=4, K=128, V=128, dtype=torch.bfloat16, seed=31,
                             cu_seqlens=[0, 70, 70, 260], name="ctx_oracle")
    tol = H.TOL[inp.dtype]
    o, hT, grads, _ = H.gpu_fwd_bwd_ctx(inp)
    ro, rhT = H.oracle_fwd(inp)
    H.check_fwd(inp, o.cpu(), hT.cpu(), ro, rhT, tol["fwd"])
    H.check_bwd(inp, {k: (None if v is None else v.cpu()) for k, v in grads[0].items()}, H.oracle_bwd(inp),
                tol["bwd"])


def test_context_pair_full_size_dense_training_layer():
    """B=8, T=4096, H=HV=32, K=V=128 bf16: the benchmark's workload and launch
    configuration, context pair against the recompute pair, every output."""
    import ctypes

    from gated_delta_rule_42_gb300 import _lib
    from gated_delta_rule_42_gb300.ops import make_inputs_struct
    inp = inputs.make_config(2)
    o, hT, grads, nctx = H.gpu_fwd_bwd_ctx(inp, want_dh0=inp.h0 is not None)
    assert nctx > 0
    lib = _lib.load()
    d = inp.to("cuda")
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens)
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    ws, wp, wb = H._poisoned_ws(lib.kda_chunk_bwd_workspace_size(ctypes.byref(s)), "cuda")
    o2 = torch.empty_like(d.v)
    _lib.check(lib, lib.kda_chunk_fwd(ctypes.byref(s), p(o2), None, wp, wb, sp))
    ref = {k: torch.empty_like(grads[0][k]) for k in ("dq", "dk", "dv", "dg", "dbeta")}
    _lib.check(lib, lib.kda_chunk_bwd(ctypes.byref(s), p(d.do), p(d.dhT), p(ref["dq"]), p(ref["dk"]), p(ref["dv"]),
                                      p(ref["dg"]), p(ref["dbeta"]), None, wp, wb, sp))
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    for k, v in ref.items():
        assert torch.equal(grads[0][k], v), k
    assert torch.isfinite(grads[0]["dg"]).all()


@pytest.mark.parametrize("keep_context", [True, False])
def test_autograd_tensor_core_path_matches_c_abi(keep_context):
    """chunk_kda on the tensor-core path, with and without the kept context,
    returns exactly what the recompute C-ABI pair returns."""
    from gated_delta_rule_42_gb300 import chunk_kda
    inp = inputs.make_inputs(B=1, T=200, H=2, HV=4, K=128, V=128, dtype=torch.bfloat16, seed=6,
                             cu_seqlens=[0, 50, 50, 200], name="autograd_tc")
    d = inp.to("cuda")
    leaves = [t.clone().requires_grad_(True) for t in (d.q, d.k, d.v, d.g, d.beta, d.h0)]
    o, hT = chunk_kda(*leaves, cu_seqlens=d.cu_seqlens, output_final_state=True, keep_context=keep_context)
    torch.autograd.backward([o, hT], [d.do, d.dhT])
    o2, hT2 = H.gpu_fwd(inp)
    assert torch.equal(o.detach().cpu(), o2) and torch.equal(hT.detach().cpu(), hT2)
    gr = H.gpu_bwd(inp)
    for t, key in zip(leaves, GRADS):
        assert torch.equal(t.grad.cpu(), gr[key]), key


STATE_CASES = [
    ("tc_varlen_empty", dict(B=1, T=300, H=2, HV=4, K=128, V=128, cu_seqlens=[0, 0, 100, 100, 300])),
    ("tc_scalar_gate", dict(B=2, T=130, H=1, HV=2, K=128, V=128, scalar_gate=True)),
    ("general_fp32", dict(B=1, T=150, H=1, HV=2, K=64, V=48, dtype=torch.float32)),
]


@pytest.mark.parametrize("name,kw", STATE_CASES, ids=[c[0] for c in STATE_CASES])
def test_start_state_gradient_alone_matches_the_full_backward(name, kw):
    """The backward with dq .. dbeta NULL (the reverse scan alone) returns the
    full backward's dh0, bit for bit, with and without a forward context."""
    from gated_delta_rule_42_gb300.ops import chunk_kda_bwd_state, chunk_kda_fwd_ctx
    kw = dict(kw)
    dtype = kw.pop("dtype", torch.bfloat16)
    inp = inputs.make_inputs(dtype=dtype, seed=zlib.crc32(name.encode()) % 1000, name=name, **kw)
    d = inp.to("cuda")
    full = H.gpu_bwd(inp)["dh0"]
    alone = chunk_kda_bwd_state(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, d.do, d.dhT)
    _, _, kctx = chunk_kda_fwd_ctx(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, True)
    alone_ctx = chunk_kda_bwd_state(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, d.do, d.dhT, kctx)
    torch.cuda.synchronize()
    assert torch.equal(alone.cpu(), full)
    assert torch.equal(alone_ctx.cpu(), full)


@pytest.mark.parametrize("name,kw", [
    ("tc_varlen_gva", dict(B=1, T=300, H=2, HV=4, K=128, V=128, cu_seqlens=[0, 0, 100, 100, 300])),
    ("general_fp32", dict(B=1, T=150, H=1, HV=2, K=64, V=48, dtype=torch.float32)),
], ids=["tc_varlen_gva", "general_fp32"])
def test_final_state_only_and_record_reuse(name, kw):
    """(1) The forward without o returns the full forward's final state, bit for
    bit.  (2) A context filled on one (v, h0), then reused for another (v', h0')
    with the same q, k, g, beta, gives what the plain pair gives on (v', h0'):
    o, hT and every gradient, bit for bit."""
    from gated_delta_rule_42_gb300.ops import (chunk_kda_bwd, chunk_kda_bwd_ctx, chunk_kda_fwd, chunk_kda_fwd_ctx,
                                               chunk_kda_fwd_reuse)
    kw = dict(kw)
    dtype = kw.pop("dtype", torch.bfloat16)
    inp = inputs.make_inputs(dtype=dtype, seed=zlib.crc32(name.encode()) % 1000, name=name, **kw)
    d = inp.to("cuda")
    args = (d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens)
    o_full, hT_full = chunk_kda_fwd(*args, True)
    none, hT_only = chunk_kda_fwd(*args, True, need_output=False)
    assert none is None and torch.equal(hT_only, hT_full)
    # another v and h0 on the same q, k, g, beta
    v2 = torch.flip(d.v, dims=[1]).contiguous()
    h2 = (0.5 * d.h0).contiguous()
    _, _, kctx = chunk_kda_fwd_ctx(*args, True, need_output=False)
    o_r, hT_r = chunk_kda_fwd_reuse(d.q, d.k, v2, d.g, d.beta, h2, d.cu_seqlens, kctx, True)
    o_p, hT_p = chunk_kda_fwd(d.q, d.k, v2, d.g, d.beta, h2, d.cu_seqlens, True)
    torch.cuda.synchronize()
    _same("o", o_r, o_p)
    _same("hT", hT_r, hT_p)
    g_r = chunk_kda_bwd_ctx(d.q, d.k, v2, d.g, d.beta, h2, d.cu_seqlens, kctx, d.do, d.dhT)
    g_p = chunk_kda_bwd(d.q, d.k, v2, d.g, d.beta, h2, d.cu_seqlens, d.do, d.dhT)
    torch.cuda.synchronize()
    for key, a, b in zip(GRADS, g_r, g_p):
        _same(key, a, b)


def test_context_pair_cuda_graph_replay_with_mutated_offsets():
    """The step the benchmark times (kda_chunk_fwd_ctx + kda_chunk_bwd_ctx on the
    tensor-core path), captured once in a CUDA graph, replays correctly after
    the offsets buffer is overwritten in place: every output equals, bit for
    bit, the eager recompute pair on the new offsets."""
    import ctypes

    from gated_delta_rule_42_gb300 import _lib
    from gated_delta_rule_42_gb300.ops import make_inputs_struct
    inp = inputs.make_inputs(B=1, T=300, H=2, HV=4, K=128, V=128, dtype=torch.bfloat16, seed=51,
                             cu_seqlens=[0, 100, 300], name="graph_ctx")
    d = inp.to("cuda")
    lib = _lib.load()
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens)
    nctx = lib.kda_chunk_ctx_size(ctypes.byref(s))
    nws = max(lib.kda_chunk_fwd_ctx_workspace_size(ctypes.byref(s)), lib.kda_chunk_bwd_ctx_workspace_size(ctypes.byref(s)))
    assert nctx > 0
    ctx, cp, cb = H._poisoned_ws(nctx, "cuda")
    ws, wp, wb = H._poisoned_ws(nws, "cuda")
    o, hT = torch.empty_like(d.v), torch.empty_like(d.h0)
    grads = [torch.empty_like(x) for x in (d.q, d.k, d.v, d.g, d.beta, d.h0)]
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    def step(stream):
        sp = ctypes.c_void_p(stream.cuda_stream)
        _lib.check(lib, lib.kda_chunk_fwd_ctx(ctypes.byref(s), p(o), p(hT), cp, cb, wp, wb, sp))
        _lib.check(lib, lib.kda_chunk_bwd_ctx(ctypes.byref(s), cp, cb, p(d.do), p(d.dhT), *[p(x) for x in grads],
                                              wp, wb, sp))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)  # warm-up outside the capture (function attributes, cached device queries)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step(side)
    torch.cuda.synchronize()
    for cu in ([0, 100, 300], [0, 3, 300], [0, 300, 300]):
        d.cu_seqlens.copy_(torch.tensor(cu, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        ref_inp = inputs.make_inputs(B=1, T=300, H=2, HV=4, K=128, V=128, dtype=torch.bfloat16, seed=51,
                                     cu_seqlens=[0, 100, 300], name="graph_ctx")
        ref_inp.cu_seqlens = torch.tensor(cu, dtype=torch.int32)
        ro, rhT = H.gpu_fwd(ref_inp)
        rg = H.gpu_bwd(ref_inp)
        _same(f"o {cu}", o, ro)
        _same(f"hT {cu}", hT, rhT)
        for key, x in zip(GRADS, grads):
            _same(f"{key} {cu}", x, rg[key])


def test_context_filled_without_output_then_reused_with_output_serves_the_backward():
    """kda_chunk_fwd_ctx with o NULL computes the final state alone and keeps
    the records; a reuse forward with o on the same inputs completes the
    context, and the backward on it equals the recompute pair's, bit for bit."""
    from gated_delta_rule_42_gb300.ops import (chunk_kda_bwd, chunk_kda_bwd_ctx, chunk_kda_fwd, chunk_kda_fwd_ctx,
                                               chunk_kda_fwd_reuse)
    inp = inputs.make_inputs(B=1, T=260, H=2, HV=4, K=128, V=128, dtype=torch.bfloat16, seed=61,
                             cu_seqlens=[0, 70, 70, 260], name="ctx_no_output")
    d = inp.to("cuda")
    args = (d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens)
    none, hT, kctx = chunk_kda_fwd_ctx(*args, True, need_output=False)
    assert none is None and kctx.numel() > 0
    o_ref, hT_ref = chunk_kda_fwd(*args, True)
    o, hT2 = chunk_kda_fwd_reuse(*args, kctx, True)
    torch.cuda.synchronize()
    _same("hT (final state alone)", hT, hT_ref)
    _same("o", o, o_ref)
    _same("hT", hT2, hT_ref)
    g_ctx = chunk_kda_bwd_ctx(*args, kctx, d.do, d.dhT)
    g_ref = chunk_kda_bwd(*args, d.do, d.dhT)
    torch.cuda.synchronize()
    for key, a, b in zip(GRADS, g_ctx, g_ref):
        _same(key, a, b)
