"""kda_chunk_fwd_noalloc: the chunked forward for callers that cannot allocate
device memory (a host program linked against libkda alone, or a runtime that
plans every device byte at start-up and forbids allocation afterwards).  It
runs on a scratch array inside the library, so it must give what
kda_chunk_fwd gives with a caller workspace, call after call."""
import ctypes

import pytest
import torch

from gated_delta_rule_42_gb300 import _lib, inputs
from gated_delta_rule_42_gb300.ops import make_inputs_struct
from tests import kda_gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_42_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return _lib.load()


def noalloc_fwd(lib, inp):
    d = inp.to("cuda")
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens)
    o = torch.full(d.v.shape, float("nan"), dtype=d.dtype, device="cuda")
    hT = torch.full((s.N, s.HV, s.K, s.V), float("nan"), dtype=torch.float32, device="cuda")
    st = lib.kda_chunk_fwd_noalloc(ctypes.byref(s), ctypes.c_void_p(o.data_ptr()),
                                   ctypes.c_void_p(hT.data_ptr()),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _lib.check(lib, st)
    torch.cuda.synchronize()
    return o.cpu(), hT.cpu()


CASES = [
    ("bf16_tensor_core_varlen", dict(B=1, T=300, H=2, HV=4, K=128, V=128, dtype=torch.bfloat16,
                                     cu_seqlens=[0, 0, 130, 130, 300])),
    ("f32_small", dict(B=2, T=100, H=1, HV=2, K=64, V=64, dtype=torch.float32)),
]
# an unrelated problem run on the scratch first, so that it holds other data
UNRELATED = dict(B=1, T=257, H=1, HV=3, K=128, V=128, dtype=torch.bfloat16, cu_seqlens=[0, 60, 257])


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry_on_consecutive_calls(lib, name, kw):
    """Both entry points run the same deterministic kernels, so their results
    must be equal bit for bit -- after the scratch held another problem's data,
    and on two calls in a row with different inputs."""
    noalloc_fwd(lib, inputs.make_inputs(seed=30, name="unrelated", **UNRELATED))
    for seed in (31, 32):
        inp = inputs.make_inputs(seed=seed, name=name, **kw)
        o1, h1 = noalloc_fwd(lib, inp)
        o2, h2 = H.gpu_fwd(inp)  # caller workspace, poisoned with 0xFF
        m = torch.from_numpy(H.valid_mask(inp))
        assert torch.equal(o1.reshape(inp.B * inp.T, -1)[m], o2.reshape(inp.B * inp.T, -1)[m])
        assert torch.equal(h1, h2)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    inp = inputs.make_inputs(B=1, T=4096, H=1, HV=4, K=128, V=128, dtype=torch.float32, seed=1)
    d = inp.to("cuda")
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(s)) > 4 << 20
    o = torch.empty_like(d.v)
    st = lib.kda_chunk_fwd_noalloc(ctypes.byref(s), ctypes.c_void_p(o.data_ptr()), None,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.KDA_ERR_WORKSPACE
    assert "static scratch" in lib.kda_last_error().decode()
