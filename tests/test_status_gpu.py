"""GPU: the device status words a call leaves in its workspace (chunks mapped,
malformed offsets, a bounded wait that gave up, slots on the exact wide-decay
path, slots on the block-reference path) and the bounded-wait path
itself, exercised by a probe that waits on an mbarrier nothing completes.
Nothing here faults, traps or hangs the GPU: malformed offsets are handled by
the chunk map as empty sequences, and the probe's wait is bounded."""
import ctypes

import numpy as np
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


def _words(ws, wp, off):
    base = wp.value - ws.data_ptr()
    return ws[base + off: base + off + 28].cpu().numpy().view(np.int32).tolist()


def _run_fwd_bwd(lib, d, s):
    """kda_chunk_fwd then kda_chunk_bwd on one workspace; the status words after each."""
    need = max(lib.kda_chunk_fwd_workspace_size(ctypes.byref(s)), lib.kda_chunk_bwd_workspace_size(ctypes.byref(s)))
    ws, wp, wb = H._poisoned_ws(need, "cuda")
    off = lib.kda_status_offset(ctypes.byref(s))
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    o, hT = torch.empty_like(d.v), torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device="cuda")
    _lib.check(lib, lib.kda_chunk_fwd(ctypes.byref(s), p(o), p(hT), wp, wb, None))
    fwd = _words(ws, wp, off)
    g = [torch.empty_like(x) for x in (d.q, d.k, d.v, d.g, d.beta)]
    _lib.check(lib, lib.kda_chunk_bwd(ctypes.byref(s), p(d.do), p(d.dhT), *[p(x) for x in g], p(hT), wp, wb, None))
    bwd = _words(ws, wp, off)
    torch.cuda.synchronize()
    return fwd, bwd, o, g


@pytest.mark.parametrize("K,dtype", [(128, torch.bfloat16), (64, torch.float32)], ids=["tensor_core", "general"])
def test_status_words_after_clean_calls(lib, K, dtype):
    inp = inputs.make_inputs(B=1, T=300, H=1, HV=2, K=K, V=K, dtype=dtype, seed=41, cu_seqlens=[0, 130, 130, 300],
                             name="status")
    d = inp.to("cuda")
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens)
    fwd, bwd, _, _ = _run_fwd_bwd(lib, d, s)
    chunks = 3 + 3  # 130 and 170 tokens
    assert fwd == [chunks, 0, 0, 0, 0, 0, 0] and bwd == [chunks, 0, 0, 0, 0, 0, 0]


def test_malformed_offsets_are_flagged_and_treated_as_empty(lib):
    """cu_seqlens [0, 100, 400, 300] on T = 300: sequence 1 ends past the token
    axis and sequence 2 ends before it starts, so both are empty; sequence 0
    is computed as usual."""
    inp = inputs.make_inputs(B=1, T=300, H=1, HV=2, K=128, V=128, dtype=torch.bfloat16, seed=42,
                             cu_seqlens=[0, 100, 300, 300], name="malformed")
    d = inp.to("cuda")
    cu = torch.tensor([0, 100, 400, 300], dtype=torch.int32, device="cuda")
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, cu)
    fwd, bwd, o, g = _run_fwd_bwd(lib, d, s)
    assert fwd == [2, 1, 0, 0, 0, 0, 0] and bwd == [2, 1, 0, 0, 0, 0, 0]
    assert torch.isfinite(o[:, :100]).all() and all(torch.isfinite(x[:, :100]).all() for x in g)


def test_bounded_wait_gives_up_and_the_context_stays_usable(lib):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.check(lib, lib.kda_debug_bounded_wait(ctypes.c_void_p(err.data_ptr()), 1000, None))
    torch.cuda.synchronize()
    assert err.item() == 1
    inp = inputs.make_inputs(B=1, T=70, H=1, HV=1, K=128, V=128, dtype=torch.bfloat16, seed=43, name="after_probe")
    o, hT = H.gpu_fwd(inp)
    ro, rhT = H.oracle_fwd(inp)
    H.check_fwd(inp, o, hT, ro, rhT, H.TOL[torch.bfloat16]["fwd"])
