"""GPU: the device chunk map, read back out of the workspace and compared bit for
bit with a host enumeration of the same offsets.

The map is what every kernel indexes by: a sequence table (first token,
length, first chunk, chunk count) per logical sequence and a chunk table
(sequence, first token, length, index in the sequence) per 64-token chunk,
chunks never straddling a sequence and empty slots producing none -- the packed
contract of the recurrent_kda / chunk_kda entry points in "kda in torchtitan
(training)" (pytorch/torchtitan PR #4164, agent note).  The enumeration below is
written from that contract, independently of the kernel's prefix scan."""
import ctypes

import numpy as np
import pytest
import torch

from gated_delta_rule_42_gb300 import _lib, inputs
from gated_delta_rule_42_gb300.ops import make_inputs_struct
from tests import kda_gpu_helpers as H

pytestmark = pytest.mark.gpu
C = 64


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_42_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return _lib.load()


def _a256(x):
    return (x + 255) // 256 * 256


def host_map(cu, T):
    """(seq table [N][4], chunk table [NC][4], chunks mapped, malformed flag) of packed
    offsets cu on a token axis of T rows.  A malformed sequence (negative start,
    end before start, or end past the axis) is empty and raises the flag."""
    N = len(cu) - 1
    NC = (T + C - 1) // C + N
    seq = np.zeros((N, 4), dtype=np.int32)
    chunk = np.tile(np.array([-1, 0, 0, 0], dtype=np.int32), (NC, 1))
    bad, nxt = 0, 0
    for n in range(N):
        a, b = int(cu[n]), int(cu[n + 1])
        if a < 0 or b < a or b > T:
            bad, a, ln = 1, 0, 0
        else:
            ln = b - a
        nch = (ln + C - 1) // C
        seq[n] = (a, ln, nxt, nch)
        for c in range(nch):
            chunk[nxt + c] = (n, a + C * c, min(C, ln - C * c), c)
        nxt += nch
    return seq, chunk, nxt, bad


def device_map(lib, inp, cu_dev):
    """Runs kda_chunk_fwd and returns (seq table, chunk table, status words) read from
    its workspace: the sequence table comes first, the chunk table at the next
    256-byte boundary, the status words after that."""
    d = inp.to("cuda")
    s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, cu_dev)
    o = torch.empty_like(d.v)
    hT = torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device="cuda")
    ws, wp, wb = H._poisoned_ws(lib.kda_chunk_fwd_workspace_size(ctypes.byref(s)), "cuda")
    _lib.check(lib, lib.kda_chunk_fwd(ctypes.byref(s), ctypes.c_void_p(o.data_ptr()),
                                      ctypes.c_void_p(hT.data_ptr()), wp, wb, None))
    torch.cuda.synchronize()
    base = wp.value - ws.data_ptr()
    N = s.N
    NC = (inp.B * inp.T + C - 1) // C + N if cu_dev is not None else inp.B * ((inp.T + C - 1) // C)
    raw = ws[base:].cpu().numpy()
    seq = raw[:16 * N].view(np.int32).reshape(N, 4)
    off = _a256(16 * max(N, 1))
    chunk = raw[off:off + 16 * NC].view(np.int32).reshape(NC, 4)
    words = H.status_words(lib, s, ws, wp)
    return seq.copy(), chunk.copy(), words


def _problem(T, cu, K=128, dtype=torch.bfloat16):
    return inputs.make_inputs(B=1, T=T, H=1, HV=1, K=K, V=K, dtype=dtype, seed=77, cu_seqlens=cu,
                              name="chunk_map")


def _lengths(n, seed, hi):
    rng = np.random.default_rng(seed)
    ln = rng.integers(0, hi + 1, size=n)
    ln[rng.random(n) < 0.2] = 0  # empty slots, some in runs
    return ln


@pytest.mark.parametrize("K,dtype", [(128, torch.bfloat16), (64, torch.float32)], ids=["tensor_core", "general"])
def test_three_thousand_sequences_bitwise(lib, K, dtype):
    """N = 3000 > 1024: the scan runs in several blocks with a carry between them."""
    ln = _lengths(3000, 5, 150)
    cu = np.concatenate([[0], np.cumsum(ln)]).astype(np.int64)
    T = int(cu[-1])
    inp = _problem(T, list(cu), K, dtype)
    seq, chunk, words = device_map(lib, inp, inp.cu_seqlens.cuda())
    hseq, hchunk, total, bad = host_map(cu, T)
    assert np.array_equal(seq, hseq)
    assert np.array_equal(chunk, hchunk)
    assert words[:2] == [total, bad] == [total, 0]


def test_terminal_offset_below_the_token_axis(lib):
    ln = _lengths(40, 6, 300)
    cu = np.concatenate([[0], np.cumsum(ln)]).astype(np.int64)
    T = int(cu[-1]) + 333  # capacity tail outside the contract
    inp = _problem(T, list(cu))
    seq, chunk, words = device_map(lib, inp, inp.cu_seqlens.cuda())
    hseq, hchunk, total, bad = host_map(cu, T)
    assert np.array_equal(seq, hseq) and np.array_equal(chunk, hchunk)
    assert words[:2] == [total, 0]


def test_malformed_offsets_bitwise(lib):
    """Decreasing offsets and an end past the token axis: those sequences map to
    no chunk, the rest map as usual, and the malformed flag is raised."""
    T = 1000
    cu = [0, 100, 90, 300, 300, 1200, 1000, 1000]
    inp = _problem(T, [0, 100, 100, 300, 300, 300, 1000, 1000])
    cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
    seq, chunk, words = device_map(lib, inp, cu_dev)
    hseq, hchunk, total, bad = host_map(np.array(cu), T)
    assert bad == 1
    assert np.array_equal(seq, hseq) and np.array_equal(chunk, hchunk)
    assert words[:2] == [total, 1]


def test_dense_batch_bitwise(lib):
    inp = inputs.make_inputs(B=3, T=200, H=1, HV=1, K=128, V=128, dtype=torch.bfloat16, seed=78, name="dense_map")
    seq, chunk, words = device_map(lib, inp, None)
    hseq, hchunk, total, bad = host_map(np.arange(4) * 200, 600)
    NC = 3 * ((200 + C - 1) // C)
    assert np.array_equal(seq, hseq) and np.array_equal(chunk, hchunk[:NC])
    assert words[:2] == [total, 0]
