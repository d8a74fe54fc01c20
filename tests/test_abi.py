"""The C-ABI library loads, exports every symbol include/kda.h declares, and
rejects bad arguments on the host (no GPU is touched: validation happens before
anything is enqueued)."""
import ctypes
import os
import re

import pytest

from gated_delta_rule_42_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n
    assert lib.kda_version() >= 100


def _inputs(**kw):
    s = _lib.KdaInputs()
    s.B, s.T, s.H, s.HV, s.K, s.V, s.N, s.dtype = 1, 128, 2, 4, 64, 64, 1, _lib.KDA_BF16
    for f in ("q", "k", "v", "g", "beta"):
        setattr(s, f, 0x1000)
    for key, val in kw.items():
        setattr(s, key, val)
    return s


@pytest.mark.parametrize("kw,status", [
    (dict(HV=3), _lib.KDA_ERR_INVALID_ARG),
    (dict(K=256), _lib.KDA_ERR_UNSUPPORTED),
    (dict(V=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(N=2), _lib.KDA_ERR_INVALID_ARG),             # dense: N must equal B
    (dict(B=2, N=2, cu_seqlens=0x2000), _lib.KDA_ERR_INVALID_ARG),  # packed needs B == 1
    (dict(q=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(dtype=7), _lib.KDA_ERR_INVALID_ARG),
    (dict(flags=4), _lib.KDA_ERR_INVALID_ARG),          # unknown flag bit
    (dict(flags=-1), _lib.KDA_ERR_INVALID_ARG),
])
def test_host_validation(lib, kw, status):
    s = _inputs(**kw)
    st = lib.kda_chunk_fwd(ctypes.byref(s), ctypes.c_void_p(0x3000), None, None, 0, None)
    assert st == status, lib.kda_last_error()
    assert lib.kda_last_error().decode() != ""
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(s)) == 0


def test_workspace_checks(lib):
    s = _inputs()
    need_f = lib.kda_chunk_fwd_workspace_size(ctypes.byref(s))
    need_b = lib.kda_chunk_bwd_workspace_size(ctypes.byref(s))
    assert 0 < need_f < need_b
    st = lib.kda_chunk_fwd(ctypes.byref(s), ctypes.c_void_p(0x3000), None, None, need_f, None)
    assert st == _lib.KDA_ERR_WORKSPACE
    st = lib.kda_chunk_fwd(ctypes.byref(s), ctypes.c_void_p(0x3000), None, ctypes.c_void_p(0x10000),
                           need_f - 1, None)
    assert st == _lib.KDA_ERR_WORKSPACE
    st = lib.kda_chunk_fwd(ctypes.byref(s), ctypes.c_void_p(0x3000), None, ctypes.c_void_p(0x10010),
                           need_f, None)
    assert st == _lib.KDA_ERR_WORKSPACE  # misaligned
    st = lib.kda_chunk_bwd(ctypes.byref(s), None, None, None, None, None, None, None, None, None, 0, None)
    assert st == _lib.KDA_ERR_INVALID_ARG


def test_status_strings(lib):
    for st in range(5):
        assert lib.kda_status_string(st).decode()


def test_struct_fields_follow_the_header(lib):
    """The ctypes mirror of kda_inputs lists the header's members in order."""
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    body = re.search(r"typedef struct kda_inputs \{(.*?)\} kda_inputs;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = []
    for decl in body.split(";"):
        decl = decl.strip()
        if decl:
            names += [re.sub(r"[*\s]", "", n).split()[-1] if n.strip() else n
                      for n in re.sub(r"^(const\s+)?[a-z0-9_]+\s+", "", decl).split(",")]
    assert [n.strip("* ") for n in names] == [f[0] for f in _lib.KdaInputs._fields_]


def test_l2norm_flag_workspace(lib):
    """The fp32 path with the q/k L2-norm prologue works on normalised copies
    of q and k (two more [T][H][K] buffers); the bf16 tensor-core path
    normalises in its kernels, and with HV = H fuses the norm's backward into
    the gradient kernel, so its workspace does not change."""
    s0 = _inputs(K=64, V=64, dtype=_lib.KDA_F32)
    s1 = _inputs(K=64, V=64, dtype=_lib.KDA_F32, flags=_lib.KDA_QK_L2NORM)
    extra = lib.kda_chunk_fwd_workspace_size(ctypes.byref(s1)) - lib.kda_chunk_fwd_workspace_size(ctypes.byref(s0))
    assert extra >= 2 * 128 * 2 * 64 * 4
    t0 = _inputs(K=128, V=128, HV=2)
    t1 = _inputs(K=128, V=128, HV=2, flags=_lib.KDA_QK_L2NORM)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(t1)) == lib.kda_chunk_fwd_workspace_size(ctypes.byref(t0))
    assert lib.kda_chunk_bwd_workspace_size(ctypes.byref(t1)) == lib.kda_chunk_bwd_workspace_size(ctypes.byref(t0))


@pytest.mark.parametrize("args,status", [
    (dict(count=-1), _lib.KDA_ERR_INVALID_ARG),
    (dict(K=129), _lib.KDA_ERR_UNSUPPORTED),
    (dict(V=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(M=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(out=0x100000 + 4 * 64), _lib.KDA_ERR_INVALID_ARG),  # out overlaps h
])
def test_state_compose_validation(lib, args, status):
    a = dict(M=0x400000, h=0x100000, c=None, out=0x800000, count=2, K=64, V=64, transpose=0)
    a.update(args)
    st = lib.kda_state_compose(a["M"], a["h"], a["c"], a["out"], a["count"], a["K"], a["V"], a["transpose"], None)
    assert st == status, lib.kda_last_error()


def test_misaligned_dO_on_the_tensor_core_path_is_rejected(lib):
    """bf16, K = V = 128 with aligned q, k, v, g selects the tensor-core kernels,
    whose TMA loads need a 16-byte aligned dO: rejected before any launch."""
    s = _inputs(K=128, V=128)
    fake = [ctypes.c_void_p(0x200000 + 0x1000 * i) for i in range(6)]
    st = lib.kda_chunk_bwd(ctypes.byref(s), ctypes.c_void_p(0x100002), None, *fake[:5], None,
                           ctypes.c_void_p(0x10000), 1 << 30, None)
    assert st == _lib.KDA_ERR_INVALID_ARG, lib.kda_last_error()
    assert b"aligned" in lib.kda_last_error()


def _a256(x):
    return (x + 255) & ~255


def test_forward_context_sizes(lib):
    """The forward context holds, per (64-token chunk, value head), the record
    (66,048 B), the bf16 chunk-start state and the X^T, D^T tiles; the _ctx
    workspaces are the plain ones minus those regions.  The general path keeps
    nothing."""
    s = _inputs(K=128, V=128, T=200)          # 4 chunks x 4 value heads, tensor-core path
    slots = 4 * 4
    ctx = lib.kda_chunk_ctx_size(ctypes.byref(s))
    assert ctx == _a256(66048 * slots) + _a256(2 * 128 * 128 * slots) + 2 * _a256(16384 * slots)
    f, b = lib.kda_chunk_fwd_workspace_size(ctypes.byref(s)), lib.kda_chunk_bwd_workspace_size(ctypes.byref(s))
    fc = lib.kda_chunk_fwd_ctx_workspace_size(ctypes.byref(s))
    bc = lib.kda_chunk_bwd_ctx_workspace_size(ctypes.byref(s))
    assert f - fc == _a256(66048 * slots)
    assert b - bc == ctx
    # a 64-wide head runs in the same 128-wide tiles: the same context
    assert lib.kda_chunk_ctx_size(ctypes.byref(_inputs(K=64, V=64, T=200))) == ctx
    for kw in (dict(K=96, V=96), dict(K=128, V=128, dtype=_lib.KDA_F32), dict(K=128, V=128, v=0x1008)):
        g = _inputs(T=200, **kw)                # general path: fp32, K not 64 or 128, or a misaligned v
        assert lib.kda_chunk_ctx_size(ctypes.byref(g)) == 0
        assert lib.kda_chunk_fwd_ctx_workspace_size(ctypes.byref(g)) == lib.kda_chunk_fwd_workspace_size(ctypes.byref(g))
        assert lib.kda_chunk_bwd_ctx_workspace_size(ctypes.byref(g)) == lib.kda_chunk_bwd_workspace_size(ctypes.byref(g))
    assert lib.kda_chunk_ctx_size(ctypes.byref(_inputs(HV=3))) == 0  # invalid problem


def test_forward_context_checks(lib):
    """A missing, short or misaligned context is KDA_ERR_WORKSPACE before any launch."""
    s = _inputs(K=128, V=128)
    need = lib.kda_chunk_ctx_size(ctypes.byref(s))
    ws = ctypes.c_void_p(0x10000)
    o = ctypes.c_void_p(0x3000)
    for ctx, nbytes in ((None, need), (ctypes.c_void_p(0x100000), need - 1), (ctypes.c_void_p(0x100010), need)):
        st = lib.kda_chunk_fwd_ctx(ctypes.byref(s), o, None, ctx, nbytes, ws, 1 << 30, None)
        assert st == _lib.KDA_ERR_WORKSPACE, lib.kda_last_error()
        assert b"forward context" in lib.kda_last_error()
        fake = [ctypes.c_void_p(0x200000 + 0x1000 * i) for i in range(6)]
        st = lib.kda_chunk_bwd_ctx(ctypes.byref(s), ctx, nbytes, fake[0], None, *fake[1:6], None, ws, 1 << 30, None)
        assert st == _lib.KDA_ERR_WORKSPACE, lib.kda_last_error()
    # a general-path problem keeps nothing: a NULL context is fine up to the workspace check
    g = _inputs(K=64, V=64, dtype=_lib.KDA_F32)
    st = lib.kda_chunk_fwd_ctx(ctypes.byref(g), o, None, None, 0, None, 0, None)
    assert st == _lib.KDA_ERR_WORKSPACE and b"workspace is NULL" in lib.kda_last_error()


@pytest.mark.parametrize("bad", ["o", "dq", "dk", "dv", "dg"])
def test_misaligned_outputs_on_the_tensor_core_path_are_rejected(lib, bad):
    """The tensor-core kernels store o and the gradients in 4- to 16-byte vectors: a
    caller pointer off a 16-byte boundary is rejected before any launch."""
    s = _inputs(K=128, V=128)
    ptr = {n: 0x200000 + 0x1000 * i for i, n in enumerate(("o", "dO", "dq", "dk", "dv", "dg", "db"))}
    ptr[bad] += 4
    ws = ctypes.c_void_p(0x10000)
    if bad == "o":
        st = lib.kda_chunk_fwd(ctypes.byref(s), ctypes.c_void_p(ptr["o"]), None, ws, 1 << 30, None)
    else:
        p = [ctypes.c_void_p(ptr[n]) for n in ("dO", "dq", "dk", "dv", "dg", "db")]
        st = lib.kda_chunk_bwd(ctypes.byref(s), p[0], None, *p[1:], None, ws, 1 << 30, None)
    assert st == _lib.KDA_ERR_INVALID_ARG, lib.kda_last_error()
    assert bad.encode() + b" must be 16-byte aligned" in lib.kda_last_error()


def test_scalar_gate_dg_needs_no_vector_alignment(lib):
    """With a scalar gate the caller's dg [B, T, HV] is written one float at a time: a
    4-byte aligned dg passes the host checks (here up to the workspace check)."""
    s = _inputs(K=128, V=128, flags=_lib.KDA_SCALAR_GATE)
    p = [ctypes.c_void_p(0x200000 + 0x1000 * i) for i in range(6)]
    p[4] = ctypes.c_void_p(0x204004)
    st = lib.kda_chunk_bwd(ctypes.byref(s), p[0], None, *p[1:], None, None, 0, None)
    assert st == _lib.KDA_ERR_WORKSPACE, lib.kda_last_error()


def test_start_state_gradient_only_mode_validation(lib):
    """dq .. dbeta all NULL with a dh0 asks for dh0 alone; a partial set of NULL
    gradients, or no dh0 either, is an invalid argument."""
    s = _inputs(K=128, V=128)
    p = [ctypes.c_void_p(0x200000 + 0x1000 * i) for i in range(7)]
    dO, dh0 = p[0], p[6]
    st = lib.kda_chunk_bwd(ctypes.byref(s), dO, None, None, None, None, None, None, dh0, None, 0, None)
    assert st == _lib.KDA_ERR_WORKSPACE, lib.kda_last_error()  # valid request: stops at the workspace check
    st = lib.kda_chunk_bwd(ctypes.byref(s), dO, None, None, None, None, None, None, None, None, 0, None)
    assert st == _lib.KDA_ERR_INVALID_ARG  # nothing to compute
    st = lib.kda_chunk_bwd(ctypes.byref(s), dO, None, p[1], None, None, None, None, dh0, None, 0, None)
    assert st == _lib.KDA_ERR_INVALID_ARG  # dq given, the rest NULL
    st = lib.kda_chunk_bwd_ctx(ctypes.byref(s), None, 0, dO, None, None, None, None, None, None, dh0, None, 0, None)
    assert st == _lib.KDA_ERR_WORKSPACE and b"forward context" in lib.kda_last_error()


def test_final_state_only_forward_validation(lib):
    """o may be NULL when hT is not (the final state alone); both NULL is an
    invalid argument.  kda_chunk_fwd_reuse checks its context like the _ctx pair."""
    s = _inputs(K=128, V=128)
    hT = ctypes.c_void_p(0x300000)
    st = lib.kda_chunk_fwd(ctypes.byref(s), None, hT, None, 0, None)
    assert st == _lib.KDA_ERR_WORKSPACE, lib.kda_last_error()  # valid request: stops at the workspace check
    st = lib.kda_chunk_fwd(ctypes.byref(s), None, None, None, 0, None)
    assert st == _lib.KDA_ERR_INVALID_ARG
    st = lib.kda_chunk_fwd_reuse(ctypes.byref(s), ctypes.c_void_p(0x3000), None, None, 0, ctypes.c_void_p(0x10000),
                                 1 << 30, None)
    assert st == _lib.KDA_ERR_WORKSPACE and b"forward context" in lib.kda_last_error()


def test_status_offset_follows_the_workspace_layout(lib):
    """The status words sit after the sequence and chunk tables: byte offset
    align256(16 N) + align256(16 NC), the same for every workspace of a problem."""
    s = _inputs(K=128, V=128, T=200)               # N = 1, 4 chunks
    assert lib.kda_status_offset(ctypes.byref(s)) == _a256(16) + _a256(16 * 4)
    v = _inputs(K=64, V=64, T=1000, N=3, cu_seqlens=0x2000)  # packed: NC = ceil(1000/64) + N = 19
    assert lib.kda_status_offset(ctypes.byref(v)) == _a256(16 * 3) + _a256(16 * 19)
    assert lib.kda_status_offset(ctypes.byref(_inputs(HV=3))) == ctypes.c_size_t(-1).value


def test_bounded_wait_probe_validation(lib):
    assert lib.kda_debug_bounded_wait(None, 100, None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_debug_bounded_wait(ctypes.c_void_p(0x1000), 0, None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_debug_bounded_wait(ctypes.c_void_p(0x1000), (1 << 24) + 1, None) == _lib.KDA_ERR_INVALID_ARG


def test_kernel_family_query(lib):
    """bf16 with K and V each 64 or 128 and 16-byte aligned q, k, v, g runs the
    tensor-core kernels; an fp32 problem, other head dims or a misaligned input
    the general ones."""
    for K, V in ((128, 128), (64, 64), (64, 128), (128, 64)):
        assert lib.kda_uses_tensor_cores(ctypes.byref(_inputs(K=K, V=V))) == 1, (K, V)
    assert lib.kda_uses_tensor_cores(ctypes.byref(_inputs(K=128, V=128, dtype=_lib.KDA_F32))) == 0
    assert lib.kda_uses_tensor_cores(ctypes.byref(_inputs(K=96, V=96))) == 0
    assert lib.kda_uses_tensor_cores(ctypes.byref(_inputs(K=128, V=128, q=0x1002))) == 0
    assert lib.kda_uses_tensor_cores(ctypes.byref(_inputs(HV=3))) == -1
