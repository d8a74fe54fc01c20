"""ctypes binding of libkda.so (the C ABI declared in include/kda.h).

Argument marshalling only.  Loading fails loudly when the library has not
been built: there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE, KDA_ERR_CUDA = range(5)
KDA_F32, KDA_BF16 = 0, 1
KDA_QK_L2NORM = 1  # kda_inputs.flags bit: q/k rows L2-normalised inside the op
KDA_SCALAR_GATE = 2  # kda_inputs.flags bit: g, dg are [B, T, HV] (one decay per token and value head)
KDA_GATE_IN_KERNEL = 4  # kda_inputs.flags bit: g holds the raw gate, the op makes the decay (kda_inputs.gate)

EXPORTS = (
    "kda_chunk_fwd_workspace_size", "kda_chunk_fwd", "kda_chunk_bwd_workspace_size",
    "kda_chunk_bwd", "kda_recurrent_fwd", "kda_status_string", "kda_last_error", "kda_version",
    "kda_launch_count", "kda_timing_enable", "kda_timing_collect", "kda_chunk_fwd_noalloc",
    "kda_state_compose", "kda_chunk_ctx_size", "kda_chunk_fwd_ctx_workspace_size",
    "kda_chunk_bwd_ctx_workspace_size", "kda_chunk_fwd_ctx", "kda_chunk_bwd_ctx", "kda_chunk_fwd_reuse",
    "kda_status_offset", "kda_debug_bounded_wait", "kda_uses_tensor_cores",
)


class KdaGate(ctypes.Structure):
    _fields_ = [
        ("A_log", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("lower_bound", ctypes.c_float),
        ("dA_log", ctypes.c_void_p), ("dbias", ctypes.c_void_p),
    ]


class KdaInputs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int), ("HV", ctypes.c_int),
        ("K", ctypes.c_int), ("V", ctypes.c_int), ("N", ctypes.c_int), ("dtype", ctypes.c_int),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("h0", ctypes.c_void_p),
        ("cu_seqlens", ctypes.c_void_p), ("flags", ctypes.c_int),
        ("gate", ctypes.POINTER(KdaGate)),
    ]


class KdaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"kda status {status}: {msg}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load libkda.so once.  Raises if it is missing (build it with
    ``python -m gated_delta_rule_42_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libkda.so not built ({path}); run python -m gated_delta_rule_42_gb300.build")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(KdaInputs)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        lib.kda_chunk_fwd_workspace_size.argtypes = [P]
        lib.kda_chunk_fwd_workspace_size.restype = sz
        lib.kda_chunk_bwd_workspace_size.argtypes = [P]
        lib.kda_chunk_bwd_workspace_size.restype = sz
        lib.kda_chunk_fwd.argtypes = [P, vp, vp, vp, sz, vp]
        lib.kda_chunk_fwd.restype = i
        lib.kda_chunk_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.kda_chunk_bwd.restype = i
        for nm in ("kda_chunk_ctx_size", "kda_chunk_fwd_ctx_workspace_size", "kda_chunk_bwd_ctx_workspace_size"):
            getattr(lib, nm).argtypes = [P]
            getattr(lib, nm).restype = sz
        for nm in ("kda_chunk_fwd_ctx", "kda_chunk_fwd_reuse"):
            getattr(lib, nm).argtypes = [P, vp, vp, vp, sz, vp, sz, vp]
            getattr(lib, nm).restype = i
        lib.kda_chunk_bwd_ctx.argtypes = [P, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.kda_chunk_bwd_ctx.restype = i
        lib.kda_uses_tensor_cores.argtypes = [P]
        lib.kda_uses_tensor_cores.restype = ctypes.c_int
        lib.kda_status_offset.argtypes = [P]
        lib.kda_status_offset.restype = sz
        lib.kda_debug_bounded_wait.argtypes = [vp, ctypes.c_longlong, vp]
        lib.kda_debug_bounded_wait.restype = i
        lib.kda_recurrent_fwd.argtypes = [P, vp, vp, vp]
        lib.kda_recurrent_fwd.restype = i
        lib.kda_chunk_fwd_noalloc.argtypes = [P, vp, vp, vp]
        lib.kda_chunk_fwd_noalloc.restype = i
        lib.kda_state_compose.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
        lib.kda_state_compose.restype = i
        lib.kda_status_string.argtypes = [i]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_last_error.argtypes = []
        lib.kda_last_error.restype = ctypes.c_char_p
        lib.kda_version.argtypes = []
        lib.kda_version.restype = i
        lib.kda_launch_count.argtypes = []
        lib.kda_launch_count.restype = ctypes.c_ulonglong
        lib.kda_timing_enable.argtypes = [i]
        lib.kda_timing_enable.restype = i
        lib.kda_timing_collect.argtypes = [i, ctypes.c_char_p, sz, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_int)]
        lib.kda_timing_collect.restype = i
        if path == LIB_PATH:
            _lib = lib
        return lib


def check(lib, status: int):
    if status != KDA_OK:
        msg = lib.kda_last_error().decode() or lib.kda_status_string(status).decode()
        raise KdaError(status, msg)


def timing_collect(lib, max_kernels: int = 64):
    """{kernel name: (total ms, launches)} for the event pairs recorded since
    the last collect."""
    stride = 96
    names = ctypes.create_string_buffer(max_kernels * stride)
    ms = (ctypes.c_double * max_kernels)()
    cnt = (ctypes.c_int * max_kernels)()
    n = lib.kda_timing_collect(max_kernels, names, stride, ms, cnt)
    out = {}
    for i in range(min(n, max_kernels)):
        nm = names.raw[i * stride:(i + 1) * stride].split(b"\0", 1)[0].decode()
        out[nm] = (ms[i], cnt[i])
    return out
