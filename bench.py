#!/usr/bin/env python3
"""Benchmark: chunked KDA forward + backward on one GB300 (or N replicas).

One step = kda_chunk_fwd_ctx + kda_chunk_bwd_ctx (the backward reads the
intermediates the forward kept; --recompute: kda_chunk_fwd + kda_chunk_bwd,
the backward recomputes them) through the C ABI on the dense
training layer (B=8, T=4096, H=HV=32, K=V=128, bf16 q/k/v, fp32 g/beta, no
initial or final state), inputs resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 it runs under torchrun, one replica per rank (no collective in the
op: independent batches, weak scaling); rank 0 prints the max-over-ranks time.
``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload), as the slow reference arm.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_delta_rule_42_gb300 import _lib, inputs  # noqa: E402
from gated_delta_rule_42_gb300.ops import make_inputs_struct  # noqa: E402

METRIC = "chunk_kda fwd+bwd tokens/s on 1 GB300 (bf16, K=V=128); % of roofline"
WORKLOAD_CFG = 2  # the dense training layer
L2_BYTES = 126 * 2 ** 20


# --------------------------------------------------------------------------
# algorithmic cost model (per token, whole layer): the bytes every step must
# move at minimum (inputs read once, outputs written once, states) and the
# flops of the chunked algorithm without recompute (triangular products at half)
# --------------------------------------------------------------------------
def algorithmic_bytes(cfg):
    e = 2 if cfg.dtype == torch.bfloat16 else 4
    H, HV, K, V = cfg.H, cfg.HV, cfg.K, cfg.V
    gb = 4 * HV if cfg.g.dim() == 3 else 4 * HV * K  # the gate (and dg): scalar or per channel
    inp = 2 * H * K * e + HV * V * e + gb + 4 * HV
    fwd = inp + HV * V * e
    bwd = inp + HV * V * e + 2 * H * K * e + HV * V * e + gb + 4 * HV
    toks = cfg.valid_tokens
    state = 4 * cfg.N * HV * K * V
    st_f = (state if cfg.h0 is not None else 0) + (state if cfg.output_final_state else 0)
    st_b = (state if cfg.h0 is not None else 0) + (2 * state if cfg.output_final_state else 0) + \
        (state if cfg.h0 is not None else 0)
    return dict(fwd=fwd * toks + st_f, bwd=bwd * toks + st_b, total=(fwd + bwd) * toks + st_f + st_b,
                per_token_head=(fwd + bwd) / HV)


def algorithmic_flops(cfg, C=64):
    d = cfg.K
    per = 18 * d * d + 15 * C * d + 2 * C * C
    return per * cfg.valid_tokens * cfg.HV


# Algorithmic bytes per launch of each tensor-core kernel, per token of the
# layer: the step's own inputs it reads and outputs it writes (the cost model
# above, split by kernel; intermediates such as the per-chunk records, saved
# states and tiles are the implementation's cost and are not counted).  This
# is what the dominant kernel's roofline divides by its time.
def kernel_algorithmic_bytes_per_token(name, cfg):
    e = 2 if cfg.dtype == torch.bfloat16 else 4
    H, HV, K, V = cfg.H, cfg.HV, cfg.K, cfg.V
    qk, vv, b = H * K * e, HV * V * e, 4 * HV
    g = 4 * HV if cfg.g.dim() == 3 else 4 * HV * K
    table = {
        "kda_prep_tc": 2 * qk + g + b,                            # reads q, k, g, beta
        "kda_fwd_tc": 2 * vv,                                     # reads v, writes o
        "kda_fwd_tc_save": 2 * vv,
        "kda_bwd_scan_tc": vv,                                    # reads dO
        "kda_bwd_intra_tc": (2 * qk + vv + g + b + vv) + (2 * qk + vv + g + b),  # q k v g beta dO -> dq dk dv dg dbeta
    }
    return table.get(name)


# Interface bytes per launch of each kernel (what the kernel must read and
# write by its own contract, intermediates included), per token of the layer:
# a diagnostic beside the algorithmic roofline, not a roofline.
def kernel_bytes_per_token(name, cfg):
    e = 2 if cfg.dtype == torch.bfloat16 else 4
    H, HV, K, V = cfg.H, cfg.HV, cfg.K, cfg.V
    qk, vv, b = H * K * e, HV * V * e, 4 * HV
    g = 4 * HV if cfg.g.dim() == 3 else 4 * HV * K  # a scalar gate: one fp32 per (token, value head)
    f32K, f32V, cc, hh = 4 * HV * K, 4 * HV * V, 4 * HV * 64, 4 * HV * K * V / 64
    hs = 2 * HV * K * V / 64            # bf16 K x V state per chunk, per token
    t16 = 16384 * HV / 64               # one 16 KB per-chunk tile (X^T or D^T), per token
    rec = (65536 + 512) * HV / 64       # the per-chunk tile record (Bk, Qg, Khat, Aqk, A, 2^G_last), per token
    recs = (40960 + 512) * HV / 64      # what the states pass reads of it (Bk, Khat, A, 2^G_last)
    dgl = 4 * HV * K / 64               # fp32 K-vector per chunk, per token
    table = {
        # tensor-core path (bf16, K = V = 128)
        "kda_prep_tc": 2 * qk + g + b + rec,
        "kda_fwd_tc": rec + 2 * vv,
        "kda_fwd_tc_states": recs + vv + hs + 2 * t16,
        "kda_fwd_tc_save": rec + 2 * vv + hs + 2 * t16,
        "kda_bwd_scan_tc": rec + vv + hs + 2 * vv,
        "kda_bwd_intra_tc": 2 * t16 + 2 * hs + 3 * vv + vv + b + g + t16 / 2 + 2 * qk + vv + 2 * qk + g + b,
        # fp32 path
        "simple_intra_kernel": 2 * qk + vv + g + b + 2 * f32K + 2 * cc + f32K + f32V,
        "simple_scan_kernel": qk + 2 * f32K + f32V + hh + f32V,
        "simple_output_kernel": qk + f32K + cc + f32V + hh + vv,
        "simple_dh_scan_kernel": 2 * qk + 2 * f32K + cc + vv + hh + f32V,
        "simple_bwd_intra_kernel": 3 * qk - qk + vv + vv + b + f32K + 2 * cc + 2 * hh + 2 * f32V
        + vv + b + g + 2 * f32K + 2 * f32K,
        "group_reduce_kernel": 2 * f32K + 2 * qk,
        "group_reduce4_kernel": 2 * f32K + 2 * qk,
        "group_reduce_l2norm_kernel": 2 * f32K + 4 * qk,
        "l2norm_rows_kernel": 4 * qk,
        "gate_expand_kernel": 4 * HV + f32K,
        "gate_grad_reduce_kernel": f32K + 4 * HV,
    }
    return table.get(name)


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the step's
# kernels, each from its own one-kernel ncu --set full capture on the dense layer
# at T = 1024, per token of the captured launch, with the SHA-256 of the sources
# the kernel was built from at capture time.  A value is reported only while
# those sources are unchanged.
NCU_TRAFFIC = {
    "kda_bwd_intra_tc": dict(
        bytes_per_token=1282263552 / 8192,  # 974.3 MB read + 308.0 MB written, B=8 T=1024 H=HV=32
        sources=("gated_delta_rule_42_gb300/csrc/tc_bwd_chunk.cu", "gated_delta_rule_42_gb300/csrc/tc_intra.cuh", "gated_delta_rule_42_gb300/csrc/tc_common.cuh", "gated_delta_rule_42_gb300/csrc/umma.cuh", "gated_delta_rule_42_gb300/csrc/kda_internal.cuh"),
        sha256="4581ef8aa45c4e51f08b58124c6303e06625a71ded908159970c1f09398680c1"),
    "kda_prep_tc": dict(
        bytes_per_token=512473856 / 8192,  # 271.0 MB read + 241.5 MB written, B=8 T=1024 H=HV=32
        sources=("gated_delta_rule_42_gb300/csrc/tc_prep.cu", "gated_delta_rule_42_gb300/csrc/tc_common.cuh", "gated_delta_rule_42_gb300/csrc/umma.cuh", "gated_delta_rule_42_gb300/csrc/kda_internal.cuh"),
        sha256="4ead00db5b17147d97749679830f43945dcd04f9f84a5c236afb3c7cbda103d6"),
    "kda_fwd_tc_save": dict(
        bytes_per_token=624946432 / 8192,  # 339.1 MB read + 285.9 MB written, B=8 T=1024 H=HV=32
        sources=("gated_delta_rule_42_gb300/csrc/tc_fwd.cu", "gated_delta_rule_42_gb300/csrc/tc_common.cuh", "gated_delta_rule_42_gb300/csrc/umma.cuh", "gated_delta_rule_42_gb300/csrc/kda_internal.cuh"),
        sha256="fae778c4ab025e760bca5f5321e1e0cfcc7c54cd81732da36474481e1753f12f"),
    "kda_bwd_scan_tc": dict(
        bytes_per_token=560227584 / 8192,  # 337.7 MB read + 222.5 MB written, B=8 T=1024 H=HV=32
        sources=("gated_delta_rule_42_gb300/csrc/tc_bwd_scan.cu", "gated_delta_rule_42_gb300/csrc/tc_common.cuh", "gated_delta_rule_42_gb300/csrc/umma.cuh", "gated_delta_rule_42_gb300/csrc/kda_internal.cuh"),
        sha256="fa160889992d5989fb10277ed479daa765b8d06e9c96eaea678e6017847af27e"),
}


def dominant_roofline(name, launch_ms, cfg, toks_launch, peaks):
    """The dominant kernel's roofline object: achieved = its algorithmic bytes
    per launch (kernel_algorithmic_bytes_per_token x the tokens one launch
    covers) / its average launch time, against the measured HBM copy peak.
    ``interface`` is the same kernel's bytes by its own contract, intermediates
    included (a diagnostic), and ``traffic`` its ncu DRAM bytes per launch while
    the capture matches the sources."""
    abpt = kernel_algorithmic_bytes_per_token(name, cfg)
    ibpt = kernel_bytes_per_token(name, cfg)
    sec = launch_ms / 1e3
    achieved = abpt * toks_launch / sec / 1e9 if abpt else None
    return dict(kernel=name, bound="hbm", achieved=None if achieved is None else round(achieved, 1),
                peak=peaks["hbm"], unit="GB/s",
                frac=None if achieved is None else round(achieved / peaks["hbm"], 4),
                algorithmic_bytes=None if abpt is None else int(round(abpt * toks_launch)),
                traffic=measured_traffic(name, toks_launch), launch_ms=round(launch_ms, 4),
                interface=None if ibpt is None else dict(
                    bytes=int(round(ibpt * toks_launch)), GBps=round(ibpt * toks_launch / sec / 1e9, 1),
                    frac=round(ibpt * toks_launch / sec / 1e9 / peaks["hbm"], 4)),
                peak_source=f"{peaks['src']} (MEASURED_PEAKS.json hbm_gbs)" if peaks["src"] == "measured"
                else "fallback 6.8 TB/s")


def sources_sha256(paths):
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def step_traffic(split, steps_split, tokens):
    """The step's DRAM bytes from the per-kernel captures: the sum over the
    kernels that take more than 1 % of the step's kernel time (the rest are a
    few-microsecond chunk map and empty fix-up launches) of their traffic per
    launch x launches per step; None unless every one of them has a capture
    that matches its sources."""
    total_ms = sum(v[0] for v in split.values())
    total = 0.0
    for name, (ms_k, n_k) in split.items():
        if ms_k < 0.01 * total_ms:
            continue
        t = measured_traffic(name, tokens)
        if t is None:
            return None
        total += t * n_k / steps_split
    return int(round(total))


def measured_traffic(name, tokens):
    """Per-launch DRAM bytes of kernel ``name`` scaled to ``tokens`` (its traffic
    grows in proportion to the (chunk, head) slots), or None when no capture of
    the current sources exists."""
    t = NCU_TRAFFIC.get(name)
    if t is None or sources_sha256(t["sources"]) != t["sha256"]:
        return None
    return int(round(t["bytes_per_token"] * tokens))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sust=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


# --------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region: every
    20 ms, each sample stamped on arrival; only the samples that arrive between
    begin() and end() (plus one interval) count, or the first one after begin()
    when the region is shorter than an interval."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []  # (arrival time, line)
        self.t_begin = self.t_end = None

    def start(self):
        """Start sampling and wait (up to 3 s) until the first sample arrives."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", str(self.INTERVAL_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
            t_stop = time.monotonic() + 3.0
            while not self.lines and time.monotonic() < t_stop and self.proc.poll() is None:
                time.sleep(0.005)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def begin(self):
        self.t_begin = time.monotonic()

    def end(self):
        self.t_end = time.monotonic()

    def stop(self):
        if self.proc is None:
            return None
        if self.t_end is not None:  # let the sample that covers the region's end arrive
            time.sleep(2 * self.INTERVAL_MS / 1e3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        lines = list(self.lines)
        if self.t_begin is not None and self.t_end is not None:
            lag = self.INTERVAL_MS / 1e3
            inside = [ln for t, ln in lines if self.t_begin <= t <= self.t_end + lag]
            after = [ln for t, ln in lines if t >= self.t_begin]
            lines = inside if inside else after[:1]
        else:
            lines = [ln for _, ln in lines]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return dict(sm_mhz=statistics.median(sm), sm_max_mhz=mx, reasons=sorted(reasons),
                    samples=len(sm), interval_ms=self.INTERVAL_MS)


# --------------------------------------------------------------------------
class Runner:
    """Preallocated device buffers and the two C-ABI calls of one step: the
    forward-context pair (kda_chunk_fwd_ctx, kda_chunk_bwd_ctx: the backward
    reads what the forward kept) or, with keep_context=False, the recompute
    pair (kda_chunk_fwd, kda_chunk_bwd)."""

    def __init__(self, cfg, device, qk_l2norm=False, keep_context=True):
        self.lib = _lib.load()
        self.cfg = cfg
        self.dev = device
        d = cfg.to(device)
        self.d = d
        gate = None  # the KDA gate inside the op: g holds raw pre-activations
        self.dA = self.dbias = None
        if d.meta.get("raw_gate"):
            from gated_delta_rule_42_gb300.ops import KdaGateParams
            gate = KdaGateParams(d.A_log, d.g_bias, d.lower_bound)
            self.dA = None if d.A_log is None else torch.empty_like(d.A_log)
            self.dbias = None if d.g_bias is None else torch.empty_like(d.g_bias)
        self.s = make_inputs_struct(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, qk_l2norm, gate, self.dA,
                                    self.dbias)
        s = self.s
        self.o = torch.empty_like(d.v)
        self.hT = (torch.empty((s.N, s.HV, s.K, s.V), dtype=torch.float32, device=device)
                   if cfg.output_final_state else None)
        self.dq, self.dk, self.dv = torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v)
        self.dg, self.db = torch.empty_like(d.g), torch.empty_like(d.beta)
        self.dh0 = torch.empty_like(d.h0) if d.h0 is not None else None
        lib = self.lib
        self.keep_context = keep_context
        if keep_context:
            need = max(lib.kda_chunk_fwd_ctx_workspace_size(ctypes.byref(s)),
                       lib.kda_chunk_bwd_ctx_workspace_size(ctypes.byref(s)))
            self.ctx_bytes = lib.kda_chunk_ctx_size(ctypes.byref(s))
        else:
            need = max(lib.kda_chunk_fwd_workspace_size(ctypes.byref(s)),
                       lib.kda_chunk_bwd_workspace_size(ctypes.byref(s)))
            self.ctx_bytes = 0
        self.ws = torch.empty(need + 256, dtype=torch.uint8, device=device)
        p = self.ws.data_ptr()
        self.wp = ctypes.c_void_p((p + 255) & ~255)
        self.wb = need
        self.ctx = torch.empty(self.ctx_bytes + 256, dtype=torch.uint8, device=device)
        p = self.ctx.data_ptr()
        self.cp = ctypes.c_void_p((p + 255) & ~255) if self.ctx_bytes else None
        self.stream = torch.cuda.current_stream(device)
        self.sp = ctypes.c_void_p(self.stream.cuda_stream)

    @staticmethod
    def _p(t):
        return None if t is None else ctypes.c_void_p(t.data_ptr())

    def fwd(self):
        p, lib, s = self._p, self.lib, self.s
        if self.keep_context:
            _lib.check(lib, lib.kda_chunk_fwd_ctx(ctypes.byref(s), p(self.o), p(self.hT), self.cp, self.ctx_bytes,
                                                  self.wp, self.wb, self.sp))
        else:
            _lib.check(lib, lib.kda_chunk_fwd(ctypes.byref(s), p(self.o), p(self.hT), self.wp, self.wb, self.sp))

    def bwd(self):
        p, lib, s = self._p, self.lib, self.s
        grads = (p(self.d.do), p(self.d.dhT), p(self.dq), p(self.dk), p(self.dv), p(self.dg), p(self.db),
                 p(self.dh0), self.wp, self.wb, self.sp)
        if self.keep_context:
            _lib.check(lib, lib.kda_chunk_bwd_ctx(ctypes.byref(s), self.cp, self.ctx_bytes, *grads))
        else:
            _lib.check(lib, lib.kda_chunk_bwd(ctypes.byref(s), *grads))

    def step(self):
        self.fwd()
        self.bwd()


def cp_step_fn(runner, R):
    """One fwd+bwd step of the context-parallel layer: every sequence split into
    R equal segments, each processed as its rank would (local pass keeping a
    forward context, transition and final pass reusing its records, relay scan;
    the mirror image
    backward: the start-state gradient by the reverse scan alone, relay scan,
    full backward, both reading that context), the ranks one after the other on
    this GPU."""
    from gated_delta_rule_42_gb300 import cp
    from gated_delta_rule_42_gb300.ops import (chunk_kda_bwd_ctx, chunk_kda_bwd_state, chunk_kda_fwd_ctx,
                                               chunk_kda_fwd_reuse)
    d = runner.d
    T = d.q.shape[1]
    bounds = [T * r // R for r in range(R + 1)]
    segs = [[x[:, bounds[r]:bounds[r + 1]].contiguous() for x in (d.q, d.k, d.v, d.g, d.beta, d.do)]
            for r in range(R)]

    def step():
        cs, Ms, ctxs = [], [], []
        for q, k, v, g, beta, _ in segs:  # local pass (final state only), the context's one record pass
            _, c, kctx = chunk_kda_fwd_ctx(q, k, v, g, beta, None, None, True, need_output=False)
            cs.append(c)
            ctxs.append(kctx)
            Ms.append(cp.segment_transition(q, k, g, beta, kctx))
        hs = [d.h0 if d.h0 is not None else torch.zeros_like(cs[0])]
        for r in range(1, R):
            hs.append(cp.compose(Ms[r - 1], hs[-1], cs[r - 1]))
        for r, (q, k, v, g, beta, _) in enumerate(segs):
            chunk_kda_fwd_reuse(q, k, v, g, beta, hs[r], None, ctxs[r], r == R - 1)
        ds = [chunk_kda_bwd_state(q, k, v, g, beta, hs[r], None, do, None, ctxs[r])
              for r, (q, k, v, g, beta, do) in enumerate(segs)]
        ends = [None] * R
        ends[R - 1] = d.dhT
        for r in range(R - 1, 0, -1):
            ends[r - 1] = cp.compose(Ms[r], ends[r] if ends[r] is not None else torch.zeros_like(ds[r]), ds[r], True)
        for r, (q, k, v, g, beta, do) in enumerate(segs):
            chunk_kda_bwd_ctx(q, k, v, g, beta, hs[r], None, ctxs[r], do, ends[r],
                              need_dh0=(r == 0 and d.h0 is not None))

    return step


def segmented_step_fn(runner, S, qk_l2norm=False):
    """One fwd+bwd step with every sequence split into S segments that run at
    once on this GPU (gated_delta_rule_42_gb300.segments)."""
    from gated_delta_rule_42_gb300.segments import chunk_kda_bwd_segmented, chunk_kda_fwd_segmented
    d = runner.d
    assert d.cu_seqlens is None, "segments: dense workloads only"

    def step():
        _, _, ctx = chunk_kda_fwd_segmented(d.q, d.k, d.v, d.g, d.beta, d.h0, S, runner.hT is not None,
                                            use_qk_l2norm=qk_l2norm)
        chunk_kda_bwd_segmented(d.q, d.k, d.v, d.g, d.beta, ctx, d.do, d.dhT, need_dh0=d.h0 is not None,
                                use_qk_l2norm=qk_l2norm)

    return step


def timed(fn, steps, stream):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def e2e_measure(cfg, runner, steps, qk_l2norm=False):
    """Same step through the public API with HOST buffers: every step copies its
    inputs in from pinned host memory and every output back out, inside the
    timed region.  The steps are pipelined the way a training loop would run
    them: copies in on one stream, the two C-ABI calls on another, copies out
    on a third, with two device sets so that step i+1's inputs arrive and step
    i-1's outputs leave while step i computes.  Timed with CUDA events from the
    first copy in to the last copy out."""
    dev = runner.dev
    host_in = {k: getattr(cfg, k).pin_memory() for k in ("q", "k", "v", "g", "beta", "do")
               if getattr(cfg, k) is not None}
    for k in ("h0", "dhT"):
        if getattr(cfg, k) is not None:
            host_in[k] = getattr(cfg, k).pin_memory()
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    with torch.cuda.stream(s_cmp):
        runners = [runner, Runner(cfg, dev, qk_l2norm=qk_l2norm, keep_context=runner.keep_context)]
    for r in runners:
        r.sp = ctypes.c_void_p(s_cmp.cuda_stream)

    def outs_of(r):
        return [r.o, r.dq, r.dk, r.dv, r.dg, r.db] + [t for t in (r.hT, r.dh0) if t is not None]

    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs_of(runner)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    ev = lambda: torch.cuda.Event()  # noqa: E731

    def run(n, start=None, end=None):
        torch.cuda.synchronize()
        done_cmp = [None, None]   # compute of the last step on each set (its inputs are free after it)
        done_out = [None, None]   # copy-out of the last step on each set (its outputs are free after it)
        if start is not None:
            start.record(s_in)
        last = None
        for i in range(n):
            b = i & 1
            r = runners[b]
            with torch.cuda.stream(s_in):
                if done_cmp[b] is not None:
                    s_in.wait_event(done_cmp[b])
                for k, t in host_in.items():
                    getattr(r.d, k).copy_(t, non_blocking=True)
                arrived = ev()
                arrived.record(s_in)
            s_cmp.wait_event(arrived)
            if done_out[b] is not None:
                s_cmp.wait_event(done_out[b])
            r.step()
            done_cmp[b] = ev()
            done_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_cmp[b])
                for dst, src in zip(host_out, outs_of(r)):
                    dst.copy_(src, non_blocking=True)
                done_out[b] = ev()
                done_out[b].record(s_out)
            last = done_out[b]
        if end is not None:
            s_in.wait_event(last)
            end.record(s_in)
        torch.cuda.synchronize()

    run(2)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(steps, a, b)
    for r in runners:
        r.sp = ctypes.c_void_p(runner.stream.cuda_stream)
    return a.elapsed_time(b) / steps, h2d, d2h


def kernel_split(runner, steps):
    """Per-kernel device time (CUDA events on the launching stream)."""
    lib = runner.lib
    _lib.timing_collect(lib)
    lib.kda_timing_enable(1)
    for _ in range(steps):
        runner.step()
    torch.cuda.synchronize()
    lib.kda_timing_enable(0)
    return _lib.timing_collect(lib)


def oracle_sample(cfg, units, seqs=1):
    """fp64 slices of the first ``seqs`` sequences holding ``units`` value heads
    (rounded up to whole q/k head groups), for the oracle, packed as one batch
    row with offsets."""
    r = cfg.HV // cfg.H
    hs = list(range((min(units, cfg.HV) + r - 1) // r))
    js = list(range(hs[0] * r, (hs[-1] + 1) * r))
    off = cfg.offsets()
    seqs = max(1, min(seqs, len(off) - 1))
    a, b = int(off[0]), int(off[seqs])
    sl = {}
    for k in ("q", "k", "v", "g", "beta", "do"):
        x = getattr(cfg, k)
        y = x.reshape(cfg.B * cfg.T, *x.shape[2:])[a:b]
        y = y[:, hs] if k in ("q", "k") else y[:, js]
        sl[k] = np.ascontiguousarray(y.to(torch.float64).numpy()[None])
    sl["cu"] = np.ascontiguousarray((off[:seqs + 1] - a).astype(np.int32))
    return sl, len(js), b - a


def run_oracle(sl, cores):
    import oracle
    oracle.kda_fwd(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], None, sl["cu"], False, nthreads=cores)
    oracle.kda_bwd(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], None, sl["do"], None, sl["cu"], nthreads=cores)


def cpu_baseline(cfg):
    """The fp64 oracle as it stands, on the host cores, on a bounded sample:
    whole (sequence, value head) units of the same workload, fwd + bwd."""
    cores = os.cpu_count() or 1
    # one sequence first, to size a sample of about ten seconds of CPU work
    sl, nj, L = oracle_sample(cfg, cfg.HV, 1)
    t0 = time.perf_counter()
    run_oracle(sl, cores)
    dt1 = time.perf_counter() - t0
    seqs = int(max(1, min(cfg.N, 10.0 // max(dt1, 1e-3))))
    if seqs > 1:
        sl, nj, L = oracle_sample(cfg, cfg.HV, seqs)
        t0 = time.perf_counter()
        run_oracle(sl, cores)
        dt = time.perf_counter() - t0
    else:
        dt = dt1
    value = L * nj / cfg.HV / dt  # a layer token needs all HV value heads
    return dict(value=round(value, 2), unit="tokens/s", cores=min(cores, seqs * nj), kind="oracle",
                sample=f"the first {seqs} of {cfg.N} sequences, {nj} of {cfg.HV} value heads, {L} tokens, "
                       f"fwd+bwd in fp64 ({dt:.1f} s); tokens/s = tokens x heads / HV / seconds")


# --------------------------------------------------------------------------
def job_throughput(ms_local, tokens_per_rank, steps, dist=None, device="cpu"):
    """Whole-job tokens/s for weak scaling: every rank processes tokens_per_rank
    per step; the job's time is the slowest rank's (max over ranks).  Returns
    (tokens/s, max ms over ranks for the timed steps)."""
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    world = 1
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        world = dist.get_world_size()
    ms = float(t.item())
    return tokens_per_rank * world / (ms / steps / 1e3), ms


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=WORKLOAD_CFG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=["step", "fwd", "bwd"], default="step",
                    help="time only the forward or only the backward call (profiling aid)")
    ap.add_argument("--qk-l2norm", action="store_true",
                    help="the same layer with the q/k L2-norm prologue inside the op")
    ap.add_argument("--scalar-gate", action="store_true",
                    help="the same layer with a scalar gate g [B, T, HV] (the GDN variant)")
    ap.add_argument("--head-dim", type=int, default=None, choices=(64, 128),
                    help="the same layer with K = V = this head dim (64: the pages' benchmark head dim)")
    ap.add_argument("--kda-gate", action="store_true",
                    help="the same layer with the KDA gate inside the op (raw gate, A_log and bias in, their "
                         "gradients out; unbounded)")
    ap.add_argument("--cp-ranks", type=int, default=0,
                    help="context parallelism: split every sequence into this many segments and run the state "
                         "relay, the ranks serialized on this GPU (measures the relay's per-rank work)")
    ap.add_argument("--recompute", action="store_true",
                    help="time the recompute pair (kda_chunk_fwd + kda_chunk_bwd) instead of the forward-context "
                         "pair: the backward re-runs the record kernel and the states pass")
    ap.add_argument("--segments", type=int, default=0,
                    help="split every sequence into this many segments that run at once on this GPU, with the "
                         "state relay (for few long sequences); the dense workloads only")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip timing the other backward mode (profiling aid: only this mode's kernels launch)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="profiling aid: the dense workload with T replaced (e.g. 1024 for small ncu captures); "
                         "the JSON line names the changed workload")
    args = ap.parse_args()
    warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return reference_arm(args, warmup)

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    if args.seq_len is not None or args.scalar_gate or args.kda_gate or args.head_dim:  # a variant of the layer
        name, kw = inputs.CONFIGS[args.config]
        if args.head_dim and args.head_dim != kw["K"]:
            kw = dict(kw, K=args.head_dim, V=args.head_dim)
            name = name.replace(f"K{inputs.CONFIGS[args.config][1]['K']}", f"K{args.head_dim}")
        if args.seq_len is not None:
            assert kw.get("cu_seqlens") is None and "T" in kw, "--seq-len needs a dense configuration"
            kw = dict(kw, T=args.seq_len)
            name = f"{name}_T{args.seq_len}"
        if args.scalar_gate:
            kw = dict(kw, scalar_gate=True)
            name = f"{name}_scalar_gate"
        if args.kda_gate:
            kw = dict(kw, raw_gate=True)
            name = f"{name}_kda_gate"
        cfg = inputs.make_inputs(seed=1000 + args.config + 7919 * rank, name=name, **kw)
    else:
        cfg = inputs.make_config(args.config, seed=1000 + args.config + 7919 * rank)
    runner = Runner(cfg, dev, qk_l2norm=args.qk_l2norm, keep_context=not args.recompute)
    if args.cp_ranks > 1:  # context parallelism, the ranks serialized on this GPU
        runner.step = cp_step_fn(runner, args.cp_ranks)
        args.no_e2e = True
    if args.segments > 1:  # every sequence in segments that run at once, with the state relay
        runner.step = segmented_step_fn(runner, args.segments, args.qk_l2norm)
        args.no_e2e = True
    if args.only != "step":  # profiling aid: time one half of the step only
        runner.step = runner.fwd if args.only == "fwd" else runner.bwd
        args.no_e2e = args.no_cpu_baseline = True
    for _ in range(warmup):
        runner.step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    n0 = runner.lib.kda_launch_count()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.begin()
    ms = timed(runner.step, args.steps, runner.stream)
    clocks.end()
    if dist:
        dist.barrier()
    launches = runner.lib.kda_launch_count() - n0
    ck = clocks.stop() if rank == 0 else None
    value, ms = job_throughput(ms, cfg.valid_tokens, args.steps, dist, device=dev)

    split = kernel_split(runner, max(3, min(args.steps, 10)))
    other = None  # the other backward mode, timed the same way, for comparison
    if args.only == "step" and args.cp_ranks <= 1 and args.segments <= 1 and not args.no_compare:
        alt = Runner(cfg, dev, qk_l2norm=args.qk_l2norm, keep_context=args.recompute)
        for _ in range(warmup):
            alt.step()
        a_ms = timed(alt.step, args.steps, alt.stream)
        a_value, a_ms = job_throughput(a_ms, cfg.valid_tokens, args.steps, dist, device=dev)
        other = dict(backward="forward context kept" if args.recompute else "recompute",
                     value=round(a_value, 1), ms_per_step=round(a_ms / args.steps, 4))
        del alt
    e2e = None
    if not args.no_e2e:
        e_ms, h2d, d2h = e2e_measure(cfg, runner, max(3, args.steps), args.qk_l2norm)  # pipeline fill amortised like a training loop
        e_value, e_ms = job_throughput(e_ms, cfg.valid_tokens, 1, dist, device=dev)  # ms per step, max over ranks
        e2e = (e_value, e_ms, h2d, d2h)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    peaks = load_peaks()
    ms_step = ms / args.steps
    toks = cfg.valid_tokens
    ab = algorithmic_bytes(cfg)
    af = algorithmic_flops(cfg)
    t_hbm = ab["total"] / (peaks["hbm"] * 1e9)
    t_tc = af / (peaks["bf16_sust"] * 1e12 if peaks.get("bf16_sust") else peaks["bf16"] * 1e12)
    roof_s = max(t_hbm, t_tc)

    # dominant kernel
    steps_split = max(3, min(args.steps, 10))
    per_step = {k: v[0] / steps_split for k, v in split.items()}
    dom = max(split, key=lambda k: split[k][0])
    dom_ms, dom_n = split[dom]
    # the captures are of the dense layer's kernels (K = V = 128, the gate as given, no L2-norm
    # prologue): their traffic per token holds for this workload and its length variants only
    captured = (cfg.K == 128 and cfg.V == 128 and cfg.H == 32 and cfg.HV == 32 and not args.qk_l2norm
                and not args.scalar_gate and not args.kda_gate and not args.recompute and args.cp_ranks == 1
                and args.segments == 1)
    roof = dominant_roofline(dom, dom_ms / dom_n, cfg, toks / max(1, args.cp_ranks), peaks)
    if not captured:
        roof["traffic"] = None
    traffic = step_traffic(split, steps_split, toks) if captured else None
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.name, "B": cfg.B, "T": cfg.T, "H": cfg.H, "HV": cfg.HV, "K": cfg.K,
                   "V": cfg.V, "global_batch": cfg.B * world, "seq_len": cfg.T,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": f"inputs {ab['fwd'] / 1e9:.2f} GB read per step > L2 (no flush)",
                   "qk_l2norm": bool(args.qk_l2norm), "scalar_gate": bool(args.scalar_gate),
                   "kda_gate": bool(args.kda_gate),
                   "backward": "recompute" if args.recompute else "forward context kept",
                   "forward_context_bytes": int(runner.ctx_bytes),
                   **({"cp_ranks": args.cp_ranks, "cp": "sequences split into cp_ranks segments, state relay, "
                       "ranks serialized on one GPU"} if args.cp_ranks > 1 else {}),
                   **({"segments": args.segments, "segmented": "every sequence split into segments that run at "
                       "once, state relay"} if args.segments > 1 else {})},
        "roofline": roof,
        "step_roofline": {"bound": "hbm" if t_hbm >= t_tc else "tensor",
                          "algorithmic_bytes": ab["total"], "algorithmic_flops": af,
                          "roofline_ms": round(roof_s * 1e3, 4),
                          "achieved_GBps": round(ab["total"] / (ms_step / 1e3) / 1e9, 1),
                          "frac": round(roof_s / (ms_step / 1e3), 4),
                          "traffic": traffic,
                          "traffic_vs_algorithmic": None if traffic is None else round(traffic / ab["total"], 3),
                          "peaks": {"hbm_gbs": peaks["hbm"], "bf16_tflops": peaks["bf16"],
                                    "source": peaks["src"]}},
        "kernel_ms_per_step": {k: round(v, 4) for k, v in sorted(per_step.items(), key=lambda x: -x[1])},
        "gpu_launches": int(launches),
        **({"other_backward_mode": other} if other is not None else {}),
        "clocks": ck,
    }
    if e2e is not None:
        e_value, e_ms, h2d, d2h = e2e
        out["e2e"] = {"value": round(e_value, 1), "unit": "tokens/s", "ms_per_step": round(e_ms, 3),
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg)
    print(json.dumps(out))
    if dist:
        dist.destroy_process_group()
    return 0


def reference_arm(args, warmup):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample of the workload (batch row 0, a few value heads, fwd+bwd)."""
    cfg = inputs.make_config(args.config)
    cores = os.cpu_count() or 1
    # one (sequence, value head) unit per host core: the oracle threads over units
    sl, nj, L = oracle_sample(cfg, cores)
    used = min(cores, nj)
    for _ in range(warmup):
        run_oracle(sl, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle(sl, cores)
    dt = (time.perf_counter() - t0) / args.steps
    value = L * nj / cfg.HV / dt
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
           "n_gpus": 0, "steps": args.steps, "warmup": warmup, "ms_per_step": round(dt * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": cfg.name, "B": cfg.B, "T": cfg.T, "H": cfg.H, "HV": cfg.HV,
                      "K": cfg.K, "V": cfg.V, "parallelism": "host threads"},
           "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": used, "kind": "oracle",
                            "sample": f"per step: the first sequence, {nj} of {cfg.HV} value heads x {L} tokens, "
                                      f"fwd+bwd fp64; tokens/s = tokens x heads / HV / seconds"},
           "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return 0


if __name__ == "__main__":
    sys.exit(main())
