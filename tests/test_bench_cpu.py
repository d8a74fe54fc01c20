"""The benchmark's roofline arithmetic, pinned on the host: the algorithmic
bytes and flops of the dense training layer (per token and value head), each
tensor-core kernel's share of them (what the dominant kernel's roofline
divides by), its interface bytes (a diagnostic), and the rule that measured
DRAM traffic (the dominant kernel's, and the step's sum over its kernels) is
reported only while each kernel's sources match its capture."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gated_delta_rule_42_gb300 import inputs  # noqa: E402


def _layer(**kw):
    # the dense training layer's head shape; per-token figures do not depend on T
    return inputs.make_inputs(B=1, T=64, H=32, HV=32, K=128, V=128, dtype=torch.bfloat16, h0=False,
                              final_state=False, seed=1, **kw)


def test_algorithmic_cost_per_token_head():
    cfg = _layer()
    # fwd: q, k, v, g, beta in, o out; bwd: the same plus dO in, dq, dk, dv, dg, dbeta out
    e, K, V = 2, 128, 128
    fwd = 2 * K * e + V * e + 4 * K + 4 + V * e
    bwd = fwd + 2 * K * e + V * e + 4 * K + 4
    assert bench.algorithmic_bytes(cfg)["per_token_head"] == fwd + bwd == 4364
    # 18 d^2 + 15 C d + 2 C^2 at d = 128, C = 64
    assert bench.algorithmic_flops(cfg) / (cfg.valid_tokens * cfg.HV) == 18 * 128 ** 2 + 15 * 64 * 128 + 2 * 64 ** 2
    # a scalar gate moves one fp32 per (token, value head) instead of K of them, three times
    assert bench.algorithmic_bytes(_layer(scalar_gate=True))["per_token_head"] == 4364 - 3 * (4 * K - 4)


def test_interface_bytes_per_token_of_the_tensor_core_kernels():
    cfg = _layer()
    want = {"kda_prep_tc": 65920, "kda_fwd_tc": 49408, "kda_fwd_tc_states": 61696, "kda_fwd_tc_save": 82176,
            "kda_bwd_scan_tc": 73984, "kda_bwd_intra_tc": 160000}
    for name, b in want.items():
        assert bench.kernel_bytes_per_token(name, cfg) == b, name
    assert bench.kernel_bytes_per_token("no_such_kernel", cfg) is None


def test_algorithmic_bytes_per_token_of_the_tensor_core_kernels():
    """The dominant kernel's roofline divides its share of the step's algorithmic
    bytes: the gradient kernel reads q, k, v, g, beta, dO and writes dq, dk, dv,
    dg, dbeta -- 90,368 bytes per token of the dense training layer."""
    cfg = _layer()
    assert bench.kernel_algorithmic_bytes_per_token("kda_bwd_intra_tc", cfg) == 90368
    assert bench.kernel_algorithmic_bytes_per_token("kda_prep_tc", cfg) == 2 * 8192 + 16384 + 128
    assert bench.kernel_algorithmic_bytes_per_token("kda_fwd_tc_save", cfg) == 2 * 8192
    assert bench.kernel_algorithmic_bytes_per_token("kda_bwd_scan_tc", cfg) == 8192
    # the forward kernels and the backward kernels together cover the step's bytes once each,
    # except dO, which the reverse scan and the gradient kernel both read
    step = bench.algorithmic_bytes(cfg)["per_token_head"] * cfg.HV
    parts = sum(bench.kernel_algorithmic_bytes_per_token(k, cfg)
                for k in ("kda_prep_tc", "kda_fwd_tc_save", "kda_bwd_scan_tc", "kda_bwd_intra_tc"))
    assert parts == step + 8192


def test_dominant_roofline_fraction_is_algorithmic_bytes_over_time():
    cfg = _layer()
    peaks = dict(hbm=6791.4, src="measured")
    r = bench.dominant_roofline("kda_bwd_intra_tc", 1.866, cfg, 32768, peaks)
    assert r["algorithmic_bytes"] == 90368 * 32768
    assert abs(r["achieved"] - 90368 * 32768 / 1.866e-3 / 1e9) < 0.1
    assert abs(r["frac"] - r["achieved"] / 6791.4) < 1e-4
    assert 0.23 < r["frac"] < 0.24  # 2.96 GB in 1.866 ms on 6.79 TB/s
    assert r["interface"]["bytes"] == 160000 * 32768


def test_traffic_is_reported_only_for_the_captured_sources():
    t = bench.NCU_TRAFFIC["kda_bwd_intra_tc"]
    current = bench.sources_sha256(t["sources"]) == t["sha256"]
    got = bench.measured_traffic("kda_bwd_intra_tc", 8192)
    assert (got is not None) == current
    if current:  # the capture's own size gives back its bytes
        assert abs(got - t["bytes_per_token"] * 8192) <= 1
    assert bench.measured_traffic("chunk_map_kernel", 8192) is None  # no capture recorded for it


def test_step_traffic_needs_a_capture_for_every_kernel_that_matters():
    split = {"kda_bwd_intra_tc": (15.6, 10), "kda_prep_tc": (5.6, 10), "kda_fwd_tc_save": (4.2, 10),
             "kda_bwd_scan_tc": (3.6, 10), "chunk_map_kernel": (0.16, 20)}
    current = all(bench.sources_sha256(bench.NCU_TRAFFIC[k]["sources"]) == bench.NCU_TRAFFIC[k]["sha256"]
                  for k in ("kda_bwd_intra_tc", "kda_prep_tc", "kda_fwd_tc_save", "kda_bwd_scan_tc"))
    got = bench.step_traffic(split, 10, 8192)
    assert (got is not None) == current
    if current:  # one launch of each per step; the chunk map (under 1 % of the time) is left out
        want = sum(bench.NCU_TRAFFIC[k]["bytes_per_token"] * 8192 for k in list(split)[:4])
        assert abs(got - want) <= 4
    assert bench.step_traffic(dict(split, other_kernel=(5.0, 10)), 10, 8192) is None


def test_clock_sampler_keeps_the_samples_of_the_timed_region():
    """Samples count only when they arrive between begin() and end() plus one
    interval (or, for a region shorter than an interval, the first one after
    begin()); a slowdown reason outside the region is not reported."""
    class _Proc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    def line(mhz, hw="Not Active"):
        return f"0, {mhz}, 2070, 900.0, 0x0, {hw}, Not Active, Not Active, Not Active"

    s = bench.ClockSampler(0)
    s.proc = _Proc()
    s.INTERVAL_MS = 0  # (no wait for a last sample in the test)
    s.t_begin, s.t_end = 10.0, 10.1
    s.lines = [(9.9, line(1200, "Active")), (10.02, line(2070)), (10.07, line(2065)), (10.5, line(1000, "Active"))]
    got = s.stop()
    assert got["samples"] == 2 and got["sm_mhz"] == 2067.5 and got["reasons"] == []
    s2 = bench.ClockSampler(0)
    s2.proc = _Proc()
    s2.INTERVAL_MS = 0
    s2.t_begin, s2.t_end = 10.0, 10.001
    s2.lines = [(9.9, line(1200)), (10.03, line(2070, "Active")), (10.06, line(2060))]
    got = s2.stop()
    assert got["samples"] == 1 and got["sm_mhz"] == 2070 and got["reasons"] == ["hw_slowdown"]
