"""Seeded synthetic inputs for chunked KDA (Kimi Delta Attention).

This module is shared by the CUDA path's tests/bench and by the fp64 oracle's
tests.  It holds no arithmetic of the method itself: it only draws random
tensors with the shapes, value distributions and packing structure of the
workloads the KDA pages test on (dense and ``cu_seqlens``-packed batches,
grouped value heads, optional initial / final state), and casts them to the
dtype the kernels consume.

Distributions (one generator, numpy PCG64, values drawn in this order:
sequence lengths (packed batches only), q, k, v, beta, g, h0, dO, dhT):

* q, k ~ N(0, 1), each (token, head) row L2-normalised, then cast;
* v ~ N(0, 1);
* beta = sigmoid(N(0, 1)), one per (token, value head);
* g = clip(-softplus(N(mu, 1)), -5, 0): a per-token, per-channel log2 decay
  (mu = 0, or -3 for the near-1 decays of the long-context case; strong-decay
  test cases widen the spread and the clip);
* h0 ~ 0.1 * N(0, 1); dO ~ N(0, 1); dhT ~ 0.1 * N(0, 1).

The packed-varlen contract (device int32 offsets, repeated offsets = empty
slots, one state per logical sequence) follows the ``recurrent_kda`` entry
point described in "kda in torchtitan (training)" (pytorch/torchtitan PR
#4164, the agent note on the public ``recurrent_kda`` interface).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

__all__ = ["KdaInputs", "make_inputs", "make_config", "CONFIGS", "packed_lengths"]


@dataclass
class KdaInputs:
    """One synthetic problem.  Tensors live on the host (CPU) in the dtype
    the GPU path consumes; ``to(device)`` moves them.

    Layout (token axis packed, like the pages' varlen contract):
      q, k  [B, T, H, K]    v, dO  [B, T, HV, V]
      g     [B, T, HV, K]   beta   [B, T, HV]       (fp32)
      h0, dhT [N, HV, K, V] (fp32, or None)
    ``cu_seqlens`` (int32 [N+1]) requires B == 1; otherwise N == B.
    """

    name: str
    B: int
    T: int
    H: int
    HV: int
    K: int
    V: int
    dtype: torch.dtype
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    h0: Optional[torch.Tensor]
    do: torch.Tensor
    dhT: Optional[torch.Tensor]
    cu_seqlens: Optional[torch.Tensor]
    output_final_state: bool
    seed: int
    meta: dict = field(default_factory=dict)
    # KDA gate inside the op: g then holds raw pre-activations, with these parameters
    A_log: Optional[torch.Tensor] = None     # [HV] fp32
    g_bias: Optional[torch.Tensor] = None    # [HV, K] fp32
    lower_bound: Optional[float] = None      # None: the unbounded gate

    @property
    def gate(self) -> Optional[dict]:
        """The oracle's gate parameters (fp64 numpy), or None without the gate."""
        if not self.meta.get("raw_gate"):
            return None
        c = (lambda x: None if x is None else x.detach().cpu().to(torch.float64).numpy())
        return dict(A_log=c(self.A_log), bias=c(self.g_bias), lower_bound=self.lower_bound)

    @property
    def N(self) -> int:
        return self.B if self.cu_seqlens is None else int(self.cu_seqlens.numel()) - 1

    @property
    def valid_tokens(self) -> int:
        if self.cu_seqlens is None:
            return self.B * self.T
        return int(self.cu_seqlens[-1])

    def offsets(self) -> np.ndarray:
        """int64 [N+1] token offsets into the packed token axis (B*T rows)."""
        if self.cu_seqlens is None:
            return np.arange(self.B + 1, dtype=np.int64) * self.T
        return self.cu_seqlens.numpy().astype(np.int64)

    def to(self, device) -> "KdaInputs":
        def mv(x):
            return None if x is None else x.to(device)

        return KdaInputs(
            self.name, self.B, self.T, self.H, self.HV, self.K, self.V, self.dtype,
            mv(self.q), mv(self.k), mv(self.v), mv(self.g), mv(self.beta), mv(self.h0),
            mv(self.do), mv(self.dhT), mv(self.cu_seqlens), self.output_final_state,
            self.seed, dict(self.meta), mv(self.A_log), mv(self.g_bias), self.lower_bound)

    def f64(self) -> dict:
        """Exact fp64 copies (numpy) of every input, as the oracle consumes them.
        bf16 -> fp64 and fp32 -> fp64 are exact, so both sides see the same
        numbers."""
        def c(x):
            return None if x is None else x.detach().cpu().to(torch.float64).numpy()

        return dict(q=c(self.q), k=c(self.k), v=c(self.v), g=c(self.g), beta=c(self.beta),
                    h0=c(self.h0), do=c(self.do), dhT=c(self.dhT))


def _normal(rng: np.random.Generator, shape, mean=0.0, std=1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x


def _l2_rows(x: np.ndarray) -> np.ndarray:
    # Row normalisation of the last axis, in fp64 for the norm.
    n = np.sqrt(np.einsum("...k,...k->...", x.astype(np.float64), x.astype(np.float64)))
    n = np.maximum(n, 1e-12)
    return (x / n[..., None]).astype(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def _neg_softplus_clipped(x: np.ndarray, lo: float = -5.0) -> np.ndarray:
    x64 = x.astype(np.float64)
    sp = np.where(x64 > 20, x64, np.log1p(np.exp(np.minimum(x64, 20))))
    return np.clip(-sp, lo, 0.0).astype(np.float32)


def packed_lengths(rng: np.random.Generator, n_seq: int, total: int, lo: int, hi: int) -> np.ndarray:
    """Log-uniform lengths in [lo, hi], rescaled so they sum to exactly ``total``.

    Draw n_seq values exp(U(ln lo, ln hi)); repeatedly rescale the unclamped
    values so the clamped sum hits ``total`` (clamping to [lo, hi]) until
    stable; floor, then hand out the remainder +1 each by largest fractional
    part (ties: lower index first)."""
    raw = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n_seq))
    scale = 1.0
    for _ in range(200):
        cl = np.clip(raw * scale, lo, hi)
        s = cl.sum()
        if abs(s - total) < 1e-9 * total:
            break
        free = (raw * scale > lo) & (raw * scale < hi)
        fs = cl[free].sum()
        if fs <= 0:
            break
        scale *= 1.0 + (total - s) / fs
    cl = np.clip(raw * scale, lo, hi)
    fl = np.floor(cl).astype(np.int64)
    fl = np.clip(fl, lo, hi)
    rem = int(total - fl.sum())
    order = sorted(range(n_seq), key=lambda i: (-(cl[i] - math.floor(cl[i])), i))
    i = 0
    guard = 0
    while rem != 0 and guard < 10 * n_seq * max(1, abs(rem)):
        j = order[i % n_seq]
        if rem > 0 and fl[j] < hi:
            fl[j] += 1
            rem -= 1
        elif rem < 0 and fl[j] > lo:
            fl[j] -= 1
            rem += 1
        i += 1
        guard += 1
    assert int(fl.sum()) == total, (fl.sum(), total)
    return fl


def make_inputs(*, B: int, T: int, H: int, HV: int, K: int, V: int, dtype=torch.bfloat16,
                cu_seqlens=None, lengths_fn=None, h0: bool = True, final_state: bool = True,
                dhT: Optional[bool] = None, g_mean: float = 0.0, seed: int = 0,
                name: str = "custom", scalar_gate: bool = False, g_std: float = 1.0,
                g_lo: float = -5.0, raw_gate: bool = False, A_log: Optional[bool] = None,
                g_bias: Optional[bool] = None, lower_bound: Optional[float] = None) -> KdaInputs:
    """Draw one problem.  ``cu_seqlens`` may be a list of offsets (B must be 1);
    ``lengths_fn(rng)`` may instead return the offsets from the generator.
    ``scalar_gate`` draws g as [B, T, HV] (one decay per token and value head).
    The gate is clip(-softplus(N(g_mean, g_std)), g_lo, 0); the workloads keep
    the defaults (std 1, clip at -5), the strong-decay cases widen both.
    ``raw_gate`` draws g as raw pre-activations N(g_mean, g_std) for the KDA
    gate inside the op instead, and then (after every other draw) A_log ~
    0.5 N(0, 1) [HV] and g_bias ~ 0.5 N(0, 1) [HV, K] unless A_log / g_bias is
    False; ``lower_bound`` selects the bounded gate."""
    rng = np.random.Generator(np.random.PCG64(seed))
    cu = None
    if lengths_fn is not None:
        cu = np.asarray(lengths_fn(rng), dtype=np.int64)
    elif cu_seqlens is not None:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
    if cu is not None:
        assert B == 1, "packed batches use B == 1"
        assert cu[0] == 0 and np.all(np.diff(cu) >= 0) and cu[-1] <= T
    N = B if cu is None else len(cu) - 1

    q = _l2_rows(_normal(rng, (B, T, H, K)))
    k = _l2_rows(_normal(rng, (B, T, H, K)))
    v = _normal(rng, (B, T, HV, V))
    beta = _sigmoid(_normal(rng, (B, T, HV)))
    graw = _normal(rng, (B, T, HV) if scalar_gate else (B, T, HV, K), mean=g_mean, std=g_std)
    g = graw if raw_gate else _neg_softplus_clipped(graw, lo=g_lo)
    h0_t = _normal(rng, (N, HV, K, V), std=0.1) if h0 else None
    do = _normal(rng, (B, T, HV, V))
    if dhT is None:
        dhT = final_state
    dhT_t = _normal(rng, (N, HV, K, V), std=0.1) if dhT else None

    def t(x, dt):
        return torch.from_numpy(x).to(dt)

    A_t = bias_t = None
    if raw_gate:
        if A_log is not False:
            A_t = torch.from_numpy(_normal(rng, (HV,), std=0.5))
        if g_bias is not False:
            bias_t = torch.from_numpy(_normal(rng, (HV, K), std=0.5))

    return KdaInputs(
        name=name, B=B, T=T, H=H, HV=HV, K=K, V=V, dtype=dtype,
        q=t(q, dtype), k=t(k, dtype), v=t(v, dtype),
        g=torch.from_numpy(g), beta=torch.from_numpy(beta),
        h0=None if h0_t is None else torch.from_numpy(h0_t),
        do=t(do, dtype),
        dhT=None if dhT_t is None else torch.from_numpy(dhT_t),
        cu_seqlens=None if cu is None else torch.from_numpy(cu.astype(np.int32)),
        output_final_state=final_state, seed=seed, meta=dict(raw_gate=raw_gate),
        A_log=A_t, g_bias=bias_t, lower_bound=lower_bound)


def _packed_varlen_offsets(rng: np.random.Generator) -> np.ndarray:
    lens = list(packed_lengths(rng, 64, 131072, 1, 8192))
    for pos in (0, 21, 42, 67):  # empty slots: leading, interior, trailing
        lens.insert(pos, 0)
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)


# The five workloads: (name, kwargs).  Seed = 1000 + index.
CONFIGS = [
    ("tiny_dense_f32_T256_H2_K64",
     dict(B=1, T=256, H=2, HV=2, K=64, V=64, dtype=torch.float32, h0=True, final_state=True)),
    ("varlen_gva_bf16_T4096_H4_HV8_K128",
     dict(B=1, T=4096, H=4, HV=8, K=128, V=128, dtype=torch.bfloat16,
          cu_seqlens=[0, 3, 73, 73, 1100, 4096], h0=True, final_state=True)),
    ("dense_train_bf16_B8_T4096_H32_K128",
     dict(B=8, T=4096, H=32, HV=32, K=128, V=128, dtype=torch.bfloat16, h0=False,
          final_state=False)),
    ("long_ctx_bf16_T65536_H16_K128",
     dict(B=1, T=65536, H=16, HV=16, K=128, V=128, dtype=torch.bfloat16, h0=True,
          final_state=True, g_mean=-3.0)),
    ("packed_varlen_bf16_T131072_H16_HV32_K128",
     dict(B=1, T=131072, H=16, HV=32, K=128, V=128, dtype=torch.bfloat16,
          lengths_fn=_packed_varlen_offsets, h0=True, final_state=True)),
]


def make_config(i: int, seed: Optional[int] = None) -> KdaInputs:
    name, kw = CONFIGS[i]
    return make_inputs(seed=1000 + i if seed is None else seed, name=name, **kw)
