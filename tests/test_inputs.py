"""Seeded input generators: shapes, determinism and the packed-batch recipe."""
import numpy as np
import torch

from gated_delta_rule_42_gb300 import inputs


def test_tiny_config_shapes_and_determinism():
    a = inputs.make_config(0)
    b = inputs.make_config(0)
    assert a.q.shape == (1, 256, 2, 64) and a.g.shape == (1, 256, 2, 64)
    assert a.h0.shape == (1, 2, 64, 64) and a.dtype == torch.float32
    for x, y in ((a.q, b.q), (a.g, b.g), (a.beta, b.beta), (a.h0, b.h0), (a.do, b.do)):
        assert torch.equal(x, y)
    assert float(a.g.max()) <= 0.0 and float(a.g.min()) >= -5.0
    assert float(a.beta.min()) > 0.0 and float(a.beta.max()) < 1.0
    n = a.q.double().norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-6)


def test_varlen_gva_config_offsets():
    c = inputs.make_inputs(name="x", seed=1001, B=1, T=4096, H=4, HV=8, K=16, V=16,
                           cu_seqlens=[0, 3, 73, 73, 1100, 4096], dtype=torch.bfloat16)
    assert c.N == 5 and c.cu_seqlens.dtype == torch.int32
    assert c.h0.shape == (5, 8, 16, 16) and c.q.dtype == torch.bfloat16


def test_packed_lengths_recipe():
    rng = np.random.Generator(np.random.PCG64(1004))
    cu = inputs._packed_varlen_offsets(rng)
    lens = np.diff(cu)
    assert len(cu) == 69 and cu[0] == 0 and cu[-1] == 131072
    assert [i for i, l in enumerate(lens) if l == 0] == [0, 21, 42, 67]
    nz = lens[lens > 0]
    assert len(nz) == 64 and nz.min() >= 1 and nz.max() <= 8192
    assert nz.max() > 1000 and nz.min() < 200  # log-uniform spread
