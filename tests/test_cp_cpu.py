"""The context-parallel state relay's host logic on CPU ranks (gloo, world
size 2): each rank runs the fp64 oracle on its segment of the sequences (in
place of the GPU kernels), and the relay's exchange and scans
(``relay_start_state``, ``relay_end_grad``) must reproduce the unsplit
oracle: the start state at the split, every output and gradient of both
segments, the final state and the initial-state gradient."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from gated_delta_rule_42_gb300 import cp

T, SPLIT, B, H, HV, K, V = 40, 23, 2, 1, 2, 3, 2


def _problem():
    rng = np.random.default_rng(41)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, HV, V))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, HV, K))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, HV))))
    h0 = rng.standard_normal((B, HV, K, V))
    do = rng.standard_normal((B, T, HV, V))
    dhT = rng.standard_normal((B, HV, K, V))
    return q, k, v, g, beta, h0, do, dhT


def _cpu_compose(M, h, c, transpose):
    return (M.transpose(-1, -2) if transpose else M) @ h + c


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, g, beta, h0, do, dhT = _problem()
        seg = slice(0, SPLIT) if rank == 0 else slice(SPLIT, T)
        qs, ks, vs, gs, bs, dos = (x[:, seg] for x in (q, k, v, g, beta, do))
        gather = cp.all_gather_fn()
        # the segment's affine map: c from a zero start, M from v = 0, h0 = I
        _, c = oracle.kda_fwd(qs, ks, vs, gs, bs, None, nthreads=1)
        eye = np.broadcast_to(np.eye(K), (B, HV, K, K)).copy()
        _, M = oracle.kda_fwd(qs, ks, np.zeros(vs.shape[:3] + (K,)), gs, bs, eye, nthreads=1)
        # h0 held by rank 0 only, dhT by the last rank only: the relay fetches them
        hs = cp.relay_start_state(torch.from_numpy(c), torch.from_numpy(M),
                                  torch.from_numpy(h0) if rank == 0 else None, rank, gather, _cpu_compose).numpy()
        o, hT = oracle.kda_fwd(qs, ks, vs, gs, bs, hs, nthreads=1)
        d = oracle.kda_bwd(qs, ks, vs, gs, bs, hs, dos, None, nthreads=1)["dh0"]
        dh_end = cp.relay_end_grad(torch.from_numpy(d), torch.from_numpy(M),
                                   torch.from_numpy(dhT) if rank == world - 1 else None, rank, world, gather,
                                   _cpu_compose).numpy()
        gr = oracle.kda_bwd(qs, ks, vs, gs, bs, hs, dos, dh_end, nthreads=1)
        out[rank] = dict(hs=hs, o=o, hT=hT, **gr)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_state_relay_two_gloo_ranks_match_the_unsplit_oracle():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:  # no fork of a multi-threaded parent
        out = mgr.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = {r: dict(out[r]) for r in (0, 1)}
    q, k, v, g, beta, h0, do, dhT = _problem()
    o, hT = oracle.kda_fwd(q, k, v, g, beta, h0, nthreads=1)
    gr = oracle.kda_bwd(q, k, v, g, beta, h0, do, dhT, nthreads=1)
    _, h_split = oracle.kda_fwd(q[:, :SPLIT], k[:, :SPLIT], v[:, :SPLIT], g[:, :SPLIT], beta[:, :SPLIT], h0,
                                nthreads=1)
    np.testing.assert_allclose(res[0]["hs"], h0, rtol=0, atol=0)
    np.testing.assert_allclose(res[1]["hs"], h_split, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.concatenate([res[0]["o"], res[1]["o"]], axis=1), o, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(res[1]["hT"], hT, rtol=1e-11, atol=1e-11)
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(np.concatenate([res[0][key], res[1][key]], axis=1), gr[key],
                                   rtol=1e-10, atol=1e-10, err_msg=key)
    np.testing.assert_allclose(res[0]["dh0"], gr["dh0"], rtol=1e-10, atol=1e-10)


def test_segment_offsets():
    from gated_delta_rule_42_gb300.segments import segment_offsets
    cu = segment_offsets(2, 1024, 4, "cpu")
    assert cu.tolist() == [0, 256, 512, 768, 1024, 1280, 1536, 1792, 2048]
    for T, S in ((1000, 4), (1024, 3), (1024, 32)):  # not whole 64-token chunks per segment
        with pytest.raises(ValueError):
            segment_offsets(1, T, S, "cpu")
