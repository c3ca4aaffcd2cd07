"""Sharded Muon on the GPU: NCCL collectives around the CUDA muon_step (one rank; GPU).

This run has one GPU, so the process group has one rank: the reduce-scatter and all-gather run
through NCCL in place on the flat buffers and the whole set is owned locally. The result must be
bitwise the one muon_step gives on the same data outside the sharded path, and match the oracle.
The exchange between several ranks is covered on CPU with gloo in test_sharded.py.
"""
import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
import workloads as wl
from gpu_util import bf16_ulp, dev, host

pytestmark = pytest.mark.gpu

CUBIC = (1.5, -0.5, 0.0)
SHAPES = [(256, 640), (640, 256), (130, 70), (384, 384), (1, 5)]


def test_sharded_single_rank_nccl_matches_plain_step():
    from muon_newton_schulz_09_b300 import Muon, ShardedMuon
    w = wl.small_workload("sh", SHAPES, kind="step", dtype="bf16", param_dtype="bf16", grad_std=1e-3,
                          spike_rank=2, spike_gain=20.0, seed=81)
    g = [wl.gradient(w, j) for j in range(w.count)]
    m = [wl.momentum_buffer(w, j) for j in range(w.count)]
    p = [wl.parameter(w, j) for j in range(w.count)]
    lr = 0.02
    dist.init_process_group("nccl", store=dist.HashStore(), rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    try:
        sm = ShardedMuon(SHAPES, 0, 1, device=0, lr=lr, beta=0.95, nesterov=True)
        for j in range(w.count):
            sm.params[j].copy_(dev(p[j], "bf16"))
            sm.grads[j].copy_(dev(g[j], "bf16"))
            sm.momentum[j].copy_(dev(m[j], "f32"))
        sm.step()
        torch.cuda.synchronize()
        assert sm.muon.get_error() == 0
        got = [t.clone() for t in sm.params]
        sm.close()
    finally:
        dist.destroy_process_group()
    P = [dev(x, "bf16") for x in p]
    with Muon(0) as mu:
        mu.step(P, [dev(x, "bf16") for x in g], [dev(x, "f32") for x in m], lr=lr, beta=0.95, nesterov=True)
        torch.cuda.synchronize()
    for j, (r, c) in enumerate(SHAPES):
        assert torch.equal(got[j], P[j]), (r, c)
        w_new, _, o = oracle.muon_step(p[j], g[j], m[j], lr, 0.95, True, 5, CUBIC)
        upd = lr * oracle.lr_scale(r, c) * np.abs(o).max()
        err = np.abs(host(got[j]) - w_new)
        assert np.all(err <= bf16_ulp(w_new) + 0.05 * upd), (r, c, float(err.max()))
