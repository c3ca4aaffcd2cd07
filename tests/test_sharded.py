"""Sharded Muon across ranks: the partition (host, C library) and the collectives (gloo, world size 2).

The local step of each rank here is the fp64 oracle on CPU tensors, so the exchange logic is
checked on its own: the gathered parameters on every rank must equal a single-rank oracle step
whose gradient is the sum of the ranks' gradients. The GPU version of the same step (CUDA local
step, NCCL) is in test_gpu_sharded.py.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads as wl
from muon_newton_schulz_09_b300 import shard_layout, sharded_step
from muon_newton_schulz_09_b300.sharded import ALIGN, views

CUBIC = (1.5, -0.5, 0.0)
GPT2_124M = wl.GPT2_124M.shapes
SMALL = [(64, 96), (96, 64), (32, 32), (48, 80), (80, 48), (16, 40), (0, 8), (40, 16), (130, 70)]


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_layout_owns_every_matrix_once_and_balances(world):
    L = shard_layout(GPT2_124M, world)
    assert len(L.owner) == len(GPT2_124M) and all(0 <= r < world for r in L.owner)
    assert sorted(sum((L.owned(r) for r in range(world)), [])) == list(range(len(GPT2_124M)))
    # balanced by algorithmic flops: the heaviest rank within 10% of the mean
    mean = sum(L.load) / world
    assert max(L.load) <= 1.10 * mean, (world, L.load)
    want = sum(n * (n + 1) * m + 2 * n * n * m for n, m in (sorted(s) for s in GPT2_124M))
    assert sum(L.load) == pytest.approx(want, rel=1e-12)
    _check_placement(L)


def _check_placement(L):
    """Aligned, non-overlapping matrices, each inside its owner's segment."""
    assert L.segment % ALIGN == 0 and L.segment >= ALIGN
    spans = []
    for j, ((r, c), o) in enumerate(zip(L.shapes, L.offset)):
        assert o % ALIGN == 0
        lo, hi = L.owner[j] * L.segment, (L.owner[j] + 1) * L.segment
        assert lo <= o and o + r * c <= hi, j
        if r * c:
            spans.append((o, o + r * c))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))


def test_layout_small_and_degenerate():
    L = shard_layout(SMALL, 2)
    _check_placement(L)
    assert L.owner[SMALL.index((0, 8))] == 0  # empty matrices cost nothing and sit on rank 0
    # the quintic's A A pass is counted when c != 0
    lc = shard_layout(SMALL, 2, with_c=True)
    assert sum(lc.load) > sum(L.load)
    # more ranks than matrices: some ranks own nothing, every segment still has the same length
    L9 = shard_layout([(32, 64), (64, 32)], 5)
    assert sorted(L9.owner)[:2] == [0, 1] and sum(1 for r in range(5) if not L9.owned(r)) == 3
    with pytest.raises(Exception):
        shard_layout(SMALL, 0)


def test_layout_is_deterministic():
    a, b = shard_layout(GPT2_124M, 8), shard_layout(list(GPT2_124M), 8)
    assert (a.owner, a.offset, a.segment) == (b.owner, b.offset, b.segment)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


LR, BETA = 0.02, 0.95


def _inputs(rank):
    """Replicated parameters and momentum (seed 61), this rank's own gradients (seed 70 + rank)."""
    common = wl.small_workload("shard", SMALL, kind="step", dtype="f32", param_dtype="f32", grad_std=1e-3,
                               seed=61)
    mine = wl.small_workload("shard", SMALL, kind="step", dtype="f32", param_dtype="f32", grad_std=1e-3,
                             spike_rank=2, spike_gain=10.0, seed=70 + rank)
    p = [wl.parameter(common, j) for j in range(len(SMALL))]
    m = [wl.momentum_buffer(common, j) for j in range(len(SMALL))]
    g = [wl.gradient(mine, j) for j in range(len(SMALL))]
    return p, m, g


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        L = shard_layout(SMALL, world)
        p, m, g = _inputs(rank)
        flat_p = torch.zeros(L.total, dtype=torch.float32)
        flat_g = torch.zeros(L.total, dtype=torch.float32)
        P, G = views(flat_p, L), views(flat_g, L)
        for j in range(len(SMALL)):
            P[j].copy_(torch.from_numpy(p[j]))
            G[j].copy_(torch.from_numpy(g[j]))
        mom = {j: m[j].astype(np.float64) for j in L.owned(rank)}  # momentum of owned matrices only
        seen = []

        def local_step(owned):
            seen.extend(owned)
            for j in owned:
                if 0 in SMALL[j]:
                    continue
                w_new, buf, _ = oracle.muon_step(P[j].numpy(), G[j].numpy(), mom[j], LR, BETA, True, 5, CUBIC)
                mom[j] = buf
                P[j].copy_(torch.from_numpy(w_new.astype(np.float32)))

        sharded_step(L, rank, flat_p, flat_g, local_step)
        q.put((rank, sorted(seen), [x.numpy().copy() for x in P]))
    finally:
        dist.destroy_process_group()


def test_sharded_step_two_gloo_ranks_equals_single_rank_step_on_summed_gradients():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict()
    for _ in range(world):
        rank, seen, params = q.get(timeout=120)
        got[rank] = (seen, params)
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    L = shard_layout(SMALL, world)
    assert got[0][0] == L.owned(0) and got[1][0] == L.owned(1)
    p, m, _ = _inputs(0)
    gsum = [sum(_inputs(r)[2][j].astype(np.float64) for r in range(world)) for j in range(len(SMALL))]
    for j, (r, c) in enumerate(SMALL):
        a, b = got[0][1][j], got[1][1][j]
        assert np.array_equal(a, b), j  # replicated: bitwise the same on both ranks
        if r * c == 0:
            continue
        want, _, o = oracle.muon_step(p[j], gsum[j], m[j], LR, BETA, True, 5, CUBIC)
        # the only differences are the fp32 sum of two gradients and the fp32 storage of W'
        assert oracle.rel_frobenius(a - p[j], want - p[j]) < 1e-5, (j, oracle.rel_frobenius(a - p[j], want - p[j]))
