"""Muon across data-parallel ranks: whole matrices sharded between one reduce-scatter and one all-gather.

The speedrun reduce-scatters gradients instead of all-reducing them (energy-efficiency article on
Modded-NanoGPT, technical-evolution section; "How to train a GPT model in 3 minutes", system
optimisations, distributed communication) and sends attention and MLP parameters through one
merged reduce_scatter call ("Muon Custom Sizing", linked from the record analysis of
2026-05-27_MuddGatedAndDC). Here every matrix's Newton-Schulz iteration is independent, so:

1. every rank holds its local gradients in one flat rank-major buffer laid out by
   ``muon_shard_layout``; one in-place reduce-scatter leaves each rank the summed gradients of
   the matrices it owns, in its own segment;
2. each rank runs ``muon_step`` (the CUDA library) on its owned matrices only, keeping momentum
   for those alone;
3. one in-place all-gather over the flat parameter buffer replicates every rank's updated
   matrices to all ranks.

The step acts on the SUMMED gradient: it equals a single-rank ``muon_step`` whose gradient is the
sum over ranks. The orthogonalised update does not depend on the gradient's scale, so dividing by
the world size (a mean) would change only the momentum buffer's scale; no extra pass does it.

This module holds the host logic and the two collectives (torch.distributed: NCCL on GPUs, gloo
for the CPU tests). It computes nothing itself: the partition comes from the C library and the
step from its CUDA kernels (or, in the CPU tests, from whatever ``local_step`` they pass).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence

from .binding import MUON_OK, Muon, MuonError, load_library

# Every matrix view starts on a multiple of this many elements (256 bytes for bf16), so TMA sees
# 16-byte aligned rows and the last combine can write the parameters directly.
ALIGN = 128


@dataclass
class ShardLayout:
    """Who owns each matrix and where it sits in the flat rank-major buffers."""
    shapes: List[tuple]
    world: int
    owner: List[int]
    offset: List[int]
    segment: int
    load: List[float]

    def owned(self, rank: int) -> List[int]:
        return [j for j, r in enumerate(self.owner) if r == rank]

    @property
    def total(self) -> int:
        return self.world * self.segment


def shard_layout(shapes: Sequence, world: int, with_c: bool = False, align: int = ALIGN) -> ShardLayout:
    """The layout muon_shard_layout computes (host only, no GPU)."""
    lib = load_library()
    n = len(shapes)
    rows = (ctypes.c_int64 * max(1, n))(*[int(r) for r, _ in shapes])
    cols = (ctypes.c_int64 * max(1, n))(*[int(c) for _, c in shapes])
    owner = (ctypes.c_int * max(1, n))()
    offset = (ctypes.c_int64 * max(1, n))()
    seg = ctypes.c_int64()
    load = (ctypes.c_double * max(1, world))()
    st = lib.muon_shard_layout(rows, cols, n, int(world), int(bool(with_c)), int(align), owner, offset,
                               ctypes.byref(seg), load)
    if st != MUON_OK:
        raise MuonError(st, f"muon_shard_layout(count={n}, world={world})")
    return ShardLayout([tuple(map(int, s)) for s in shapes], int(world), list(owner[:n]), list(offset[:n]),
                       seg.value, list(load[:world]))


def views(flat, layout: ShardLayout, which: Optional[Sequence[int]] = None, base: int = 0) -> list:
    """2-D views of the matrices `which` (all by default) inside a flat buffer; `base` is the buffer's
    first element's offset in the layout (the own segment's start for a segment-sized buffer)."""
    idx = range(len(layout.shapes)) if which is None else which
    out = []
    for j in idx:
        r, c = layout.shapes[j]
        o = layout.offset[j] - base
        out.append(flat[o:o + r * c].view(r, c))
    return out


def sharded_step(layout: ShardLayout, rank: int, flat_params, flat_grads, local_step: Callable[[List[int]], None],
                 group=None):
    """One sharded Muon step on flat rank-major buffers (both world * segment long).

    flat_grads holds this rank's local gradients on entry; afterwards its own segment holds the
    gradients summed over ranks (the other segments are left as the reduce-scatter leaves them).
    local_step(owned) must update the owned matrices' parameters (views of flat_params) in place
    from the summed gradients (views of flat_grads). On return flat_params is the same on every rank.
    """
    import torch.distributed as dist
    seg = layout.segment
    lo, hi = rank * seg, (rank + 1) * seg
    dist.reduce_scatter_tensor(flat_grads[lo:hi], flat_grads, op=dist.ReduceOp.SUM, group=group)
    local_step(layout.owned(rank))
    dist.all_gather_into_tensor(flat_params, flat_params[lo:hi], group=group)


class ShardedMuon:
    """A Muon step sharded over the ranks of a process group, one GPU per rank.

    Owns the flat parameter and gradient buffers (``params`` and ``grads`` are per-matrix views the
    training loop reads and fills) and the momentum of this rank's own matrices. ``step`` runs the
    reduce-scatter, ``muon_step`` on the owned matrices through the CUDA library, and the all-gather.
    """

    def __init__(self, shapes: Sequence, rank: int, world: int, device: int, group=None, lr: float = 0.02,
                 beta: float = 0.95, nesterov: bool = True, param_dtype=None, grad_dtype=None, **config):
        import torch
        self.layout = shard_layout(shapes, world, with_c=config.get("c", 0.0) != 0.0)
        self.rank, self.world, self.group = rank, world, group
        self.device = torch.device("cuda", device)
        pdt = param_dtype or torch.bfloat16
        gdt = grad_dtype or torch.bfloat16
        L = self.layout
        self.flat_params = torch.zeros(L.total, dtype=pdt, device=self.device)
        self.flat_grads = torch.zeros(L.total, dtype=gdt, device=self.device)
        self.own = L.owned(rank)
        self.flat_momentum = torch.zeros(max(L.segment, 1), dtype=torch.float32, device=self.device)
        self.params = views(self.flat_params, L)
        self.grads = views(self.flat_grads, L)
        base = rank * L.segment
        self.momentum = views(self.flat_momentum, L, self.own, base)
        self.muon = Muon(device, **config)
        own_p = [self.params[j] for j in self.own]
        own_g = [self.grads[j] for j in self.own]
        self._local = (self.muon.prepare_step(own_p, own_g, self.momentum, lr=lr, beta=beta, nesterov=nesterov)
                       if self.own else (lambda: None))

    def step(self):
        sharded_step(self.layout, self.rank, self.flat_params, self.flat_grads, lambda owned: self._local(),
                     self.group)

    def close(self):
        self.muon.close()
