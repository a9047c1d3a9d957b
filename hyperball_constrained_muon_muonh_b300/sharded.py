"""Data-parallel sharding of the MuonH step across ranks.

Every weight matrix is an independent unit of the step, so a data-parallel
job can split the optimizer work: each rank steps the matrices it owns
(muonh_partition, greedy by Newton-Schulz cost), then every matrix's updated
weight is sent from its owner to the other ranks.  Momenta live only on the
owner; weights stay replicated.  The exchange is one broadcast per rank of a
flat buffer holding that rank's matrices (torch.distributed: NCCL on GPUs,
gloo on CPUs).
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import check, lib


def partition(shapes, world_size: int) -> list[int]:
    """owner[i] = rank that steps matrix i (muonh_partition)."""
    n = len(shapes)
    arr = (_lib.MatrixT * n)()
    for i, (r, c) in enumerate(shapes):
        arr[i].rows, arr[i].cols = r, c
        arr[i].w = 256  # any aligned non-null value: only shapes are read
    out = (ctypes.c_int * n)()
    check(lib.muonh_partition(arr, n, world_size, out), "muonh_partition")
    return list(out)


def exchange_weights(weights, owners, group=None) -> None:
    """Make every rank's copy of weights[i] equal to its owner's.

    For each rank k, the matrices it owns are packed into one flat buffer on
    rank k, broadcast, and unpacked on the others.  All ranks must call this
    with the same owners list and tensors of the same shapes and dtype."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    for k in range(world):
        mine = [w for w, o in zip(weights, owners) if o == k]
        if not mine:
            continue
        numel = sum(w.numel() for w in mine)
        if rank == k:
            flat = torch.cat([w.reshape(-1) for w in mine])
        else:
            flat = torch.empty(numel, dtype=mine[0].dtype, device=mine[0].device)
        src = k if group is None else dist.get_global_rank(group, k)
        dist.broadcast(flat, src=src, group=group)
        if rank != k:
            off = 0
            for w in mine:
                w.copy_(flat[off:off + w.numel()].view_as(w))
                off += w.numel()


class ShardedMuonH:
    """MuonH with the step split across the ranks of a process group: this
    rank runs the library's step on the matrices it owns, then the updated
    weights are exchanged.  The result equals every rank running the whole
    step (each matrix's step is independent of the others)."""

    def __init__(self, weights, group=None, **kwargs):
        import torch.distributed as dist
        from . import MuonH
        self.weights = list(weights)
        self.group = group
        self.owners = partition([tuple(w.shape) for w in self.weights], dist.get_world_size(group))
        rank = dist.get_rank(group)
        self.mine = [i for i, o in enumerate(self.owners) if o == rank]
        self.local = MuonH([self.weights[i] for i in self.mine], **kwargs) if self.mine else None

    def step(self, grads) -> None:
        if self.local is not None:
            self.local.step([grads[i] for i in self.mine])
        exchange_weights(self.weights, self.owners, self.group)
