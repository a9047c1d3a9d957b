"""Data-parallel sharding of the step (no GPU): the partition function and
the weight exchange, on CPU.

* partition: every matrix gets exactly one owner; greedy longest-processing-
  time assignment keeps the largest load within Graham's bound
  (4/3 - 1/(3m)) x the optimal makespan, checked against brute force on small
  inputs, and the loads within one item's cost of each other;
* exchange: gloo jobs of 2, 3 and 8 ranks (with 8, one rank owns no
  matrix) where each rank steps only the matrices it owns (the float64 oracle stands in for the GPU step) and the exchange
  makes every rank hold the weights of the unsharded step, bit for bit.
"""

import itertools
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import muonh_workloads as wl
from hyperball_constrained_muon_muonh_b300 import exchange_weights, partition


def _cost(shape):
    s, l = min(shape), max(shape)
    return 3 * s * s * l + s ** 3


def _loads(shapes, owners, world):
    load = [0.0] * world
    for sh, o in zip(shapes, owners):
        load[o] += _cost(sh)
    return load


def test_partition_covers_and_balances_the_2b_set():
    shapes = wl.qwen3_2b().shapes
    for world in range(1, 9):
        owners = partition(shapes, world)
        assert len(owners) == len(shapes) and all(0 <= o < world for o in owners)
        load = _loads(shapes, owners, world)
        assert max(load) - min(load) <= max(_cost(s) for s in shapes)
        assert owners == partition(shapes, world)          # deterministic
    assert set(partition(shapes, 1)) == {0}


def test_partition_within_graham_bound_of_optimum():
    rng = np.random.default_rng(5)
    for trial in range(30):
        n = int(rng.integers(2, 8))
        world = int(rng.integers(2, 4))
        shapes = [(int(rng.integers(1, 9)) * 16, int(rng.integers(1, 9)) * 16) for _ in range(n)]
        owners = partition(shapes, world)
        got = max(_loads(shapes, owners, world))
        best = min(max(_loads(shapes, assign, world)) for assign in itertools.product(range(world), repeat=n))
        assert got <= (4 / 3 - 1 / (3 * world)) * best + 1e-9


def test_partition_rejects_bad_arguments():
    with pytest.raises(Exception):
        partition([(4, 4)], 0)
    with pytest.raises(Exception):
        partition([(0, 4)], 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import muonh as om
        work = wl.ragged(EXCHANGE_SHAPES)
        ws = [w for w in work.weights("cpu")]
        gs = [g for g in work.grads(0, "cpu")]
        w0 = [w.numpy().copy() for w in ws]
        r0 = om.capture_norms(w0)
        owners = partition(work.shapes, world)
        mine = [i for i, o in enumerate(owners) if o == rank]
        # this rank's share of the step (the oracle stands in for the GPU step);
        # with more ranks than matrices a rank may own none
        if mine:
            out = om.muonh_step([w0[i] for i in mine], [gs[i].numpy() for i in mine],
                                [np.zeros_like(w0[i]) for i in mine], r0[mine], work.lr, work.beta, work.ns_steps,
                                work.coeffs, work.eps)
            for k, i in enumerate(mine):
                ws[i].copy_(torch.from_numpy(out["w"][k]))
        for i in range(len(ws)):
            if owners[i] != rank:
                ws[i].fill_(float("nan"))                   # must be overwritten by the exchange
        exchange_weights(ws, owners)
        full = om.muonh_step(w0, [g.numpy() for g in gs], [np.zeros_like(w) for w in w0], r0, work.lr, work.beta,
                             work.ns_steps, work.coeffs, work.eps)
        ok = all(np.array_equal(ws[i].numpy(), full["w"][i]) for i in range(len(ws)))
        digest = torch.tensor([float(sum(w.double().sum() for w in ws))])
        got = [torch.zeros(1, dtype=digest.dtype) for _ in range(world)]
        dist.all_gather(got, digest)
        result[rank] = int(ok and all(torch.equal(got[0], d) for d in got))
    finally:
        dist.destroy_process_group()


EXCHANGE_SHAPES = [(48, 32), (32, 48), (64, 64), (16, 40), (40, 16), (24, 24), (96, 8)]


@pytest.mark.parametrize("world", [2, 3, 8])
def test_exchange_gloo(world):
    owners = partition(EXCHANGE_SHAPES, world)
    if world > len(EXCHANGE_SHAPES):
        assert len(set(owners)) < world          # some rank owns nothing and still takes part
    ctx = mp.get_context("spawn")
    result = ctx.Manager().dict()
    mp.start_processes(_worker, args=(world, _free_port(), result), nprocs=world, start_method="spawn", join=True)
    assert dict(result) == {r: 1 for r in range(world)}
