"""The multi-GPU host logic of bench.py on CPU ranks (gloo, world size 2).

Each rank processes its own requests (its own seed) and nothing crosses ranks
on the data path; only the step time (max) and the token count (sum) are
reduced for the whole-job rate.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from sparse_long_context_tail_gb300 import workload as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        spec = bench.rank_spec(wl.scaled_spec(wl.named_spec("small-L4096"), [700, 300], planted=[1, 1]), rank)
        w = wl.generate(spec)
        # a rank-dependent fake step time: rank 1 is the slow one
        sec, tokens, rate = bench.aggregate_over_ranks(0.010 * (rank + 1), w.total_tokens, dist)
        out[rank] = (sec, tokens, rate, hash(w.k_bits.tobytes()), spec.seed)
    finally:
        dist.destroy_process_group()


def test_two_ranks_aggregate_and_own_requests():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    (s0, n0, r0, k0, seed0), (s1, n1, r1, k1, seed1) = out[0], out[1]
    assert s0 == s1 == pytest.approx(0.020)          # max over ranks
    assert n0 == n1 == 2000                          # units of both ranks
    assert r0 == pytest.approx(2000 / 0.020)
    assert seed0 != seed1 and k0 != k1               # each rank has its own requests


def test_single_process_aggregate_is_local():
    assert bench.aggregate_over_ranks(0.5, 100) == (0.5, 100, 200.0)
