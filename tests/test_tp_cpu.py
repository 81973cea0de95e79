"""Tensor-parallel score exchange on CPU ranks (gloo, world size 2).

Each rank scores only its own heads (here with the oracle, on the CPU,
normalised by the total head count as ``upf_score_shard`` does), the ranks sum
their shard scores with one all-reduce, and the result must be the all-heads
score on every rank, bit-identical across ranks, with the same selection.  A rank that dies before the exchange makes the other rank's
exchange fail with an error instead of hanging.
"""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from sparse_long_context_tail_gb300 import tp
from sparse_long_context_tail_gb300 import workload as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _spec():
    return wl.WorkloadSpec("tp-cpu", [700, 1300], 8, 4, 64, 64, n_tail=32, block=32, planted=[2, 3],
                           strength_range=(1.0, 4.0), seed=91)


def _local_scores(w, rank, world):
    """The oracle's score over this rank's heads, normalised by all H_q heads
    (the oracle normalises by the heads it is given: rescale by H_local / H_q)."""
    s = w.spec
    qs, ks = tp.shard_heads(s.num_q_heads, s.num_kv_heads, rank, world)
    local = oracle.token_scores(np.ascontiguousarray(w.k_bits[:, ks]), np.ascontiguousarray(w.q_tail_bits[:, qs]),
                                w.cu_seqlens, qs.stop - qs.start, ks.stop - ks.start, s.head_dim, s.n_tail)
    return local * ((qs.stop - qs.start) / s.num_q_heads)


def _exchange_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        w = wl.generate(_spec())
        local = torch.from_numpy(_local_scores(w, rank, world))
        tp.allreduce_scores(local)
        out[rank] = local.numpy().tobytes()
    finally:
        dist.destroy_process_group()


def test_shard_heads_covers_every_group_once():
    seen_q, seen_kv = [], []
    for r in range(4):
        qs, ks = tp.shard_heads(32, 8, r, 4)
        assert (qs.stop - qs.start, ks.stop - ks.start) == (8, 2)
        # every q head of the shard reads a kv head of the same shard (contiguous GQA groups)
        assert all(ks.start <= h // 4 < ks.stop for h in range(qs.start, qs.stop))
        seen_q += list(range(qs.start, qs.stop))
        seen_kv += list(range(ks.start, ks.stop))
    assert seen_q == list(range(32)) and seen_kv == list(range(8))
    with pytest.raises(ValueError):
        tp.shard_heads(32, 8, 0, 3)
    with pytest.raises(ValueError):
        tp.shard_heads(32, 8, 2, 2)


def test_sum_of_shard_scores_is_the_all_heads_score():
    w = wl.generate(_spec())
    s = w.spec
    full = oracle.token_scores(w.k_bits, w.q_tail_bits, w.cu_seqlens, s.num_q_heads, s.num_kv_heads, s.head_dim,
                               s.n_tail)
    for world in (2, 4):
        got = tp.sum_of_partials([torch.from_numpy(_local_scores(w, r, world)) for r in range(world)]).numpy()
        np.testing.assert_allclose(got, full, rtol=1e-12, atol=1e-300)


def test_two_ranks_exchange_scores():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_exchange_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    assert out[0] == out[1]                          # every rank holds the same bits
    w = wl.generate(_spec())
    s = w.spec
    got = np.frombuffer(out[0], dtype=np.float64)
    full = oracle.token_scores(w.k_bits, w.q_tail_bits, w.cu_seqlens, s.num_q_heads, s.num_kv_heads, s.head_dim,
                               s.n_tail)
    np.testing.assert_allclose(got, full, rtol=1e-12, atol=1e-300)
    a = oracle.select(got, w.cu_seqlens, s.block, s.top_p, s.sink_keep, s.tail_keep)
    b = oracle.select(full, w.cu_seqlens, s.block, s.top_p, s.sink_keep, s.tail_keep)
    np.testing.assert_array_equal(a["mask"], b["mask"])


class _FakeSelector:
    """Stands in for TokenSelector on the CPU: records what tp_select_tokens passes."""

    def __init__(self, local_scores):
        self.local_scores = local_scores
        self.calls = []

    def score(self, q, k, cu_host, cu_dev, hq, hkv, d, params=None, total_q_heads=None):
        self.calls.append(("score", hq, hkv, d, tuple(q.shape), tuple(k.shape), total_q_heads))
        return self.local_scores.clone()

    def select_compact(self, scores, cu_host, cu_dev, hidden, positions, slots, layer_id, history, history_len,
                       params, out):
        self.calls.append(("select_compact", layer_id))
        return scores


def _glue_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        T, hq, hkv, d = 50, 8, 4, 64
        qs, ks = tp.shard_heads(hq, hkv, rank, world)
        q = torch.zeros(T, hq, d)[:, qs]
        k = torch.zeros(T, hkv, d)[:, ks]
        sel = _FakeSelector(torch.arange(T, dtype=torch.float32) * (rank + 1))
        got = tp.tp_select_tokens(sel, q, k, np.array([0, T]), torch.tensor([0, T]), qs.stop - qs.start,
                                  ks.stop - ks.start, d, layer_id=7)
        out[rank] = (got.numpy().tobytes(), sel.calls)
    finally:
        dist.destroy_process_group()


def test_tp_select_tokens_scores_locally_then_selects_on_the_sum():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_glue_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    (b0, c0), (b1, c1) = out[0], out[1]
    assert b0 == b1
    want = (np.arange(50, dtype=np.float32) * 3.0)          # sum of 1x and 2x the shard scores
    np.testing.assert_array_equal(np.frombuffer(b0, dtype=np.float32), want)
    for calls in (c0, c1):
        assert calls == [("score", 4, 2, 64, (50, 4, 64), (50, 2, 64), 8), ("select_compact", 7)]


def test_tp_select_tokens_rejects_a_wrong_head_slice_before_any_exchange():
    sel = _FakeSelector(torch.zeros(50))
    q, k = torch.zeros(50, 4, 64), torch.zeros(50, 2, 64)
    cu = np.array([0, 50])
    with pytest.raises(ValueError, match="q_local"):
        tp.tp_select_tokens(sel, q, k, cu, torch.tensor(cu), 8, 2, 64)
    with pytest.raises(ValueError, match="k_local"):
        tp.tp_select_tokens(sel, q, k, cu, torch.tensor(cu), 4, 4, 64)
    with pytest.raises(ValueError, match="token count"):
        tp.tp_select_tokens(sel, q, k, np.array([0, 49]), torch.tensor([0, 49]), 4, 2, 64)
    assert sel.calls == []                           # nothing was scored, no collective was entered


def _dead_peer_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=10))
    if rank == 1:
        os._exit(0)                                  # dies before the exchange
    try:
        tp.allreduce_scores(torch.ones(64, dtype=torch.float64))
        out[rank] = "returned"
    except Exception as e:                           # noqa: BLE001 - any error is the expected outcome
        out[rank] = "raised: " + type(e).__name__
    os._exit(0)


def test_dead_rank_fails_the_exchange_instead_of_hanging():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_dead_peer_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.kill()
    assert not alive, "a rank hung in the exchange"
    assert out.get(0, "").startswith("raised"), out.get(0)
