"""The bench's tensor-parallel mode and roofline rules, host side, on CPU.

Two gloo ranks run the TP step the way ``bench.py --tp`` does: each takes its
head slices of the same batch (``tp_shard_inputs``), scores them (here with
the float64 oracle normalised by the total head count, standing in for
``upf_score_shard``), sums the scores with one all-reduce inside
``tp.tp_select_tokens``, selects, and checks that every rank holds the same
mask (``tp_masks_agree``).  A rank whose mask differs must be caught.
"""
import datetime
import os
import socket
import types

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from oracle import compare as C
from sparse_long_context_tail_gb300 import workload as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _spec():
    return wl.WorkloadSpec("tp-bench", [900, 1500], 8, 4, 64, 64, n_tail=32, block=32, planted=[2, 3],
                           strength_range=(1.0, 4.0), seed=93)


class _OracleShardSelector:
    """CPU stand-in for TokenSelector: shard scores from the oracle."""

    def __init__(self, w, q_bits, k_bits):
        self.w, self.q_bits, self.k_bits = w, q_bits, k_bits

    def score(self, q, k, cu_host, cu_dev, hq, hkv, d, params=None, total_q_heads=None):
        s = oracle.token_scores(self.k_bits, self.q_bits, cu_host, hq, hkv, d, self.w.spec.n_tail)
        return torch.from_numpy(s * (hq / total_q_heads))

    def select_compact(self, scores, cu_host, cu_dev, hidden, positions, slots, layer_id, history, history_len,
                       params, out):
        s = self.w.spec
        sel = oracle.select(scores.numpy(), cu_host, s.block, s.top_p, s.sink_keep, s.tail_keep)
        return types.SimpleNamespace(scores=scores, keep_bits=torch.from_numpy(C.pack_bits(sel["mask"]).view(np.int32)))


def _tp_worker(rank, world, port, out, corrupt_rank):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        from sparse_long_context_tail_gb300 import tp
        w = wl.generate(_spec())
        qs, ks, q_bits, k_bits = bench.tp_shard_inputs(w, rank, world)
        s = w.spec
        T = w.total_tokens
        q_local = torch.zeros(T, qs.stop - qs.start, s.head_dim)
        k_local = torch.zeros(T, ks.stop - ks.start, s.head_dim)
        sel = _OracleShardSelector(w, q_bits, k_bits)
        res = tp.tp_select_tokens(sel, q_local, k_local, w.cu_seqlens, torch.from_numpy(w.cu_seqlens),
                                  qs.stop - qs.start, ks.stop - ks.start, s.head_dim)
        bits = res.keep_bits.clone()
        if rank == corrupt_rank:
            bits[0] ^= 1
        out[rank] = (bench.tp_masks_agree(bits, dist), res.scores.numpy().tobytes(), (qs.start, qs.stop, ks.start,
                                                                                      ks.stop))
    finally:
        dist.destroy_process_group()


def _run(corrupt_rank):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_tp_worker, args=(r, 2, port, out, corrupt_rank)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    return dict(out)


def test_tp_mode_on_two_ranks_gives_the_all_heads_selection_on_both():
    out = _run(corrupt_rank=-1)
    (a0, s0, sh0), (a1, s1, sh1) = out[0], out[1]
    assert a0 and a1
    assert s0 == s1
    assert sh0 == (0, 4, 0, 2) and sh1 == (4, 8, 2, 4)
    w = wl.generate(_spec())
    s = w.spec
    full = oracle.token_scores(w.k_bits, w.q_tail_bits, w.cu_seqlens, s.num_q_heads, s.num_kv_heads, s.head_dim,
                               s.n_tail)
    np.testing.assert_allclose(np.frombuffer(s0, dtype=np.float64), full, rtol=1e-12, atol=1e-300)


def test_tp_mask_check_catches_a_rank_that_differs():
    out = _run(corrupt_rank=1)
    assert out[0][0] is False and out[1][0] is False


def test_tp_mask_check_is_true_without_a_process_group():
    assert bench.tp_masks_agree(torch.zeros(4, dtype=torch.int32), dist)


# ------------------------------------------------------------- rooflines ----

PEAKS = {"bf16_tflops": 2240.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 8000.0}


def test_scoring_pass_bound_follows_arithmetic_intensity():
    # ridge = 2240e12 / 8000e9 = 280 flop per byte; intensity of a pass ~ H_q n / H_kv
    for name, want in (("llama8b-L131072", "tensor"),        # 32 * 128 / 8 = 512
                       ("qwen3next-G64-n512", "tensor"),     # 16 * 512 / 2 = 4096
                       ("qwen3next-G64-n32", "hbm"),         # 16 * 32 / 2 = 256 (255.5 with the tail Q bytes)
                       ("gemma3-G64-n128", "hbm"),           # 16 * 128 / 8 = 256, idem
                       ("gemma3-G64-n32", "hbm")):           # 64
        spec = wl.named_spec(name)
        work = bench.algorithmic_work(spec, [0, spec.lengths[0]], 0, 2 * spec.hidden, spec.top_p)
        got = bench.scoring_bound(work["score_pass1"], PEAKS)
        assert got == want, (name, work["score_pass1"]["flops"] / work["score_pass1"]["bytes"])


def test_tensor_bound_pass_takes_the_burst_peak():
    spec = wl.named_spec("llama8b-L131072")
    work = bench.algorithmic_work(spec, [0, 131072], 0, 2 * spec.hidden, spec.top_p)
    r = bench.kernel_roofline("score_pass1", work, 100e-6, PEAKS, "measured", spec.name)
    want = work["score_pass1"]["flops"] / 100e-6 / 1e12
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 2240.0
    assert r["achieved"] == pytest.approx(want) and r["frac"] == pytest.approx(want / 2240.0)
    assert r["frac_of_sustained_peak"] == pytest.approx(want / 1700.0)
    g = bench.kernel_roofline("compact_gather", bench.algorithmic_work(spec, [0, 131072], 1000, 8192, 0.99), 1e-6,
                              PEAKS, "measured", spec.name)
    assert g["bound"] == "hbm" and g["peak"] == 8000.0 and g["achieved"] == pytest.approx(1000 * (2 * 8192 + 36) / 1e-6 / 1e9)
