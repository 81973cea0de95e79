"""The C ABI without a GPU: the library builds, loads, exports every declared
entry point, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

from sparse_long_context_tail_gb300 import _binding as B
from sparse_long_context_tail_gb300 import build as build_mod

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "upf.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(upf_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
        assert n in B._SIGNATURES, f"binding lacks {n}"


def test_version_and_defaults(lib):
    assert B.upf_version() == 1
    p = B.upf_default_params()
    assert (p.n_tail, p.block, p.sink_keep, p.tail_keep) == (128, 64, 128, 128)
    assert abs(p.top_p - 0.99) < 1e-7 and p.softmax_scale == 0.0
    assert B.upf_status_name(0) == "UPF_OK" and B.upf_status_name(4) == "UPF_ERR_CAPACITY"


def _batch(cu, Hq=32, Hkv=8, d=128, kv=None):
    return B.make_batch(0x1000, np.asarray(cu, np.int32), Hq, Hkv, d, kv)


def test_workspace_bytes_valid_and_invalid(lib):
    b, keep = _batch([0, 131072])
    n = B.upf_workspace_bytes(b, B.make_params())
    assert n > 131072 * 8 * 4    # at least the per-group partial scores
    b2, k2 = _batch([0, 5000, 9000])
    assert B.upf_workspace_bytes(b2, B.make_params()) > 0
    bad = [(_batch([0, 100], Hq=6, Hkv=4), B.make_params(), "H_q"),
           (_batch([0, 100], d=96), B.make_params(), "head_dim"),
           (_batch([0, 100, 50]), B.make_params(), "non-decreasing"),
           (_batch([0, 100]), B.make_params(top_p=0.0), "top_p"),
           (_batch([0, 100]), B.make_params(top_p=1.5), "top_p"),
           (_batch([0, 100]), B.make_params(block=0), "block"),
           (_batch([0, 16385 * 64]), B.make_params(), "blocks"),
           (_batch([0, 100], Hq=4, Hkv=2, kv=[0, 0, 0, 1]), B.make_params(), "kv_of_q")]
    for (bb, kk), p, word in bad:
        with pytest.raises(B.UpfError) as e:
            B.upf_workspace_bytes(bb, p)
        assert word in e.value.message, (word, e.value.message)


def test_workspace_size_is_device_independent(lib):
    b, keep = _batch([0, 70000, 90000])
    assert B.upf_workspace_bytes(b, B.make_params()) == B.upf_workspace_bytes(b, B.make_params())


def test_calls_without_context_fail_before_launch(lib):
    b, keep = _batch([0, 1000])
    p = B.make_params()
    with pytest.raises(B.UpfError) as e:
        B.upf_score(None, b, p, 16, 4096, 16, 1024, 16, 256, 1 << 20)
    assert e.value.status == 1 and "context" in e.value.message
    io = B.make_compact_io(cu_seqlens_out=16, total_kept=16)
    with pytest.raises(B.UpfError):
        B.upf_compact(None, b, 16, io, 256, 1 << 20)
    with pytest.raises(B.UpfError):
        B.upf_select_tokens(None, b, p, 16, 4096, 16, 1024, 0, 0, 16, 16, io, 256, 1 << 20)


def test_create_without_gpu_reports_an_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(B.UpfError) as e:
        B.upf_create(0)
    assert e.value.status in (1, 3)


def test_destroy_null_is_an_argument_error(lib):
    assert lib.upf_destroy(None) == 1
    assert "NULL" in B.upf_last_error()


def test_wait_limit_and_shard_scoring_check_their_arguments(lib):
    assert lib.upf_set_wait_limit(None, 100) == 1 and "context" in B.upf_last_error()
    b, keep = _batch([0, 1000], Hq=8, Hkv=2)
    with pytest.raises(B.UpfError) as e:
        B.upf_score_shard(None, b, B.make_params(), 32, 16, 4096, 16, 1024, 16, 256, 1 << 20)
    assert e.value.status == 1


def _greedy_makespan(lengths, hkv, nqc, ks, ovh, sms):
    """Items in launch order (request, kv head, split, query chunk) dealt to the
    first free of `sms` slots; an item costs its keys plus ovh."""
    import heapq
    heap = [0] * sms
    for L in lengths:
        for _ in range(hkv):
            for sp in range(-(-L // ks)):
                for _ in range(nqc):
                    t = heapq.heappop(heap)
                    heapq.heappush(heap, t + min(ks, L - sp * ks) + ovh)
    return max(heap)


def test_scoring_work_split_is_near_the_best_whole_tile_split(lib):
    """The tensor-core passes run one item per CTA (or CTA pair) and one CTA per
    SM: 160 equal items on 152 SMs take two item-times.  Over every whole-tile
    split, simulated independently here, the planner's pick must be within 2 %
    of the best estimated duration, on every benchmark workload."""
    from sparse_long_context_tail_gb300 import workload as wl
    for name in wl.NAMED:
        s = wl.named_spec(name)
        cu = np.concatenate([[0], np.cumsum(s.lengths)]).astype(np.int32)
        b, keep = B.make_batch(0x1000, cu, s.num_q_heads, s.num_kv_heads, s.head_dim)
        p = B.make_params(s.n_tail, s.block, s.sink_keep, s.tail_keep, s.top_p)
        ks1, ks2, n1, n2, ctas1, ctas2 = B.upf_plan_info(b, p)
        gamma = s.num_q_heads // s.num_kv_heads
        qr = gamma * s.n_tail
        qc = min(-(-qr // 128) * 128, 512 if s.head_dim <= 128 else (128 if qr <= 256 else 256))
        tile1 = 256 if s.head_dim <= 128 else 128      # pass-1 key tile of the single-CTA kernels
        # small batches: halve the chunk while even one tile per item leaves SMs idle
        while qc > 128 and s.num_kv_heads * -(-qr // qc) * sum(-(-L // tile1) for L in s.lengths) < 152:
            qc = -(-(qc // 2) // 128) * 128
        nqc = -(-qr // qc)
        # pairs when the chunk is whole 256-row units at d = 256; a d = 256
        # group of 129..256 rows in a long pass (kv heads x tokens >= 2^19)
        # runs pass 1 in two 128-row chunks on single CTAs and pass 2 in one
        # 256-row chunk on pairs
        pair1 = s.head_dim == 256 and qc % 256 == 0
        split = (s.head_dim == 256 and qc == 128 and 128 < qr <= 256
                 and s.num_kv_heads * sum(s.lengths) >= 1 << 19)
        assert (ctas1, ctas2) == ((2 if pair1 else 1), (2 if pair1 or split else 1)), name
        nqc2 = 1 if split else nqc
        for ks, n, tile, nq, ctas in ((ks1, n1, 256 if ctas1 == 2 or s.head_dim <= 128 else 128, nqc, ctas1),
                                      (ks2, n2, 256 if ctas2 == 2 else 128, nqc2, ctas2)):
            sms = 152 // ctas
            units = s.num_kv_heads * nq
            assert ks % tile == 0 and ks >= 256, (name, ks)
            assert n == units * sum(-(-L // ks) for L in s.lengths), name
            ovh = 2 * tile
            lo = max(256, -(-sum(s.lengths) * units // (4 * sms) // tile) * tile)
            cand = range(lo, -(-max(s.lengths) // tile) * tile + tile, tile)
            best = min(_greedy_makespan(s.lengths, s.num_kv_heads, nq, c, ovh, sms) for c in cand)
            assert _greedy_makespan(s.lengths, s.num_kv_heads, nq, ks, ovh, sms) <= 1.02 * best, (name, ks)
