"""upf_select_noalloc: the selection step for callers that cannot allocate.

Callers such as a serving engine that has reserved nearly all GPU memory for
its own pools, or a plugin living inside such an engine, cannot allocate a
workspace or hold a library context; upf_select_noalloc keeps its scratch in a
fixed array inside the library instead.  Its results must be those of
upf_select (context + caller workspace) on the same inputs, on consecutive
calls that share that array.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare as C
from sparse_long_context_tail_gb300 import _binding as B

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return B.load()


def synthetic_scores(seed, lengths):
    """Per-request scores that sum to 1: a few strong blocks over a noisy floor."""
    rng = np.random.default_rng(seed)
    parts = []
    for L in lengths:
        s = rng.exponential(1.0, size=L)
        for _ in range(max(1, L // 4000)):
            a = int(rng.integers(0, max(1, L - 64)))
            s[a:a + 64] *= 200.0
        parts.append(s / s.sum() if L else s)
    return np.concatenate(parts).astype(np.float32)


def run_both(lengths, seed, block, top_p, pass_block_scores):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, R = int(cu[-1]), len(lengths)
    cu_dev = torch.from_numpy(cu).to(DEV)
    scores = torch.from_numpy(synthetic_scores(seed, lengths)).to(DEV)
    batch, keep = B.make_batch(cu_dev.data_ptr(), cu, 32, 8, 128)
    params = B.make_params(block=block, top_p=top_p)
    nb = int(sum(-(-int(L) // block) for L in lengths))
    stream = torch.cuda.current_stream().cuda_stream

    ctx = B.upf_create(0)
    try:
        nbytes = B.upf_workspace_bytes(batch, params)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        bits_a = torch.empty((T + 31) // 32, dtype=torch.int32, device=DEV)
        cnt_a = torch.empty(R, dtype=torch.int32, device=DEV)
        bs_a = torch.empty(max(1, nb), dtype=torch.float32, device=DEV)
        B.upf_select(ctx, batch, params, scores.data_ptr(), bs_a.data_ptr(), bits_a.data_ptr(), cnt_a.data_ptr(),
                     ws.data_ptr(), nbytes, stream)
        assert B.upf_sync_status(ctx, stream) == 0
    finally:
        torch.cuda.synchronize()
        B.upf_destroy(ctx)

    bits_b = torch.full(((T + 31) // 32,), -1, dtype=torch.int32, device=DEV)
    cnt_b = torch.full((R,), -1, dtype=torch.int32, device=DEV)
    bs_b = torch.full((max(1, nb),), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.upf_select_noalloc(batch, params, scores.data_ptr(), bs_b.data_ptr() if pass_block_scores else 0,
                         bits_b.data_ptr(), cnt_b.data_ptr(), status.data_ptr(), stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(bits_a, bits_b)
    assert torch.equal(cnt_a, cnt_b)
    if pass_block_scores:
        # same kernels on the same scores: block means agree within the score tolerance (in fact exactly)
        assert torch.allclose(bs_a, bs_b, rtol=1e-3, atol=1e-6 / max(lengths))
    # and against the float64 oracle on the same float32 scores: the mask is the
    # oracle's outside boundary blocks and exactly the top-p rule on the block
    # means the call produced; the counts follow the mask
    scores_np = scores.cpu().numpy().astype(np.float64)
    ref = oracle.select(scores_np, cu, block, params.top_p, params.sink_keep, params.tail_keep)
    mask = C.unpack_bits(bits_b.cpu().numpy(), T)
    assert C.mask_mismatches(mask, ref, cu, block, params.top_p, params.sink_keep, params.tail_keep) == []
    own_bs = (bs_b if pass_block_scores else bs_a).cpu().numpy()[:nb]
    ref_bs = np.concatenate(ref["block_scores"])
    assert np.all(np.abs(own_bs - ref_bs) <= 1e-3 * np.abs(ref_bs) + 1e-6 / max(lengths))
    assert C.self_consistency_mismatches(mask, own_bs, cu, block, params.top_p, params.sink_keep,
                                         params.tail_keep) == []
    assert cnt_b.cpu().numpy().tolist() == [int(mask[cu[r]:cu[r + 1]].sum()) for r in range(R)]
    return int(cnt_b.sum().item())


def test_noalloc_select_matches_upf_select_on_two_calls_in_a_row(lib):
    # first call: a long batch; second call: a shorter one, so that anything left
    # in the shared array by the first call would show up in the second
    kept1 = run_both([131072, 5000, 70000], seed=1, block=64, top_p=0.99, pass_block_scores=False)
    kept2 = run_both([3000, 41, 9000], seed=2, block=32, top_p=0.9, pass_block_scores=True)
    assert kept1 > 0 and kept2 > 0


def test_noalloc_rejects_batches_over_its_limits(lib):
    cu = np.arange(0, 1026 * 10, 10, dtype=np.int32)       # 1025 requests
    batch, keep = B.make_batch(0x1000, cu, 32, 8, 128)
    with pytest.raises(B.UpfError) as e:
        B.upf_select_noalloc(batch, B.make_params(), 0x1000, 0, 0x1000, 0x1000)
    assert e.value.status == 2 and "UPF_NOALLOC_MAX_REQS" in e.value.message
    cu = np.array([0, 16384 * 64, 2 * 16384 * 64, 5 * 16384 * 64], dtype=np.int32)   # > 65536 blocks
    batch, keep = B.make_batch(0x1000, cu, 32, 8, 128)
    with pytest.raises(B.UpfError) as e:
        B.upf_select_noalloc(batch, B.make_params(), 0x1000, 0, 0x1000, 0x1000)
    assert e.value.status == 2
