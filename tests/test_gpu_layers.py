"""GPU parity of the cross-layer helpers against the float64 oracle.

Revival of frozen tokens and re-selection on the compacted batch (UniPrefill
article, section 2, third step), and per-layer KV lengths read from the drop
history (section 3, last paragraph).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare as C
from sparse_long_context_tail_gb300 import _binding as B
from sparse_long_context_tail_gb300 import workload as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def sel():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_long_context_tail_gb300.selector import TokenSelector
    s = TokenSelector(0)
    yield s
    s.close()


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _run(sel, k_bits, q_full_bits, cu, spec, hidden, layer_id, history=None, history_len=None):
    q = _up(q_full_bits.view(np.int16)).view(torch.bfloat16)
    k = _up(k_bits.view(np.int16)).view(torch.bfloat16)
    params = B.make_params(spec.n_tail, spec.block, spec.sink_keep, spec.tail_keep, spec.top_p)
    out = sel.select_tokens(q, k, cu, _up(cu), spec.num_q_heads, spec.num_kv_heads, spec.head_dim, hidden,
                            layer_id=layer_id, history=history, history_len=history_len, params=params)
    torch.cuda.synchronize()
    assert sel.status() == 0
    return out


def test_revive_matches_oracle(sel):
    spec = wl.WorkloadSpec("rev", [1500, 700], 8, 2, 128, 264, planted=[2, 1], seed=21)
    w = wl.generate(spec)
    hid = _up(w.hidden_bits().view(np.int16))
    out = _run(sel, w.k_bits, w.q_full_bits(), w.cu_seqlens, spec, hid, 0)
    total = int(out.total_kept.item())
    # "later layers" change the kept rows; dropped rows stay frozen
    rows = out.hidden_out[:total] ^ torch.tensor(0x1234, dtype=torch.int16, device=DEV)
    full = hid.clone()
    batch, keep = B.make_batch(_up(w.cu_seqlens).data_ptr(), w.cu_seqlens, 8, 2, 128)
    B.upf_revive(sel.ctx, batch, out.kept_index.data_ptr(), out.total_kept.data_ptr(), rows.data_ptr(),
                 hid.stride(0) * 2, full.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    want = oracle.revive(w.hidden_bits().view(np.int16), out.kept_index[:total].cpu().numpy(), rows.cpu().numpy())
    np.testing.assert_array_equal(full.cpu().numpy(), want)


def test_history_kv_len_after_two_drops(sel):
    spec = wl.WorkloadSpec("hist", [2000, 900, 1300], 8, 2, 128, 64, planted=[2, 1, 1], seed=22)
    w = wl.generate(spec)
    R, cap = 3, 4
    hist = torch.zeros((R, cap, 2), dtype=torch.int32, device=DEV)
    hlen = torch.zeros(R, dtype=torch.int32, device=DEV)
    hid = _up(w.hidden_bits().view(np.int16))
    _run(sel, w.k_bits, w.q_full_bits(), w.cu_seqlens, spec, hid, 3, hist, hlen)
    _run(sel, w.k_bits, w.q_full_bits(), w.cu_seqlens, spec, hid, 11, hist, hlen)
    h_np, l_np = hist.cpu().numpy(), hlen.cpu().numpy()
    assert l_np.tolist() == [2, 2, 2]
    cu_dev = _up(w.cu_seqlens)
    batch, keep = B.make_batch(cu_dev.data_ptr(), w.cu_seqlens, 8, 2, 128)
    kv = torch.empty(R, dtype=torch.int32, device=DEV)
    for layer in (0, 2, 3, 7, 11, 30):
        B.upf_history_kv_len(sel.ctx, batch, hist.data_ptr(), hlen.data_ptr(), cap, layer, kv.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert kv.cpu().numpy().tolist() == oracle.history_kv_len(h_np, l_np, w.cu_seqlens, layer).tolist(), layer


def test_second_layer_selects_on_the_compacted_batch(sel):
    """Layer A drops tokens; the next full-attention layer scores the compacted batch only."""
    spec = wl.WorkloadSpec("chain", [3000, 1800], 8, 2, 128, 128, planted=[4, 2], block=32, seed=23)
    w = wl.generate(spec)
    hid = _up(w.hidden_bits().view(np.int16))
    first = _run(sel, w.k_bits, w.q_full_bits(), w.cu_seqlens, spec, hid, 0)
    total = int(first.total_kept.item())
    kept = first.kept_index[:total].cpu().numpy()
    cu2 = first.cu_seqlens_out.cpu().numpy().astype(np.int32)
    # Next layer's keys: the kept tokens' rows (random new values would do as well); the
    # tail is exempt, so each request's questioners are the last n rows of its compacted part.
    k2 = w.k_bits[kept]
    q2 = w.q_full_bits()[kept]
    tails = np.concatenate([np.arange(cu2[r + 1] - min(spec.n_tail, cu2[r + 1] - cu2[r]), cu2[r + 1])
                            for r in range(len(cu2) - 1)])
    second = _run(sel, k2, q2, cu2, spec, _up(w.hidden_bits().view(np.int16)[kept]), 5)
    ref_s = oracle.token_scores(k2, q2[tails], cu2, 8, 2, 128, spec.n_tail)
    assert C.score_violations(second.scores.cpu().numpy(), ref_s, cu2)["ok"]
    ref = oracle.select(ref_s, cu2, spec.block, spec.top_p, spec.sink_keep, spec.tail_keep)
    mask2 = C.unpack_bits(second.keep_bits.cpu().numpy(), int(cu2[-1]))
    assert not C.mask_mismatches(mask2, ref, cu2, spec.block, spec.top_p, spec.sink_keep, spec.tail_keep)
    assert int(second.total_kept.item()) <= total
