"""GPU parity: libupf (through its C ABI) against the float64 oracle.

Scores within 1e-3 relative (+1e-6/L absolute floor); the keep mask equal to
the oracle's outside boundary blocks and exactly the top-p rule on the GPU's own
block scores; compaction, metadata and drop history bit-exact given the mask.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import compare as C
from sparse_long_context_tail_gb300 import _binding as B
from sparse_long_context_tail_gb300 import workload as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sel():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_long_context_tail_gb300.selector import TokenSelector
    s = TokenSelector(0)
    yield s
    s.close()


DEV = torch.device("cuda", 0)


def _up(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


def params_of(spec, **kw):
    d = dict(n_tail=spec.n_tail, block=spec.block, sink_keep=spec.sink_keep, tail_keep=spec.tail_keep,
             top_p=spec.top_p)
    d.update(kw)
    return B.make_params(**d)


def run_gpu(sel, w, params, hidden=True, layer_id=5, history=None, history_len=None, kv_of_q=None):
    s = w.spec
    q = _up(w.q_full_bits().view(np.int16)).view(torch.bfloat16)
    k = _up(w.k_bits.view(np.int16)).view(torch.bfloat16)
    hid = _up(w.hidden_bits().view(np.int16)) if hidden else None
    pos = _up(w.positions()) if hidden else None
    slots = _up(w.slots()) if hidden else None
    out = sel.select_tokens(q, k, w.cu_seqlens, _up(w.cu_seqlens), s.num_q_heads, s.num_kv_heads, s.head_dim,
                            hid, pos, slots, layer_id=layer_id, history=history, history_len=history_len,
                            params=params, kv_of_q=kv_of_q)
    torch.cuda.synchronize()
    status = sel.status()
    return out, status, (hid, pos, slots)


def ref_of(w, params, kv_of_q=None):
    s = w.spec
    scores = oracle.token_scores(w.k_bits, w.q_tail_bits, w.cu_seqlens, s.num_q_heads, s.num_kv_heads,
                                 s.head_dim, params.n_tail, None, kv_of_q)
    sel = oracle.select(scores, w.cu_seqlens, params.block, params.top_p, params.sink_keep, params.tail_keep)
    return scores, sel


def check(w, params, out, status, inputs, kv_of_q=None, check_hidden=True):
    assert status == 0, B.STATUS_NAMES.get(status)
    cu = w.cu_seqlens
    T = w.total_tokens
    scores, sel = ref_of(w, params, kv_of_q)
    got = out.scores.cpu().numpy()
    v = C.score_violations(got, scores, cu)
    assert v["ok"], v
    mask = C.unpack_bits(out.keep_bits.cpu().numpy(), T)
    bad = C.mask_mismatches(mask, sel, cu, params.block, params.top_p, params.sink_keep, params.tail_keep)
    assert not bad, bad[:10]
    nb = TokenSelectorBlocks(cu, params.block)
    bs = out.block_scores.cpu().numpy()[:nb]
    bad2 = C.self_consistency_mismatches(mask, bs, cu, params.block, params.top_p, params.sink_keep,
                                         params.tail_keep)
    assert not bad2, bad2[:10]
    # block scores against the oracle's block means of its own scores
    ref_bs = np.concatenate([b for b in sel["block_scores"]]) if nb else np.zeros(0)
    assert np.all(np.abs(bs - ref_bs) <= 1e-3 * np.abs(ref_bs) + 1e-6 / max(1, T)), "block means"
    # compaction and metadata, bit-exact given the GPU's mask
    comp = oracle.compact(mask, cu)
    total = int(out.total_kept.item())
    assert total == comp["total_kept"]
    assert out.kept_count.cpu().numpy().tolist() == comp["kept_count"].tolist()
    assert out.cu_seqlens_out.cpu().numpy().tolist() == comp["cu_seqlens_out"].tolist()
    kidx = out.kept_index.cpu().numpy()[:total]
    np.testing.assert_array_equal(kidx, comp["kept_index"])
    hid, pos, slots = inputs
    if hid is not None:
        idx = torch.from_numpy(comp["kept_index"]).to(DEV)
        np.testing.assert_array_equal(out.pos_out[:total].cpu().numpy(), w.positions()[comp["kept_index"]])
        np.testing.assert_array_equal(out.slot_out[:total].cpu().numpy(), w.slots()[comp["kept_index"]])
        if check_hidden:
            assert torch.equal(out.hidden_out[:total], hid.index_select(0, idx))
    return mask, sel


def TokenSelectorBlocks(cu, G):
    L = np.diff(np.asarray(cu, dtype=np.int64))
    return int(sum(-(-int(x) // G) for x in L))


# ----------------------------------------------------------- small cases ----

SMALL = [
    ("ragged-d64", dict(lengths=[1, 77, 300, 0, 1029, 4200], H=(4, 2, 64), hidden=512, n=128, G=64, planted=[0, 0, 1, 0, 3, 6])),
    ("llama-2req", dict(lengths=[3000, 1700], H=(32, 8, 128), hidden=4096, n=128, G=64, planted=[4, 2])),
    ("qwen-n512-G32", dict(lengths=[2500], H=(16, 2, 256), hidden=2048, n=512, G=32, planted=[5])),
    ("gemma-n32-G128", dict(lengths=[2000, 640], H=(16, 8, 256), hidden=3840, n=32, G=128, planted=[2, 1])),
    # 256 rows per group at d = 256 over 8 kv heads x 65536+ tokens: pass 1 in two 128-row chunks,
    # pass 2 in one 256-row chunk on CTA pairs
    ("d256-rows256", dict(lengths=[40000, 0, 25600], H=(16, 8, 256), hidden=512, n=128, G=64, planted=[2, 0, 1])),
    ("tail-only", dict(lengths=[100, 129, 257], H=(8, 2, 128), hidden=256, n=128, G=64, planted=[0, 0, 0])),
    ("odd-hidden", dict(lengths=[3333], H=(8, 1, 128), hidden=520, n=64, G=16, planted=[7])),
    # 384 query rows per chunk: pass-2 units of 128 columns, three per key tile
    ("gqa3-rows384", dict(lengths=[2600, 1500], H=(6, 2, 128), hidden=256, n=128, G=64, planted=[3, 2])),
    # 64 query rows: one unit per key tile in both passes
    ("rows64-d128", dict(lengths=[3100, 900, 2049], H=(8, 4, 128), hidden=256, n=32, G=32, planted=[2, 1, 1])),
]


def small_spec(name, c, seed=77):
    Hq, Hkv, d = c["H"]
    return wl.WorkloadSpec(name, c["lengths"], Hq, Hkv, d, c["hidden"], n_tail=c["n"], block=c["G"],
                           planted=c["planted"], strength_range=(1.0, 4.0), seed=seed)


@pytest.mark.parametrize("name,c", SMALL, ids=[s[0] for s in SMALL])
def test_small_parity(sel, name, c):
    spec = small_spec(name, c)
    w = wl.generate(spec)
    p = params_of(spec)
    out, status, inputs = run_gpu(sel, w, p)
    check(w, p, out, status, inputs)


@pytest.mark.parametrize("name,c", [SMALL[0], SMALL[2]], ids=["ragged-d64", "qwen-n512-G32"])
def test_cuda_core_fallback_parity(sel, name, c, monkeypatch):
    """The CUDA-core scoring kernels (used when n is not a multiple of 16) against the oracle."""
    monkeypatch.setenv("UPF_SCORE_PATH", "simt")
    spec = small_spec(name, c)
    w = wl.generate(spec)
    p = params_of(spec)
    out, status, inputs = run_gpu(sel, w, p)
    check(w, p, out, status, inputs)


@pytest.mark.parametrize("pairs", ["0", "1"])
@pytest.mark.parametrize("name,c", [SMALL[1], SMALL[2], SMALL[0], SMALL[4]],
                         ids=["llama-2req", "qwen-n512-G32", "ragged-d64", "d256-rows256"])
def test_scoring_on_single_ctas_and_on_pairs(sel, name, c, pairs, monkeypatch):
    """d = 256 chunks of whole 256-row units run on CTA pairs by default (and
    a d = 256 group of 256 rows runs pass 2 on pairs after pass 1 on single
    CTAs), the rest on single CTAs; both kernel families must match the oracle
    at every head dim (UPF_SCORE_PAIRS=0: single CTAs only, =1: pairs wherever
    the chunk allows)."""
    monkeypatch.setenv("UPF_SCORE_PAIRS", pairs)
    spec = small_spec(name, c)
    w = wl.generate(spec)
    p = params_of(spec)
    out, status, inputs = run_gpu(sel, w, p)
    check(w, p, out, status, inputs)


def test_pair_scoring_full_size_at_d128(sel, monkeypatch):
    monkeypatch.setenv("UPF_SCORE_PAIRS", "1")
    spec = wl.named_spec("llama8b-L131072")
    w = wl.generate(spec)
    p = params_of(spec)
    out, status, inputs = run_gpu(sel, w, p)
    check(w, p, out, status, inputs)


def test_odd_tail_count_uses_fallback(sel):
    """n = 100 (not a multiple of 16) runs on the CUDA-core kernels."""
    spec = wl.WorkloadSpec("n100", [900, 2048], 8, 2, 128, 256, n_tail=100, block=64, planted=[1, 2], seed=9)
    w = wl.generate(spec)
    p = params_of(spec)
    out, status, inputs = run_gpu(sel, w, p)
    check(w, p, out, status, inputs)


def test_explicit_kv_map(sel):
    spec = wl.WorkloadSpec("kvmap", [1500, 900], 8, 2, 128, 256, planted=[2, 1], seed=5,
                           kv_of_q=[0, 1, 0, 1, 0, 1, 0, 1])
    w = wl.generate(spec)
    p = params_of(spec)
    out, status, inputs = run_gpu(sel, w, p, kv_of_q=spec.kv_of_q)
    check(w, p, out, status, inputs, kv_of_q=spec.kv_of_q)


def test_top_p_one_and_small_p(sel):
    spec = small_spec("p1", SMALL[1][1])
    w = wl.generate(spec)
    for top_p in (1.0, 0.5):
        p = params_of(spec, top_p=top_p)
        out, status, inputs = run_gpu(sel, w, p)
        check(w, p, out, status, inputs)


def test_scale_parameter(sel):
    spec = small_spec("scale", SMALL[0][1])
    w = wl.generate(spec)
    p = params_of(spec, softmax_scale=0.05)
    out, status, inputs = run_gpu(sel, w, p, hidden=False)
    s = w.spec
    ref = oracle.token_scores(w.k_bits, w.q_tail_bits, w.cu_seqlens, s.num_q_heads, s.num_kv_heads, s.head_dim,
                              s.n_tail, 0.05)
    assert status == 0
    assert C.score_violations(out.scores.cpu().numpy(), ref, w.cu_seqlens)["ok"]


def test_entry_points_separately_match_fused(sel):
    """upf_score, upf_select and upf_compact called one by one give the fused call's results."""
    spec = small_spec("sep", SMALL[0][1])
    w = wl.generate(spec)
    p = params_of(spec)
    fused, status, (hid, pos, slots) = run_gpu(sel, w, p)
    s = w.spec
    T = w.total_tokens
    cu_dev = _up(w.cu_seqlens)
    batch, keep = B.make_batch(cu_dev.data_ptr(), w.cu_seqlens, s.num_q_heads, s.num_kv_heads, s.head_dim)
    nbytes = B.upf_workspace_bytes(batch, p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    q = _up(w.q_full_bits().view(np.int16)).view(torch.bfloat16)
    k = _up(w.k_bits.view(np.int16)).view(torch.bfloat16)
    scores = torch.empty(T, dtype=torch.float32, device=DEV)
    B.upf_score(sel.ctx, batch, p, q.data_ptr(), q.stride(0), k.data_ptr(), k.stride(0), scores.data_ptr(),
                ws.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
    bits = torch.empty((T + 31) // 32, dtype=torch.int32, device=DEV)
    cnt = torch.empty(len(w.cu_seqlens) - 1, dtype=torch.int32, device=DEV)
    B.upf_select(sel.ctx, batch, p, scores.data_ptr(), 0, bits.data_ptr(), cnt.data_ptr(), ws.data_ptr(), nbytes,
                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(scores, fused.scores)
    assert torch.equal(bits, fused.keep_bits)
    assert torch.equal(cnt, fused.kept_count)


def test_compact_with_oracle_mask(sel):
    """Feed the oracle's mask to upf_compact: outputs and history are bit-exact."""
    spec = small_spec("cmp", SMALL[0][1])
    w = wl.generate(spec)
    p = params_of(spec)
    scores, ref = ref_of(w, p)
    T, R = w.total_tokens, len(w.cu_seqlens) - 1
    bits = _up(C.pack_bits(ref["mask"]).view(np.int32))
    cu_dev = _up(w.cu_seqlens)
    batch, keep = B.make_batch(cu_dev.data_ptr(), w.cu_seqlens, 1, 1, 64)
    nbytes = B.upf_workspace_bytes(batch, B.make_params())
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    hid = _up(w.hidden_bits().view(np.int16))
    pos, slots = _up(w.positions()), _up(w.slots())
    hout, pout, sout = torch.empty_like(hid), torch.empty_like(pos), torch.empty_like(slots)
    kidx = torch.empty(T, dtype=torch.int32, device=DEV)
    cuo = torch.empty(R + 1, dtype=torch.int32, device=DEV)
    tot = torch.empty(1, dtype=torch.int32, device=DEV)
    cap = 3
    hist0 = np.zeros((R, cap, 2), dtype=np.int32)
    hist0[:, 0] = [[1, 11]] * R
    hlen0 = np.ones(R, dtype=np.int32)
    hist, hlen = _up(hist0), _up(hlen0)
    io = B.make_compact_io(hid.stride(0) * 2, hid.data_ptr(), hout.data_ptr(), pos.data_ptr(), pout.data_ptr(),
                           slots.data_ptr(), sout.data_ptr(), kidx.data_ptr(), cuo.data_ptr(), tot.data_ptr(), 9,
                           cap, hist.data_ptr(), hlen.data_ptr())
    stream = torch.cuda.current_stream().cuda_stream
    B.upf_compact(sel.ctx, batch, bits.data_ptr(), io, ws.data_ptr(), nbytes, stream)
    torch.cuda.synchronize()
    assert sel.status() == 0
    comp = oracle.compact(ref["mask"], w.cu_seqlens, w.hidden_bits(), w.positions(), w.slots(), 9, hist0, hlen0)
    total = comp["total_kept"]
    assert int(tot.item()) == total
    np.testing.assert_array_equal(kidx[:total].cpu().numpy(), comp["kept_index"])
    np.testing.assert_array_equal(cuo.cpu().numpy(), comp["cu_seqlens_out"])
    np.testing.assert_array_equal(hout[:total].cpu().numpy().view(np.uint16), comp["hidden_out"])
    np.testing.assert_array_equal(pout[:total].cpu().numpy(), comp["positions_out"])
    np.testing.assert_array_equal(sout[:total].cpu().numpy(), comp["slots_out"])
    np.testing.assert_array_equal(hist.cpu().numpy(), comp["history"])
    np.testing.assert_array_equal(hlen.cpu().numpy(), comp["history_len"])
    # fill the history to capacity, then one more call must report CAPACITY and write nothing
    B.upf_compact(sel.ctx, batch, bits.data_ptr(), io, ws.data_ptr(), nbytes, stream)
    torch.cuda.synchronize()
    assert sel.status() == 0
    before = hist.clone(), hlen.clone()
    B.upf_compact(sel.ctx, batch, bits.data_ptr(), io, ws.data_ptr(), nbytes, stream)
    torch.cuda.synchronize()
    assert sel.status() == 4
    assert torch.equal(hist, before[0]) and torch.equal(hlen, before[1])
    assert sel.status() == 0   # the status word was cleared by the read


def test_compact_all_and_none(sel):
    T = 5000
    cu = np.array([0, 1234, 1234, 5000], dtype=np.int32)
    cu_dev = _up(cu)
    batch, keep = B.make_batch(cu_dev.data_ptr(), cu, 1, 1, 64)
    nbytes = B.upf_workspace_bytes(batch, B.make_params())
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    hid = torch.randint(-30000, 30000, (T, 24), dtype=torch.int16, device=DEV)
    for fill in (0, -1):
        bits = torch.full(((T + 31) // 32,), fill, dtype=torch.int32, device=DEV)
        hout = torch.zeros_like(hid)
        kidx = torch.empty(T, dtype=torch.int32, device=DEV)
        cuo = torch.empty(4, dtype=torch.int32, device=DEV)
        tot = torch.empty(1, dtype=torch.int32, device=DEV)
        io = B.make_compact_io(48, hid.data_ptr(), hout.data_ptr(), kept_index=kidx.data_ptr(),
                               cu_seqlens_out=cuo.data_ptr(), total_kept=tot.data_ptr())
        B.upf_compact(sel.ctx, batch, bits.data_ptr(), io, ws.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        n = int(tot.item())
        if fill == 0:
            assert n == 0 and cuo.cpu().tolist() == [0, 0, 0, 0]
        else:   # all bits set, including stray bits past T in the last word
            assert n == T and cuo.cpu().tolist() == cu.tolist()
            assert torch.equal(hout, hid) and torch.equal(kidx.cpu(), torch.arange(T, dtype=torch.int32))



def test_compact_spans_several_chunks(sel):
    """Random keep bits over more tokens than one scan chunk holds (131072), with
    request boundaries on, just before and just after the chunk edges and an
    empty request: every output is bit-exact against the oracle."""
    rng = np.random.default_rng(11)
    T = 3 * 131072 + 4321
    cu = np.array([0, 5, 131071, 131072, 131073, 131073, 262144, 262175, 300000, T], dtype=np.int32)
    R = len(cu) - 1
    mask = rng.random(T) < 0.3
    mask[131000:131200] = True
    mask[262100:262200] = False
    cu_dev = _up(cu)
    batch, keep = B.make_batch(cu_dev.data_ptr(), cu, 1, 1, 64)
    nbytes = B.upf_workspace_bytes(batch, B.make_params())
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    bits = _up(C.pack_bits(mask).view(np.int32))
    hid_np = rng.integers(-30000, 30000, size=(T, 8), dtype=np.int16)
    pos_np = rng.integers(0, 1 << 40, size=T, dtype=np.int64)
    hid, pos = _up(hid_np), _up(pos_np)
    hout, pout = torch.empty_like(hid), torch.empty_like(pos)
    kidx = torch.empty(T, dtype=torch.int32, device=DEV)
    cuo = torch.empty(R + 1, dtype=torch.int32, device=DEV)
    tot = torch.empty(1, dtype=torch.int32, device=DEV)
    io = B.make_compact_io(16, hid.data_ptr(), hout.data_ptr(), pos.data_ptr(), pout.data_ptr(),
                           kept_index=kidx.data_ptr(), cu_seqlens_out=cuo.data_ptr(), total_kept=tot.data_ptr())
    B.upf_compact(sel.ctx, batch, bits.data_ptr(), io, ws.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert sel.status() == 0
    comp = oracle.compact(mask, cu, hid_np, pos_np)
    total = comp["total_kept"]
    assert int(tot.item()) == total
    np.testing.assert_array_equal(cuo.cpu().numpy(), comp["cu_seqlens_out"])
    np.testing.assert_array_equal(kidx[:total].cpu().numpy(), comp["kept_index"])
    np.testing.assert_array_equal(hout[:total].cpu().numpy(), comp["hidden_out"])
    np.testing.assert_array_equal(pout[:total].cpu().numpy(), comp["positions_out"])


@pytest.mark.parametrize("name,world", [("ragged-d64", 2), ("llama-2req", 2), ("llama-2req", 4)])
def test_tensor_parallel_heads_on_one_gpu(sel, name, world):
    """Heads sharded over `world` ranks, run one after another on this GPU:
    each rank scores its own heads (``upf_score_shard`` on head-range views,
    normalised by all H_q heads), the shard scores are summed in rank order
    (what the all-reduce computes), and selection plus compaction follow.
    Everything is checked against the oracle's all-heads result."""
    from sparse_long_context_tail_gb300 import tp
    c = dict(SMALL)[name]
    spec = small_spec("tp-" + name, c)
    w = wl.generate(spec)
    p = params_of(spec)
    q = _up(w.q_full_bits().view(np.int16)).view(torch.bfloat16)
    k = _up(w.k_bits.view(np.int16)).view(torch.bfloat16)
    cu_dev = _up(w.cu_seqlens)
    partials = []
    for r in range(world):
        qs, ks = tp.shard_heads(spec.num_q_heads, spec.num_kv_heads, r, world)
        partials.append(sel.score(q[:, qs], k[:, ks], w.cu_seqlens, cu_dev, qs.stop - qs.start, ks.stop - ks.start,
                                  spec.head_dim, params=p, total_q_heads=spec.num_q_heads))
    scores = tp.sum_of_partials(partials)
    hid, pos, slots = _up(w.hidden_bits().view(np.int16)), _up(w.positions()), _up(w.slots())
    out = sel.select_compact(scores, w.cu_seqlens, cu_dev, hid, pos, slots, layer_id=3, params=p)
    torch.cuda.synchronize()
    check(w, p, out, sel.status(), (hid, pos, slots))

def test_nonfinite_scores_are_reported(sel):
    cu = np.array([0, 640, 1000], dtype=np.int32)
    T = 1000
    cu_dev = _up(cu)
    batch, keep = B.make_batch(cu_dev.data_ptr(), cu, 1, 1, 64)
    p = B.make_params()
    nbytes = B.upf_workspace_bytes(batch, p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    scores = torch.full((T,), 1.0 / 640, device=DEV)
    scores[700] = float("nan")
    bits = torch.empty((T + 31) // 32, dtype=torch.int32, device=DEV)
    cnt = torch.empty(2, dtype=torch.int32, device=DEV)
    B.upf_select(sel.ctx, batch, p, scores.data_ptr(), 0, bits.data_ptr(), cnt.data_ptr(), ws.data_ptr(), nbytes,
                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert sel.status() == 5
    assert cnt.cpu().tolist()[1] == 360      # the request with the NaN keeps everything


def test_inconsistent_device_cu_seqlens_is_reported(sel):
    cu_host = np.array([0, 500, 1000], dtype=np.int32)
    cu_dev = _up(np.array([0, 700, 900], dtype=np.int32))    # device copy disagrees on the total
    batch, keep = B.make_batch(cu_dev.data_ptr(), cu_host, 1, 1, 64)
    p = B.make_params()
    nbytes = B.upf_workspace_bytes(batch, p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    scores = torch.full((1000,), 1e-3, device=DEV)
    bits = torch.empty(32, dtype=torch.int32, device=DEV)
    cnt = torch.empty(2, dtype=torch.int32, device=DEV)
    B.upf_select(sel.ctx, batch, p, scores.data_ptr(), 0, bits.data_ptr(), cnt.data_ptr(), ws.data_ptr(), nbytes,
                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert sel.status() == 1


@pytest.mark.parametrize("R", [64, 70])
def test_batches_at_and_past_the_carried_descriptor_limit(sel, R):
    """Up to 64 requests the fused call carries the batch's descriptor tables in
    the kernel parameters; past that the describe kernel builds them on the
    device.  Both routes against the oracle, with requests shorter than n."""
    rng = np.random.default_rng(20 + R)
    lengths = [int(x) for x in rng.integers(1, 400, size=R)]
    spec = wl.WorkloadSpec(f"many-{R}", lengths, 8, 2, 64, 64, n_tail=32, block=16, seed=R)
    w = wl.generate(spec)
    p = params_of(spec)
    out, status, inputs = run_gpu(sel, w, p)
    check(w, p, out, status, inputs)


@pytest.mark.parametrize("R", [2, 70])
def test_inconsistent_device_cu_seqlens_in_the_fused_call(sel, R):
    """A device cu_seqlens whose total disagrees with the host copy is reported
    by both descriptor routes (carried tables and device-built ones)."""
    spec = wl.WorkloadSpec("cu-mismatch", [300] * R, 8, 2, 64, 64, n_tail=32, block=16, seed=9)
    w = wl.generate(spec)
    q = _up(w.q_full_bits().view(np.int16)).view(torch.bfloat16)
    k = _up(w.k_bits.view(np.int16)).view(torch.bfloat16)
    bad = w.cu_seqlens.copy()
    bad[-1] -= 7
    sel.select_tokens(q, k, w.cu_seqlens, _up(bad), spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                      params=params_of(spec))
    torch.cuda.synchronize()
    assert sel.status() == 1
    # the context stays usable
    out, status, inputs = run_gpu(sel, w, params_of(spec), hidden=False)
    assert status == 0


def test_repeat_calls_are_deterministic(sel):
    spec = small_spec("det", SMALL[1][1])
    w = wl.generate(spec)
    p = params_of(spec)
    a, _, _ = run_gpu(sel, w, p, hidden=False)
    sa, ba = a.scores.clone(), a.keep_bits.clone()
    b, _, _ = run_gpu(sel, w, p, hidden=False)
    assert torch.equal(sa, b.scores) and torch.equal(ba, b.keep_bits)


# ----------------------------------------------- the benchmark workloads ----

# Every benchmark workload at full size: the four LLaMA-shaped / small ones and
# all eighteen Qwen3-Next / Gemma-3 sweep points (G in {32, 64, 128} x n in
# {32, 128, 512} for each shape).
FULL = ["small-L4096", "llama8b-L32768", "llama8b-L131072", "llama8b-batch16"] + list(wl.SWEEP_NAMES)
assert len(FULL) == 22


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(sel, name):
    spec = wl.named_spec(name)
    w = wl.generate(spec)
    p = params_of(spec)
    out, status, inputs = run_gpu(sel, w, p)
    check(w, p, out, status, inputs)


def _select_only(sel, scores_np, cu, block, top_p, sink=128, tail=128):
    cu = np.asarray(cu, dtype=np.int32)
    T, R = int(cu[-1]), len(cu) - 1
    cu_dev = _up(cu)
    batch, keep = B.make_batch(cu_dev.data_ptr(), cu, 1, 1, 64)
    p = B.make_params(block=block, top_p=top_p, sink_keep=sink, tail_keep=tail)
    nbytes = B.upf_workspace_bytes(batch, p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    scores = _up(np.asarray(scores_np, dtype=np.float32))
    nb = TokenSelectorBlocks(cu, block)
    bs = torch.empty(max(1, nb), dtype=torch.float32, device=DEV)
    bits = torch.empty((T + 31) // 32, dtype=torch.int32, device=DEV)
    cnt = torch.empty(R, dtype=torch.int32, device=DEV)
    B.upf_select(sel.ctx, batch, p, scores.data_ptr(), bs.data_ptr(), bits.data_ptr(), cnt.data_ptr(),
                 ws.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return sel.status(), C.unpack_bits(bits.cpu().numpy(), T), bs.cpu().numpy()[:nb], cnt.cpu().numpy()


def test_select_ties_take_lower_blocks_first(sel):
    """Equal block scores at the boundary enter in block-index order (the oracle's tie rule)."""
    rng = np.random.default_rng(3)
    # large and small requests, partial last blocks
    for G, L, top_p in [(64, 64 * 300, 0.5), (32, 32 * 1000 + 17, 0.37), (16, 16 * 5000, 0.9),
                        (64, 64 * 200, 0.5), (32, 32 * 37 + 5, 0.9), (16, 16 * 256, 0.3), (8, 8 * 257, 0.6),
                        (64, 64 * 3 + 1, 0.99)]:
        nb = -(-L // G)
        levels = np.array([0.0, 1.0, 2.0, 4.0], dtype=np.float32)    # few distinct values: many ties
        b = levels[rng.integers(0, 4, size=nb)]
        scores = np.repeat(b, G)[:L]
        status, mask, bs, cnt = _select_only(sel, scores, [0, L], G, top_p, sink=0, tail=0)
        assert status == 0
        want = oracle.select(scores.astype(np.float64), [0, L], G, top_p, 0, 0)["mask"]
        np.testing.assert_array_equal(mask, want)


def test_select_boundary_bucket_small_after_each_round(sel):
    """Score sets whose boundary bucket drops to at most 256 blocks after the
    first, second, third or fourth 8-bit round of the radix select (and one
    where it never does: over 256 equal scores), against the oracle's rule.
    One token per block and scores exact in float32, so the block means are
    the scores themselves."""
    rng = np.random.default_rng(11)
    nb = 2000
    cases = [
        (rng.exponential(1.0, nb) ** 4).astype(np.float32).astype(np.float64),   # exponents differ: first round
        1.0 + rng.integers(0, 128, nb) * 2.0 ** -7,          # bits 16-22 differ: second round
        1.5 + rng.integers(0, 512, nb) * 2.0 ** -16,         # bits 7-15 differ: third round
        1.5 + rng.integers(0, 256, nb) * 2.0 ** -23,         # low byte differs: fourth round
        np.array([1.0, 2.0, 3.0, 4.0])[rng.integers(0, 4, nb)],   # ~500 equal scores per value
    ]
    for vals in cases:
        scores = vals.astype(np.float32)
        assert np.array_equal(scores.astype(np.float64), vals)   # exact in float32
        for top_p in (0.3, 0.9, 0.99):
            status, mask, bs, cnt = _select_only(sel, scores, [0, nb], 1, top_p, sink=0, tail=0)
            assert status == 0
            want = oracle.select(scores.astype(np.float64), [0, nb], 1, top_p, 0, 0)["mask"]
            np.testing.assert_array_equal(mask, want)


def test_select_rejects_negative_scores(sel):
    scores = np.full(2000, 1.0 / 2000, dtype=np.float32)
    scores[768:832] = -1e-3          # block 12 has a negative mean
    status, mask, bs, cnt = _select_only(sel, scores, [0, 2000], 64, 0.99)
    assert status == 5 and mask.all() and cnt.tolist() == [2000]


def test_select_large_request_many_blocks(sel):
    """16384 blocks (the per-request maximum) against the oracle's rule."""
    rng = np.random.default_rng(4)
    G, nb = 8, 16384
    b = rng.exponential(1.0, size=nb).astype(np.float32) ** 4
    scores = np.repeat(b, G)
    status, mask, bs, cnt = _select_only(sel, scores, [0, nb * G], G, 0.95)
    assert status == 0
    bad = C.self_consistency_mismatches(mask, bs, [0, nb * G], G, 0.95, 128, 128)
    assert not bad, bad[:5]


def test_compaction_with_host_buffers(sel):
    """Hidden rows, positions and slots in page-locked host memory (read and
    written by the gather over the host link) give the device buffers' results."""
    spec = small_spec("hostbuf", SMALL[1][1])
    w = wl.generate(spec)
    p = params_of(spec)
    dev_out, status, _ = run_gpu(sel, w, p)
    assert status == 0
    q = _up(w.q_full_bits().view(np.int16)).view(torch.bfloat16)
    k = _up(w.k_bits.view(np.int16)).view(torch.bfloat16)
    hid_h = torch.from_numpy(w.hidden_bits().view(np.int16)).pin_memory()
    pos_h = torch.from_numpy(w.positions()).pin_memory()
    slot_h = torch.from_numpy(w.slots()).pin_memory()
    out = sel.alloc_outputs(w.cu_seqlens, spec.block)
    out.hidden_out = torch.empty_like(hid_h).pin_memory()
    out.pos_out = torch.empty_like(pos_h).pin_memory()
    out.slot_out = torch.empty_like(slot_h).pin_memory()
    s = w.spec
    sel.select_tokens(q, k, w.cu_seqlens, _up(w.cu_seqlens), s.num_q_heads, s.num_kv_heads, s.head_dim, hid_h,
                      pos_h, slot_h, params=p, kv_of_q=s.kv_of_q, out=out)
    torch.cuda.synchronize()
    assert sel.status() == 0
    total = int(out.total_kept.item())
    assert total == int(dev_out.total_kept.item())
    assert torch.equal(out.keep_bits, dev_out.keep_bits)
    assert torch.equal(out.hidden_out[:total], dev_out.hidden_out[:total].cpu())
    assert torch.equal(out.pos_out[:total], dev_out.pos_out[:total].cpu())
    assert torch.equal(out.slot_out[:total], dev_out.slot_out[:total].cpu())


def test_compaction_pageable_host_memory_is_refused_or_exact(sel):
    """An ordinary (pageable) host buffer is refused with a clear error, unless
    the device reads pageable host memory itself; then the rows are exact."""
    spec = small_spec("pageable", SMALL[4][1])
    w = wl.generate(spec)
    p = params_of(spec)
    dev_out, status, _ = run_gpu(sel, w, p)
    assert status == 0
    q = _up(w.q_full_bits().view(np.int16)).view(torch.bfloat16)
    k = _up(w.k_bits.view(np.int16)).view(torch.bfloat16)
    hid = torch.from_numpy(w.hidden_bits().view(np.int16)).clone()   # pageable host memory
    out = sel.alloc_outputs(w.cu_seqlens, spec.block)
    out.hidden_out = torch.empty(hid.shape, dtype=hid.dtype, device=DEV)
    s = w.spec
    try:
        sel.select_tokens(q, k, w.cu_seqlens, _up(w.cu_seqlens), s.num_q_heads, s.num_kv_heads, s.head_dim, hid,
                          params=p, kv_of_q=s.kv_of_q, out=out)
        torch.cuda.synchronize()
    except B.UpfError as e:
        assert "cannot access" in str(e)
        return
    assert sel.status() == 0
    total = int(out.total_kept.item())
    assert torch.equal(out.hidden_out[:total], dev_out.hidden_out[:total])


def test_pass1_sweeps_again_after_a_huge_logit_jump(sel):
    """One key with a logit about 2900 (log2 units) above every key of its
    item's first tile overflows pass 1's fast-path sums; that item is swept
    again on the checked path and every score still matches the oracle."""
    L, Hq, Hkv, d, n = 40000, 2, 1, 64, 32       # key splits of 512 keys: two 256-key tiles per item
    rng = np.random.default_rng(31)
    q = (0.5 * rng.standard_normal((L, Hq, d))).astype(np.float32)
    k = (0.5 * rng.standard_normal((L, Hkv, d))).astype(np.float32)
    q[L - n:] = 4.0
    big = 512 * 40 + 300                          # second tile of its item
    k[big] = 64.0
    q_bits, k_bits = wl.f32_to_bf16_bits(q), wl.f32_to_bf16_bits(k)
    cu = np.array([0, L], dtype=np.int32)
    p = B.make_params(n_tail=n, block=64, top_p=0.99)
    qd = _up(q_bits.view(np.int16)).view(torch.bfloat16)
    kd = _up(k_bits.view(np.int16)).view(torch.bfloat16)
    out = sel.select_tokens(qd, kd, cu, _up(cu), Hq, Hkv, d, params=p)
    torch.cuda.synchronize()
    assert sel.status() == 0
    ref = oracle.token_scores(k_bits, q_bits[L - n:], cu, Hq, Hkv, d, n)
    got = out.scores.cpu().numpy()
    assert C.score_violations(got, ref, cu)["ok"]
    assert got[big] > 0.99


def test_select_tokens_replays_from_a_cuda_graph(sel):
    """The fused call captured once in a CUDA graph and replayed gives the eager call's results."""
    spec = small_spec("graph", SMALL[1][1])
    w = wl.generate(spec)
    p = params_of(spec)
    s = w.spec
    q = _up(w.q_full_bits().view(np.int16)).view(torch.bfloat16)
    k = _up(w.k_bits.view(np.int16)).view(torch.bfloat16)
    hid = _up(w.hidden_bits().view(np.int16))
    pos, slots, cu_dev = _up(w.positions()), _up(w.slots()), _up(w.cu_seqlens)
    eager = sel.select_tokens(q, k, w.cu_seqlens, cu_dev, s.num_q_heads, s.num_kv_heads, s.head_dim, hid, pos, slots,
                              params=p, kv_of_q=s.kv_of_q)
    torch.cuda.synchronize()
    eager = {f: getattr(eager, f).clone() for f in ("scores", "keep_bits", "kept_count", "cu_seqlens_out",
                                                     "total_kept", "hidden_out", "pos_out", "slot_out")}
    out = sel.alloc_outputs(w.cu_seqlens, s.block, hid, pos, slots)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        sel.select_tokens(q, k, w.cu_seqlens, cu_dev, s.num_q_heads, s.num_kv_heads, s.head_dim, hid, pos, slots,
                          params=p, kv_of_q=s.kv_of_q, out=out)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            sel.select_tokens(q, k, w.cu_seqlens, cu_dev, s.num_q_heads, s.num_kv_heads, s.head_dim, hid, pos,
                              slots, params=p, kv_of_q=s.kv_of_q, out=out)
    for f in eager:
        getattr(out, f).zero_()
    g.replay()
    torch.cuda.synchronize()
    assert sel.status() == 0
    total = int(eager["total_kept"].item())
    for f in ("scores", "keep_bits", "kept_count", "cu_seqlens_out", "total_kept"):
        assert torch.equal(getattr(out, f), eager[f]), f
    for f in ("hidden_out", "pos_out", "slot_out"):
        assert torch.equal(getattr(out, f)[:total], eager[f][:total]), f
