"""Pins of the float64 oracle against things other than itself.

Each test fixes one part of the oracle by an independent route: a pure-Python
brute force, a library routine, a closed form, an exhaustive enumeration, a
hand-worked fixture, or an invariant of the method (UniPrefill article, section
2).  A plausible slip in the oracle (a dropped causal mask, a wrong softmax
axis, head grouping by modulo instead of contiguous groups, a missing scale,
mean over the wrong count, the wrong end of the ranking, an off-by-one in the
exempt ranges, a reordered compaction) fails at least one of them.
"""
import itertools
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle
from sparse_long_context_tail_gb300 import workload as wl

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers ----

def _bf16_py(bits):
    """bf16 -> float via struct (independent of the oracle's numpy conversion)."""
    return struct.unpack(">f", struct.pack(">I", int(bits) << 16))[0]


def _brute_scores(k_bits, q_bits, cu, Hq, Hkv, d, n, scale, kv_map):
    """Pure-Python loops: full causal softmax per (request, head, tail query)."""
    T = cu[-1]
    K = [[[_bf16_py(k_bits[t, g, e]) for e in range(d)] for g in range(Hkv)] for t in range(T)]
    s = [0.0] * T
    qrow = 0
    for r in range(len(cu) - 1):
        L = cu[r + 1] - cu[r]
        n_eff = min(n, L)
        for h in range(Hq):
            g = kv_map[h]
            for j in range(n_eff):
                t = L - n_eff + j
                q = [_bf16_py(q_bits[qrow + j, h, e]) for e in range(d)]
                logits = [scale * sum(q[e] * K[cu[r] + kk][g][e] for e in range(d)) for kk in range(t + 1)]
                mx = max(logits)
                den = sum(math.exp(x - mx) for x in logits)
                for kk in range(t + 1):
                    s[cu[r] + kk] += math.exp(logits[kk] - mx) / den / (Hq * n_eff)
        qrow += n_eff
    return np.array(s)


def _bits(x):
    return wl.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _rand_case(seed, lengths, Hq, Hkv, d, n):
    rng = np.random.default_rng(seed)
    cu = [0] + list(np.cumsum(lengths))
    T = cu[-1]
    k = _bits(rng.standard_normal((T, Hkv, d)))
    nq = sum(min(n, L) for L in lengths)
    q = _bits(rng.standard_normal((nq, Hq, d)) * 1.5)
    return cu, k, q


# ----------------------------------------------------------- input layer ----

def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F, 0x0001], dtype=np.uint16)
    want = [1.0, -2.0, 1.0078125, 0.0, -0.0, _bf16_py(0x7F7F), _bf16_py(0x0001)]
    got = oracle.bf16_to_f64(bits)
    assert [float(x) for x in got] == want


def test_tail_positions():
    assert list(oracle.tail_positions(10, 4)) == [6, 7, 8, 9]
    assert list(oracle.tail_positions(3, 128)) == [0, 1, 2]
    assert list(oracle.tail_positions(0, 128)) == []


# ----------------------------------------------------- scores [§2 step 1] ----

@pytest.mark.parametrize("lengths,Hq,Hkv,d,n", [
    ([9], 1, 1, 4, 3),
    ([1, 7, 12], 4, 2, 4, 5),
    ([13, 2], 6, 3, 8, 4),
    ([5], 2, 1, 4, 8),      # L < n: every token is a questioner
])
def test_scores_match_pure_python_brute_force(lengths, Hq, Hkv, d, n):
    cu, k, q = _rand_case(11 + len(lengths), lengths, Hq, Hkv, d, n)
    scale = 1.0 / math.sqrt(d)
    got = oracle.token_scores(k, q, cu, Hq, Hkv, d, n, threads=1)
    kv_map = [h // (Hq // Hkv) for h in range(Hq)]
    want = _brute_scores(k, q, cu, Hq, Hkv, d, n, scale, kv_map)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)


def test_single_query_single_head_is_one_softmax_row():
    """n=1, H_q=H_kv=1: the scores are scipy's softmax of the last query's logits."""
    rng = np.random.default_rng(5)
    L, d = 50, 16
    k = _bits(rng.standard_normal((L, 1, d)))
    q = _bits(rng.standard_normal((1, 1, d)))
    scale = 0.3
    got = oracle.token_scores(k, q, [0, L], 1, 1, d, 1, softmax_scale=scale, threads=1)
    Kf = np.array([[_bf16_py(k[t, 0, e]) for e in range(d)] for t in range(L)])
    qf = np.array([_bf16_py(q[0, 0, e]) for e in range(d)])
    want = scipy.special.softmax(scale * (Kf @ qf))
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-17)


@pytest.mark.parametrize("L,n,Hq,Hkv", [(40, 8, 2, 1), (6, 8, 4, 2), (300, 128, 8, 2)])
def test_uniform_attention_closed_form(L, n, Hq, Hkv):
    """K = 0 -> every visible logit is 0 -> P_j(k) = 1/(t_j+1) for k <= t_j.

    s_k = (1/n_eff) * sum_{j : t_j >= k} 1/(t_j + 1), the same for every head.
    """
    d = 8
    rng = np.random.default_rng(3)
    k = np.zeros((L, Hkv, d), dtype=np.uint16)
    n_eff = min(n, L)
    q = _bits(rng.standard_normal((n_eff, Hq, d)))
    got = oracle.token_scores(k, q, [0, L], Hq, Hkv, d, n, threads=1)
    tails = range(L - n_eff, L)
    want = [float(sum(Fraction(1, t + 1) for t in tails if t >= kk) / n_eff) for kk in range(L)]
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=0)


def test_scale_zero_gives_uniform_attention():
    cu, k, q = _rand_case(2, [30], 2, 1, 4, 6)
    got = oracle.token_scores(k, q, cu, 2, 1, 4, 6, softmax_scale=0.0, threads=1)
    want = [sum(1.0 / (t + 1) for t in range(24, 30) if t >= kk) / 6 for kk in range(30)]
    np.testing.assert_allclose(got, want, rtol=1e-13)


@pytest.mark.parametrize("lengths", [[1], [17], [3, 64, 129, 2]])
def test_scores_sum_to_one_per_request(lengths):
    """Each query's probabilities sum to 1, so the mean over (h, j) sums to 1 per request."""
    cu, k, q = _rand_case(7, lengths, 4, 2, 8, 16)
    s = oracle.token_scores(k, q, cu, 4, 2, 8, 16, threads=2)
    for r in range(len(lengths)):
        assert abs(s[cu[r]:cu[r + 1]].sum() - 1.0) < 1e-12
    assert (s >= 0).all()


def test_causal_keys_after_every_questioner_get_nothing_but_later_ones_do():
    """Keys seen only by later questioners get less mass than under full visibility."""
    cu, k, q = _rand_case(9, [20], 1, 1, 4, 5)
    s = oracle.token_scores(k, q, cu, 1, 1, 4, 5, threads=1)
    # the last key is seen only by the last questioner
    kf = oracle.bf16_to_f64(k).reshape(20, 4)
    qf = oracle.bf16_to_f64(q).reshape(5, 4)
    last = scipy.special.softmax(0.5 * (kf @ qf[4]))[19] / 5
    assert abs(s[19] - last) < 1e-15


def test_planted_key_takes_all_attention():
    """One key with logit +64 above every other: softmax puts 1 - O(L e^-64) on it."""
    L, d, n = 200, 4, 16
    k = np.zeros((L, 1, d), dtype=np.uint16)
    k[37, 0] = _bits([2.0, 0, 0, 0])
    q = np.tile(_bits([64.0, 0, 0, 0]), (n, 1, 1)).reshape(n, 1, d)
    s = oracle.token_scores(k, q, [0, L], 1, 1, d, n, threads=1)   # scale 1/2 -> logit 64
    assert abs(s[37] - 1.0) < 1e-15
    assert np.delete(s, 37).max() < 1e-26


def test_gqa_groups_are_contiguous():
    """H_q=4, H_kv=2: q-heads 0,1 read kv-head 0 and 2,3 read kv-head 1.

    Heads 0,1 have q = 0 (uniform attention).  Heads 2,3 have a strong q that
    picks key a under kv-head 0 and key b under kv-head 1.  Contiguous grouping
    gives 0.5*uniform + 0.5*delta_b; grouping by h % H_kv would give
    0.5*uniform + 0.25*delta_a + 0.25*delta_b.
    """
    L, d, n, a, b = 64, 4, 4, 10, 20
    k = np.zeros((L, 2, d), dtype=np.uint16)
    k[a, 0] = _bits([2.0, 0, 0, 0])
    k[b, 1] = _bits([2.0, 0, 0, 0])
    q = np.zeros((n, 4, d), dtype=np.uint16)
    q[:, 2] = _bits([64.0, 0, 0, 0])
    q[:, 3] = _bits([64.0, 0, 0, 0])
    s = oracle.token_scores(k, q, [0, L], 4, 2, d, n, threads=1)
    uni = np.array([sum(1.0 / (t + 1) for t in range(L - n, L) if t >= kk) / n for kk in range(L)])
    want = 0.5 * uni
    want[b] += 0.5
    np.testing.assert_allclose(s, want, rtol=1e-12, atol=1e-20)
    # an explicit map reproduces the other grouping
    s2 = oracle.token_scores(k, q, [0, L], 4, 2, d, n, kv_of_q=[0, 1, 0, 1], threads=1)
    want2 = 0.5 * uni
    want2[a] += 0.25
    want2[b] += 0.25
    np.testing.assert_allclose(s2, want2, rtol=1e-12, atol=1e-20)


def test_requests_are_independent():
    """Packing requests together changes nothing for each of them."""
    cu, k, q = _rand_case(4, [33, 70], 2, 1, 8, 8)
    both = oracle.token_scores(k, q, cu, 2, 1, 8, 8, threads=1)
    first = oracle.token_scores(k[:33], q[:8], [0, 33], 2, 1, 8, 8, threads=1)
    second = oracle.token_scores(k[33:], q[8:], [0, 70], 2, 1, 8, 8, threads=1)
    np.testing.assert_array_equal(both, np.concatenate([first, second]))


def test_threads_do_not_change_the_result():
    cu, k, q = _rand_case(8, [50, 10, 90], 4, 2, 8, 16)
    a = oracle.token_scores(k, q, cu, 4, 2, 8, 16, threads=1)
    b = oracle.token_scores(k, q, cu, 4, 2, 8, 16, threads=8)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------ block means [§2 step 2] ----

def test_block_means_brute_force_and_partial_last_block():
    s = np.arange(1.0, 11.0)           # 1..10
    got = oracle.block_means(s, 4)     # [1..4], [5..8], [9, 10]
    assert list(got) == [2.5, 6.5, 9.5]
    assert list(oracle.block_means(np.ones(5), 2)) == [1.0, 1.0, 1.0]
    assert len(oracle.block_means(np.zeros(0), 64)) == 0


@pytest.mark.parametrize("L,G", [(1, 64), (64, 64), (65, 64), (1000, 64), (130, 32)])
def test_sum_of_block_means_weighted_by_size_is_total_score(L, G):
    rng = np.random.default_rng(L)
    s = rng.random(L)
    b = oracle.block_means(s, G)
    sizes = [min(L, (i + 1) * G) - i * G for i in range(len(b))]
    assert abs(sum(bi * ni for bi, ni in zip(b, sizes)) - s.sum()) < 1e-10


def test_block_size_one_is_token_level():
    s = np.random.default_rng(0).random(37)
    np.testing.assert_array_equal(oracle.block_means(s, 1), s)


# ------------------------------------------------ top-p set [§2 step 2] -----

def test_top_p_golden_examples():
    with open(os.path.join(GOLDEN, "top_p_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        keep = oracle.top_p_blocks(np.array(c["b"], dtype=np.float64), c["p"])
        assert sorted(np.nonzero(keep)[0].tolist()) == c["keep"], c


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("p", [0.3, 0.75, 0.99])
def test_top_p_is_a_minimum_cardinality_max_mass_set(seed, p):
    """Exhaustive enumeration of every subset (nb <= 10).

    Scores are multiples of 1/1024 so every sum is exact.  The oracle's set must
    reach p of the total, no smaller set may reach it, and no set of the same
    size may carry more mass.
    """
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(1, 11))
    b = rng.integers(0, 64, size=nb) / 1024.0
    if seed % 3 == 0:
        b[rng.integers(0, nb)] = b[0]           # force a tie sometimes
    keep = oracle.top_p_blocks(b, p)
    total = b.sum()
    target = p * total
    best = {}
    for mask in range(1 << nb):
        idx = [i for i in range(nb) if mask >> i & 1]
        m = sum(b[i] for i in idx)
        if m >= target:
            best[len(idx)] = max(best.get(len(idx), -1.0), m)
    kstar = min(best)
    assert keep.sum() == kstar
    assert b[keep].sum() == best[kstar]
    assert b[keep].sum() >= target


def test_top_p_ties_rank_lower_index_first():
    keep = oracle.top_p_blocks(np.full(8, 0.125), 0.3)   # needs 3 of 8 equal blocks
    assert np.nonzero(keep)[0].tolist() == [0, 1, 2]


def test_top_p_one_keeps_every_block_with_mass():
    b = np.array([0.0, 0.1, 0.0, 0.3, 0.6, 0.0])
    assert np.nonzero(oracle.top_p_blocks(b, 1.0))[0].tolist() == [1, 3, 4]


def test_top_p_tiny_keeps_only_the_top_block():
    b = np.array([0.1, 0.2, 0.7, 0.0])
    assert np.nonzero(oracle.top_p_blocks(b, 1e-9))[0].tolist() == [2]


# ------------------------------------------------ exempt [§2 exemption] -----

def test_exempt_blocks_golden_table():
    n = 0
    with open(os.path.join(GOLDEN, "exempt_blocks.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            lhs, rhs = line.split("|")
            L, G, sink, tail = (int(x) for x in lhs.split())
            want = [int(x) for x in rhs.split()]
            got = np.nonzero(oracle.exempt_blocks(L, G, sink, tail))[0].tolist()
            assert got == want, line
            n += 1
    assert n >= 8


def test_defaults_are_the_articles():
    with open(os.path.join(GOLDEN, "defaults.json")) as f:
        d = json.load(f)
    import inspect
    sig = inspect.signature(oracle.select_tokens)
    for key in ("n_tail", "block", "top_p", "sink_keep", "tail_keep"):
        assert sig.parameters[key].default == d[key]["value"], key
        assert getattr(wl.WorkloadSpec("x", [1], 1, 1, 8, 8), key) == d[key]["value"], key


# --------------------------------------------------------- whole mask -------

def test_planted_block_plus_exempt_is_the_kept_set():
    """One block carries (to e^-32) all the attention: kept = it + sink + tail blocks."""
    L, d, n, G = 1024, 4, 128, 64
    k = np.zeros((L, 1, d), dtype=np.uint16)
    k[512:576, 0] = _bits([4.0, 0, 0, 0])
    q = np.tile(_bits([16.0, 0, 0, 0]), (n, 2, 1)).reshape(n, 2, d)
    out = oracle.select_tokens(k, q, [0, L], 2, 1, d, n, G, 0.99, 128, 128, threads=1)
    kept_blocks = np.nonzero(out["block_keep"][0])[0].tolist()
    assert kept_blocks == [0, 1, 8, 14, 15]
    assert out["kept_count"].tolist() == [5 * 64]
    assert out["mask"].sum() == 320


@pytest.mark.parametrize("seed", range(4))
def test_mask_invariants_on_random_requests(seed):
    """kept mass >= p; dropping the smallest kept top-p block falls below p; exempt kept."""
    rng = np.random.default_rng(100 + seed)
    lengths = [int(x) for x in rng.integers(1, 700, size=3)]
    cu, k, q = _rand_case(seed, lengths, 4, 2, 8, 32)
    p = 0.9
    out = oracle.select_tokens(k, q, cu, 4, 2, 8, 32, 16, p, 48, 40, threads=2)
    for r, L in enumerate(lengths):
        b = out["block_scores"][r]
        S = out["top_p_set"][r]
        keep = out["block_keep"][r]
        total = b.sum()
        assert b[S].sum() >= p * total * (1 - 1e-12)
        if S.any():
            assert b[S].sum() - b[S].min() < p * total
            assert b[S].min() >= b[~S].max(initial=-1.0)
        ex = oracle.exempt_blocks(L, 16, 48, 40)
        assert (keep >= ex).all() and (keep == (S | ex)).all()
        tok = out["mask"][cu[r]:cu[r + 1]]
        assert tok.sum() == out["kept_count"][r]
        for i in range(len(b)):
            assert (tok[i * 16:(i + 1) * 16] == keep[i]).all()


# ------------------------------------------- compaction [§2 step 3, §3] -----

def test_compaction_golden_example():
    with open(os.path.join(GOLDEN, "compaction_example.json")) as f:
        g = json.load(f)
    mask = np.array(g["mask"], dtype=bool)
    hidden = np.arange(10 * 8, dtype=np.uint16).reshape(10, 8)
    hist = np.array(g["history_in"], dtype=np.int64)
    hlen = np.array(g["history_len_in"], dtype=np.int64)
    out = oracle.compact(mask, g["cu_seqlens"], hidden, np.array(g["positions"]), np.array(g["slots"]),
                         g["layer_id"], hist, hlen)
    e = g["expect"]
    assert out["kept_index"].tolist() == e["kept_index"]
    assert out["positions_out"].tolist() == e["positions_out"]
    assert out["slots_out"].tolist() == e["slots_out"]
    assert out["cu_seqlens_out"].tolist() == e["cu_seqlens_out"]
    assert out["total_kept"] == e["total_kept"]
    assert out["history"].tolist() == e["history"]
    assert out["history_len"].tolist() == e["history_len"]
    assert not out["capacity_error"]
    np.testing.assert_array_equal(out["hidden_out"], hidden[e["kept_index"]])
    again = oracle.compact(mask, g["cu_seqlens"], layer_id=8, history=out["history"],
                           history_len=out["history_len"])
    assert again["capacity_error"] == g["second_call"]["capacity_error"]
    np.testing.assert_array_equal(again["history"], out["history"])
    np.testing.assert_array_equal(again["history_len"], out["history_len"])


def test_compaction_all_and_nothing():
    cu = [0, 5, 5, 9]
    allk = oracle.compact(np.ones(9, bool), cu)
    assert allk["kept_index"].tolist() == list(range(9)) and allk["cu_seqlens_out"].tolist() == [0, 5, 5, 9]
    none = oracle.compact(np.zeros(9, bool), cu)
    assert none["total_kept"] == 0 and none["cu_seqlens_out"].tolist() == [0, 0, 0, 0]


def test_empty_request_in_a_batch():
    cu, k, q = _rand_case(1, [20, 0, 15], 2, 1, 4, 8)
    out = oracle.select_tokens(k, q, cu, 2, 1, 4, 8, 4, 0.9, 4, 4, threads=1)
    assert out["kept_count"].tolist()[1] == 0
    assert abs(out["scores"][:20].sum() - 1) < 1e-12 and abs(out["scores"][20:].sum() - 1) < 1e-12


def test_history_kv_len_hand_worked():
    """Two requests of 1000 and 600 tokens; drops at layers 3 and 11 for request 0, layer 3 only for request 1.

    Layers 0-2 hold the prompt; layers 3-10 hold the first drop's kept count;
    layer 11 on holds the second drop's (UniPrefill article, section 3: the
    drop history tells decode how many KV entries each layer wrote).
    """
    hist = np.array([[[3, 400], [11, 150], [0, 0]], [[3, 90], [0, 0], [0, 0]]])
    hlen = np.array([2, 1])
    cu = [0, 1000, 1600]
    want = {0: [1000, 600], 2: [1000, 600], 3: [400, 90], 10: [400, 90], 11: [150, 90], 40: [150, 90]}
    for layer, kv in want.items():
        assert oracle.history_kv_len(hist, hlen, cu, layer).tolist() == kv
    assert oracle.history_kv_len(hist, np.array([0, 0]), cu, 40).tolist() == [1000, 600]


def test_revive_hand_worked_and_round_trip():
    """Kept rows return to their token positions; dropped rows stay frozen (section 2, third step)."""
    full = np.arange(6 * 2).reshape(6, 2)            # 6 tokens, 2 values each
    rows = np.array([[100, 101], [102, 103]])        # later layers' output for the kept tokens 1 and 4
    got = oracle.revive(full, [1, 4], rows)
    assert got.tolist() == [[0, 1], [100, 101], [4, 5], [6, 7], [102, 103], [10, 11]]
    assert full.tolist()[1] == [2, 3]                 # input untouched
    # compacting then reviving unchanged rows reproduces the original exactly
    rng = np.random.default_rng(0)
    h = rng.integers(0, 1 << 15, size=(50, 8))
    mask = rng.random(50) < 0.3
    comp = oracle.compact(mask, [0, 20, 50], hidden=h)
    np.testing.assert_array_equal(oracle.revive(h, comp["kept_index"], comp["hidden_out"]), h)
