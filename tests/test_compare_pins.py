"""Pins of the acceptance checker (``oracle/compare.py``).

Every GPU parity verdict passes through these rules, so each rule is fixed
here by hand-built candidates it must reject and ones it must accept.  A slip
in the checker (an ``or`` for an ``and``, a band that excuses too many blocks,
a missing partial-block or exempt-block check, a per-request sum taken over
the whole batch) fails at least one case below.

Method being checked: the UniPrefill article (m.youleyou.com/wenzhang/2886770),
section 2 second step (block means, the smallest block set reaching p of the
total) and the paragraph after it (the first and last 128 tokens are never
dropped).
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import compare as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------- bit packing ----

def test_pack_and_unpack_bits_by_hand():
    mask = np.zeros(40, dtype=bool)
    mask[[0, 3, 31, 32, 39]] = True
    words = C.pack_bits(mask)
    assert words.tolist() == [(1 << 0) | (1 << 3) | (1 << 31), (1 << 0) | (1 << 7)]
    assert C.unpack_bits(words, 40).tolist() == mask.tolist()
    # bits past T are ignored by unpacking
    assert C.unpack_bits(np.array([0xFFFFFFFF], dtype=np.uint32), 5).tolist() == [True] * 5


# ------------------------------------------------------- token scores ----

def _ref_two_requests():
    rng = np.random.default_rng(0)
    a = rng.exponential(1.0, 300)
    b = rng.exponential(1.0, 200)
    return np.concatenate([a / a.sum(), b / b.sum()]), [0, 300, 500]


def test_scores_identical_candidate_is_accepted():
    ref, cu = _ref_two_requests()
    v = C.score_violations(ref.astype(np.float32), ref, cu)
    assert v["ok"] and v["worst"] <= 0 and v["sum_err"] < 1e-6


def test_scores_one_token_off_by_1p2e_3_relative_is_rejected():
    ref, cu = _ref_two_requests()
    s = ref.copy()
    s[417] *= 1.0012
    v = C.score_violations(s, ref, cu)
    assert not v["ok"] and v["at"] == 417 and v["worst"] > 0
    assert v["sum_err"] < 1e-3          # the sum alone would have passed


def test_scores_one_token_off_by_0p8e_3_relative_is_accepted():
    ref, cu = _ref_two_requests()
    s = ref.copy()
    s[417] *= 1.0008
    assert C.score_violations(s, ref, cu)["ok"]


def test_scores_absolute_floor_is_one_millionth_of_the_mean_score():
    L = 1000
    ref = np.full(L, 1.0 / L)
    ref[10] = 0.0                       # a score that underflows: only the floor 1e-6 / L applies
    ref /= ref.sum()
    s = ref.copy()
    s[10] = 0.5e-6 / L
    assert C.score_violations(s, ref, [0, L])["ok"]
    s[10] = 2e-6 / L
    v = C.score_violations(s, ref, [0, L])
    assert not v["ok"] and v["at"] == 10


def test_scores_request_sum_off_by_2e_3_is_rejected():
    """Every token within its tolerance of the reference, but the request's
    scores sum to 1.002 (a reference that does not sum to 1 shows this)."""
    L = 500
    ref = np.full(L, 1.002 / L)
    v = C.score_violations(ref.copy(), ref, [0, L])
    assert v["worst"] <= 0 and not v["ok"] and abs(v["sum_err"] - 0.002) < 1e-9


def test_scores_sum_is_checked_per_request_not_over_the_batch():
    """0.5 + 1.5 = 2 = the number of requests: only a per-request sum sees it."""
    ref = np.concatenate([np.full(100, 0.5 / 100), np.full(100, 1.5 / 100)])
    v = C.score_violations(ref.copy(), ref, [0, 100, 200])
    assert not v["ok"] and abs(v["sum_err"] - 0.5) < 1e-12


def test_scores_empty_request_is_skipped():
    ref, cu = _ref_two_requests()
    cu3 = [0, 300, 300, 500]
    assert C.score_violations(ref.astype(np.float32), ref, cu3)["ok"]


# ---------------------------------------------------- boundary blocks ----

def test_boundary_blocks_hand_worked_fixture():
    with open(os.path.join(GOLDEN, "boundary_blocks.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = C.boundary_blocks(np.array(c["b"], dtype=np.float64), c["p"], c["tol"])
        assert got.tolist() == c["boundary"], c["name"]


def test_boundary_band_edges():
    """Running mass after the block at p + 0.0015: outside; at p + 0.0005: inside."""
    for after, want in ((0.9915, False), (0.9905, True), (0.9885, False), (0.9895, True)):
        b = np.array([after, 1.0 - after])            # b0 ends at `after`, b1 starts there
        got = C.boundary_blocks(b, 0.99)
        assert bool(got[0]) == want and bool(got[1]) == want, after


# ------------------------------------------------------ mask vs oracle ----

G = 4


def _fixture_mask_case():
    """8 blocks of 4 tokens; the first and last block are exempt (sink = tail = 4).

    Block means b = [0.01, 0.40, 0.30, 0.20, 0.0895, 0.0005, 0, 0] (total 1).
    Ranking 1, 2, 3, 4, 0, 5, 6, 7 with running mass after each block 0.4, 0.7,
    0.9, 0.9895, 0.9995, 1, 1, 1.  p = 0.99 is first reached after block 0,
    so the top-p set is {1, 2, 3, 4, 0}; with the exempt blocks the kept set is
    {0, 1, 2, 3, 4, 7}.  Boundary blocks (band 1e-3 around p): block 4 (ends at
    0.9895) and block 0 (starts there)."""
    b = np.array([0.01, 0.40, 0.30, 0.20, 0.0895, 0.0005, 0.0, 0.0])
    scores = np.repeat(b, G)
    cu = [0, len(scores)]
    ref = oracle.select(scores, cu, G, 0.99, 4, 4)
    assert ref["block_keep"][0].tolist() == [True, True, True, True, True, False, False, True]
    return scores, cu, ref


def _mask_of_blocks(keep):
    return np.repeat(np.asarray(keep, dtype=bool), G)


def test_mask_identical_to_the_oracle_is_accepted():
    scores, cu, ref = _fixture_mask_case()
    assert C.mask_mismatches(ref["mask"], ref, cu, G, 0.99, 4, 4) == []


def test_mask_flip_of_a_boundary_block_is_excused():
    scores, cu, ref = _fixture_mask_case()
    keep = ref["block_keep"][0].copy()
    keep[4] = False
    assert C.mask_mismatches(_mask_of_blocks(keep), ref, cu, G, 0.99, 4, 4) == []


def test_mask_flip_of_an_interior_block_is_reported():
    scores, cu, ref = _fixture_mask_case()
    for i in (2, 5, 6):
        keep = ref["block_keep"][0].copy()
        keep[i] = not keep[i]
        bad = C.mask_mismatches(_mask_of_blocks(keep), ref, cu, G, 0.99, 4, 4)
        assert [(r, j) for r, j, _ in bad] == [(0, i)], i


def test_mask_dropped_exempt_block_is_reported_even_on_the_boundary():
    scores, cu, ref = _fixture_mask_case()
    for i in (0, 7):                      # block 0 is also a boundary block
        keep = ref["block_keep"][0].copy()
        keep[i] = False
        bad = C.mask_mismatches(_mask_of_blocks(keep), ref, cu, G, 0.99, 4, 4)
        assert bad == [(0, i, "exempt block dropped")], i


def test_mask_half_kept_block_is_reported():
    scores, cu, ref = _fixture_mask_case()
    mask = ref["mask"].copy()
    mask[3 * G + 2:4 * G] = False         # block 3: tokens 12, 13 kept, 14, 15 dropped
    assert C.mask_mismatches(mask, ref, cu, G, 0.99, 4, 4) == [(0, 3, "partial block")]
    mask = ref["mask"].copy()
    mask[5 * G + 1] = True                # block 5: one stray kept token
    assert C.mask_mismatches(mask, ref, cu, G, 0.99, 4, 4) == [(0, 5, "partial block")]


def test_mask_drop_of_a_block_5e_3_from_p_is_reported():
    """b = [0.5, 0.485, 0.01, 0.005]: block 2 runs from 0.985 to 0.995, so it
    is needed to reach 0.99 and lies outside the band either way."""
    b = np.array([0.5, 0.485, 0.01, 0.005])
    scores = np.repeat(b, G)
    cu = [0, len(scores)]
    ref = oracle.select(scores, cu, G, 0.99, 0, 0)
    assert ref["block_keep"][0].tolist() == [True, True, True, False]
    keep = [True, True, False, False]
    assert C.mask_mismatches(_mask_of_blocks(keep), ref, cu, G, 0.99, 0, 0) == [(0, 2, "kept=False oracle=True")]


def test_mask_rules_apply_per_request():
    """Two requests packed back to back; a flip in the second is reported at its own block index."""
    scores1, _, _ = _fixture_mask_case()
    scores = np.concatenate([scores1, scores1])
    cu = [0, len(scores1), 2 * len(scores1)]
    ref = oracle.select(scores, cu, G, 0.99, 4, 4)
    mask = ref["mask"].copy()
    mask[len(scores1) + 2 * G:len(scores1) + 3 * G] = False
    assert [(r, i) for r, i, _ in C.mask_mismatches(mask, ref, cu, G, 0.99, 4, 4)] == [(1, 2)]


# ------------------------------------------------- self-consistency ----

def test_self_consistency_accepts_the_rule_on_the_candidates_own_scores():
    b = np.array([0.01, 0.40, 0.30, 0.20, 0.0895, 0.0005, 0.0, 0.0])
    keep = oracle.top_p_blocks(b, 0.99) | oracle.exempt_blocks(8 * G, G, 4, 4)
    assert C.self_consistency_mismatches(_mask_of_blocks(keep), b, [0, 8 * G], G, 0.99, 4, 4) == []


def test_self_consistency_rejects_a_mask_that_is_not_the_rule():
    b = np.array([0.01, 0.40, 0.30, 0.20, 0.0895, 0.0005, 0.0, 0.0])
    keep = oracle.top_p_blocks(b, 0.99) | oracle.exempt_blocks(8 * G, G, 4, 4)
    keep[4] = False                      # a boundary block for the oracle comparison, but not ambiguous here
    bad = C.self_consistency_mismatches(_mask_of_blocks(keep), b, [0, 8 * G], G, 0.99, 4, 4)
    assert bad == [(0, 4, "kept=False rule=True")]


def test_self_consistency_enforces_the_tie_rule_away_from_the_target():
    """b = [0.3, 0.3, 0.3, 0.1], p = 0.5: the rule keeps blocks 0 and 1 (ties
    by lower index); keeping 0 and 2 instead is reported."""
    b = np.array([0.3, 0.3, 0.3, 0.1])
    bad = C.self_consistency_mismatches(_mask_of_blocks([True, False, True, False]), b, [0, 4 * G], G, 0.5, 0, 0)
    assert sorted(i for _, i, _ in bad) == [1, 2]


def test_self_consistency_excuses_only_the_1e_9_band():
    """b = [0.25] * 4, p = 0.5: the running sum meets the target exactly after
    block 1, so blocks 1 and 2 are ambiguous and either choice passes; block
    0 is not."""
    b = np.full(4, 0.25)
    cu = [0, 4 * G]
    assert C.self_consistency_mismatches(_mask_of_blocks([True, False, True, False]), b, cu, G, 0.5, 0, 0) == []
    bad = C.self_consistency_mismatches(_mask_of_blocks([False, True, True, False]), b, cu, G, 0.5, 0, 0)
    assert [i for _, i, _ in bad] == [0]
    # a target 1e-6 above 0.5 leaves nothing ambiguous: the rule now needs
    # blocks 0, 1 and 2, so dropping block 1 is reported
    bad = C.self_consistency_mismatches(_mask_of_blocks([True, False, True, False]), b, cu, G, 0.5 + 1e-6, 0, 0)
    assert [i for _, i, _ in bad] == [1]


def test_self_consistency_checks_exempt_blocks():
    b = np.array([0.0, 0.5, 0.5, 0.0])
    keep = [False, True, True, True]     # block 0 is exempt (sink = 4) and was dropped
    bad = C.self_consistency_mismatches(_mask_of_blocks(keep), b, [0, 4 * G], G, 0.99, 4, 4)
    assert [i for _, i, _ in bad] == [0]


# ----------------------------------------- end to end on a tiny workload ----

def test_perturbed_oracle_output_is_accepted_and_a_shifted_one_is_not():
    """Scores within 5e-4 relative noise of the oracle's, with the mask taken by
    the rule on the candidate's own block means, pass every check; a copy whose
    scores are shifted by one token does not."""
    from sparse_long_context_tail_gb300 import workload as wl
    spec = wl.WorkloadSpec("tiny", [700, 333], 4, 2, 64, 64, n_tail=32, block=16, planted=[3, 1],
                           strength_range=(1.0, 4.0), seed=21)
    w = wl.generate(spec)
    cu = w.cu_seqlens
    ref_s = oracle.token_scores(w.k_bits, w.q_tail_bits, cu, 4, 2, 64, 32)
    ref = oracle.select(ref_s, cu, 16, 0.99, 128, 128)
    rng = np.random.default_rng(5)
    cand = ref_s * (1.0 + 5e-4 * rng.uniform(-1, 1, ref_s.shape))
    assert C.score_violations(cand, ref_s, cu)["ok"]
    mine = oracle.select(cand, cu, 16, 0.99, 128, 128)
    bs = np.concatenate(mine["block_scores"])
    assert C.mask_mismatches(mine["mask"], ref, cu, 16, 0.99, 128, 128) == []
    assert C.self_consistency_mismatches(mine["mask"], bs, cu, 16, 0.99, 128, 128) == []
    shifted = np.roll(ref_s, 1)
    assert not C.score_violations(shifted, ref_s, cu)["ok"]
