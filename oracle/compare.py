"""Acceptance rules for comparing a candidate implementation with the oracle.

TEST INFRASTRUCTURE ONLY (same restriction as ``upf_oracle``).

* Token scores: |s - s_ref| <= 1e-3 |s_ref| + 1e-6 / L_r per token (bf16 inputs
  with fp32 accumulation against float64; the absolute floor, 1e-6 of the mean
  score 1/L_r, covers scores that underflow in fp32), and the scores of each
  request sum to 1 within 1e-3.
* Keep mask: equal to the oracle's except on boundary blocks -- blocks whose
  normalised running mass in the oracle's ranking, before or after adding the
  block, lies within 1e-3 of p.  Exempt blocks must always be kept.
* Self-consistency: the candidate's mask must be exactly the oracle's top-p rule
  applied to the candidate's own block scores (float64 running sums), except
  where that rule's running sum is within 1e-9 of the target.
"""
from __future__ import annotations

from typing import Dict, List, Sequence

import numpy as np

from . import upf_oracle as O


def unpack_bits(words: np.ndarray, T: int) -> np.ndarray:
    w = np.asarray(words).view(np.uint32).reshape(-1)
    bits = ((w[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & np.uint32(1)).astype(bool)
    return bits.reshape(-1)[:T]


def pack_bits(mask: np.ndarray) -> np.ndarray:
    m = np.asarray(mask, dtype=bool)
    nw = max(1, -(-len(m) // 32))
    pad = np.zeros(nw * 32, dtype=np.uint32)
    pad[:len(m)] = m
    return (pad.reshape(nw, 32) << np.arange(32, dtype=np.uint32)[None, :]).sum(axis=1).astype(np.uint32)


def score_violations(s: np.ndarray, ref: np.ndarray, cu_seqlens: Sequence[int]) -> Dict:
    """Worst normalised violation of the score tolerance (<= 0 means within tolerance)."""
    cu = [int(x) for x in cu_seqlens]
    worst, worst_at, sum_err = -np.inf, -1, 0.0
    for r in range(len(cu) - 1):
        a, b = cu[r], cu[r + 1]
        if b == a:
            continue
        tol = 1e-3 * np.abs(ref[a:b]) + 1e-6 / (b - a)
        v = np.abs(s[a:b].astype(np.float64) - ref[a:b]) - tol
        i = int(np.argmax(v))
        if v[i] > worst:
            worst, worst_at = float(v[i]), a + i
        sum_err = max(sum_err, abs(float(s[a:b].astype(np.float64).sum()) - 1.0))
    return dict(worst=worst, at=worst_at, sum_err=sum_err, ok=(worst <= 0 and sum_err <= 1e-3))


def boundary_blocks(b: np.ndarray, top_p: float, tol: float = 1e-3) -> np.ndarray:
    nb = len(b)
    out = np.zeros(nb, dtype=bool)
    if nb == 0:
        return out
    order = sorted(range(nb), key=lambda i: (-b[i], i))
    cum = np.concatenate([[0.0], np.cumsum(np.asarray(b, dtype=np.float64)[order])])
    total = cum[-1]
    if total <= 0:
        return out
    c = cum / total
    for pos, i in enumerate(order):
        out[i] = abs(c[pos] - top_p) <= tol or abs(c[pos + 1] - top_p) <= tol
    return out


def mask_mismatches(mask: np.ndarray, ref_sel: Dict, cu_seqlens: Sequence[int], block: int, top_p: float,
                    sink_keep: int, tail_keep: int) -> List[tuple]:
    """Blocks where the candidate mask disagrees with the oracle outside the boundary tolerance."""
    cu = [int(x) for x in cu_seqlens]
    bad = []
    for r in range(len(cu) - 1):
        L = cu[r + 1] - cu[r]
        tok = mask[cu[r]:cu[r + 1]]
        keep_ref = ref_sel["block_keep"][r]
        nb = len(keep_ref)
        bnd = boundary_blocks(ref_sel["block_scores"][r], top_p)
        ex = O.exempt_blocks(L, block, sink_keep, tail_keep)
        for i in range(nb):
            seg = tok[i * block:min(L, (i + 1) * block)]
            if not (seg.all() or not seg.any()):
                bad.append((r, i, "partial block"))
                continue
            got = bool(seg[0]) if len(seg) else False
            if ex[i] and not got:
                bad.append((r, i, "exempt block dropped"))
            elif got != bool(keep_ref[i]) and not bnd[i]:
                bad.append((r, i, f"kept={got} oracle={bool(keep_ref[i])}"))
    return bad


def self_consistency_mismatches(mask: np.ndarray, block_scores: np.ndarray, cu_seqlens: Sequence[int], block: int,
                                top_p: float, sink_keep: int, tail_keep: int) -> List[tuple]:
    """Blocks where the mask is not the top-p rule applied to the candidate's own block scores."""
    cu = [int(x) for x in cu_seqlens]
    bad = []
    off = 0
    for r in range(len(cu) - 1):
        L = cu[r + 1] - cu[r]
        nb = -(-L // block)
        b = np.asarray(block_scores[off:off + nb], dtype=np.float64)
        off += nb
        S = O.top_p_blocks(b, top_p)
        keep = S | O.exempt_blocks(L, block, sink_keep, tail_keep)
        order = sorted(range(nb), key=lambda i: (-b[i], i))
        cum = np.concatenate([[0.0], np.cumsum(b[order])]) if nb else np.zeros(1)
        target = top_p * cum[-1]
        ambiguous = np.zeros(nb, dtype=bool)
        for pos, i in enumerate(order):
            ambiguous[i] = abs(cum[pos + 1] - target) <= 1e-9 * max(abs(cum[-1]), 1e-300) or \
                abs(cum[pos] - target) <= 1e-9 * max(abs(cum[-1]), 1e-300)
        tok = mask[cu[r]:cu[r + 1]]
        for i in range(nb):
            got = bool(tok[i * block])
            if got != bool(keep[i]) and not ambiguous[i]:
                bad.append((r, i, f"kept={got} rule={bool(keep[i])}"))
    return bad
