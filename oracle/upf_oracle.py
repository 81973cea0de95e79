"""Float64 CPU oracle of UniPrefill's per-full-attention-layer token selection.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or runs
this module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg (``cpu_baseline`` and ``--impl reference``) may use it.  It shares
no code with the CUDA path; both sides receive the same bfloat16 bit patterns
from the seeded generator and nothing else.

Source.  The only description of the method is the article "中国科学院与腾讯微信
合作解决AI排队等待问题" (m.youleyou.com/wenzhang/2886770, a reprint of a 163.com
piece on UniPrefill, arXiv:2605.06221).  Citations below name its sections:

* [§2 step 1]  section 二, first step: the last n tokens (default 128) act as
  questioners, attend to every token, and give each token a preliminary
  importance score.
* [§2 step 2]  section 二, second step: cut the sequence into blocks of G tokens
  (default 64), average the token scores inside each block, sort blocks from
  most to least important and keep the smallest set whose importance sum just
  reaches 99% of the total; drop the rest.
* [§2 exempt]  section 二, paragraph after step 2: the first 128 tokens (anchors)
  and the last 128 tokens (the questioners) are never dropped.
* [§2 step 3]  section 二, third step: dropped tokens are skipped by every later
  layer until the next full-attention layer; their hidden states are frozen.
* [§3 kernels] section 三: scores, online normalisation, in-block aggregation and
  a binary mask, all on the GPU.
* [§3 history] section 三, last paragraph: each drop records the layer id and the
  number of kept tokens (the drop-history bill); positions and KV slot addresses
  of the batch are updated to match.

Readings where the article is silent (each one is listed in the design notes):
causal visibility (tail query j at position t_j sees keys 0..t_j); softmax scale
1/sqrt(d) unless given; the token score is the arithmetic mean of the normalised
attention probabilities over all q-heads and all n_eff = min(n, L) tail queries;
GQA groups are contiguous (q-head h reads kv-head floor(h / (H_q/H_kv))) unless a
map is given; blocks start at token 0 and the last block averages its valid
tokens only; "reaches p" means cumulative >= p * total, with the total taken as
the sum of all block means in sorted order; ties in block score rank the lower
block index first; the exempt blocks are OR-ed in after the top-p set is chosen
over all blocks, and a block is exempt when it overlaps the first ``sink_keep`` or
the last ``tail_keep`` tokens; compaction is out of place and order preserving.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# Inputs
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64, exactly (bf16 is the top half of float32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def tail_positions(L: int, n_tail: int) -> np.ndarray:
    """Positions (within the request) of the questioners: the last min(n, L) tokens [§2 step 1]."""
    n_eff = min(n_tail, L)
    return np.arange(L - n_eff, L, dtype=np.int64)


def kv_head_map(num_q_heads: int, num_kv_heads: int, kv_of_q: Optional[Sequence[int]] = None) -> np.ndarray:
    """q-head -> kv-head.  Contiguous groups unless an explicit map is given (a reading)."""
    if kv_of_q is not None:
        return np.asarray(kv_of_q, dtype=np.int64)
    gamma = num_q_heads // num_kv_heads
    return np.arange(num_q_heads, dtype=np.int64) // gamma


# ---------------------------------------------------------------------------
# [§2 step 1] + [§3 kernels]: tail-query importance of every token
# ---------------------------------------------------------------------------

def _head_contribution(Qt: np.ndarray, Kh: np.ndarray, tpos: np.ndarray, scale: float) -> np.ndarray:
    """Sum over tail queries of the causal softmax probabilities one head gives each key.

    Qt: [n_eff, d] tail queries of one q-head; Kh: [L, d] keys of its kv-head.
    Row j is the softmax over keys 0..tpos[j] of scale * (q_j . k); the
    normalisation is the plain max-subtracted softmax, which is what an online
    normalisation reaches exactly.
    """
    L = Kh.shape[0]
    logits = scale * (Qt @ Kh.T)                                   # [n_eff, L]
    visible = np.arange(L)[None, :] <= tpos[:, None]               # causal
    logits = np.where(visible, logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    P = e / e.sum(axis=1, keepdims=True)
    return P.sum(axis=0)                                           # [L]


def token_scores(k_bits: np.ndarray, q_tail_bits: np.ndarray, cu_seqlens: Sequence[int],
                 num_q_heads: int, num_kv_heads: int, head_dim: int, n_tail: int,
                 softmax_scale: Optional[float] = None, kv_of_q: Optional[Sequence[int]] = None,
                 threads: Optional[int] = None) -> np.ndarray:
    """Per-token importance s_k of every packed token, float64 [T].

    s_k = (1 / (H_q * n_eff)) * sum over q-heads h and tail queries j with
    t_j >= k of softmax_j(k), per request.

    k_bits: uint16 [T, H_kv, d]; q_tail_bits: uint16 [sum_r n_eff_r, H_q, d], the
    tail query rows of each request in request order.
    """
    cu = [int(x) for x in cu_seqlens]
    R = len(cu) - 1
    T = cu[-1]
    scale = 1.0 / math.sqrt(head_dim) if softmax_scale is None else float(softmax_scale)
    g_of = kv_head_map(num_q_heads, num_kv_heads, kv_of_q)
    K = bf16_to_f64(k_bits).reshape(T, num_kv_heads, head_dim)
    Q = bf16_to_f64(q_tail_bits).reshape(-1, num_q_heads, head_dim)
    scores = np.zeros(T, dtype=np.float64)
    jobs = []
    q_off = 0
    for r in range(R):
        L = cu[r + 1] - cu[r]
        tpos = tail_positions(L, n_tail)
        n_eff = len(tpos)
        for h in range(num_q_heads):
            jobs.append((r, h, q_off, n_eff, tpos))
        q_off += n_eff

    def run(job):
        r, h, qo, n_eff, tpos = job
        if n_eff == 0:
            return np.zeros(0)
        Kh = K[cu[r]:cu[r + 1], g_of[h], :]
        Qt = Q[qo:qo + n_eff, h, :]
        return _head_contribution(Qt, Kh, tpos, scale)

    workers = threads if threads is not None else min(32, os.cpu_count() or 1)
    if workers > 1 and len(jobs) > 1:
        with ThreadPoolExecutor(max_workers=workers) as ex:
            parts = list(ex.map(run, jobs))
    else:
        parts = [run(j) for j in jobs]
    # Sum per request in head order, then take the mean over (h, j).
    for (r, h, qo, n_eff, tpos), part in zip(jobs, parts):
        if n_eff:
            scores[cu[r]:cu[r + 1]] += part
    for r in range(R):
        L = cu[r + 1] - cu[r]
        n_eff = min(n_tail, L)
        if n_eff:
            scores[cu[r]:cu[r + 1]] /= (num_q_heads * n_eff)
    return scores


# ---------------------------------------------------------------------------
# [§2 step 2]: block means
# ---------------------------------------------------------------------------

def block_means(scores_r: np.ndarray, block: int) -> np.ndarray:
    """Mean token score of each block of G tokens of one request (last block: its valid tokens)."""
    L = len(scores_r)
    nb = -(-L // block)
    return np.array([scores_r[i * block:min(L, (i + 1) * block)].mean() for i in range(nb)], dtype=np.float64)


# ---------------------------------------------------------------------------
# [§2 step 2]: smallest block set reaching p of the total importance
# ---------------------------------------------------------------------------

def top_p_blocks(b: np.ndarray, top_p: float) -> np.ndarray:
    """bool [nb]: the top-p block set S of one request.

    Blocks are ranked by score, highest first (equal scores: lower index first).
    S is the shortest prefix of that ranking whose running sum reaches
    top_p * total, where total is the running sum over all blocks.  The empty
    prefix (sum 0) counts, so a zero total selects nothing.
    """
    nb = len(b)
    order = sorted(range(nb), key=lambda i: (-b[i], i))
    cum = np.zeros(nb + 1, dtype=np.float64)
    for pos, i in enumerate(order):
        cum[pos + 1] = cum[pos] + b[i]
    target = top_p * cum[nb]
    k = nb
    for pos in range(nb + 1):
        if cum[pos] >= target:
            k = pos
            break
    keep = np.zeros(nb, dtype=bool)
    keep[order[:k]] = True
    return keep


# ---------------------------------------------------------------------------
# [§2 exempt]: sink and tail blocks
# ---------------------------------------------------------------------------

def exempt_blocks(L: int, block: int, sink_keep: int, tail_keep: int) -> np.ndarray:
    """bool [nb]: blocks overlapping the first sink_keep or the last tail_keep tokens."""
    nb = -(-L // block)
    out = np.zeros(nb, dtype=bool)
    for i in range(nb):
        lo, hi = i * block, min(L, (i + 1) * block)
        if lo < min(sink_keep, L):
            out[i] = True
        if hi > max(0, L - tail_keep):
            out[i] = True
    return out


# ---------------------------------------------------------------------------
# [§2 step 2] + [§2 exempt] + [§3 kernels]: the binary keep mask
# ---------------------------------------------------------------------------

def select(scores: np.ndarray, cu_seqlens: Sequence[int], block: int, top_p: float,
           sink_keep: int, tail_keep: int, block_scores: Optional[List[np.ndarray]] = None) -> Dict:
    """Keep mask of every packed token, per-request kept counts and the block scores.

    If ``block_scores`` is given (one float array per request) the selection runs
    on those values instead of the block means of ``scores``.
    """
    cu = [int(x) for x in cu_seqlens]
    R = len(cu) - 1
    T = cu[-1]
    mask = np.zeros(T, dtype=bool)
    kept_count = np.zeros(R, dtype=np.int64)
    all_b, all_s, all_keep = [], [], []
    for r in range(R):
        L = cu[r + 1] - cu[r]
        b = (np.asarray(block_scores[r], dtype=np.float64) if block_scores is not None
             else block_means(scores[cu[r]:cu[r + 1]], block))
        S = top_p_blocks(b, top_p)
        keep = S | exempt_blocks(L, block, sink_keep, tail_keep)
        tok = np.repeat(keep, block)[:L]
        mask[cu[r]:cu[r + 1]] = tok
        kept_count[r] = int(tok.sum())
        all_b.append(b)
        all_s.append(S)
        all_keep.append(keep)
    return dict(mask=mask, kept_count=kept_count, block_scores=all_b, top_p_set=all_s, block_keep=all_keep)


# ---------------------------------------------------------------------------
# [§2 step 3] + [§3 history]: compaction and the drop-history record
# ---------------------------------------------------------------------------

def compact(mask: np.ndarray, cu_seqlens: Sequence[int], hidden: Optional[np.ndarray] = None,
            positions: Optional[np.ndarray] = None, slots: Optional[np.ndarray] = None,
            layer_id: int = 0, history: Optional[np.ndarray] = None,
            history_len: Optional[np.ndarray] = None) -> Dict:
    """Gather the kept tokens in their original order; append one history record per request.

    history: int [R, cap, 2] and history_len: int [R] are updated in copies:
    record (layer_id, kept count of r) goes to history[r, history_len[r]] and the
    length grows by one.  A full history (history_len[r] == cap) is an error:
    nothing is written for any request and ``capacity_error`` is True.
    """
    cu = [int(x) for x in cu_seqlens]
    R = len(cu) - 1
    mask = np.asarray(mask, dtype=bool)
    kept_index = np.nonzero(mask)[0].astype(np.int64)
    counts = np.array([int(mask[cu[r]:cu[r + 1]].sum()) for r in range(R)], dtype=np.int64)
    cu_out = np.zeros(R + 1, dtype=np.int64)
    for r in range(R):
        cu_out[r + 1] = cu_out[r] + counts[r]
    out = dict(kept_index=kept_index, cu_seqlens_out=cu_out, total_kept=int(cu_out[-1]), kept_count=counts)
    if hidden is not None:
        out["hidden_out"] = hidden[kept_index]
    if positions is not None:
        out["positions_out"] = positions[kept_index]
    if slots is not None:
        out["slots_out"] = slots[kept_index]
    if history is not None:
        hist = np.array(history, copy=True)
        hlen = np.array(history_len, copy=True)
        cap = hist.shape[1]
        full = any(int(hlen[r]) >= cap for r in range(R))
        if not full:
            for r in range(R):
                hist[r, int(hlen[r]), 0] = layer_id
                hist[r, int(hlen[r]), 1] = counts[r]
                hlen[r] += 1
        out.update(history=hist, history_len=hlen, capacity_error=full)
    return out


def revive(full: np.ndarray, kept_index: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Write a compacted batch's rows back into the full-length buffer [§2 step 3].

    Dropped tokens keep their frozen hidden states; kept token kept_index[o]
    takes row o of the compacted batch.  Returns an updated copy of `full`.
    """
    out = np.array(full, copy=True)
    out[np.asarray(kept_index, dtype=np.int64)] = rows
    return out


def history_kv_len(history: np.ndarray, history_len: np.ndarray, cu_seqlens: Sequence[int], layer_id: int) -> np.ndarray:
    """KV entries each request's layer `layer_id` holds, read from the drop history [§3 history].

    A drop at full-attention layer l_i keeps c_i tokens; that layer and every
    later one up to the next drop process (and cache) only those tokens, so
    layer `layer_id` holds c_i of the latest record with l_i <= layer_id, and
    the prompt length L_r when no drop happened at or before it.  Records are
    in append order (non-decreasing layer ids).
    """
    cu = [int(x) for x in cu_seqlens]
    R = len(cu) - 1
    out = np.zeros(R, dtype=np.int64)
    for r in range(R):
        kv = cu[r + 1] - cu[r]
        for i in range(int(history_len[r])):
            if int(history[r][i][0]) <= layer_id:
                kv = int(history[r][i][1])
        out[r] = kv
    return out


def select_tokens(k_bits, q_tail_bits, cu_seqlens, num_q_heads, num_kv_heads, head_dim, n_tail=128,
                  block=64, top_p=0.99, sink_keep=128, tail_keep=128, softmax_scale=None, kv_of_q=None,
                  hidden=None, positions=None, slots=None, layer_id=0, history=None, history_len=None,
                  threads=None) -> Dict:
    """The whole path: scores, block means, top-p + exempt mask, compaction, history."""
    s = token_scores(k_bits, q_tail_bits, cu_seqlens, num_q_heads, num_kv_heads, head_dim, n_tail,
                     softmax_scale, kv_of_q, threads)
    sel = select(s, cu_seqlens, block, top_p, sink_keep, tail_keep)
    comp = compact(sel["mask"], cu_seqlens, hidden, positions, slots, layer_id, history, history_len)
    return dict(scores=s, **sel, **{k: v for k, v in comp.items() if k != "kept_count"})
