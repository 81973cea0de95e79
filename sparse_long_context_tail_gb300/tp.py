"""Tensor-parallel token selection: heads sharded over ranks, one score exchange.

UniPrefill article, section 三 (multi-GPU): under tensor parallelism every GPU
holds a slice of the attention heads, computes the importance scores of its
own heads, and the per-GPU scores are summed before the keep decision, so all
GPUs take the same decision and drop the same tokens.

Here rank r of P owns the contiguous kv heads [r H_kv/P, (r+1) H_kv/P) and the
q heads that read them.  ``upf_score_shard`` on the local heads, normalised by
the total head count H_q, gives s^(r)_k = 1/(H_q n_eff) sum_{h of r} ..., so
the global score (the average over all H_q heads) is the plain sum of the P
rank scores.  One sum all-reduce of the fp32 [T] scores is the only exchange
and the only arithmetic outside the library's kernels is that sum; every rank
then runs the same selection and compaction on its own copy of the hidden
rows.  The all-reduce leaves the same bits on every rank, so the masks agree.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np
import torch

from . import _binding as B
from .selector import SelectOutputs, TokenSelector


def shard_heads(num_q_heads: int, num_kv_heads: int, rank: int, world: int) -> Tuple[slice, slice]:
    """(q heads, kv heads) of `rank` for contiguous GQA groups (q head h reads
    kv head h // (H_q / H_kv)).  H_kv must divide evenly over the ranks."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if num_kv_heads % world or num_q_heads % num_kv_heads:
        raise ValueError(f"{num_q_heads} q heads / {num_kv_heads} kv heads do not shard over {world} ranks")
    kv = num_kv_heads // world
    q = num_q_heads // world
    return slice(rank * q, (rank + 1) * q), slice(rank * kv, (rank + 1) * kv)


def sum_of_partials(partials: Sequence[torch.Tensor]) -> torch.Tensor:
    """Global scores from the P ranks' shard scores, summed in rank order."""
    total = partials[0].clone()
    for p in partials[1:]:
        total += p
    return total


def _group_size(group=None) -> int:
    """Ranks in `group`; 1 when no process group is running (a single GPU)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return 1
    return dist.get_world_size(group)


def allreduce_scores(local: torch.Tensor, group=None) -> torch.Tensor:
    """In place: the sum over the group's ranks of their shard scores."""
    import torch.distributed as dist
    if _group_size(group) > 1:
        dist.all_reduce(local, op=dist.ReduceOp.SUM, group=group)
    return local


def tp_select_tokens(sel: TokenSelector, q_local: torch.Tensor, k_local: torch.Tensor,
                     cu_seqlens_host: np.ndarray, cu_seqlens_dev: torch.Tensor, local_q_heads: int,
                     local_kv_heads: int, head_dim: int, hidden: Optional[torch.Tensor] = None,
                     positions: Optional[torch.Tensor] = None, slots: Optional[torch.Tensor] = None,
                     layer_id: int = 0, history: Optional[torch.Tensor] = None,
                     history_len: Optional[torch.Tensor] = None, params: Optional[B.UpfParams] = None,
                     group=None, out: Optional[SelectOutputs] = None) -> SelectOutputs:
    """One full-attention layer's selection on this rank's heads.

    q_local / k_local: this rank's head slices ([T, H_q/P, d] / [T, H_kv/P, d],
    views with the full row strides are fine).  Scores the local heads
    normalised by all H_q = P * local_q_heads heads, sums the scores over the
    ranks of `group` (one all-reduce), then selects and compacts exactly as the
    single-GPU call does.  Shapes are checked before the exchange: a rank given
    the wrong slice raises without entering it, and the other ranks' exchange
    then fails on the process group's timeout."""
    for name, t, heads in (("q_local", q_local, local_q_heads), ("k_local", k_local, local_kv_heads)):
        if t.dim() != 3 or t.shape[1] != heads or t.shape[2] != head_dim:
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected [T, {heads}, {head_dim}]")
    if q_local.shape[0] != k_local.shape[0] or q_local.shape[0] != int(cu_seqlens_host[-1]):
        raise ValueError("q_local, k_local and cu_seqlens disagree on the token count")
    world = _group_size(group)
    scores = sel.score(q_local, k_local, cu_seqlens_host, cu_seqlens_dev, local_q_heads, local_kv_heads,
                       head_dim, params=params, total_q_heads=world * local_q_heads)
    allreduce_scores(scores, group)
    return sel.select_compact(scores, cu_seqlens_host, cu_seqlens_dev, hidden, positions, slots, layer_id,
                              history, history_len, params, out)
