"""Torch-tensor front end of libupf: output allocation and pointer passing only.

``TokenSelector.select_tokens`` is the call a layer makes at a full-attention
layer: it runs the whole per-layer path of UniPrefill (article section 二,
steps 1-3; section 三) through ``upf_select_tokens`` on the current CUDA stream
and returns the keep mask, the compacted tensors and the batch metadata of the
kept tokens.  Tensors must already live on the selector's GPU.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

from . import _binding as B


@dataclasses.dataclass
class SelectOutputs:
    scores: torch.Tensor          # float32 [T]
    block_scores: torch.Tensor    # float32 [sum_r ceil(L_r/G)]
    keep_bits: torch.Tensor       # int32 [ceil(T/32)] (uint32 bit patterns)
    kept_count: torch.Tensor      # int32 [R]
    cu_seqlens_out: torch.Tensor  # int32 [R+1]
    total_kept: torch.Tensor      # int32 [1]
    kept_index: torch.Tensor      # int32 [T]
    hidden_out: Optional[torch.Tensor] = None
    pos_out: Optional[torch.Tensor] = None
    slot_out: Optional[torch.Tensor] = None


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


class TokenSelector:
    """Owns one libupf context on one GPU and a reusable workspace."""

    def __init__(self, device: int = 0):
        self.device = torch.device("cuda", device)
        self.ctx = B.upf_create(device)
        self._ws = None

    def close(self) -> None:
        if self.ctx:
            torch.cuda.synchronize(self.device)
            B.upf_destroy(self.ctx)
            self.ctx = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------------
    def workspace(self, nbytes: int) -> torch.Tensor:
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def status(self) -> int:
        """Device status word of the context (0 = OK); waits for the current stream."""
        return B.upf_sync_status(self.ctx, torch.cuda.current_stream(self.device).cuda_stream)

    @staticmethod
    def num_blocks(cu_seqlens_host: np.ndarray, block: int) -> int:
        L = np.diff(np.asarray(cu_seqlens_host, dtype=np.int64))
        return int(sum(-(-int(x) // block) for x in L))

    def alloc_outputs(self, cu_seqlens_host: np.ndarray, block: int, hidden: Optional[torch.Tensor] = None,
                      positions: Optional[torch.Tensor] = None, slots: Optional[torch.Tensor] = None) -> SelectOutputs:
        T = int(cu_seqlens_host[-1])
        R = len(cu_seqlens_host) - 1
        dev = self.device
        return SelectOutputs(
            scores=torch.empty(T, dtype=torch.float32, device=dev),
            block_scores=torch.empty(max(1, self.num_blocks(cu_seqlens_host, block)), dtype=torch.float32, device=dev),
            keep_bits=torch.empty(max(1, math.ceil(T / 32)), dtype=torch.int32, device=dev),
            kept_count=torch.empty(R, dtype=torch.int32, device=dev),
            cu_seqlens_out=torch.empty(R + 1, dtype=torch.int32, device=dev),
            total_kept=torch.empty(1, dtype=torch.int32, device=dev),
            kept_index=torch.empty(max(1, T), dtype=torch.int32, device=dev),
            hidden_out=None if hidden is None else torch.empty_like(hidden),
            pos_out=None if positions is None else torch.empty_like(positions),
            slot_out=None if slots is None else torch.empty_like(slots),
        )

    def select_tokens(self, q: torch.Tensor, k: torch.Tensor, cu_seqlens_host: np.ndarray,
                      cu_seqlens_dev: torch.Tensor, num_q_heads: int, num_kv_heads: int, head_dim: int,
                      hidden: Optional[torch.Tensor] = None, positions: Optional[torch.Tensor] = None,
                      slots: Optional[torch.Tensor] = None, layer_id: int = 0,
                      history: Optional[torch.Tensor] = None, history_len: Optional[torch.Tensor] = None,
                      params: Optional[B.UpfParams] = None, kv_of_q: Optional[Sequence[int]] = None,
                      out: Optional[SelectOutputs] = None) -> SelectOutputs:
        """q: bf16 [T, H_q, d] (rows may be strided), k: bf16 [T, H_kv, d]; hidden: [T, hidden]."""
        params = params or B.make_params()
        batch, keep = B.make_batch(cu_seqlens_dev.data_ptr(), cu_seqlens_host, num_q_heads, num_kv_heads,
                                   head_dim, kv_of_q)
        nbytes = B.upf_workspace_bytes(batch, params)
        ws = self.workspace(nbytes)
        if out is None:
            out = self.alloc_outputs(cu_seqlens_host, params.block, hidden, positions, slots)
        io = B.make_compact_io(
            row_bytes=0 if hidden is None else hidden.stride(0) * hidden.element_size(),
            hidden_in=_ptr(hidden), hidden_out=_ptr(out.hidden_out), pos_in=_ptr(positions),
            pos_out=_ptr(out.pos_out), slot_in=_ptr(slots), slot_out=_ptr(out.slot_out),
            kept_index=_ptr(out.kept_index), cu_seqlens_out=_ptr(out.cu_seqlens_out),
            total_kept=_ptr(out.total_kept), layer_id=layer_id,
            history_cap=0 if history is None else history.shape[1], history=_ptr(history),
            history_len=_ptr(history_len))
        stream = torch.cuda.current_stream(self.device).cuda_stream
        B.upf_select_tokens(self.ctx, batch, params, q.data_ptr(), q.stride(0), k.data_ptr(), k.stride(0),
                            _ptr(out.scores), _ptr(out.block_scores), _ptr(out.keep_bits), _ptr(out.kept_count),
                            io, ws.data_ptr(), ws.numel(), stream)
        del keep
        return out

    def score(self, q: torch.Tensor, k: torch.Tensor, cu_seqlens_host: np.ndarray, cu_seqlens_dev: torch.Tensor,
              num_q_heads: int, num_kv_heads: int, head_dim: int, params: Optional[B.UpfParams] = None,
              kv_of_q: Optional[Sequence[int]] = None, scores: Optional[torch.Tensor] = None,
              total_q_heads: Optional[int] = None) -> torch.Tensor:
        """Token importances alone (``upf_score``): float32 [T] on the selector's GPU.

        q and k may be views of a wider tensor (a head range of every row): the
        row strides are passed through.  With ``total_q_heads`` (a tensor-
        parallel rank's share of the heads) the scores are normalised by that
        many q heads (``upf_score_shard``), so the ranks' scores sum to the
        all-heads score."""
        params = params or B.make_params()
        batch, keep = B.make_batch(cu_seqlens_dev.data_ptr(), cu_seqlens_host, num_q_heads, num_kv_heads,
                                   head_dim, kv_of_q)
        nbytes = B.upf_workspace_bytes(batch, params)
        ws = self.workspace(nbytes)
        T = int(cu_seqlens_host[-1])
        if scores is None:
            scores = torch.empty(T, dtype=torch.float32, device=self.device)
        stream = torch.cuda.current_stream(self.device).cuda_stream
        if total_q_heads is None:
            B.upf_score(self.ctx, batch, params, q.data_ptr(), q.stride(0), k.data_ptr(), k.stride(0),
                        scores.data_ptr(), ws.data_ptr(), ws.numel(), stream)
        else:
            B.upf_score_shard(self.ctx, batch, params, int(total_q_heads), q.data_ptr(), q.stride(0), k.data_ptr(),
                              k.stride(0), scores.data_ptr(), ws.data_ptr(), ws.numel(), stream)
        del keep
        return scores

    def select_compact(self, scores: torch.Tensor, cu_seqlens_host: np.ndarray, cu_seqlens_dev: torch.Tensor,
                       hidden: Optional[torch.Tensor] = None, positions: Optional[torch.Tensor] = None,
                       slots: Optional[torch.Tensor] = None, layer_id: int = 0,
                       history: Optional[torch.Tensor] = None, history_len: Optional[torch.Tensor] = None,
                       params: Optional[B.UpfParams] = None, out: Optional[SelectOutputs] = None) -> SelectOutputs:
        """``upf_select`` then ``upf_compact`` on given token scores (e.g. scores
        summed over tensor-parallel ranks); ``out.scores`` is set to ``scores``."""
        params = params or B.make_params()
        # selection and compaction read only the request layout from the batch
        batch, keep = B.make_batch(cu_seqlens_dev.data_ptr(), cu_seqlens_host, 1, 1, 64)
        nbytes = B.upf_workspace_bytes(batch, params)
        ws = self.workspace(nbytes)
        if out is None:
            out = self.alloc_outputs(cu_seqlens_host, params.block, hidden, positions, slots)
        out.scores = scores
        stream = torch.cuda.current_stream(self.device).cuda_stream
        B.upf_select(self.ctx, batch, params, scores.data_ptr(), _ptr(out.block_scores), _ptr(out.keep_bits),
                     _ptr(out.kept_count), ws.data_ptr(), ws.numel(), stream)
        io = B.make_compact_io(
            row_bytes=0 if hidden is None else hidden.stride(0) * hidden.element_size(),
            hidden_in=_ptr(hidden), hidden_out=_ptr(out.hidden_out), pos_in=_ptr(positions),
            pos_out=_ptr(out.pos_out), slot_in=_ptr(slots), slot_out=_ptr(out.slot_out),
            kept_index=_ptr(out.kept_index), cu_seqlens_out=_ptr(out.cu_seqlens_out),
            total_kept=_ptr(out.total_kept), layer_id=layer_id,
            history_cap=0 if history is None else history.shape[1], history=_ptr(history),
            history_len=_ptr(history_len))
        B.upf_compact(self.ctx, batch, out.keep_bits.data_ptr(), io, ws.data_ptr(), ws.numel(), stream)
        del keep
        return out
