"""Seeded synthetic inputs for the token-selection path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no logits, softmax, pooling, selection or compaction).
Both the float64 oracle (via the tests and the bench's CPU leg) and the CUDA
path consume exactly the bit patterns produced here, so a parity test compares
the two on identical inputs.

Recipe (one request ``r`` of a workload with seed ``S``):

* ``numpy.random.Generator(PCG64(1000 * S + r))`` draws, in this order,
  K ``[L, H_kv, d]``, the tail query rows ``[n_eff, H_q, d]`` and one direction
  ``u[g]`` per kv head, all float32 N(0, 1).
* Planted structure: ``count`` distinct blocks of ``G`` tokens are drawn without
  replacement from the blocks that lie wholly between the first ``sink_keep``
  and the last ``tail_keep`` tokens; every key row of a planted block gets
  ``+ s_b * u[g]`` (``s_b`` fixed, or U[lo, hi] per block), the tail query rows
  of every q-head of group ``g`` get ``+ u[g]``, and optionally key 0 gets
  ``+ sink_boost * u[g]``.  With ``|u|^2 ~ d`` the logit boost of a planted key
  is about ``s_b * sqrt(d)``, so planted blocks carry most of the attention.
* Everything is rounded once to bfloat16 (round-to-nearest-even) and stored as
  uint16 bit patterns.
* Hidden states ``[T, hidden]`` are N(0, 1) bf16 from ``PCG64(1000 * S + 999)``;
  positions are ``0..L_r-1`` per request; slot ids are a random permutation of
  ``[0, T)`` from ``PCG64(1000 * S + 998)`` so that the gather is not an identity.

The named workloads mirror the shapes of the full-attention layers of
LLaMA-3.1-8B (32/8 heads, d=128, hidden 4096), Qwen3-Next-80B-A3B (16/2, d=256,
hidden 2048) and Gemma-3-12B (16/8, d=256, hidden 3840) that the UniPrefill
article evaluates (section 4, results), with random values in place of trained
activations.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits.

    Finite inputs only (the generator never produces NaN/Inf).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class WorkloadSpec:
    name: str
    lengths: Sequence[int]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    hidden: int
    n_tail: int = 128
    block: int = 64
    top_p: float = 0.99
    sink_keep: int = 128
    tail_keep: int = 128
    planted: Optional[Sequence[int]] = None   # planted block count per request
    strength: float = 3.0                     # fixed s_b, used when strength_range is None
    strength_range: Optional[tuple] = None    # (lo, hi): s_b ~ U[lo, hi] per block
    sink_boost: float = 0.0                   # + sink_boost * u on key 0 of every request
    seed: int = 0
    kv_of_q: Optional[Sequence[int]] = None   # q-head -> kv-head; None = contiguous groups

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def group_map(self) -> np.ndarray:
        if self.kv_of_q is not None:
            return np.asarray(self.kv_of_q, dtype=np.int32)
        gamma = self.num_q_heads // self.num_kv_heads
        return (np.arange(self.num_q_heads) // gamma).astype(np.int32)


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    cu_seqlens: np.ndarray        # int32 [R+1]
    k_bits: np.ndarray            # uint16 [T, H_kv, d]
    q_tail_bits: np.ndarray       # uint16 [sum n_eff, H_q, d]  (tail rows, request order)
    tail_rows: np.ndarray         # int64 [sum n_eff]: packed token index of each tail row
    planted_blocks: List[np.ndarray]  # per request: planted block indices
    _hidden: Optional[np.ndarray] = None
    _positions: Optional[np.ndarray] = None
    _slots: Optional[np.ndarray] = None

    @property
    def num_reqs(self) -> int:
        return len(self.spec.lengths)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    def hidden_bits(self) -> np.ndarray:
        """uint16 [T, hidden] bf16 N(0, 1) hidden states (generated on first use)."""
        if self._hidden is None:
            T, H = self.total_tokens, self.spec.hidden
            rng = np.random.Generator(np.random.PCG64(1000 * self.spec.seed + 999))
            out = np.empty((T, H), dtype=np.uint16)
            step = max(1, (1 << 24) // H)
            for s in range(0, T, step):
                e = min(T, s + step)
                out[s:e] = f32_to_bf16_bits(rng.standard_normal((e - s, H), dtype=np.float32))
            self._hidden = out
        return self._hidden

    def positions(self) -> np.ndarray:
        if self._positions is None:
            self._positions = np.concatenate(
                [np.arange(L, dtype=np.int64) for L in self.spec.lengths]) if self.num_reqs else np.zeros(0, np.int64)
        return self._positions

    def slots(self) -> np.ndarray:
        if self._slots is None:
            rng = np.random.Generator(np.random.PCG64(1000 * self.spec.seed + 998))
            self._slots = rng.permutation(self.total_tokens).astype(np.int64)
        return self._slots

    def q_full_bits(self) -> np.ndarray:
        """uint16 [T, H_q, d] with the tail rows filled and every other row zero.

        Only tail rows are read by the method; this layout is for callers that
        want the packed [T, H_q, d] query tensor a real layer would hold.
        """
        s = self.spec
        q = np.zeros((self.total_tokens, s.num_q_heads, s.head_dim), dtype=np.uint16)
        q[self.tail_rows] = self.q_tail_bits
        return q


def _eligible_blocks(L: int, G: int, sink: int, tail: int) -> np.ndarray:
    """Blocks lying wholly inside [sink, L - tail): where planting is allowed."""
    nb = -(-L // G)
    i = np.arange(nb)
    ok = (i * G >= sink) & ((i + 1) * G <= L - tail)
    return i[ok]


def generate(spec: WorkloadSpec) -> Workload:
    R = len(spec.lengths)
    H_q, H_kv, d = spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    if H_q % H_kv != 0:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    gmap = spec.group_map()
    lengths = [int(L) for L in spec.lengths]
    cu = np.zeros(R + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    k_bits = np.empty((T, H_kv, d), dtype=np.uint16)
    q_tail, tail_rows, planted_all = [], [], []
    for r, L in enumerate(lengths):
        rng = np.random.Generator(np.random.PCG64(1000 * spec.seed + r))
        n_eff = min(spec.n_tail, L)
        K = rng.standard_normal((L, H_kv, d), dtype=np.float32)
        Qt = rng.standard_normal((n_eff, H_q, d), dtype=np.float32)
        u = rng.standard_normal((H_kv, d), dtype=np.float32)
        count = 0 if spec.planted is None else int(spec.planted[r])
        elig = _eligible_blocks(L, spec.block, spec.sink_keep, spec.tail_keep)
        count = min(count, len(elig))
        blocks = np.sort(rng.choice(elig, size=count, replace=False)) if count > 0 else np.zeros(0, np.int64)
        if spec.strength_range is not None:
            strengths = rng.uniform(spec.strength_range[0], spec.strength_range[1], size=count).astype(np.float32)
        else:
            strengths = np.full(count, spec.strength, dtype=np.float32)
        if count > 0:
            for b, s_b in zip(blocks, strengths):
                lo, hi = int(b) * spec.block, min(L, (int(b) + 1) * spec.block)
                K[lo:hi] += s_b * u[None, :, :]
            Qt += u[gmap][None, :, :]
        if spec.sink_boost:
            K[0] += np.float32(spec.sink_boost) * u
            if count == 0:
                Qt += u[gmap][None, :, :]
        k_bits[cu[r]:cu[r + 1]] = f32_to_bf16_bits(K)
        q_tail.append(f32_to_bf16_bits(Qt))
        tail_rows.append(np.arange(cu[r] + L - n_eff, cu[r] + L, dtype=np.int64))
        planted_all.append(blocks.astype(np.int64))
    q_tail_bits = np.concatenate(q_tail, axis=0) if q_tail else np.zeros((0, H_q, d), np.uint16)
    tails = np.concatenate(tail_rows) if tail_rows else np.zeros(0, np.int64)
    return Workload(spec=spec, cu_seqlens=cu, k_bits=k_bits, q_tail_bits=q_tail_bits,
                    tail_rows=tails, planted_blocks=planted_all)


# ---------------------------------------------------------------------------
# Named workloads.  Shapes: the full-attention layers of the models the
# UniPrefill article evaluates; defaults n=128, G=64, p=0.99 and 128 sink/tail
# tokens from its section 2 (algorithm) and section 5 (hyper-parameters).
# ---------------------------------------------------------------------------

LLAMA = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, hidden=4096)
QWEN3_NEXT = dict(num_q_heads=16, num_kv_heads=2, head_dim=256, hidden=2048)
GEMMA3 = dict(num_q_heads=16, num_kv_heads=8, head_dim=256, hidden=3840)


def _varlen_lengths(seed: int, count: int, lo: int, hi: int) -> List[int]:
    rng = np.random.Generator(np.random.PCG64(1000 * seed + 997))
    return [int(round(math.exp(x))) for x in rng.uniform(math.log(lo), math.log(hi), size=count)]


def named_spec(name: str) -> WorkloadSpec:
    """The benchmark workloads by name.

    * ``small-L4096``: 1 x 4096, 8/2 heads, d=64, hidden 512, 4 planted blocks s=3.
    * ``llama8b-L32768``: LLaMA-3.1-8B layer shape, 1 x 32768, 16 planted s=3, sink +5u.
    * ``llama8b-L131072``: same shape, 1 x 131072, 64 planted, s ~ U[1, 4].
    * ``llama8b-batch16``: 16 requests, lengths log-uniform in [4096, 131072],
      max(1, round(64 L / 131072)) planted per request, s ~ U[1, 4].
    * ``qwen3next-G{G}-n{n}`` / ``gemma3-G{G}-n{n}``: 1 x 131072, 64 planted,
      s ~ U[1, 4], G in {32, 64, 128}, n in {32, 128, 512}.
    """
    if name == "small-L4096":
        return WorkloadSpec(name, [4096], 8, 2, 64, 512, planted=[4], strength=3.0, seed=1)
    if name == "llama8b-L32768":
        return WorkloadSpec(name, [32768], **LLAMA, planted=[16], strength=3.0, sink_boost=5.0, seed=2)
    if name == "llama8b-L131072":
        return WorkloadSpec(name, [131072], **LLAMA, planted=[64], strength_range=(1.0, 4.0), seed=3)
    if name == "llama8b-batch16":
        lengths = _varlen_lengths(4, 16, 4096, 131072)
        planted = [max(1, int(round(64 * L / 131072))) for L in lengths]
        return WorkloadSpec(name, lengths, **LLAMA, planted=planted, strength_range=(1.0, 4.0), seed=4)
    for prefix, shape, base in (("qwen3next", QWEN3_NEXT, 50), ("gemma3", GEMMA3, 60)):
        if name.startswith(prefix + "-G"):
            G, n = name[len(prefix) + 2:].split("-n")
            G, n = int(G), int(n)
            if G not in (32, 64, 128) or n not in (32, 128, 512):
                break
            point = (32, 64, 128).index(G) * 3 + (32, 128, 512).index(n)
            return WorkloadSpec(name, [131072], **shape, n_tail=n, block=G, planted=[64],
                                strength_range=(1.0, 4.0), seed=base + point)
    raise KeyError(f"unknown workload {name!r}")


SWEEP_NAMES = [f"{m}-G{G}-n{n}" for m in ("qwen3next", "gemma3") for G in (32, 64, 128) for n in (32, 128, 512)]
NAMED = ["small-L4096", "llama8b-L32768", "llama8b-L131072", "llama8b-batch16"] + SWEEP_NAMES


def scaled_spec(spec: WorkloadSpec, lengths: Sequence[int], name: Optional[str] = None,
                planted: Optional[Sequence[int]] = None) -> WorkloadSpec:
    """The same head shape and hyper-parameters at other request lengths (for tests)."""
    return dataclasses.replace(spec, name=name or f"{spec.name}-scaled", lengths=list(lengths),
                               planted=list(planted) if planted is not None else
                               [max(1, (spec.planted[0] if spec.planted else 0) * L // max(1, spec.lengths[0]))
                                for L in lengths])
