"""ctypes binding of libupf (include/upf.h): argument marshalling only.

Every function here has the name of the C entry point it calls and passes
plain integers (device pointers, sizes, the CUDA stream handle) through.  All
computation happens in libupf's CUDA kernels; if the library is missing or
cannot be loaded, every call raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p
from typing import Optional, Sequence

import numpy as np

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("UPF_LIBRARY", os.path.join(_PKG_DIR, "libupf.so"))

UPF_OK = 0
STATUS_NAMES = {0: "UPF_OK", 1: "UPF_ERR_INVALID_ARG", 2: "UPF_ERR_UNSUPPORTED", 3: "UPF_ERR_CUDA",
                4: "UPF_ERR_CAPACITY", 5: "UPF_ERR_NONFINITE", 6: "UPF_ERR_TIMEOUT"}


class UpfError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


class UpfBatch(ctypes.Structure):
    _fields_ = [("num_reqs", c_int32), ("cu_seqlens_dev", c_void_p), ("cu_seqlens_host", POINTER(c_int32)),
                ("num_q_heads", c_int32), ("num_kv_heads", c_int32), ("head_dim", c_int32),
                ("kv_of_q", POINTER(c_int32))]


class UpfParams(ctypes.Structure):
    _fields_ = [("n_tail", c_int32), ("block", c_int32), ("sink_keep", c_int32), ("tail_keep", c_int32),
                ("top_p", c_float), ("softmax_scale", c_float)]


class UpfCompactIO(ctypes.Structure):
    _fields_ = [("row_bytes", c_int64), ("hidden_in", c_void_p), ("hidden_out", c_void_p),
                ("pos_in", c_void_p), ("pos_out", c_void_p), ("slot_in", c_void_p), ("slot_out", c_void_p),
                ("kept_index", c_void_p), ("cu_seqlens_out", c_void_p), ("total_kept", c_void_p),
                ("layer_id", c_int32), ("history_cap", c_int32), ("history", c_void_p), ("history_len", c_void_p)]


_SIGNATURES = {
    "upf_version": ([], c_int),
    "upf_default_params": ([POINTER(UpfParams)], None),
    "upf_status_name": ([c_int], c_char_p),
    "upf_last_error": ([], c_char_p),
    "upf_create": ([POINTER(c_void_p), c_int], c_int),
    "upf_destroy": ([c_void_p], c_int),
    "upf_sync_status": ([c_void_p, c_void_p], c_int),
    "upf_workspace_bytes": ([POINTER(UpfBatch), POINTER(UpfParams)], c_size_t),
    "upf_score": ([c_void_p, POINTER(UpfBatch), POINTER(UpfParams), c_void_p, c_int64, c_void_p, c_int64,
                   c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "upf_score_shard": ([c_void_p, POINTER(UpfBatch), POINTER(UpfParams), c_int32, c_void_p, c_int64, c_void_p,
                         c_int64, c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "upf_set_wait_limit": ([c_void_p, c_int64], c_int),
    "upf_plan_info": ([POINTER(UpfBatch), POINTER(UpfParams), POINTER(c_int32), POINTER(c_int32), POINTER(c_int64),
                       POINTER(c_int64), POINTER(c_int32), POINTER(c_int32)], c_int),
    "upf_select": ([c_void_p, POINTER(UpfBatch), POINTER(UpfParams), c_void_p, c_void_p, c_void_p, c_void_p,
                    c_void_p, c_size_t, c_void_p], c_int),
    "upf_compact": ([c_void_p, POINTER(UpfBatch), c_void_p, POINTER(UpfCompactIO), c_void_p, c_size_t, c_void_p],
                    c_int),
    "upf_select_noalloc": ([POINTER(UpfBatch), POINTER(UpfParams), c_void_p, c_void_p, c_void_p, c_void_p,
                            c_void_p, c_void_p], c_int),
    "upf_revive": ([c_void_p, POINTER(UpfBatch), c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p], c_int),
    "upf_history_kv_len": ([c_void_p, POINTER(UpfBatch), c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p],
                           c_int),
    "upf_stage_name": ([c_int32], c_char_p),
    "upf_profile_enable": ([c_void_p, c_int32], c_int),
    "upf_profile_read": ([c_void_p, c_void_p, c_void_p, c_int32], c_int),
    "upf_select_tokens": ([c_void_p, POINTER(UpfBatch), POINTER(UpfParams), c_void_p, c_int64, c_void_p, c_int64,
                           c_void_p, c_void_p, c_void_p, c_void_p, POINTER(UpfCompactIO), c_void_p, c_size_t,
                           c_void_p], c_int),
}

_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libupf.so (built by ``sparse_long_context_tail_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libupf is not built ({p} missing): run __graft_entry__.build() or "
                           f"python -m sparse_long_context_tail_gb300.build")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


def _check(status: int) -> None:
    if status != UPF_OK:
        raise UpfError(status, load().upf_last_error().decode())


# ------------------------------------------------------------------ structs --

def make_batch(cu_seqlens_dev: int, cu_seqlens_host: np.ndarray, num_q_heads: int, num_kv_heads: int,
               head_dim: int, kv_of_q: Optional[Sequence[int]] = None):
    """Build a upf_batch; returns (struct, keepalive) -- keep both alive during the call."""
    cu = np.ascontiguousarray(cu_seqlens_host, dtype=np.int32)
    kv = None if kv_of_q is None else np.ascontiguousarray(kv_of_q, dtype=np.int32)
    b = UpfBatch(len(cu) - 1, ctypes.c_void_p(cu_seqlens_dev), cu.ctypes.data_as(POINTER(c_int32)),
                 num_q_heads, num_kv_heads, head_dim,
                 kv.ctypes.data_as(POINTER(c_int32)) if kv is not None else POINTER(c_int32)())
    return b, (cu, kv)


def make_params(n_tail: int = 128, block: int = 64, sink_keep: int = 128, tail_keep: int = 128,
                top_p: float = 0.99, softmax_scale: float = 0.0) -> UpfParams:
    return UpfParams(n_tail, block, sink_keep, tail_keep, top_p, softmax_scale)


def make_compact_io(row_bytes=0, hidden_in=0, hidden_out=0, pos_in=0, pos_out=0, slot_in=0, slot_out=0,
                    kept_index=0, cu_seqlens_out=0, total_kept=0, layer_id=0, history_cap=0, history=0,
                    history_len=0) -> UpfCompactIO:
    return UpfCompactIO(row_bytes, hidden_in or None, hidden_out or None, pos_in or None, pos_out or None,
                        slot_in or None, slot_out or None, kept_index or None, cu_seqlens_out or None,
                        total_kept or None, layer_id, history_cap, history or None, history_len or None)


# ------------------------------------------------------- entry points (C ABI) --

def upf_version() -> int:
    return load().upf_version()


def upf_default_params() -> UpfParams:
    p = UpfParams()
    load().upf_default_params(ctypes.byref(p))
    return p


def upf_status_name(status: int) -> str:
    return load().upf_status_name(status).decode()


def upf_last_error() -> str:
    return load().upf_last_error().decode()


def upf_create(device: int = 0) -> int:
    h = c_void_p()
    _check(load().upf_create(ctypes.byref(h), device))
    return h.value


def upf_destroy(ctx: int) -> None:
    _check(load().upf_destroy(ctx))


def upf_sync_status(ctx: int, stream: int = 0) -> int:
    """Return the device status code (0 = OK) without raising."""
    return load().upf_sync_status(ctx, stream or None)


def upf_workspace_bytes(batch: UpfBatch, params: UpfParams) -> int:
    n = load().upf_workspace_bytes(ctypes.byref(batch), ctypes.byref(params))
    if n == 0:
        raise UpfError(1, upf_last_error())
    return n


def upf_score(ctx, batch, params, q, q_row_stride, k, k_row_stride, scores, ws, ws_bytes, stream=0):
    _check(load().upf_score(ctx, ctypes.byref(batch), ctypes.byref(params), q, q_row_stride, k, k_row_stride,
                            scores, ws, ws_bytes, stream or None))


def upf_score_shard(ctx, batch, params, num_q_heads_total, q, q_row_stride, k, k_row_stride, scores, ws, ws_bytes,
                    stream=0):
    _check(load().upf_score_shard(ctx, ctypes.byref(batch), ctypes.byref(params), num_q_heads_total, q, q_row_stride,
                                  k, k_row_stride, scores, ws, ws_bytes, stream or None))


def upf_plan_info(batch: UpfBatch, params: UpfParams):
    """(keys per split of pass 1, of pass 2, items of pass 1, items of pass 2,
    CTAs per item of pass 1, of pass 2)."""
    k1, k2, i1, i2, c1, c2 = c_int32(), c_int32(), c_int64(), c_int64(), c_int32(), c_int32()
    _check(load().upf_plan_info(ctypes.byref(batch), ctypes.byref(params), ctypes.byref(k1), ctypes.byref(k2),
                                ctypes.byref(i1), ctypes.byref(i2), ctypes.byref(c1), ctypes.byref(c2)))
    return k1.value, k2.value, i1.value, i2.value, c1.value, c2.value


def upf_set_wait_limit(ctx: int, cycles: int) -> None:
    _check(load().upf_set_wait_limit(ctx, cycles))


def upf_select(ctx, batch, params, scores, block_scores, keep_bits, kept_count, ws, ws_bytes, stream=0):
    _check(load().upf_select(ctx, ctypes.byref(batch), ctypes.byref(params), scores, block_scores or None,
                             keep_bits, kept_count, ws, ws_bytes, stream or None))


def upf_select_noalloc(batch, params, scores, block_scores, keep_bits, kept_count, status_dev=0, stream=0):
    """upf_select without a context or workspace (scratch in a fixed array inside the library)."""
    _check(load().upf_select_noalloc(ctypes.byref(batch), ctypes.byref(params), scores, block_scores or None,
                                     keep_bits, kept_count, status_dev or None, stream or None))


def upf_compact(ctx, batch, keep_bits, io: UpfCompactIO, ws, ws_bytes, stream=0):
    _check(load().upf_compact(ctx, ctypes.byref(batch), keep_bits, ctypes.byref(io), ws, ws_bytes, stream or None))


def upf_revive(ctx, batch, kept_index, total_kept, rows, row_bytes, full, stream=0):
    _check(load().upf_revive(ctx, ctypes.byref(batch), kept_index, total_kept, rows, row_bytes, full, stream or None))


def upf_history_kv_len(ctx, batch, history, history_len, history_cap, layer_id, kv_len, stream=0):
    _check(load().upf_history_kv_len(ctx, ctypes.byref(batch), history, history_len, history_cap, layer_id, kv_len,
                                     stream or None))


NUM_STAGES = 8


def upf_stage_name(stage: int) -> str:
    return load().upf_stage_name(stage).decode()


def upf_profile_enable(ctx: int, on: bool = True) -> None:
    _check(load().upf_profile_enable(ctx, 1 if on else 0))


def upf_profile_read(ctx: int):
    """Per-stage (launches, device ms) since the previous read, as two lists."""
    launches = (c_int32 * NUM_STAGES)()
    ms = (ctypes.c_double * NUM_STAGES)()
    _check(load().upf_profile_read(ctx, ctypes.byref(launches), ctypes.byref(ms), NUM_STAGES))
    return list(launches), list(ms)


def upf_select_tokens(ctx, batch, params, q, q_row_stride, k, k_row_stride, scores, block_scores, keep_bits,
                      kept_count, io: UpfCompactIO, ws, ws_bytes, stream=0):
    _check(load().upf_select_tokens(ctx, ctypes.byref(batch), ctypes.byref(params), q, q_row_stride, k,
                                    k_row_stride, scores or None, block_scores or None, keep_bits, kept_count,
                                    ctypes.byref(io), ws, ws_bytes, stream or None))
