"""Failure detection on the GPU without a fault: a bounded wait that expires.

Every wait inside the tensor-core scoring kernels is bounded.  Here the
pipeline waits' limit is lowered to 64 SM cycles for one call, far below the
time a key tile takes to arrive or to be consumed, so a wait expires: the
kernel must report UPF_ERR_TIMEOUT through the status word, wind down (its
outstanding copies and MMAs are waited for with the full limit, its tensor
memory is freed) and leave the context usable.  The next call on the same
context, with the default limit back, must match the float64 oracle.
"""
import pytest

from sparse_long_context_tail_gb300 import _binding as B
from sparse_long_context_tail_gb300 import workload as wl

from test_gpu_parity import check, params_of, run_gpu, sel  # noqa: F401  (sel is a fixture)

pytestmark = pytest.mark.gpu

UPF_ERR_TIMEOUT = 6


def _spec():
    # LLaMA-shaped heads, 8192 tokens: every work item streams more key tiles
    # than the ring holds, so the producer has to wait for a free stage.
    return wl.WorkloadSpec("timeout", [8192, 3000], 32, 8, 128, 512, planted=[4, 2], strength_range=(1.0, 4.0),
                           seed=41)


def test_expired_pipeline_wait_is_reported_and_the_context_recovers(sel):  # noqa: F811
    w = wl.generate(_spec())
    p = params_of(w.spec)
    B.upf_set_wait_limit(sel.ctx, 64)
    try:
        _, status, _ = run_gpu(sel, w, p)
    finally:
        B.upf_set_wait_limit(sel.ctx, 0)
    assert status == UPF_ERR_TIMEOUT, B.STATUS_NAMES.get(status)
    assert sel.status() == 0                     # the read cleared the status word
    for _ in range(2):                           # the context and the GPU are fine afterwards
        out, status, inputs = run_gpu(sel, w, p)
        check(w, p, out, status, inputs)

