"""GPU parity on seeded random batches: head shapes and dims, GQA ratios, tail
sizes (including one the tensor-core path cannot tile, which takes the
CUDA-core kernels), block sizes, top-p, sink and tail exemptions, hidden row
sizes, ragged and empty requests and batches of more than 64 requests, each
checked against the oracle as in test_gpu_parity.check().  The configurations
are drawn from a fixed seed, so a failure names a reproducible case.
"""
import random

import pytest

from sparse_long_context_tail_gb300 import workload as wl
from test_gpu_parity import check, params_of, run_gpu

pytestmark = pytest.mark.gpu

HEADS = [(4, 2, 64), (8, 2, 128), (32, 8, 128), (6, 2, 128), (16, 8, 256), (16, 2, 256), (8, 8, 128), (12, 4, 64)]
LENS = [0, 1, 17, 100, 129, 257, 1000, 2049, 3000, 4096, 6000, 9000]
NCASES = 48


def random_spec(case, seed=20261203):
    rng = random.Random(seed * 1000 + case)
    Hq, Hkv, d = rng.choice(HEADS)
    many = rng.random() < 0.1
    R = rng.randint(65, 72) if many else rng.randint(1, 5)
    if many:
        lengths = [rng.randint(0, 300) for _ in range(R)]
    else:
        lengths = [rng.choice(LENS) if rng.random() < 0.6 else rng.randint(0, 7000) for _ in range(R)]
    budget = 24000 if d <= 128 and Hq <= 8 else 12000
    while sum(lengths) > budget:
        i = rng.randrange(R)
        lengths[i] //= 2
    if sum(lengths) == 0:
        lengths[0] = 300
    n = rng.choice([16, 32, 48, 64, 128, 128, 20])
    G = rng.choice([16, 32, 64, 64, 128])
    planted = [rng.randint(0, max(0, (L // G) // 4)) for L in lengths]
    return wl.WorkloadSpec(f"random-{case}", lengths, Hq, Hkv, d, rng.choice([256, 512, 520, 1040]), n_tail=n,
                           block=G, top_p=rng.choice([0.5, 0.8, 0.95, 0.99]), sink_keep=rng.choice([0, 64, 128]),
                           tail_keep=rng.choice([0, 64, 128]), planted=planted, strength_range=(1.0, 4.0),
                           seed=7000 + case)


@pytest.fixture(scope="module")
def sel():
    import __graft_entry__
    __graft_entry__.build()
    from sparse_long_context_tail_gb300.selector import TokenSelector
    s = TokenSelector(0)
    yield s
    s.close()


@pytest.mark.parametrize("case", range(NCASES))
def test_random_batch_parity(sel, case):
    spec = random_spec(case)
    w = wl.generate(spec)
    p = params_of(spec)
    out, status, inputs = run_gpu(sel, w, p)
    check(w, p, out, status, inputs)
