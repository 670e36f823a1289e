"""Seeded random shapes against the checker, element by element: N, the
tensor list, the bucket size, the rank window, micro-batches, the gradient
format and the path are drawn at random (fixed seed), so that owners start
at every phase of the 16-byte grid, windows start at odd owners and bucket
boundaries fall anywhere. Small sizes, two steps each."""
import numpy as np
import pytest
import torch

import oracle
from fsdp_sharded_mixed_shard_gb300 import workloads as W
from parity_util import run_small

pytestmark = pytest.mark.gpu

N_CASES = 96


def _case(i):
    rng = np.random.default_rng(20_261_202 + i)
    n = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 13, 16, 31, 64]))
    n_tensors = int(rng.integers(1, 5))
    numels = [int(x) for x in rng.integers(0, 60_000, size=n_tensors)]
    if sum(numels) == 0:
        numels[0] = 1
    bucket = int(rng.choice([0, 0, 7, 4096, 10_001, 32_768]))
    lo = int(rng.integers(0, n))
    hi = int(rng.integers(lo + 1, n + 1))
    micro = int(rng.choice([1, 1, 2, 3]))
    bf16 = bool(rng.integers(0, 2))
    clip = float(rng.choice([0.0, 0.0, 0.3]))
    per_bucket = clip > 0 and bucket > 0 and bool(rng.integers(0, 2))
    return dict(n=n, numels=numels, bucket=bucket, lo=lo, hi=hi, micro=micro, bf16=bf16,
                clip=clip, per_bucket=per_bucket)


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_matches_checker(i):
    c = _case(i)
    wl = W.Workload("random%d" % i, c["numels"], c["n"], c["bucket"], c["bf16"], 100 + i, 1e-3,
                    init_scale=1.0 if c["bf16"] else 1024.0, steps=2, rank_lo=c["lo"],
                    rank_hi=c["hi"], n_micro=c["micro"], max_grad_norm=c["clip"])
    p, _, _ = oracle.make_plan(wl.numels, wl.n_ranks, wl.bucket_elems)
    assert p.shard >= 1
    run_small(wl, per_bucket=c["per_bucket"], two_pass=c["clip"] > 0)


def test_random_cases_cover_the_grid_phases():
    """The drawn cases include owners at several phases of the 8-element
    grid, rank windows that do not start at 0 and micro-batches (checked on
    the CPU, from the case list alone)."""
    phases, windows, micro = set(), 0, 0
    for i in range(N_CASES):
        c = _case(i)
        p, _, _ = oracle.make_plan(c["numels"], c["n"], c["bucket"])
        for r in range(c["lo"], c["hi"]):
            phases.add(((r - c["lo"]) * p.shard) % 8)
        windows += c["lo"] > 0
        micro += c["micro"] > 1
    assert len(phases) >= 6 and windows >= 4 and micro >= 4
