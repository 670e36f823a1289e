"""Seeded random shapes against the checker, element by element: N, the
tensor list, the bucket size, the rank window, micro-batches, the gradient
format and the path are drawn at random (fixed seed), so that owners start
at every phase of the 16-byte grid, windows start at odd owners and bucket
boundaries fall anywhere. Small sizes, two steps each."""
import pytest
import torch

import oracle
from parity_util import random_workload, run_small

pytestmark = pytest.mark.gpu

N_CASES = 96


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_matches_checker(i):
    wl, per_bucket, two_pass = random_workload(i)
    p, _, _ = oracle.make_plan(wl.numels, wl.n_ranks, wl.bucket_elems)
    assert p.shard >= 1
    run_small(wl, per_bucket=per_bucket, two_pass=two_pass)
