"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times: the checker regenerates every replica value on the host,
computes the global flags, overflow and norm over all elements, and the
updates of sampled elements (slice and bucket edges, padding, the injected
element, random ones)."""
import pytest
import torch

from fsdp_sharded_mixed_shard_gb300 import workloads as W
from parity_util import run_sampled

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_gpt2_small_full():
    dev, orc = run_sampled(W.GPT2_SMALL)
    assert dev.t == 10


def test_flat_1p5b_full():
    dev, orc = run_sampled(W.FLAT_1P5B)
    assert dev.t == 4 and dev.n_skipped == 1 and dev.scale == 32768.0


def test_stage3_slice_full():
    dev, orc = run_sampled(W.STAGE3_SLICE)
    assert dev.t == 5


def test_llama_2b_full():
    dev, orc = run_sampled(W.LLAMA_2B)
    assert dev.t == 5 and dev.clip_apply == 1
