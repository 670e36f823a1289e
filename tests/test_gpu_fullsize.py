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


def test_indices_beyond_2p31_fused():
    """2^31 + 12,345 parameters at N = 2 (about 64 GB on the device): every
    window, shard and tile index passes 2^31 on the way."""
    wl = W.Workload("int64_fused", [2 ** 31 + 12_345], 2, 0, True, 41, 1e-3, steps=2)
    dev, orc = run_sampled(wl)
    assert dev.t == 2


def test_indices_beyond_2p31_two_pass_clip():
    """One rank whose shard alone holds 2^31 + 12,345 elements, fp16 with a
    dynamic scale and an active clip: the two-pass path, norm records and
    the update (in place, one state set) address past 2^31 within a shard."""
    wl = W.Workload("int64_clip", [2 ** 31 + 12_345], 1, 0, False, 42, 1e-4, init_scale=4096.0,
                    dynamic_scale=True, max_grad_norm=1.0, steps=2)
    dev, orc = run_sampled(wl, n_sets=1)
    assert dev.t == 2 and dev.clip_apply == 1
