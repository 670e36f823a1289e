"""The checked build (libzero_checked.so: every kernel tests the memory ranges
it touches) on parity cases that cover fused and two-pass paths, both
formats, 8 to 64 ranks, a rank subset with its own window, micro-batches,
the scalar head/tail paths, the short-step kernel with an overflowed step's
re-cast, the unit all-gather / shard at every 16-byte
phase and the norm entry points (workspace, no-allocation, export / import):
results still match the checker and no kernel records a violation;
the planted self-test violation is reported."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_checked_build_records_no_violation():
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_runner.py")],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    got = {x["case"]: x for x in lines}
    assert got["selftest"]["violations"] == 1
    assert got["selftest"]["first"] == (1 << 48) | 42
    assert got["library"]["loaded"].endswith("libzero_checked.so")
    cases = [x for x in lines if x["case"] not in ("selftest", "library")]
    assert len(cases) == 14
    assert {"odd_shard_two_pass_n8", "shard_4_mod_8_fused_n64", "odd_shard_micro_fused_n8",
            "random_shapes_24", "norm_entries", "short_step_overflow_recast_n12"} <= \
        {x["case"] for x in cases}
    for x in cases:
        assert x["violations"] == 0, x
