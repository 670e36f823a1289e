"""The kernels' integer form of the fp64 step scalars (csrc/f64emu.h: the
rounded product beta^t * beta, 1 - p and the narrowing to fp32) against the
host's IEEE double and float arithmetic, bit for bit, over Adam's beta
power chains to the normal limit, random operands of every exponent and
exact ties (CPU only)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "fsdp_sharded_mixed_shard_gb300", "csrc")


def test_integer_fp64_scalars_match_ieee(tmp_path):
    if not shutil.which("g++"):
        pytest.skip("needs g++")
    exe = str(tmp_path / "f64emu_test")
    subprocess.run(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-Wall", "-I", CSRC,
                    os.path.join(ROOT, "tests", "native", "f64emu_test.cpp"), "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe, "3"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "f64emu ok" in r.stdout, r.stdout + r.stderr
