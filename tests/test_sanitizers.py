"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer (CPU only):
the library's host planner (plan.cpp, units.cpp) and the CPU checker
(oracle/*.c with the host generator), each driven by a small random-input
program under tests/native. Any sanitizer report fails the run."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NATIVE = os.path.join(ROOT, "tests", "native")
CSRC = os.path.join(ROOT, "fsdp_sharded_mixed_shard_gb300", "csrc")
SYNTH = os.path.join(ROOT, "fsdp_sharded_mixed_shard_gb300", "synth")
SAN = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer",
       "-g", "-O1"]
ENV = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=1",
           UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")


def _run(cmd, tmp_path, exe, arg):
    out = str(tmp_path / exe)
    subprocess.run(cmd + ["-o", out], check=True, capture_output=True, text=True)
    r = subprocess.run([out, str(arg)], capture_output=True, text=True, env=ENV, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "runtime error" not in r.stderr and "ERROR: AddressSanitizer" not in r.stderr
    return r.stdout


@pytest.fixture(scope="module")
def have_asan(tmp_path_factory):
    if not shutil.which("g++") or not shutil.which("gcc"):
        pytest.skip("needs gcc and g++")
    d = tmp_path_factory.mktemp("probe")
    src = d / "p.c"
    src.write_text("int main(void){return 0;}\n")
    r = subprocess.run(["gcc"] + SAN + [str(src), "-o", str(d / "p")], capture_output=True)
    if r.returncode != 0:
        pytest.skip("sanitizer runtime not available")


def test_host_planner_under_sanitizers(have_asan, tmp_path):
    cmd = ["g++", "-std=c++17"] + SAN + [
        "-I", os.path.join(ROOT, "include"), "-I", CSRC,
        os.path.join(NATIVE, "planner_fuzz.cpp"), os.path.join(CSRC, "plan.cpp"),
        os.path.join(CSRC, "units.cpp")]
    assert "planner_fuzz ok" in _run(cmd, tmp_path, "planner_fuzz", 2000)


def test_checker_under_sanitizers(have_asan, tmp_path):
    cmd = ["gcc", "-std=c11", "-ffp-contract=off", "-pthread"] + SAN + [
        "-I", os.path.join(ROOT, "oracle"), "-I", SYNTH,
        os.path.join(NATIVE, "oracle_fuzz.c"), os.path.join(ROOT, "oracle", "oracle.c"),
        os.path.join(ROOT, "oracle", "units.c"), "-lm"]
    assert "oracle_fuzz ok" in _run(cmd, tmp_path, "oracle_fuzz", 200)
