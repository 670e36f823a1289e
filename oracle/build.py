"""Build the CPU checker library (test infrastructure only).

Compiles oracle.c and units.c with gcc into oracle/_build/liboracle.so. Flags: -O2,
-ffp-contract=off and no fast-math, so every C statement of the checker is one
IEEE operation rounded to nearest-even (gcc would otherwise fuse multiply-adds
on Arm hosts).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SYNTH_DIR = os.path.join(ROOT, "fsdp_sharded_mixed_shard_gb300", "synth")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")
SOURCES = [os.path.join(HERE, "oracle.c"), os.path.join(HERE, "units.c")]
HEADERS = [os.path.join(HERE, "oracle.h"), os.path.join(SYNTH_DIR, "synth.h")]

CFLAGS = ["-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-pthread"]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False):
    """Compile liboracle.so if it is missing or older than its sources."""
    if not force and not _stale(LIB, SOURCES + HEADERS + [__file__]):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc"] + CFLAGS + ["-I", SYNTH_DIR] + SOURCES + ["-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
