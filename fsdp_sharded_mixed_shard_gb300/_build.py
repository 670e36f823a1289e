"""In-tree build of the native libraries (no pip install, no cmake).

  _lib/libzero.so          the C-ABI library: host planner + sm_103a kernels
  _lib/libzero_checked.so  the same built with -DZERO_CHECKED: every kernel tests
                           the memory ranges it touches and counts violations
  _lib/libzsynth_gpu.so    synthetic-input generator kernels (harness only)
  _lib/libzsynth_host.so   host build of the same generator (harness only)

Device code: nvcc for sm_103a only, -O3 -lineinfo, --fmad=false (no fused
multiply-add contraction: each fp32 statement of the step is one IEEE
operation), no fast-math, no flush-to-zero. Host code: -ffp-contract=off for
the same reason. Libraries are rebuilt only when a source is newer.
"""
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
SYNTH = os.path.join(PKG, "synth")
LIBDIR = os.path.join(PKG, "_lib")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-shared",
                     "-Xcompiler", "-fPIC,-ffp-contract=off,-fvisibility=hidden"]

ZERO_LIB = os.path.join(LIBDIR, "libzero.so")
ZERO_CHECKED_LIB = os.path.join(LIBDIR, "libzero_checked.so")
SYNTH_GPU_LIB = os.path.join(LIBDIR, "libzsynth_gpu.so")
SYNTH_HOST_LIB = os.path.join(LIBDIR, "libzsynth_host.so")


def _files(d, exts):
    return sorted(os.path.join(d, f) for f in os.listdir(d) if f.endswith(exts))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _jobs():
    """(target, deps, command) for each library."""
    zero_src = _files(CSRC, (".cu", ".cpp"))
    zero_dep = zero_src + _files(CSRC, (".h", ".cuh")) + _files(INCLUDE, (".h",)) + [__file__]
    synth_h = os.path.join(SYNTH, "synth.h")
    jobs = []
    if zero_src:
        jobs.append((ZERO_LIB, zero_dep,
                     [NVCC] + NVCC_FLAGS + ["-I", INCLUDE, "-I", CSRC] + zero_src))
        jobs.append((ZERO_CHECKED_LIB, zero_dep,
                     [NVCC] + NVCC_FLAGS + ["-DZERO_CHECKED", "-I", INCLUDE, "-I", CSRC] +
                     zero_src))
    jobs += [
        (SYNTH_GPU_LIB, [os.path.join(SYNTH, "synth_gpu.cu"), synth_h, __file__],
         [NVCC] + NVCC_FLAGS + ["-I", SYNTH, os.path.join(SYNTH, "synth_gpu.cu")]),
        (SYNTH_HOST_LIB, [os.path.join(SYNTH, "synth_host.c"), synth_h, __file__],
         ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-I", SYNTH, os.path.join(SYNTH, "synth_host.c")]),
    ]
    return jobs


def build(force=False, verbose=False):
    """Compile every stale library in parallel; raise on any failure."""
    os.makedirs(LIBDIR, exist_ok=True)
    procs = []
    for target, deps, cmd in _jobs():
        if not force and not _stale(target, deps):
            continue
        tmp = target + ".tmp%d" % os.getpid()
        full = cmd + ["-o", tmp]
        if verbose:
            print(" ".join(full))
        procs.append((target, tmp, full, subprocess.Popen(
            full, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for target, tmp, full, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append("%s\n%s" % (" ".join(full), out.decode(errors="replace")))
        else:
            os.replace(tmp, target)
            if verbose and out:
                print(out.decode(errors="replace"))
    if errors:
        raise RuntimeError("native build failed:\n" + "\n".join(errors))
    return [ZERO_LIB, SYNTH_GPU_LIB, SYNTH_HOST_LIB]


if __name__ == "__main__":
    build(force=True, verbose=True)
