"""Pins of the checker's bf16/fp16 conversions: the pages' format facts and
an exhaustive comparison with the compiler's own _Float16 / __bf16 types and
with numpy / torch CPU conversions."""
import json
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "page_figures.json")))


def _f16(x):
    return float(oracle.widen16(oracle.cast16([x], False), False)[0])


def _bf16(x):
    return float(oracle.widen16(oracle.cast16([x], True), True)[0])


@pytest.mark.parametrize("e", GOLD["formats"], ids=lambda e: e["id"])
def test_format_facts_from_pages(e):
    conv = _f16 if e["format"] == "fp16" else _bf16
    if "largest_finite" in e:
        big = e["largest_finite"]
        assert conv(big) == big
        assert math.isinf(conv(np.nextafter(np.float32(big), np.float32(np.inf)) * 1.01))
    if "largest_finite_approx" in e:
        mx = float(oracle.widen16([0x7F7F], True)[0])
        assert abs(mx - e["largest_finite_approx"]) <= e["tol_rel"] * mx
        assert conv(mx) == mx
    if "gap_after_one" in e:
        nxt = float(oracle.widen16([0x3C01 if e["format"] == "fp16" else 0x3F81],
                                  e["format"] == "bf16")[0])
        assert nxt - 1.0 == e["gap_after_one"]
        assert conv(1.0 + e["gap_after_one"]) == 1.0 + e["gap_after_one"]
    if "rounds_to" in e:
        want = math.inf if e["rounds_to"] == "inf" else e["rounds_to"]
        assert conv(e["value"]) == want


def test_widening_all_patterns_against_numpy_and_torch():
    pats = np.arange(65536, dtype=np.uint16)
    f16 = oracle.widen16(pats, False)
    ref16 = pats.view(np.float16).astype(np.float32)
    assert np.array_equal(f16, ref16, equal_nan=True)
    bf = oracle.widen16(pats, True)
    refbf = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(bf, refbf, equal_nan=True)


def test_narrowing_sampled_against_numpy_and_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    got16 = oracle.cast16(x, False)
    want16 = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got16, want16)
    gotbf = oracle.cast16(x, True)
    wantbf = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gotbf, wantbf)


CHECKER_C = r"""
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <math.h>
#include "oracle.h"
static uint64_t bad[64];
static int nth;
static void* work(void* a) {
  int w = (int)(intptr_t)a;
  for (uint64_t b = (uint64_t)w; b < (1ull << 32); b += (uint64_t)nth) {
    uint32_t u = (uint32_t)b; float x; memcpy(&x, &u, 4);
    if (isnan(x)) continue;
    _Float16 h = (_Float16)x; uint16_t hb; memcpy(&hb, &h, 2);
    __bf16 q = (__bf16)x; uint16_t qb; memcpy(&qb, &q, 2);
    if (orc_f32_to_f16(x) != hb) bad[w]++;
    if (orc_f32_to_bf16(x) != qb) bad[w]++;
  }
  return NULL;
}
int main(int argc, char** argv) {
  nth = argc > 1 ? atoi(argv[1]) : 8; if (nth > 64) nth = 64;
  pthread_t t[64];
  for (int w = 0; w < nth; ++w) pthread_create(&t[w], NULL, work, (void*)(intptr_t)w);
  uint64_t tot = 0;
  for (int w = 0; w < nth; ++w) { pthread_join(t[w], NULL); tot += bad[w]; }
  printf("%llu\n", (unsigned long long)tot);
  return 0;
}
"""


def test_narrowing_exhaustive_against_compiler_types():
    """All 2^32 fp32 patterns except NaNs: the checker's RNE conversions equal
    gcc's _Float16 and __bf16 conversions."""
    root = os.path.dirname(HERE)
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "chk.c")
        exe = os.path.join(d, "chk")
        open(src, "w").write(CHECKER_C.replace("#include <math.h>", "#include <math.h>\n#include <stdlib.h>"))
        cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-pthread",
               "-I", os.path.join(root, "oracle"),
               "-I", os.path.join(root, "fsdp_sharded_mixed_shard_gb300", "synth"),
               src, os.path.join(root, "oracle", "oracle.c"), "-o", exe, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            pytest.skip("compiler lacks _Float16/__bf16: " + r.stderr[-300:])
        out = subprocess.run([exe, str(os.cpu_count() or 8)], capture_output=True, text=True,
                             check=True, timeout=900)
        assert int(out.stdout.strip()) == 0


def test_special_values():
    inf = float("inf")
    for bf in (False, True):
        h = oracle.cast16([0.0, -0.0, inf, -inf, float("nan")], bf)
        w = oracle.widen16(h, bf)
        assert w[0] == 0 and not np.signbit(w[0]) and np.signbit(w[1])
        assert w[2] == inf and w[3] == -inf and np.isnan(w[4])
    # fp16 subnormals survive (no flush to zero)
    assert _f16(2.0 ** -24) == 2.0 ** -24
    assert _f16(2.0 ** -25) == 0.0          # tie to even rounds down to 0
    assert _f16(1.5 * 2.0 ** -25) == 2.0 ** -24
    # bf16 keeps fp32 subnormals it can represent
    assert _bf16(2.0 ** -133) == 2.0 ** -133
