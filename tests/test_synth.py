"""Checks of the shared seeded input generator (synth.h): known SplitMix64
outputs, the normal approximation's moments and bounds, outlier rate,
master-weight range, padding."""
import json
import math
import os

import numpy as np
import pytest

from fsdp_sharded_mixed_shard_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
G = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1


def test_splitmix64_reference_outputs():
    gold = json.load(open(os.path.join(HERE, "golden", "splitmix64.json")))
    for k, hx in enumerate(gold["state0_outputs_hex"], start=1):
        assert synth.mix64((k * G) & M64) == int(hx, 16)


def test_normal_constant():
    # lanes 0x8000, 0x7fff, 0x7fff, 0x8001 sum to the mean + 1: z = C0 exactly
    assert synth.normal_from_hash(0x80017FFF7FFF8000) == np.float32(math.sqrt(3.0) / 65536.0)
    # lanes summing to the mean give exactly 0
    h = 0x7FFF7FFF7FFF8001  # lanes 0x8001, 0x7fff, 0x7fff, 0x7fff -> 131070
    assert synth.normal_from_hash(h) == 0.0


def test_gradient_moments_and_bounds():
    spec = synth.grad_spec(seed=1, sigma=1.0, psi=1 << 22)
    x = synth.grad_f32(1 << 22, 0, spec, 1, 0).astype(np.float64)
    assert abs(x.mean()) < 2e-3
    assert abs(x.std() - 1.0) < 2e-3
    assert np.abs(x).max() <= 131070 * math.sqrt(3.0) / 65536.0 * (1 + 1e-6)


def test_streams_differ_by_step_rank_seed():
    spec = synth.grad_spec(seed=1, psi=1000)
    a = synth.grad_f32(1000, 0, spec, 1, 0)
    assert not np.array_equal(a, synth.grad_f32(1000, 0, spec, 2, 0))
    assert not np.array_equal(a, synth.grad_f32(1000, 0, spec, 1, 1))
    assert not np.array_equal(a, synth.grad_f32(1000, 0, synth.grad_spec(seed=2, psi=1000), 1, 0))
    assert np.array_equal(a, synth.grad_f32(1000, 0, spec, 1, 0))
    assert np.array_equal(a[500:], synth.grad_f32(500, 500, spec, 1, 0))
    assert np.array_equal(a[[3, 999]], synth.grad_f32_at([3, 999], spec, 1, 0))


def test_outlier_rate_and_bias():
    n = 1 << 21
    base = synth.grad_f32(n, 0, synth.grad_spec(seed=4, psi=n), 1, 3)
    out = synth.grad_f32(n, 0, synth.grad_spec(seed=4, psi=n, outliers=True), 1, 3)
    hit = out != base
    rate = hit.mean()
    assert abs(rate - 1049 / 2**20) < 4 * math.sqrt(1049 / 2**20 / n)
    assert np.array_equal(out[hit], (base[hit] * np.float32(100.0)).astype(np.float32))
    biased = synth.grad_f32(n, 0, synth.grad_spec(seed=4, psi=n, bias_sigma=1e-5), 1, 3)
    d = (biased - base).astype(np.float64)
    assert np.ptp(d) < 1e-9 + 1e-6 * 4e-3  # one offset per (step, rank) up to fp32 rounding


def test_master_range_and_padding():
    x = synth.master_f32(1 << 20, 0, 0, 1000)
    assert np.all(x[1000:] == 0)
    y = synth.master_f32(1 << 20, 0, 0, 1 << 20)
    assert y.min() > -0.05 and y.max() < 0.05 and abs(y.mean()) < 2e-4
    spec = synth.grad_spec(seed=1, psi=10)
    assert np.all(synth.grad_f32(20, 0, spec, 1, 0)[10:] == 0)


def test_stream_form_matches_direct_form():
    import ctypes as C
    L = synth.host()
    L.zs_host_fill_grad_stream.argtypes = [C.c_void_p, C.c_int64, C.c_int64,
                                           C.POINTER(synth.GradSpec), C.c_uint32, C.c_uint32]
    for kw in (dict(), dict(bias_sigma=1e-5), dict(outliers=True, loss_scale=65536.0)):
        spec = synth.grad_spec(seed=3, psi=5000, **kw)
        a = synth.grad_f32(6000, 17, spec, 2, 5)
        b = np.empty(6000, np.float32)
        L.zs_host_fill_grad_stream(b.ctypes.data, 6000, 17, C.byref(spec), 2, 5)
        assert np.array_equal(a, b)
