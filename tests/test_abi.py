"""C ABI checks that need no GPU: the library loads, exports every function
include/zero.h declares, struct layouts agree with the Python mirrors, and the
planner matches the CPU checker's planner bit for bit."""
import ctypes as C
import os
import random
import re
import subprocess

import pytest

import oracle
import fsdp_sharded_mixed_shard_gb300 as Z
from fsdp_sharded_mixed_shard_gb300 import _build, workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"ZERO_API\s+[\w\s\*]+?\b(zero_\w+)\s*\(", txt))
    return names


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert {"zero_plan_create", "zero_reduce_scatter", "zero_grad_norm", "zero_step"} <= names
    L = C.CDLL(_build.ZERO_LIB)
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", _build.ZERO_LIB], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (zero_\w+)", out))
    assert names <= exported
    assert exported <= names, "exported but undeclared: %s" % (exported - names)
    out = subprocess.run(["nm", "-D", "--defined-only", _build.ZERO_CHECKED_LIB],
                         capture_output=True, text=True).stdout
    assert set(re.findall(r" T (zero_\w+)", out)) == exported


def test_release_build_has_no_checks():
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_checked_status()
    assert e.value.status == -6
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_selftest_check()
    assert e.value.status == -6


def test_struct_sizes():
    assert C.sizeof(Z.ZeroUnit) == 56
    assert C.sizeof(Z.ZeroUnitPlanInfo) == 120
    assert C.sizeof(Z.ZeroStrategyCost) == 56
    assert C.sizeof(Z.ZeroScaler) == 80
    assert C.sizeof(Z.ZeroPlanInfo) == 168
    assert C.sizeof(Z.ZeroHParams) == 64
    assert C.sizeof(Z.ZeroSegment) == 24
    assert C.sizeof(Z.ZeroBucket) == 24
    assert C.sizeof(Z.ZeroNormRecord) == 16
    assert C.sizeof(Z.ZeroExchange) == 16 + 16 * Z.ZERO_MAX_RANKS


def _compare(numels, n, bsz, dtype=Z.ZERO_BF16):
    p = Z.zero_plan_create(numels, n, bsz, dtype)
    try:
        info = Z.zero_plan_get_info(p)
        op, ooffs, osegs = oracle.make_plan(numels, n, bsz)
        assert (info.psi, info.pad, info.psi_pad, info.shard_elems, info.n_buckets,
                info.n_segments) == (op.psi, op.pad, op.psi_pad, op.shard, op.n_buckets,
                                     op.n_segments)
        assert Z.zero_plan_tensor_offsets(p) == list(ooffs)
        assert Z.zero_plan_segments(p) == [tuple(s) for s in osegs]
        for k in range(info.n_buckets):
            lo, hi = Z.zero_plan_bucket_range(p, k)
            assert lo == (k * bsz if bsz else 0)
            assert hi == (min((k + 1) * bsz, info.psi_pad) if bsz else info.psi_pad)
        for a, b in ((info.bill_ddp, op.bill_ddp), (info.bill_z1, op.bill_z1),
                     (info.bill_z2, op.bill_z2), (info.bill_z3, op.bill_z3),
                     (info.ring_bytes_per_rank, op.ring_bytes_per_rank),
                     (info.ring_hops, op.ring_hops), (info.comm_elems_z3, op.comm_z3)):
            assert a == pytest.approx(b, rel=1e-15, abs=0)
        assert info.step_bytes_fused == 2 * n + 26
        assert info.n_tiles == sum(-(-(hi - lo) // Z.ZERO_TILE_ELEMS) for lo, hi, _, _ in osegs)
        ws = Z.zero_workspace_bytes(p, 1)
        assert ws >= 16 * (info.n_tiles + n * Z.ZERO_NORM_OWNER_BLOCKS) and ws % 256 == 0
        assert Z.zero_workspace_bytes(p, 0) == 0
        # the names the boundary lists: zero_plan_info_get, zero_plan_buckets
        alias = Z.zero_plan_info_get(p)
        assert bytes(alias) == bytes(info)
        buckets, segs = Z.zero_plan_buckets(p)
        assert segs == [tuple(s) for s in osegs]
        assert len(buckets) == op.n_buckets
        of_bucket = {}
        for i, sg in enumerate(osegs):
            of_bucket.setdefault(sg[3], []).append(i)
        for k, (lo, hi, first, count) in enumerate(buckets):
            assert (lo, hi) == Z.zero_plan_bucket_range(p, k)
            mine = of_bucket.get(k, [])
            assert count == len(mine) and (not mine or first == mine[0])
            assert mine == list(range(first, first + count))
            # the bucket's segments tile [lo, hi) (a bucket past psi_pad is empty)
            assert sum(osegs[i][1] - osegs[i][0] for i in mine) == hi - lo
    finally:
        Z.zero_plan_destroy(p)


def test_planner_matches_checker_on_workloads():
    for wl in W.ALL:
        _compare(wl.numels, wl.n_ranks, wl.bucket_elems)


def test_planner_matches_checker_random():
    rng = random.Random(7)
    for _ in range(400):
        n = rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 16, 63, 64])
        numels = [rng.choice([0, 1, 2, 5, 31, 4096, 10007]) for _ in range(rng.randint(0, 7))]
        bsz = rng.choice([0, 1, 2, 7, 64, 1000, 4096, 99991])
        _compare(numels, n, bsz)


def test_planner_rejects_bad_arguments():
    for args, status in ((([10], 0, 0), -1), (([10], 65, 0), -3), (([-1], 2, 0), -1),
                         (([10], 2, -3), -1)):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_plan_create(*args)
        assert e.value.status == status
    with pytest.raises(Z.ZeroError):
        Z.zero_plan_create([10], 2, 0, 7)


def test_scaler_init_and_strerror():
    hp = Z.ZeroHParams(1e-3, 0.9, 0.999, 1e-8, 0.01, 0.0, 1, 2000, 65536.0)
    s = Z.zero_scaler_init(hp)
    assert s.scale == 65536.0 and s.t == 0 and s.beta1_pow == 1.0 and s.state_index == 0
    assert Z.zero_strerror(-2).startswith("device pointer")
    assert Z.zero_version() >= 100
    bad = Z.ZeroHParams(1e-3, 0.9, 0.999, 1e-8, 0.01, 0.0, 1, 0, 65536.0)
    with pytest.raises(Z.ZeroError):
        Z.zero_scaler_init(bad)


def test_host_validation_without_gpu():
    """Argument checks run before any CUDA call, so they work on a CPU host."""
    p = Z.zero_plan_create([1000], 4, 0)
    hp = Z.ZeroHParams(1e-3, 0.9, 0.999, 1e-8, 0.01, 0.0, 0, 2000, 1.0)
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_step(p, 0, 5, [None] * 8, [None] * 8, [None] * 8, 2, None, [None] * 4, 0, 16, hp,
                    16)
    assert e.value.status == -1
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_step(p, 0, 4, [16] * 8, [16] * 8, [16] * 8, 2, None, [16] * 4, 0, 24, hp, 16)
    assert e.value.status == -2
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_grad_norm(p, 0, 4, None, hp, 16, 16)
    assert e.value.status == -1
    clip = Z.ZeroHParams(1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0, 0, 2000, 1.0)
    # exchange export: no exchange buffer; a clipped export without a
    # workspace; a misaligned exchange buffer
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_grad_norm_local(p, 0, 2, None, hp, 16, 0, 0)
    assert e.value.status == -1
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_grad_norm_local(p, 0, 2, None, clip, 16, 0, 16)
    assert e.value.status == -1
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_grad_norm_local(p, 2, 1, None, hp, 16, 0, 16)
    assert e.value.status == -1
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_grad_norm_local(p, 0, 2, None, hp, 16, 0, 24)
    assert e.value.status == -2
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_grad_norm_apply(p, 0, clip, 16)
    assert e.value.status == -1
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_grad_norm_apply(p, 24, clip, 16)
    assert e.value.status == -2
    for bad_limit in (0, 999, 10**11):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_selftest_wait_timeout(16, bad_limit)
        assert e.value.status == -1
    Z.zero_plan_destroy(p)


def _compare_units(numels, uot, n_units, n, align):
    p = Z.zero_unit_plan_create(numels, uot, n_units, n, align)
    try:
        info = Z.zero_unit_plan_get_info(p)
        units = Z.zero_unit_plan_units(p)
        slots, offs = Z.zero_unit_plan_tensors(p)
        op, ounits, oslots, ooffs = oracle.make_unit_plan(numels, uot, n_units, n, align)
        for f in ("psi", "psi_pad", "max_unit_psi_pad", "n_units", "n_ranks", "n_tensors",
                  "align_elems", "persistent_bytes", "peak_one_bytes", "peak_two_bytes",
                  "peak_backward_bytes", "max_unit_fraction", "comm_elems", "comm_bytes",
                  "ring_bytes", "n_gathers"):
            assert getattr(info, f) == getattr(op, f), f
        assert info.shard_elems == op.shard
        for a, b in zip(units, ounits):
            assert (a.psi, a.pad, a.psi_pad, a.shard_elems, a.shard_offset, a.flat_offset,
                    a.n_tensors, a.first_slot) == (b.psi, b.pad, b.psi_pad, b.shard,
                                                   b.shard_offset, b.flat_offset, b.n_tensors,
                                                   b.first_slot)
        assert slots == list(oslots) and offs == list(ooffs)
        for strat in range(5):
            for reps in ((1, 2, 5) if strat == Z.ZERO_HYBRID_SHARD else (1,)):
                a = Z.zero_unit_plan_strategy_cost(p, strat, reps)
                b = oracle.strategy_cost(op, strat, reps)
                for f, _ in Z.ZeroStrategyCost._fields_:
                    assert getattr(a, f) == pytest.approx(getattr(b, f), rel=1e-15, abs=0), f
        for strat, reps in ((5, 1), (-1, 1), (Z.ZERO_FULL_SHARD, 2), (Z.ZERO_HYBRID_SHARD, 0)):
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_unit_plan_strategy_cost(p, strat, reps)
            assert e.value.status == -1
    finally:
        Z.zero_unit_plan_destroy(p)


def test_unit_planner_matches_checker():
    for uw in (W.gpt2_small_units(), W.gpt2_small_units(8, 8), W.llama_2b_units(),
               W.stage3_8p81b_units(), W.stage3_8p81b_units(64, 8)):
        _compare_units(uw.numels, uw.unit_of_tensor, uw.n_units, uw.n_ranks, uw.align_elems)
    rng = random.Random(3)
    for _ in range(300):
        n_t = rng.randint(1, 9)
        n_units = rng.randint(1, n_t)
        uot = list(range(n_units)) + [rng.randrange(n_units) for _ in range(n_t - n_units)]
        rng.shuffle(uot)
        numels = [rng.choice([0, 1, 3, 8, 255, 4096, 10007]) for _ in range(n_t)]
        _compare_units(numels, uot, n_units, rng.choice([1, 2, 3, 8, 13, 64]),
                       rng.choice([1, 2, 8, 64]))


def test_unit_planner_and_gather_reject_bad_arguments():
    for args, status in ((([4], [1], 1, 2, 1), -1), (([4, 4], [0, 0], 2, 2, 1), -1),
                         (([4], [0], 1, 65, 1), -3), (([4], [0], 1, 2, 0), -1),
                         (([4], [0], 1, 2, 8192), -3), (([-4], [0], 1, 2, 1), -1)):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_unit_plan_create(*args)
        assert e.value.status == status
    p = Z.zero_unit_plan_create([100, 50], [0, 1], 2, 4, 1)
    try:
        for lo, hi in ((0, 0), (1, 3), (-1, 1), (2, 1)):
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_gather_units(p, lo, hi, [16] * 4, [16] * 2)
            assert e.value.status == -1
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_gather_units(p, 0, 2, [16, 16, None, 16], [16, 16])
        assert e.value.status == -1
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_gather_units(p, 0, 2, [16, 16, 18, 16], [16, 16])
        assert e.value.status == -2
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_shard_units(p, 0, 2, [16, 24], [16] * 4)
        assert e.value.status == -2
    finally:
        Z.zero_unit_plan_destroy(p)


def test_binding_refuses_short_pointer_lists():
    """The C calls read N (or n_sets * N) entries of every per-rank pointer
    array and cannot see a list's length, so the binding checks it before
    the call. Nothing reaches a device: the check fails first."""
    plan = Z.zero_plan_create([1000], 4, 0, Z.ZERO_BF16)
    try:
        four, eight = [16] * 4, [16] * 8
        hp = Z.ZeroHParams(1e-3, 0.9, 0.999, 1e-8, 0.0, 0.0, 0, 2000, 1.0)
        with pytest.raises(ValueError, match="master"):
            Z.zero_step(plan, 0, 4, four, eight, eight, 2, None, four, 0, 16, hp, 16)
        with pytest.raises(ValueError, match="replicas"):
            Z.zero_step(plan, 0, 4, eight, eight, eight, 2, None, [16] * 3, 0, 16, hp, 16)
        with pytest.raises(ValueError, match="grad_shards"):
            Z.zero_reduce_scatter(plan, -1, 0, 4, four, 0, [16] * 2, 16)
        with pytest.raises(ValueError, match="accum"):
            Z.zero_accumulate(plan, 0, 4, four, [16], 0, True)
    finally:
        Z.zero_plan_destroy(plan)
    uplan = Z.zero_unit_plan_create([10, 20], [0, 1], 2, 4, 1)
    try:
        with pytest.raises(ValueError, match="shards"):
            Z.zero_gather_units(uplan, 0, 2, [16] * 3, [16, 16])
        with pytest.raises(ValueError, match="unit_buffers"):
            Z.zero_gather_units(uplan, 0, 2, four, [16])
    finally:
        Z.zero_unit_plan_destroy(uplan)


def test_binding_accepts_prebuilt_pointer_tables():
    """A caller may build a per-rank pointer table once as a uint64 numpy
    array; lists of int or None marshal to the same values."""
    import numpy as np
    p = Z._ptrs([16, None, 48])
    assert [p[i] for i in range(3)] == [16, None, 48]
    q = Z._ptrs(np.array([16, 0, 48], dtype=np.uint64))
    assert [q[i] for i in range(3)] == [16, None, 48]
    with pytest.raises(ValueError, match="master"):
        Z._ptrs(np.zeros(3, dtype=np.uint64), 4, "master")
