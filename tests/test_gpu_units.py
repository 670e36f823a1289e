"""GPU parity of the stage-3 unit all-gather and its inverse (zero_gather_units,
zero_shard_units) against the CPU checker, byte for byte: small layouts that
cover both alignments, every 16-byte phase, ragged slices, empty units,
more than one launch's worth of slices, and the full 8.81B-parameter layout
at 64 ranks on sampled units."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import fsdp_sharded_mixed_shard_gb300 as Z
from fsdp_sharded_mixed_shard_gb300 import harness, workloads as W

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A5A


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _r8(x):
    return (x + 7) // 8 * 8


def _tiny_transformer_units(layers=3, d=64, vocab=503, ctx=128):
    numels = [vocab * d, ctx * d]
    for _ in range(layers):
        numels += [d, d, d * 3 * d, 3 * d, d * d, d, d, d, d * 4 * d, 4 * d, 4 * d * d, d]
    numels += [d, d]
    root = {0, 1, len(numels) - 2, len(numels) - 1}
    uot, b = [], 0
    for k in range(len(numels)):
        if k in root:
            uot.append(0)
        else:
            uot.append(1 + b // 12)
            b += 1
    return numels, uot, 1 + layers


CASES = {
    "tiny_transformer_n8_a1": _tiny_transformer_units() + (8, 1),
    "tiny_transformer_n8_a8": _tiny_transformer_units() + (8, 8),
    # ragged sizes: every rank's slice lands on a different 16-byte phase
    "ragged_n3_a1": ([1, 3, 5, 7, 1001, 4097, 3, 11], [0, 1, 1, 2, 3, 2, 4, 0], 5, 3, 1),
    "ragged_n7_a2": ([1, 3, 5, 7, 1001, 4097, 3, 11], [0, 1, 1, 2, 3, 2, 4, 0], 5, 7, 2),
    # a unit whose tensors are all empty, and a one-element unit
    "empty_unit_n4": ([0, 0, 17, 1, 90001], [1, 1, 0, 2, 3], 4, 4, 1),
    # 64 ranks x 5 units = 320 slices: more than one launch
    "many_slices_n64": ([100_003, 99_991, 64, 200_000, 12_345], [0, 1, 2, 3, 4], 5, 64, 1),
    # one rank (a plain copy) and a slice spanning hundreds of tiles
    "single_rank": ([3_000_001, 5], [0, 1], 2, 1, 1),
    "long_slices_n2": ([3_000_001, 7], [0, 0], 1, 2, 1),
}


def _setup(case, rng):
    numels, uot, n_units, n, align = case
    plan = Z.zero_unit_plan_create(numels, uot, n_units, n, align)
    info = Z.zero_unit_plan_get_info(plan)
    _, ounits, _, _ = oracle.make_unit_plan(numels, uot, n_units, n, align)
    row = _r8(max(info.shard_elems, 1))
    host = [rng.integers(0, 65536, size=row, dtype=np.uint16) for _ in range(n)]
    dev = torch.from_numpy(np.stack(host).view(np.int16)).cuda()
    return plan, info, ounits, host, dev, row


@pytest.mark.parametrize("name", sorted(CASES))
def test_gather_matches_checker(name):
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    plan, info, ounits, host, dev, row = _setup(CASES[name], rng)
    try:
        n = info.n_ranks
        shard_ptrs = [dev.data_ptr() + r * row * 2 for r in range(n)]
        # one buffer per unit with 8 guard elements past the end
        bufs = [torch.full((_r8(u.psi_pad) + 8,), SENTINEL, dtype=torch.int16, device="cuda")
                for u in ounits]
        # windows of 1..3 units over all units
        lo = 0
        while lo < info.n_units:
            hi = min(info.n_units, lo + int(rng.integers(1, 4)))
            Z.zero_gather_units(plan, lo, hi, shard_ptrs, [b.data_ptr() for b in bufs[lo:hi]])
            lo = hi
        torch.cuda.synchronize()
        for u, b in zip(ounits, bufs):
            got = b.cpu().numpy().view(np.uint16)
            want = oracle.gather_unit(u, host)
            assert np.array_equal(got[:u.psi_pad], want)
            assert np.all(got[u.psi_pad:] == SENTINEL)   # nothing written past the unit
        # the shards are read only
        assert np.array_equal(dev.cpu().numpy().view(np.uint16), np.stack(host))
    finally:
        Z.zero_unit_plan_destroy(plan)


@pytest.mark.parametrize("name", sorted(CASES))
def test_shard_matches_checker(name):
    rng = np.random.default_rng(1 + zlib.crc32(name.encode()))
    plan, info, ounits, host, dev, row = _setup(CASES[name], rng)
    try:
        n = info.n_ranks
        shard_ptrs = [dev.data_ptr() + r * row * 2 for r in range(n)]
        fulls = [rng.integers(0, 65536, size=max(u.psi_pad, 1), dtype=np.uint16) for u in ounits]
        bufs = [torch.from_numpy(np.concatenate([f, np.zeros(8, np.uint16)]).view(np.int16))
                .cuda() for f in fulls]
        # scatter every unit back in one call
        Z.zero_shard_units(plan, 0, info.n_units, [b.data_ptr() for b in bufs], shard_ptrs)
        torch.cuda.synchronize()
        want = [h.copy() for h in host]
        for u, f in zip(ounits, fulls):
            if u.psi_pad:
                oracle.shard_unit(u, f[:u.psi_pad], want)
        got = dev.cpu().numpy().view(np.uint16)
        for r in range(n):
            assert np.array_equal(got[r], want[r])   # including the untouched row tail
    finally:
        Z.zero_unit_plan_destroy(plan)


def test_gather_then_shard_round_trip_on_gpt2_units():
    uw = W.gpt2_small_units(8, 1)
    g = harness.UnitGroup(uw, window=1)
    try:
        g.fill_shards()
        torch.cuda.synchronize()   # the fill runs on the group's stream
        before = g.shards.clone()
        for u in range(uw.n_units):
            g.gather(u, u + 1)
            g.shard(u, u + 1)
        torch.cuda.synchronize()
        assert torch.equal(before, g.shards)
    finally:
        g.close()


@pytest.mark.parametrize("align", [1, 8])
def test_full_size_8p81b_units_sampled(align):
    """The 8.81B-parameter share at 64 ranks (17.6 GB of shards): gather the
    root unit with the first block, then the last block, and compare each
    whole gathered unit with the checker run on host copies of its slices."""
    uw = W.stage3_8p81b_units(64, align)
    g = harness.UnitGroup(uw, window=2)
    try:
        g.fill_shards()
        torch.cuda.synchronize()
        _, ounits, _, _ = oracle.make_unit_plan(uw.numels, uw.unit_of_tensor, uw.n_units, 64,
                                                align)
        for lo, hi in ((0, 2), (80, 81)):
            g.gather(lo, hi)
            torch.cuda.synchronize()
            for i, u in enumerate(range(lo, hi)):
                ou = ounits[u]
                sl = g.shards[:, ou.shard_offset:ou.shard_offset + ou.shard].cpu().numpy()
                slices = [np.ascontiguousarray(sl[r]).view(np.uint16) for r in range(64)]
                local = oracle.Unit(ou.psi, ou.pad, ou.psi_pad, ou.shard, 0, 0, ou.n_tensors, 0)
                want = oracle.gather_unit(local, slices)
                got = g.buffers[i, :ou.psi_pad].cpu().numpy().view(np.uint16)
                assert np.array_equal(got, want)
    finally:
        g.close()
