"""Pins of the checker's stage-3 FSDP unit planner and unit all-gather:
printed page figures (tests/golden/unit_figures.json), brute-force layouts
built with numpy, the one-unit case against the flat planner, and round
trips."""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(__file__)
GOLD = {e["id"]: e for e in json.load(open(os.path.join(HERE, "golden", "unit_figures.json")))
        ["entries"]}


def _uniform_units(psi_total, n_units):
    size = psi_total // n_units
    assert size * n_units == psi_total
    return [size] * n_units, list(range(n_units))


def test_sixty_layers_materialise_one_sixtieth():
    e = GOLD["z3_peak_60_layers"]
    numels, uot = _uniform_units(60 * 1_000_000, e["n_layers"])
    p, _, _, _ = oracle.make_unit_plan(numels, uot, e["n_layers"], 8)
    assert p.max_unit_fraction == pytest.approx(e["fraction"], rel=1e-15)
    # the transient bump is one unit: 2 bytes per element of one layer
    assert p.peak_one_bytes - p.persistent_bytes == 2 * 1_000_000


def test_worked_10b_and_7p5b_persistent_shard():
    for key, n_units in (("z3_worked_10b_n64", 50), ("zf_selfcheck_7p5b_n64", 30)):
        e = GOLD[key]
        numels, uot = _uniform_units(int(e["psi"]), n_units)
        p, _, _, _ = oracle.make_unit_plan(numels, uot, n_units, e["n"])
        assert abs(p.persistent_bytes / 1e9 - e["printed_gb"]) <= e["tol_gb"]
        # no padding needed: exactly 16 psi / N
        assert p.persistent_bytes == 16 * e["psi"] / e["n"]


def test_stage3_wire_volume():
    e = GOLD["sb_stage3_wire_8p81b"]
    # 8.81e9 in 81 units (80 blocks of 110M and a 10M root unit), one rank's view
    numels = [10_000_000] + [110_000_000] * 80
    p, _, _, _ = oracle.make_unit_plan(numels, list(range(81)), 81, 64)
    assert p.psi == int(e["psi"])
    assert p.comm_elems == e["elems_per_param"] * e["psi"]
    assert p.comm_bytes == e["bytes_per_param"] * e["psi"]
    assert abs(p.comm_bytes / 1e9 - e["printed_gb"]) <= e["tol_gb"]
    r = GOLD["sr_layer_native_3psi"]
    assert p.comm_elems / (2 * p.psi) == r["ratio_to_ddp"]
    # each ring collective moves (N - 1) of the N slices per rank
    assert p.ring_bytes == 3 * 2 * 63 * p.shard
    assert p.n_gathers == 2 * 81


def test_block_gathered_bytes_and_state_ladder():
    e = GOLD["sb_block_220mb"]
    block = e["printed_mb"] * 1_000_000 // e["bytes_per_elem"]
    numels = [10_000_000] + [block] * 80
    p, units, _, _ = oracle.make_unit_plan(numels, list(range(81)), 81, 64)
    assert (p.peak_one_bytes - p.persistent_bytes) / 1e6 == e["printed_mb"]
    s = GOLD["sb_states_141_to_2p2"]
    assert abs(16 * s["psi"] / 1e9 - s["printed_full_gb"]) <= 0.5
    assert abs(p.persistent_bytes / 1e9 - s["printed_gb"]) <= s["tol_gb"]


def test_one_or_two_gathered_units():
    assert GOLD["zf_one_or_two_units"]["units_gathered"] == [1, 2]
    numels = [5, 300, 40, 700, 650, 2]
    p, units, _, _ = oracle.make_unit_plan(numels, list(range(6)), 6, 4)
    pads = [u.psi_pad for u in units]
    assert p.peak_one_bytes == p.persistent_bytes + 2 * max(pads)
    pairs = [pads[0]] + [pads[i] + pads[i + 1] for i in range(5)]
    assert p.peak_two_bytes == p.persistent_bytes + 2 * max(pairs)
    assert p.peak_backward_bytes == p.persistent_bytes + 4 * max(pads)
    # a single unit: nothing to prefetch
    q, _, _, _ = oracle.make_unit_plan([123], [0], 1, 4)
    assert q.peak_two_bytes == q.peak_one_bytes


def test_single_unit_is_the_flat_layout():
    rng = np.random.default_rng(5)
    for _ in range(20):
        numels = list(rng.integers(0, 5000, size=int(rng.integers(1, 9))))
        n = int(rng.integers(1, 17))
        flat, offs, _ = oracle.make_plan(numels, n)
        p, units, slots, toff = oracle.make_unit_plan(numels, [0] * len(numels), 1, n)
        u = units[0]
        assert (u.psi, u.pad, u.psi_pad, u.shard) == (flat.psi, flat.pad, flat.psi_pad, flat.shard)
        assert np.array_equal(toff, offs[:len(numels)])
        assert list(slots) == list(range(len(numels)))
        assert p.persistent_bytes == 16 * flat.shard


def _brute_layout(numels, uot, n_units, n, align):
    """numpy restatement: tag every element with a unique 16-bit-safe id,
    concatenate each unit's tensors in list order, pad with zeros, split
    into N equal slices, and concatenate a rank's slices unit by unit."""
    tensors, nxt = [], 1
    for k, c in enumerate(numels):
        tensors.append(np.arange(nxt, nxt + c, dtype=np.int64))
        nxt += c
    fulls, offs = [], {}
    for u in range(n_units):
        parts, pos = [], 0
        for k in range(len(numels)):
            if uot[k] == u:
                offs[k] = pos
                parts.append(tensors[k])
                pos += numels[k]
        flat = np.concatenate(parts) if parts else np.zeros(0, np.int64)
        g = n * align
        padded = -(-len(flat) // g) * g if len(flat) else 0
        flat = np.concatenate([flat, np.zeros(padded - len(flat), np.int64)])
        fulls.append(flat)
    shards = [np.concatenate([f.reshape(n, -1)[r] for f in fulls]) for r in range(n)]
    return tensors, fulls, shards, offs


@pytest.mark.parametrize("align", [1, 8])
def test_brute_force_layout_and_gather(align):
    rng = np.random.default_rng(11 + align)
    for trial in range(40):
        n_t = int(rng.integers(1, 12))
        n_units = int(rng.integers(1, n_t + 1))
        uot = list(rng.permutation(np.concatenate([np.arange(n_units),
                                                   rng.integers(0, n_units, n_t - n_units)])))
        numels = [int(x) for x in rng.integers(0, 3000, size=n_t)]
        if all(numels[k] == 0 for k in range(n_t)):
            numels[0] = 1
        n = int(rng.choice([1, 2, 3, 4, 7, 8, 16]))
        tensors, fulls, bshards, boffs = _brute_layout(numels, uot, n_units, n, align)
        p, units, slots, toff = oracle.make_unit_plan(numels, uot, n_units, n, align)
        assert p.psi == sum(numels)
        assert p.psi_pad == sum(len(f) for f in fulls)
        assert p.shard == len(bshards[0])
        flat_off = held = 0
        for u, f in zip(units, fulls):
            assert u.psi_pad == len(f) and u.psi_pad % (n * align) == 0
            assert 0 <= u.pad < n * align
            assert u.shard * n == u.psi_pad
            assert u.flat_offset == flat_off and u.shard_offset == held
            flat_off += u.psi_pad
            held += u.shard
        for k in range(n_t):
            assert toff[k] == boffs[k]
        for u_i, u in enumerate(units):
            members = [int(x) for x in slots[u.first_slot:u.first_slot + u.n_tensors]]
            assert members == [k for k in range(n_t) if uot[k] == u_i]
        # gather from shards built by the brute force: the unit's full copy
        shards16 = [s.astype(np.uint16) for s in bshards]
        for u_i, u in enumerate(units):
            full = oracle.gather_unit(u, shards16)
            assert np.array_equal(full, fulls[u_i].astype(np.uint16))
            for k in range(n_t):
                if uot[k] == u_i:
                    seg = full[toff[k]:toff[k] + numels[k]]
                    assert np.array_equal(seg, tensors[k].astype(np.uint16))
        # shard_unit is the inverse of gather_unit
        back = [np.zeros(p.shard, np.uint16) for _ in range(n)]
        for u_i, u in enumerate(units):
            oracle.shard_unit(u, fulls[u_i].astype(np.uint16), back)
        for a, b in zip(back, shards16):
            assert np.array_equal(a, b)


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.make_unit_plan([3, 4], [0, 2], 2, 4)      # unit id out of range
    with pytest.raises(ValueError):
        oracle.make_unit_plan([3, 4], [0, 0], 2, 4)      # unit 1 has no tensor
    with pytest.raises(ValueError):
        oracle.make_unit_plan([3], [0], 1, 0)            # no ranks
    with pytest.raises(ValueError):
        oracle.make_unit_plan([3], [0], 1, 4, 0)         # align < 1
