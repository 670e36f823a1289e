"""Pins of the checker's sharding-strategy accounting (FULL_SHARD,
SHARD_GRAD_OP, NO_SHARD, HYBRID_SHARD, no reshard after forward): printed
page figures, equality with the pinned flat-plan bills and ring formula, and
a literal ring simulation that counts what every rank sends."""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(__file__)
GOLD = {e["id"]: e for e in json.load(open(os.path.join(HERE, "golden", "unit_figures.json")))
        ["entries"]}
NAMES = {"FULL_SHARD": oracle.FULL_SHARD, "SHARD_GRAD_OP": oracle.SHARD_GRAD_OP,
         "NO_SHARD": oracle.NO_SHARD, "HYBRID_SHARD": oracle.HYBRID_SHARD,
         "NO_RESHARD_AFTER_FORWARD": oracle.NO_RESHARD_AFTER_FORWARD}


def _layout_8p81b(n=64):
    return oracle.make_unit_plan([10_000_000] + [110_000_000] * 80, list(range(81)), 81, n)[0]


def test_strategies_are_the_stage_bills():
    """FULL_SHARD = stage 3, SHARD_GRAD_OP = stage 2, NO_SHARD = DDP (the
    flat planner's bills, themselves pinned to the printed 7.5B figures)."""
    e = GOLD["zf_strategy_names"]
    for psi, n in ((7.5e9, 64), (1.5e9, 8), (8.81e9, 64)):
        blocks = 50
        p, _, _, _ = oracle.make_unit_plan([int(psi) // blocks] * blocks, list(range(blocks)),
                                           blocks, n)
        assert p.psi_pad == p.psi  # no padding: the closed forms apply exactly
        flat, _, _ = oracle.make_plan([int(psi)], n)
        bill = {"z3": flat.bill_z3, "z2": flat.bill_z2, "ddp": flat.bill_ddp}
        for name, stage in e["map"].items():
            c = oracle.strategy_cost(p, NAMES[name])
            assert c.persistent_bytes == pytest.approx(bill[stage], rel=1e-15)


def test_wire_volumes_match_the_printed_figures():
    p = _layout_8p81b()
    s3 = GOLD["sb_stage3_wire_8p81b"]
    s2 = GOLD["sb_stage2_wire_8p81b"]
    full = oracle.strategy_cost(p, oracle.FULL_SHARD)
    grad_op = oracle.strategy_cost(p, oracle.SHARD_GRAD_OP)
    ddp = oracle.strategy_cost(p, oracle.NO_SHARD)
    assert full.comm_elems == s3["elems_per_param"] * s3["psi"]
    assert abs(2 * full.comm_elems / 1e9 - s3["printed_gb"]) <= s3["tol_gb"]
    for c in (grad_op, ddp):
        assert c.comm_elems == s2["elems_per_param"] * s2["psi"]
        assert abs(2 * c.comm_elems / 1e9 - s2["printed_gb"]) <= s2["tol_gb"]
    assert full.gathers_per_unit == 2 and grad_op.gathers_per_unit == 1


def test_llama3_no_reshard_is_stage3_memory_stage2_traffic():
    e = GOLD["sb_llama3_no_reshard"]
    p = _layout_8p81b()
    nr = oracle.strategy_cost(p, oracle.NO_RESHARD_AFTER_FORWARD)
    mem = oracle.strategy_cost(p, NAMES[e["memory_like"]])
    wire = oracle.strategy_cost(p, NAMES[e["traffic_like"]])
    assert nr.persistent_bytes == mem.persistent_bytes
    assert nr.comm_elems == wire.comm_elems and nr.ring_bytes == wire.ring_bytes
    s = GOLD["sb_states_141_to_2p2"]
    assert abs(nr.persistent_bytes / 1e9 - s["printed_gb"]) <= s["tol_gb"]
    # every unit gathered in the forward pass is still held at the turn
    assert nr.peak_bytes == nr.persistent_bytes + 2 * p.psi_pad
    assert nr.gathers_per_unit == 1


def test_no_shard_ring_is_the_printed_all_reduce():
    e = GOLD["sb_ring_30p8"]
    psi = int(e["grad_gb"] * 1e9 / 2)        # 16-bit gradient of 17.6 GB
    p, _, _, _ = oracle.make_unit_plan([psi], [0], 1, e["d"])
    c = oracle.strategy_cost(p, oracle.NO_SHARD)
    assert abs(c.ring_bytes / 1e9 - e["printed_gb"]) <= e["tol_gb"]
    assert c.ring_bytes < e["bound_gb"] * 1e9
    assert c.ring_bytes == oracle.ring_bytes(2.0 * psi, e["d"])


def test_hybrid_of_one_group_is_full_shard_and_hybrid_memory_is_per_group():
    p = _layout_8p81b(8)      # shard group = one node of 8
    full = oracle.strategy_cost(p, oracle.FULL_SHARD)
    one = oracle.strategy_cost(p, oracle.HYBRID_SHARD, 1)
    for f in ("persistent_bytes", "peak_bytes", "comm_elems", "comm_elems_inter", "ring_bytes",
              "ring_bytes_inter", "shard_ranks", "gathers_per_unit"):
        assert getattr(one, f) == getattr(full, f), f
    h = oracle.strategy_cost(p, oracle.HYBRID_SHARD, 8)   # 64 ranks as 8 nodes x 8
    assert h.persistent_bytes == 16 * p.shard == 16 * 8.81e9 / 8
    assert h.comm_elems_inter == 2 * p.shard
    # more memory than FULL_SHARD over all 64 ranks, less inter-node traffic
    p64 = _layout_8p81b(64)
    f64 = oracle.strategy_cost(p64, oracle.FULL_SHARD)
    assert h.persistent_bytes == 8 * f64.persistent_bytes
    assert h.ring_bytes_inter < f64.ring_bytes


# ---------------------------------------------------------------- ring ------

def _ring_all_gather(chunks):
    """chunks[i] starts on rank i; returns (what every rank holds, elements
    each rank sent). Step k: rank i forwards chunk (i - k) mod g to i + 1."""
    g = len(chunks)
    have = [{i: chunks[i]} for i in range(g)]
    sent = [0] * g
    for k in range(g - 1):
        msgs = [(i, (i - k) % g) for i in range(g)]
        for i, c in msgs:
            have[(i + 1) % g][c] = have[i][c]
            sent[i] += len(have[i][c])
    return [np.concatenate([h[c] for c in range(g)]) for h in have], sent


def _ring_reduce_scatter(vals):
    """vals[i] is rank i's full vector, cut into g chunks; afterwards rank i
    holds the sum of chunk i. Step k: rank i sends its running partial of
    chunk (i - k - 1) mod g to rank i + 1."""
    g = len(vals)
    parts = [np.array_split(v.astype(np.float64), g) for v in vals]
    sent = [0] * g
    for k in range(g - 1):
        msgs = [(i, (i - k - 1) % g, parts[i][(i - k - 1) % g].copy()) for i in range(g)]
        for i, c, data in msgs:
            parts[(i + 1) % g][c] = parts[(i + 1) % g][c] + data
            sent[i] += len(data)
    return [parts[i][i] for i in range(g)], sent


@pytest.mark.parametrize("g,R", [(2, 1), (4, 1), (4, 2), (2, 4), (3, 3), (8, 2)])
def test_ring_bytes_by_literal_simulation(g, R):
    """Simulate one stage-3 step of a tiny model (three units) on a g x R
    rank grid and count the elements every rank sends: two all-gathers and a
    reduce-scatter per unit inside its group, then an all-reduce (reduce-
    scatter + all-gather) of each rank's reduced shard across the R groups.
    Every simulated collective's result is checked too."""
    rng = np.random.default_rng(g * 10 + R)
    numels = [5 * g * R, 3 * g * R + 1, 7]
    p, units, _, _ = oracle.make_unit_plan(numels, [0, 1, 2], 3, g, R)  # shard divisible by R
    assert p.shard % R == 0
    sent = np.zeros((R, g), np.int64)
    for u in units:
        full = rng.integers(0, 1000, size=u.psi_pad)
        slices = [full[i * u.shard:(i + 1) * u.shard] for i in range(g)]
        for grp in range(R):
            for _ in range(2):  # forward and backward gathers
                got, s = _ring_all_gather(slices)
                assert all(np.array_equal(x, full) for x in got)
                sent[grp] += s
            grads = [rng.integers(0, 100, size=u.psi_pad) for _ in range(g)]
            red, s = _ring_reduce_scatter(grads)
            total = np.sum(grads, axis=0)
            for i in range(g):
                assert np.array_equal(red[i], np.array_split(total, g)[i])
            sent[grp] += s
    # all-reduce across the R groups of each rank's S held gradient elements
    if R > 1:
        for i in range(g):
            vecs = [rng.integers(0, 100, size=p.shard) for _ in range(R)]
            red, s1 = _ring_reduce_scatter(vecs)
            got, s2 = _ring_all_gather(red)
            assert all(np.array_equal(x, np.sum(vecs, axis=0)) for x in got)
            for grp in range(R):
                sent[grp, i] += s1[grp] + s2[grp]
    c = oracle.strategy_cost(p, oracle.HYBRID_SHARD, R)
    assert np.all(sent * 2 == c.ring_bytes)
    inter = 2.0 * (R - 1) / R * 2 * p.shard
    assert c.ring_bytes_inter == inter


def test_rejects_bad_arguments():
    p = _layout_8p81b(8)
    with pytest.raises(ValueError):
        oracle.strategy_cost(p, 7)
    with pytest.raises(ValueError):
        oracle.strategy_cost(p, oracle.FULL_SHARD, 2)
    with pytest.raises(ValueError):
        oracle.strategy_cost(p, oracle.HYBRID_SHARD, 0)
