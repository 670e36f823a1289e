"""Pins of the checker's planner and accounting against the pages' printed
figures (tests/golden/page_figures.json) and brute force."""
import json
import os
import random

import pytest

import oracle
from fsdp_sharded_mixed_shard_gb300 import workloads as W

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))
STAGE = {"ddp": 0, "z1": 1, "z2": 2, "z3": 3}


@pytest.mark.parametrize("e", GOLD["bills"], ids=lambda e: e["id"])
def test_bills_match_printed_figures(e):
    got = oracle.bills(e["psi"], e["n"])[STAGE[e["stage"]]] / 1e9
    assert abs(got - e["printed_gb"]) <= e["tol_gb"], (e["id"], got)


@pytest.mark.parametrize("e", GOLD["ring"], ids=lambda e: e["id"])
def test_ring_bytes_match_printed_figures(e):
    got = oracle.ring_bytes(e["m_gb"] * 1e9, e["d"]) / 1e9
    assert abs(got - e["printed_gb"]) <= e["tol_gb"], (e["id"], got)


def test_ring_hops_and_bound():
    e = GOLD["hops"][0]
    p, _, _ = oracle.make_plan([1000], e["d"])
    assert p.ring_hops == e["printed"]
    # bytes sent per rank stay below 2M for every ring size
    for d in (2, 3, 8, 64, 1024):
        assert oracle.ring_bytes(1e9, d) < 2e9
    assert oracle.ring_bytes(1e9, 1) == 0.0


@pytest.mark.parametrize("e", GOLD["wire"], ids=lambda e: e["id"])
def test_wire_volume_matches_printed_figures(e):
    p, _, _ = oracle.make_plan([int(e["psi"])], 8)
    elems = {"z2": p.comm_z2, "z3": p.comm_z3}[e["stage"]]
    got = elems * e["bytes_per_elem"] / 1e9
    assert abs(got - e["printed_gb"]) <= e["tol_gb"], (e["id"], got)


def test_grad_bytes_printed():
    e = GOLD["grad_bytes"][0]
    assert abs(e["psi"] * e["bytes_per_param"] / 1e9 - e["printed_gb"]) <= e["tol_gb"]


def test_bill_formulas_exact_special_cases():
    # N = 1: every stage equals plain data parallelism (16 bytes/param)
    b = oracle.bills(1e6, 1)
    assert b == [16e6, 16e6, 16e6, 16e6]
    # stage 3 divides the whole bill by N
    for n in (2, 8, 64):
        b = oracle.bills(7.5e9, n)
        assert b[3] * n == pytest.approx(b[0], rel=1e-15)
        # stage floors as N grows: 4 psi and 2 psi
        assert b[1] > 4 * 7.5e9 and b[2] > 2 * 7.5e9
    # exact worked values (N = 64 is a power of two: exact in fp64)
    b = oracle.bills(7.5e9, 64)
    assert b == [120e9, 31.40625e9, 16.640625e9, 1.875e9]


def _brute_plan(numels, n, bsz):
    psi = sum(numels)
    pad = (-psi) % n
    psip = psi + pad
    S = psip // n
    owner = [j // S for j in range(psip)] if S else []
    bucket = [(j // bsz if bsz else 0) for j in range(psip)]
    segs = []
    for j in range(psip):
        key = (bucket[j], owner[j])
        if segs and segs[-1][3] == key[0] and segs[-1][2] == key[1] and segs[-1][1] == j:
            segs[-1][1] = j + 1
        else:
            segs.append([j, j + 1, key[1], key[0]])
    return psi, pad, psip, S, [tuple(s) for s in segs]


def test_plan_brute_force_small():
    rng = random.Random(1234)
    for trial in range(300):
        n = rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 64])
        numels = [rng.choice([0, 1, 2, 3, 7, 31, 64, 100]) for _ in range(rng.randint(0, 6))]
        bsz = rng.choice([0, 1, 3, 5, 16, 37, 1000])
        p, offs, segs = oracle.make_plan(numels, n, bsz)
        psi, pad, psip, S, bsegs = _brute_plan(numels, n, bsz)
        assert (p.psi, p.pad, p.psi_pad, p.shard) == (psi, pad, psip, S)
        assert list(offs) == [sum(numels[:k]) for k in range(len(numels))]
        assert [tuple(s) for s in segs] == bsegs, (numels, n, bsz)
        nb = 0 if psip == 0 else (1 if bsz == 0 else -(-psip // bsz))
        assert p.n_buckets == nb


def test_plan_segments_tile_exactly_once():
    for numels, n, bsz in [([1_000_003], 4, 0), (W.gpt2_small_numels(), 8, 25_000_000),
                           (W.llama_2b_numels(), 16, 50_000_000), ([12345], 7, 1000)]:
        p, _, segs = oracle.make_plan(numels, n, bsz)
        pos = 0
        for lo, hi, r, k in segs:
            assert lo == pos and hi > lo
            assert r * p.shard <= lo and hi <= (r + 1) * p.shard
            if bsz:
                assert k * bsz <= lo and hi <= min((k + 1) * bsz, p.psi_pad)
            pos = hi
        assert pos == p.psi_pad


def test_workload_plans():
    p, _, _ = oracle.make_plan(W.TINY_FLAT.numels, 4)
    assert (p.pad, p.psi_pad, p.shard) == (1, 1_000_004, 250_001)
    p, _, segs = oracle.make_plan(W.GPT2_SMALL.numels, 8, 25_000_000)
    assert p.psi == 124_439_808 and p.pad == 0 and p.shard == 15_554_976 and p.n_buckets == 5
    p, _, _ = oracle.make_plan(W.FLAT_1P5B.numels, 8)
    assert p.shard == 187_500_000
    p, _, _ = oracle.make_plan(W.STAGE3_SLICE.numels, 64)
    assert p.shard == 137_656_250 and p.pad == 0
    assert p.bill_z3 / 1e9 == pytest.approx(2.2025, rel=1e-12)
    p, _, _ = oracle.make_plan(W.LLAMA_2B.numels, 16, 50_000_000)
    assert p.psi == 1_336_477_696 and p.shard == 83_529_856 and p.n_buckets == 27


def test_plan_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.make_plan([10], 0)
    with pytest.raises(ValueError):
        oracle.make_plan([-1], 2)
    with pytest.raises(ValueError):
        oracle.make_plan([10], 2, -5)


def test_empty_plan():
    p, offs, segs = oracle.make_plan([], 4)
    assert (p.psi, p.psi_pad, p.shard, p.n_buckets, p.n_segments) == (0, 0, 0, 0, 0)
    p, offs, segs = oracle.make_plan([0, 0], 3, 10)
    assert list(offs) == [0, 0] and segs == []
