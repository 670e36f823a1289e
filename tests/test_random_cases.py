"""The random-shape parity cases (drawn on the CPU from a fixed seed) cover
what they are meant to: owners at most phases of the 8-element grid, rank
windows that do not start at 0, micro-batches and both paths."""
import oracle
from parity_util import random_case

N_CASES = 96   # as in test_gpu_random_shapes.py


def test_random_cases_cover_the_grid_phases():
    phases, windows, micro, clipped = set(), 0, 0, 0
    for i in range(N_CASES):
        c = random_case(i)
        p, _, _ = oracle.make_plan(c["numels"], c["n"], c["bucket"])
        for r in range(c["lo"], c["hi"]):
            phases.add(((r - c["lo"]) * p.shard) % 8)
        windows += c["lo"] > 0
        micro += c["micro"] > 1
        clipped += c["clip"] > 0
    assert len(phases) == 8 and windows >= 20 and micro >= 20 and clipped >= 20


def test_random_cases_are_reproducible():
    assert random_case(7) == random_case(7)
    assert random_case(7) != random_case(8)
