"""Runs GPU parity cases through libzero_checked.so in its own process (the
library variant is fixed per process) and prints one JSON line per case
with the violations the kernels recorded. Used by tests/test_gpu_checked.py."""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import fsdp_sharded_mixed_shard_gb300 as Z  # noqa: E402

Z.use_checked_library()

from fsdp_sharded_mixed_shard_gb300 import workloads as W  # noqa: E402
from parity_util import random_workload, run_small  # noqa: E402


def tiny_transformer_numels(d=64, vocab=503, ctx=128, layers=3):
    out = [vocab * d, ctx * d]
    for _ in range(layers):
        out += [d, d, d * 3 * d, 3 * d, d * d, d, d, d, d * 4 * d, 4 * d, 4 * d * d, d]
    return out + [d, d]


def cases():
    t = tiny_transformer_numels()
    yield "fused_bf16_n8", dict(wl=W.GPT2_SMALL.scaled(numels=t, bucket_elems=50_000, steps=2))
    yield "two_pass_clip_fp16_n8", dict(wl=W.GPT2_SMALL.scaled(
        numels=t, bucket_elems=50_000, steps=2, is_bf16=False, max_grad_norm=0.5,
        init_scale=1024.0))
    yield "two_pass_clip_n16", dict(wl=W.GPT2_SMALL.scaled(
        numels=t, n_ranks=16, bucket_elems=0, steps=2, max_grad_norm=0.5))
    yield "fused_n64_ragged", dict(wl=W.Workload("n64", [300_007], 64, 0, True, 5, 1e-3,
                                                 steps=2))
    yield "rank_subset_window", dict(wl=W.Workload("subset", [200_003], 8, 0, True, 7, 1e-3,
                                                   steps=2, rank_lo=3, rank_hi=6))
    yield "micro_batches_two_pass", dict(wl=W.GPT2_SMALL.scaled(
        numels=t, bucket_elems=0, steps=2, max_grad_norm=0.5, n_micro=3))
    yield "odd_shard_scalar_paths", dict(wl=W.TINY_FLAT.scaled(numels=[100_003], steps=2))
    yield "odd_shard_two_pass_n8", dict(wl=W.Workload("odd2", [8 * 25_001 - 3], 8, 0, True, 9,
                                                      1e-3, steps=2, max_grad_norm=0.5))
    yield "odd_shard_micro_fused_n8", dict(wl=W.Workload("oddm", [8 * 25_001 - 5], 8, 0, True,
                                                         13, 1e-3, steps=2, n_micro=3))
    yield "shard_4_mod_8_fused_n64", dict(wl=W.Workload("s4", [64 * 3_004], 64, 0, True, 11,
                                                        1e-3, steps=2))
    yield "short_step_overflow_recast_n12", dict(wl=W.Workload(
        "sov", [12 * 20_002], 12, 0, False, 17, 1e-3, init_scale=1000.0, dynamic_scale=True,
        steps=3, inject=(2, 11, 12 * 20_002 - 1, 0xFC00)))


def gather_case():
    """All-gather and shard every unit of a pad-to-N layout whose slices sit
    at every 16-byte phase; compare with the checker byte for byte."""
    import numpy as np
    import torch
    import oracle
    from fsdp_sharded_mixed_shard_gb300 import harness
    uw = W.UnitWorkload("ragged_units", [1, 3, 5, 7, 1001, 40_097, 3, 11, 77_777],
                        [0, 1, 1, 2, 3, 2, 4, 0, 4], 5, 7, 1, seed=3)
    g = harness.UnitGroup(uw, window=1)
    g.fill_shards()
    torch.cuda.synchronize()
    shards = [np.ascontiguousarray(g.shards[r].cpu().numpy().view(np.uint16)) for r in range(7)]
    _, units, _, _ = oracle.make_unit_plan(uw.numels, uw.unit_of_tensor, uw.n_units, 7, 1)
    for u, ou in enumerate(units):
        g.gather(u, u + 1)
        torch.cuda.synchronize()
        got = g.buffers[0, :ou.psi_pad].cpu().numpy().view(np.uint16)
        assert np.array_equal(got, oracle.gather_unit(ou, shards)), u
        g.shard(u, u + 1)
    torch.cuda.synchronize()
    assert all(np.array_equal(g.shards[r].cpu().numpy().view(np.uint16), shards[r])
               for r in range(7))
    g.close()


def norm_entries_case():
    """The norm entry points on many segments: the workspace form, the
    no-allocation form (records in the library's fixed array, numbered from
    the call's first tile, several launches) over all owners and then over a
    window, and the export / import pair; the forms must agree bit for bit."""
    import torch
    from fsdp_sharded_mixed_shard_gb300 import harness
    numels = [97 + (k * 37) % 500 for k in range(400)]
    wl = W.Workload("noalloc_chk", numels, 8, 101, True, 33, 1e-2, max_grad_norm=0.1, steps=1)
    g = harness.Group(wl)
    g.init_state()
    g.gen_grads(1)
    sc, ws, st = g.scaler.data_ptr(), g.workspace.data_ptr(), g.sptr
    Z.zero_reduce_scatter(g.plan, -1, 0, 8, g.rep_ptrs(), 0, g.ghat_ptrs(), sc, 0, ws, st)
    ex = g.exchange.data_ptr()
    Z.zero_grad_norm_local(g.plan, 0, 8, None, g.hp, sc, ws, ex, st)
    Z.zero_grad_norm_apply(g.plan, ex, g.hp, sc, st)
    for lo, hi in ((0, 8), (3, 8)):
        Z.zero_grad_norm(g.plan, lo, hi, g.ghat_ptrs(), g.hp, sc, ws, st)
        want = g.read_scaler().norm_sq
        Z.zero_grad_norm_noalloc(g.plan, lo, hi, g.ghat_ptrs(), g.hp, sc, st)
        assert g.read_scaler().norm_sq == want, (lo, hi)
    torch.cuda.synchronize()
    g.close()


def main():
    Z.zero_selftest_check()
    n, first = Z.zero_checked_status()
    print(json.dumps({"case": "selftest", "violations": n, "first": first}), flush=True)
    for name, kw in cases():
        run_small(kw["wl"])
        n, first = Z.zero_checked_status()
        print(json.dumps({"case": name, "violations": n, "first": first}), flush=True)
    # the first 24 random shapes of the random-shape parity test
    for i in range(24):
        wl, per_bucket, two_pass = random_workload(i)
        run_small(wl, per_bucket=per_bucket, two_pass=two_pass)
    n, first = Z.zero_checked_status()
    print(json.dumps({"case": "random_shapes_24", "violations": n, "first": first}), flush=True)
    gather_case()
    n, first = Z.zero_checked_status()
    print(json.dumps({"case": "unit_gather", "violations": n, "first": first}), flush=True)
    norm_entries_case()
    n, first = Z.zero_checked_status()
    print(json.dumps({"case": "norm_entries", "violations": n, "first": first}), flush=True)
    print(json.dumps({"case": "library", "path": Z._build.ZERO_CHECKED_LIB,
                      "loaded": Z.lib()._name}), flush=True)


if __name__ == "__main__":
    main()
