"""Owners split over processes: each process holds the N replicas of its own
window of owners, runs the step on that window and exchanges only the step's
global scalars (the overflow word and, when clipping, the owners' norm
records) with the others over torch.distributed (gloo, through host memory).
The result must equal one process running every owner, bit for bit: master,
m, v and the 16-bit parameters of every window, the scaler (t, scale, norm,
clip coefficient, skip count) and the OR of the bucket flags, including a
step that overflows only in another process's window.

The processes share the one GPU of the box; their kernels never wait on one
another (the exchange is a host all-reduce between steps)."""
import datetime
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from fsdp_sharded_mixed_shard_gb300 import harness, workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _snapshot(g):
    m, mm, v = (t.numpy().copy() for t in g.current_state())
    sc = g.read_scaler()
    return {"lo": g.lo, "hi": g.hi, "master": m, "exp_avg": mm, "exp_avg_sq": v,
            "params": g.params_u16().copy(), "flags": g.flags_u32().copy(),
            "scaler": (sc.t, sc.scale, sc.overflow, sc.n_skipped, sc.good_steps, sc.norm_sq,
                       sc.clip_coef, sc.clip_apply, sc.state_index, sc.error)}


def _run_window(wl, steps, exchange=None):
    g = harness.Group(wl)
    try:
        g.init_state()
        for step in range(1, steps + 1):
            g.gen_grads(step)
            g.step(exchange=exchange)
        return _snapshot(g)
    finally:
        g.close()


def _child(rank, world, port, wl, steps, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as tdist
    from fsdp_sharded_mixed_shard_gb300 import dist as zdist
    try:
        tdist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                                 world_size=world, timeout=datetime.timedelta(seconds=120))
        wins = zdist.windows(wl.n_ranks, world)
        zdist.check_partition(wins, wl.n_ranks)
        lo, hi = wins[rank]
        torch.cuda.set_device(0)
        mine = wl.scaled(rank_lo=lo, rank_hi=hi)
        stream = torch.cuda.current_stream()
        q.put((rank, _run_window(mine, steps, lambda blob: zdist.sum_exchange(blob, stream))))
        tdist.barrier()
        tdist.destroy_process_group()
    except BaseException as e:  # reported to the parent, which fails the test
        q.put((rank, "error: %r" % (e,)))
        raise


def _split_run(wl, steps, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_child, args=(r, world, port, wl, steps, q))
             for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in procs:
            rank, snap = q.get(timeout=600)
            assert not isinstance(snap, str), snap
            out[rank] = snap
    finally:
        for p in procs:
            p.join(timeout=120)
            if p.is_alive():
                p.terminate()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return [out[r] for r in range(world)]


def _compare(whole, parts, S):
    for part in parts:
        a, b = (part["lo"] - whole["lo"]) * S, (part["hi"] - whole["lo"]) * S
        for k in ("master", "exp_avg", "exp_avg_sq"):
            assert np.array_equal(part[k][:b - a].view(np.uint32), whole[k][a:b].view(np.uint32)), k
        assert np.array_equal(part["params"][:b - a], whole["params"][a:b])
        assert part["scaler"] == whole["scaler"], (part["scaler"], whole["scaler"])
    flags = np.bitwise_or.reduce([p["flags"] for p in parts])
    assert np.array_equal(flags, whole["flags"])


CASES = {
    # two-pass with clipping, fp16 under a dynamic scale; at step 2 an +inf
    # in owner 6's slice: only the second process sees it, both skip
    "clip_fp16_inject_other_window": (
        W.Workload("split_clip", [8 * 25_001 - 3], 8, 30_000, False, 61, 1e-4,
                   init_scale=65536.0, dynamic_scale=True, max_grad_norm=0.05, steps=3,
                   inject=(2, 1, 6 * 25_001 + 17, W.FP16_POS_INF)), 2),
    # fused, bf16, a NaN at step 2 in owner 1's slice: the second process
    # re-casts its parameters from the kept state set
    "fused_bf16_inject_other_window": (
        W.Workload("split_fused", [8 * 40_003], 8, 0, True, 62, 1e-3, steps=3,
                   inject=(2, 4, 40_003 + 5, 0x7FC1)), 2),
    # three uneven windows (2, 3, 3 owners), clipping, several buckets
    "clip_three_windows": (
        W.Workload("split_three", [8 * 30_011, 77], 8, 20_000, True, 63, 1e-3,
                   max_grad_norm=0.1, steps=2), 3),
}


@pytest.mark.parametrize("name", list(CASES))
def test_split_windows_equal_one_process(name):
    wl, world = CASES[name]
    whole = _run_window(wl, wl.steps)
    parts = _split_run(wl, wl.steps, world)
    S = (wl.psi + (-wl.psi) % wl.n_ranks) // wl.n_ranks
    _compare(whole, parts, S)
    if wl.inject is not None:
        assert whole["scaler"][3] == 1  # one step skipped everywhere


def _nccl_child(port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as tdist
    from fsdp_sharded_mixed_shard_gb300 import dist as zdist
    try:
        torch.cuda.set_device(0)
        tdist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % port, rank=0,
                                 world_size=1, timeout=datetime.timedelta(seconds=120))
        wl = CASES["clip_fp16_inject_other_window"][0]
        stream = torch.cuda.current_stream()
        snap = _run_window(wl, wl.steps, lambda blob: zdist.sum_exchange(blob, stream))
        # the parameter all-gather's NCCL branch, one rank: the buffer is unchanged
        flat = torch.arange(64, dtype=torch.int16, device="cuda")
        before = flat.clone()
        zdist.all_gather_params(flat, 0, 1, 64, stream)
        torch.cuda.synchronize()
        q.put(("ok", snap, bool(torch.equal(flat, before))))
        tdist.destroy_process_group()
    except BaseException as e:
        q.put(("error: %r" % (e,), None, None))
        raise


def test_exchange_over_nccl_single_rank():
    """The exchange's NCCL branch (an all-reduce on the stream) and the
    parameter all-gather's (all_gather_into_tensor) with a one-rank NCCL
    group: the step equals the one-process step without an exchange, bit
    for bit. One rank waits on nobody; more ranks need more GPUs."""
    wl = CASES["clip_fp16_inject_other_window"][0]
    whole = _run_window(wl, wl.steps)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_nccl_child, args=(_free_port(), q))
    p.start()
    try:
        status, snap, gathered = q.get(timeout=600)
    finally:
        p.join(timeout=120)
        if p.is_alive():
            p.terminate()
    assert status == "ok", status
    assert p.exitcode == 0
    _compare(whole, [snap], (wl.psi + (-wl.psi) % wl.n_ranks) // wl.n_ranks)
    assert gathered
