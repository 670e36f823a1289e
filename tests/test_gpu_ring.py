"""The ring reduce-scatter with the ranks in separate processes, one 16-bit
gradient replica each ("How far does splitting the batch get you?", "Why
does the all-reduce not get more expensive with more ranks?"): every hop's
arithmetic in libzero's zero_ring_hop, the fp32 partials passed between
neighbours over torch.distributed (gloo, through host memory: the processes
share the box's one GPU and no kernel waits on another process), then the
scalar exchange, the update of each rank's slice and the all-gather of the
parameters. The result must equal one process reducing all N replicas
resident on the GPU, bit for bit: every rank's master, m, v, all 16-bit
parameters, the scaler, and the OR of the bucket flags, including a step
skipped for a +inf in one replica.

The one-process reference recomputes the norm records from the reduced
gradients (zero_grad_norm with grad_shards), as the ring path does, so the
two norms are formed from identical records."""
import datetime
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import fsdp_sharded_mixed_shard_gb300 as Z
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


def _rank_proc(rank, world, port, wl, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as tdist
    from fsdp_sharded_mixed_shard_gb300 import dist as zdist
    try:
        tdist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                                 world_size=world, timeout=datetime.timedelta(seconds=120))
        torch.cuda.set_device(0)
        g = harness.RingRank(wl, rank)
        g.init_state()
        zdist.all_gather_params(g.flat, rank, world, g.S, g.stream)
        for step in range(1, wl.steps + 1):
            g.gen_grads(step)
            g.step()
        m, mm, v = (t.numpy().copy() for t in g.current_state())
        sc = g.read_scaler()
        q.put((rank, {"master": m, "exp_avg": mm, "exp_avg_sq": v,
                      "params": g.flat[:g.info.psi_pad].cpu().numpy().view(np.uint16).copy(),
                      "flags": g.flags[:g.info.n_buckets].cpu().numpy().view(np.uint32).copy(),
                      "scaler": _scaler_fields(sc)}))
        g.close()
        tdist.barrier()
        tdist.destroy_process_group()
    except BaseException as e:
        q.put((rank, "error: %r" % (e,)))
        raise


def _scaler_fields(sc):
    return (sc.t, sc.scale, sc.overflow, sc.n_skipped, sc.good_steps, sc.norm_sq, sc.clip_coef,
            sc.clip_apply, sc.state_index, sc.error)


def _one_process(wl):
    """All N replicas on the GPU, reduced in one launch; the norm from
    records recomputed from the reduced gradients."""
    g = harness.Group(wl, two_pass=True)
    try:
        g.init_state()
        st, sc, ws = g.sptr, g.scaler.data_ptr(), g.workspace.data_ptr()
        clip = wl.max_grad_norm > 0
        flags = []
        for step in range(1, wl.steps + 1):
            g.gen_grads(step)
            g.flags.zero_()
            Z.zero_reduce_scatter(g.plan, -1, 0, g.N, g.rep_ptrs(), 0, g.ghat_ptrs(), sc,
                                  g.flags.data_ptr(), 0, st)
            if clip:
                Z.zero_grad_norm(g.plan, 0, g.N, g.ghat_ptrs(), g.hp, sc, ws, st)
            Z.zero_step(g.plan, 0, g.N, g._state_ptrs(0), g._state_ptrs(1), g._state_ptrs(2),
                        g.n_sets, g.ghat_ptrs(), None, 0, g.flat.data_ptr(), g.hp, sc,
                        g.flags.data_ptr(), st)
            flags.append(g.flags_u32().copy())
        m, mm, v = (t.numpy().copy() for t in g.current_state())
        return {"master": m, "exp_avg": mm, "exp_avg_sq": v, "params": g.params_u16().copy(),
                "flags": flags[-1], "scaler": _scaler_fields(g.read_scaler()), "S": g.S}
    finally:
        g.close()


def _ring(wl):
    world = wl.n_ranks
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_proc, args=(r, world, port, wl, q)) for r in range(world)]
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


CASES = {
    # fp16 under a dynamic scale, clip, odd shards, buckets; +inf in rank 2's
    # replica at step 2 (in owner 0's slice): every rank skips the step
    "n4_fp16_clip_inject": W.Workload("ring4", [4 * 30_001 - 1], 4, 50_000, False, 71, 1e-4,
                                      init_scale=65536.0, dynamic_scale=True, max_grad_norm=0.05,
                                      steps=3, inject=(2, 2, 777, W.FP16_POS_INF)),
    "n2_bf16_no_clip": W.Workload("ring2", [2 * 40_000 + 6, 10], 2, 0, True, 72, 1e-3, steps=3),
    "n3_bf16_clip_list": W.Workload("ring3", [5_003, 30_000, 7, 12_345], 3, 9_999, True, 73,
                                    1e-2, max_grad_norm=0.2, steps=2),
}


@pytest.mark.parametrize("name", list(CASES))
def test_ring_processes_equal_one_process(name):
    wl = CASES[name]
    whole = _one_process(wl)
    ranks = _ring(wl)
    S = whole["S"]
    for r, part in enumerate(ranks):
        for k in ("master", "exp_avg", "exp_avg_sq"):
            assert np.array_equal(part[k][:S].view(np.uint32),
                                  whole[k][r * S:(r + 1) * S].view(np.uint32)), (r, k)
        assert np.array_equal(part["params"], whole["params"]), r
        assert part["scaler"] == whole["scaler"], (r, part["scaler"], whole["scaler"])
    assert np.array_equal(np.bitwise_or.reduce([p["flags"] for p in ranks]), whole["flags"])
    if wl.inject is not None:
        assert whole["scaler"][3] == 1


def test_ring_hop_rejects_bad_arguments():
    p = Z.zero_plan_create([1000], 4, 0)
    buf = torch.zeros(256, dtype=torch.float32, device="cuda")
    sc = torch.zeros(80, dtype=torch.uint8, device="cuda")
    grad = torch.zeros(1008, dtype=torch.int16, device="cuda")
    a, b, s = buf.data_ptr(), buf[64:].data_ptr(), sc.data_ptr()
    try:
        for rank, hop, recv, status in ((4, 1, 0, -1), (0, 0, 0, -1), (0, 5, b, -1),
                                        (0, 1, b, -1), (0, 2, 0, -1), (0, 2, b + 4, -2)):
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_ring_hop(p, rank, hop, grad.data_ptr(), recv, a, s)
            assert e.value.status == status, (rank, hop)
    finally:
        Z.zero_plan_destroy(p)
