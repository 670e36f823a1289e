"""Host side of the ring reduce-scatter on CPU ranks (gloo, world sizes 2 to
5): the schedule (which chunk each rank works on at each hop) and the
neighbour exchange of the product (dist.ring_schedule, dist.ring_pass),
with the hop arithmetic done here in numpy fp32 as the kernel does it
(widen, add, one rounding per add). Every rank must end with its own chunk
summed in the checker's ring order, bit for bit, on values chosen so that
the order matters."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _values(world, S):
    """fp32 values of every rank's whole gradient (world * S elements): wide
    magnitudes, so that the order of the additions changes the result."""
    rng = np.random.default_rng(world * 1000 + S)
    v = rng.standard_normal((world, world * S)).astype(np.float32)
    v *= (2.0 ** rng.integers(-30, 30, size=(world, world * S))).astype(np.float32)
    return v


def _worker(rank, world, port, S, q):
    sys.path.insert(0, ROOT)
    from fsdp_sharded_mixed_shard_gb300 import dist as zdist
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    own = _values(world, S)[rank]
    send = torch.zeros(S, dtype=torch.float32)
    recv = torch.zeros(S, dtype=torch.float32)
    sched = zdist.ring_schedule(rank, world)
    for hop, chunk in sched:
        part = own[chunk * S:(chunk + 1) * S]
        if hop == 1:
            out = part.copy()
        else:
            out = (recv.numpy() + part).astype(np.float32)
        if hop < world:
            send.copy_(torch.from_numpy(out))
            zdist.ring_pass(send, recv, rank, world)
        else:
            q.put((rank, chunk, out))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3, 4, 5])
def test_ring_schedule_and_exchange_give_the_ring_order_sum(world):
    S = 257
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, S, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, chunk, out = q.get(timeout=120)
        got[rank] = (chunk, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    vals = _values(world, S)
    for rank in range(world):
        chunk, out = got[rank]
        assert chunk == rank
        want = np.array([oracle.ring_sum(vals[:, rank * S + k], rank) for k in range(S)],
                        dtype=np.float32)
        assert np.array_equal(out.view(np.uint32), want.view(np.uint32)), rank
        # another order (plain rank order 0, 1, ..., N-1) differs somewhere,
        # so the order is pinned; for owner N-1 the ring order is that order
        plain = vals[0, rank * S:(rank + 1) * S].copy()
        for r in range(1, world):
            plain = (plain + vals[r, rank * S:(rank + 1) * S]).astype(np.float32)
        if world > 2 and rank != world - 1:
            assert not np.array_equal(plain, want)


def test_ring_schedule_covers_every_chunk_once():
    from fsdp_sharded_mixed_shard_gb300 import dist as zdist
    for world in range(1, 9):
        for rank in range(world):
            sched = zdist.ring_schedule(rank, world)
            assert [h for h, _ in sched] == list(range(1, world + 1))
            assert sorted(c for _, c in sched) == list(range(world))
            assert sched[-1] == (world, rank)
        # at every hop the ranks work on distinct chunks, and what rank r
        # sends at hop h is what rank r + 1 works on at hop h + 1
        for h in range(1, world):
            chunks = [zdist.ring_schedule(r, world)[h - 1][1] for r in range(world)]
            assert sorted(chunks) == list(range(world))
            for r in range(world):
                assert zdist.ring_schedule((r + 1) % world, world)[h][1] == chunks[r]


def _gather_worker(rank, world, port, S, q):
    sys.path.insert(0, ROOT)
    from fsdp_sharded_mixed_shard_gb300 import dist as zdist
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    flat = torch.full((world * S + 5,), -1, dtype=torch.int16)
    flat[rank * S:(rank + 1) * S] = torch.arange(S, dtype=torch.int16) * 7 + rank * 1000 - 30000
    zdist.all_gather_params(flat, rank, world, S)
    q.put((rank, flat.numpy().copy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,S", [(2, 5), (3, 1001), (4, 1)])
def test_all_gather_params_fills_every_slot(world, S):
    """The parameter all-gather on CPU ranks: every rank ends with every
    rank's 16-bit slot, and nothing past world * S is touched."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, world, port, S, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = np.concatenate([np.arange(S, dtype=np.int16) * 7 + r * 1000 - 30000
                           for r in range(world)]).astype(np.int16)
    for r in range(world):
        assert np.array_equal(got[r][:world * S], want)
        assert (got[r][world * S:] == -1).all()
