"""Host side of splitting the owners over processes, on CPU ranks (gloo,
world sizes 2 and 3): the windows partition the owners, and summing the
processes' zero_exchange blobs as int32 words reproduces every owner's
record bit for bit (each is non-zero in one process only) and counts the
windows that saw an overflow. No GPU is involved: the blobs are built on
the host with arbitrary float bit patterns, NaN and negative zero included."""
import ctypes as C
import os
import socket
import struct
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import fsdp_sharded_mixed_shard_gb300 as Z
from fsdp_sharded_mixed_shard_gb300 import dist as zdist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _records(n_ranks, seed):
    """Per owner four float32 bit patterns, some of them special."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=(n_ranks, 4), dtype=np.uint64).astype(np.uint32)
    bits[0, 0] = 0x80000000  # -0.0
    bits[-1, 2] = 0x7FC00001  # a NaN with a payload
    return bits


def _blob_for(lo, hi, recs, overflow):
    ex = Z.ZeroExchange()
    ex.overflow = overflow
    for o in range(lo, hi):
        r = ex.owner[o]
        r.hi, r.lo, r.big_hi, r.big_lo = (struct.unpack("<f", struct.pack("<I", int(b)))[0]
                                          for b in recs[o])
    return torch.frombuffer(bytearray(bytes(ex)), dtype=torch.uint8)


def _worker(rank, world, port, n_ranks, q):
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    wins = zdist.windows(n_ranks, world)
    lo, hi = wins[rank]
    recs = _records(n_ranks, 5)
    blob = _blob_for(lo, hi, recs, 1 if rank == world - 1 else 0)
    zdist.sum_exchange(blob)
    q.put((rank, bytes(blob.numpy().tobytes())))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,n_ranks", [(2, 8), (3, 8), (2, 64), (3, 5)])
def test_sum_of_exports_is_every_owner_record(world, n_ranks):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n_ranks, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = bytes(_blob_for(0, n_ranks, _records(n_ranks, 5), 1).numpy().tobytes())
    for r in range(world):
        assert got[r] == want
    ex = Z.ZeroExchange.from_buffer_copy(got[0])
    assert ex.overflow == 1 and C.sizeof(ex) == zdist.EXCHANGE_BYTES


def test_windows_partition_the_owners():
    for n in (1, 2, 5, 8, 64):
        for world in range(1, n + 1):
            wins = zdist.windows(n, world)
            zdist.check_partition(wins, n)
            assert len(wins) == world
            sizes = [hi - lo for lo, hi in wins]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    with pytest.raises(ValueError):
        zdist.windows(4, 5)
    for bad in ([(0, 2), (1, 4)], [(0, 2), (3, 4)], [(0, 4), (4, 5)], [(2, 2), (0, 4)]):
        with pytest.raises(ValueError):
            zdist.check_partition(bad, 4)


def test_sum_exchange_rejects_other_buffers():
    with pytest.raises(ValueError):
        zdist.sum_exchange(torch.zeros(1024, dtype=torch.uint8))
    with pytest.raises(ValueError):
        zdist.sum_exchange(torch.zeros(zdist.EXCHANGE_BYTES // 4, dtype=torch.int32))
