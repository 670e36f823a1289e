"""Cross-process plumbing for a step whose owners are split over processes.

Each process owns a window [rank_lo, rank_hi) of the N ranks and holds the N
replicas of its owners' slices. Only the step's global scalars cross
processes ("Training models too big for one GPU: ZeRO & FSDP", "ZeRO stages
1, 2 and 3": each rank updates its own slice): libzero's
zero_grad_norm_local writes a process's share into a 1040-byte
zero_exchange blob, the blobs of all processes are summed as int32 words,
and zero_grad_norm_apply imports the sum. This module does the summing with
torch.distributed; it moves bytes and adds integers, nothing else.
"""
import ctypes as C

import torch
import torch.distributed as dist

from . import ZeroExchange

EXCHANGE_BYTES = C.sizeof(ZeroExchange)


def windows(n_ranks, world):
    """Contiguous owner windows [lo, hi) of `world` processes over n_ranks
    owners, sizes differing by at most one (every process gets >= 1 owner
    when world <= n_ranks)."""
    if not 1 <= world <= n_ranks:
        raise ValueError("need 1 <= world (%d) <= n_ranks (%d)" % (world, n_ranks))
    cuts = [n_ranks * k // world for k in range(world + 1)]
    return [(cuts[k], cuts[k + 1]) for k in range(world)]


def check_partition(wins, n_ranks):
    """The windows must cover [0, n_ranks) exactly once: an owner exported by
    two processes would be summed twice, one exported by none would be
    missing from the norm."""
    seen = [0] * n_ranks
    for lo, hi in wins:
        if not 0 <= lo < hi <= n_ranks:
            raise ValueError("window [%d, %d) outside [0, %d)" % (lo, hi, n_ranks))
        for o in range(lo, hi):
            seen[o] += 1
    if any(c != 1 for c in seen):
        raise ValueError("windows do not partition the owners: %s" % wins)


def sum_exchange(blob, stream=None, group=None):
    """Sum a device zero_exchange blob (uint8 tensor of EXCHANGE_BYTES bytes)
    over the processes of `group`, in place, as int32 words. With NCCL the
    all-reduce runs on `stream`; with another backend (gloo) the blob goes
    through host memory after `stream` is synchronized."""
    if blob.numel() != EXCHANGE_BYTES or blob.dtype != torch.uint8:
        raise ValueError("not a zero_exchange blob")
    words = blob.view(torch.int32)
    if words.is_cuda and dist.get_backend(group) == "nccl":
        s = stream if stream is not None else torch.cuda.current_stream(words.device)
        with torch.cuda.stream(s):
            dist.all_reduce(words, op=dist.ReduceOp.SUM, group=group)
        return
    if words.is_cuda:
        (stream or torch.cuda.current_stream(words.device)).synchronize()
        host = words.cpu()
        dist.all_reduce(host, op=dist.ReduceOp.SUM, group=group)
        words.copy_(host)
        return
    dist.all_reduce(words, op=dist.ReduceOp.SUM, group=group)


# ------------------------------------------------- ring reduce-scatter ----
#
# "How far does splitting the batch get you?", "Why does the all-reduce not
# get more expensive with more ranks?": with one gradient replica per
# process, chunk i (owner i's slice) starts at rank i+1, collects every
# rank's values hop by hop and ends, complete, at rank i after N - 1 hops.
# libzero's zero_ring_hop does each rank's arithmetic; this driver moves the
# fp32 partials between neighbours.

def ring_schedule(rank, world):
    """[(hop, chunk)] of one rank: at hop h (1 .. world) it works on chunk
    (rank - h) mod world; after hops 1 .. world-1 it sends that partial to
    rank + 1 and receives the next chunk's from rank - 1; hop `world` is its
    own chunk."""
    return [(h, (rank - h) % world) for h in range(1, world + 1)]


def ring_pass(send, recv, rank, world, stream=None, group=None):
    """Send `send` to rank + 1 and receive `recv` from rank - 1 (device or
    host tensors of the same size). With NCCL the pair runs on `stream`;
    otherwise (gloo) the device buffers go through host memory after
    `stream` is synchronized."""
    nxt, prv = (rank + 1) % world, (rank - 1) % world
    if send.is_cuda and dist.get_backend(group) == "nccl":
        s = stream if stream is not None else torch.cuda.current_stream(send.device)
        with torch.cuda.stream(s):
            reqs = dist.batch_isend_irecv([dist.P2POp(dist.isend, send, nxt, group),
                                           dist.P2POp(dist.irecv, recv, prv, group)])
            for r in reqs:
                r.wait()
        return
    if send.is_cuda:
        (stream or torch.cuda.current_stream(send.device)).synchronize()
        hs, hr = send.cpu(), torch.empty(recv.shape, dtype=recv.dtype)
    else:
        hs, hr = send, recv
    reqs = [dist.isend(hs, nxt, group=group), dist.irecv(hr, prv, group=group)]
    for r in reqs:
        r.wait()
    if send.is_cuda:
        recv.copy_(hr)


def ring_reduce_scatter(plan, rank, world, grad, shard, bufs, d_scaler, d_flags=0, stream=None,
                        group=None):
    """The reduce-scatter of one step over `world` processes (world == the
    plan's N): grad is this rank's 16-bit gradient (device address of flat
    element 0), shard receives this rank's reduced gradient (a float32 device
    tensor of S elements), bufs two float32 device tensors of S elements."""
    from . import zero_ring_hop
    send, recv = bufs
    sptr = 0 if stream is None else stream.cuda_stream
    for hop, _ in ring_schedule(rank, world)[:-1]:
        zero_ring_hop(plan, rank, hop, grad, recv.data_ptr() if hop > 1 else 0,
                      send.data_ptr(), d_scaler, d_flags, sptr)
        ring_pass(send, recv, rank, world, stream, group)
    zero_ring_hop(plan, rank, world, grad, recv.data_ptr() if world > 1 else 0,
                  shard.data_ptr(), d_scaler, d_flags, sptr)


def all_gather_params(flat, rank, world, shard_elems, stream=None, group=None):
    """Every rank's slot [r*S, (r+1)*S) of the 16-bit parameter buffer `flat`
    (a device int16 tensor of at least world*S elements) from its owner: the
    all-gather of the updated weights ("Training models too big for one GPU:
    ZeRO & FSDP", "ZeRO stages 1, 2 and 3")."""
    n = world * shard_elems
    mine = flat[rank * shard_elems:(rank + 1) * shard_elems]
    # the slots travel as bytes: neither NCCL nor gloo gathers int16 tensors
    if flat.is_cuda and dist.get_backend(group) == "nccl":
        s = stream if stream is not None else torch.cuda.current_stream(flat.device)
        with torch.cuda.stream(s):
            dist.all_gather_into_tensor(flat[:n].view(torch.uint8),
                                        mine.clone().view(torch.uint8), group=group)
        return
    if flat.is_cuda:
        (stream or torch.cuda.current_stream(flat.device)).synchronize()
    nbytes = shard_elems * flat.element_size()
    parts = [torch.empty(nbytes, dtype=torch.uint8) for _ in range(world)]
    dist.all_gather(parts, mine.cpu().contiguous().view(torch.uint8), group=group)
    flat[:n].copy_(torch.cat(parts).view(flat.dtype))
