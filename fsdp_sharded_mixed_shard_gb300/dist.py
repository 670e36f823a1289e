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
