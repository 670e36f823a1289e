"""GPU parity of the global-norm paths against the CPU checker's fp64 norm.

The checker's norm (plain fp64 sum of the squares of the reduced gradients,
ascending element order in fixed chunks) is compared with every device way
of forming it on the same seeded inputs:
  - zero_grad_norm from the tile records the reduce pass left,
  - zero_grad_norm recomputing the records from the reduced gradients,
  - zero_grad_norm_noalloc (recomputes into the library's fixed array),
  - zero_grad_norm_local + zero_grad_norm_apply in one process (the export /
    import pair, which must equal the first bit for bit).
The scaler's norm fields are poisoned before each call, so a call that wrote
nothing cannot pass. The clip convention is not on the pages; the checker's
reading of it is pinned against torch.nn.utils.clip_grad_norm_ on the CPU
(tests/test_oracle_step.py)."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import fsdp_sharded_mixed_shard_gb300 as Z
from fsdp_sharded_mixed_shard_gb300 import harness, synth, workloads as W
from parity_util import norm_tol, oracle_hp

pytestmark = pytest.mark.gpu

BF16_2P60 = 0x5D80   # bf16 bit patterns of 2^60, -2^59 and 2^58
BF16_M2P59 = 0xDD00
BF16_2P58 = 0x5C80


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def poison_norm_fields(g):
    """Overwrite the norm fields of the device scaler with values no norm
    call produces."""
    s = g.read_scaler()
    s.norm_sq, s.norm, s.clip_coef, s.clip_apply, s.norm_step = -1.0, -1.0, -1.0, -7, -7
    g.scaler.copy_(torch.frombuffer(bytearray(bytes(s)), dtype=torch.uint8).to(g.device))
    torch.cuda.synchronize()


def host_replicas(g, wl, step):
    """The replicas the device generator writes for `step`, rebuilt on the
    host (16-bit patterns, indexed by flat element - window base)."""
    spec = synth.grad_spec(seed=wl.seed, sigma=wl.sigma, bias_sigma=wl.bias_sigma,
                           loss_scale=wl.init_scale, outliers=wl.outliers, psi=wl.psi)
    return [oracle.cast16(synth.grad_f32(g.wlen, g.wbase, spec, step, r), wl.is_bf16)
            for r in range(wl.n_ranks)]


CASES = {
    # all owners, several buckets (segments cut at bucket edges)
    "full_n4_buckets": dict(wl=W.Workload("norm_full", [300_007, 4096, 13], 4, 50_000, True,
                                          41, 1e-2, max_grad_norm=0.5, steps=1), big=()),
    # a window of owners whose first tile is not tile 0
    "window_3_6_of_8": dict(wl=W.Workload("norm_win", [8 * 70_001 - 5], 8, 0, True, 42, 1e-3,
                                          max_grad_norm=0.05, steps=1, rank_lo=3, rank_hi=6),
                            big=()),
    # reduced gradients of 2^56 and more (squares of 2^112 and more, the
    # scaled side of the records) next to ordinary ones: at a tile edge,
    # inside tiles, in three owners, and g = 2^56 exactly
    "big_squares": dict(wl=W.Workload("norm_big", [4 * 50_003], 4, 0, True, 43, 1e-3,
                                      max_grad_norm=1.0, steps=1),
                        big=((0, 4095, BF16_2P60), (1, 4096, BF16_2P60),
                             (2, 77_777, BF16_M2P59), (3, 120_000, BF16_2P58))),
    # fp16, many segments (1-element-grained buckets of 7)
    "fp16_small_buckets": dict(wl=W.Workload("norm_fp16", [9_001, 3], 3, 7, False, 44, 1e-4,
                                             init_scale=1024.0, max_grad_norm=0.001, steps=1),
                               big=()),
}


@pytest.mark.parametrize("name", list(CASES))
def test_norm_paths_against_checker(name):
    wl, big = CASES[name]["wl"], CASES[name]["big"]
    g = harness.Group(wl)
    try:
        g.init_state()
        g.gen_grads(1, scale=wl.init_scale)
        reps = host_replicas(g, wl, 1)
        for r, e, bits in big:  # the same big values on both sides
            reps[r][e - g.wbase] = bits
            g.replicas[r, e - g.wbase] = bits - 65536 if bits >= 32768 else bits
        torch.cuda.synchronize()
        assert np.array_equal(g.replicas_u16(), np.stack(reps))

        # checker: the step with clipping, which reports the fp64 norm and ĝ
        p, _, _ = oracle.make_plan(wl.numels, wl.n_ranks, wl.bucket_elems)
        lo, hi = wl.ranks
        n = g.wlen
        master = synth.master_f32(n, g.wbase, wl.seed, wl.psi)
        ghat_host = np.zeros(n, np.float32)
        sc = oracle.scaler(wl.init_scale)
        oracle.step_arrays(p, lo, hi, wl.is_bf16, reps, g.wbase, master, np.zeros(n, np.float32),
                           np.zeros(n, np.float32), oracle.cast16(master, wl.is_bf16),
                           oracle_hp(wl), sc, ghat=ghat_host)
        assert sc.overflow == 0 and sc.norm_sq > 0
        if big:
            assert sc.norm_sq >= 2.0 ** 112

        d_sc, ws, st = g.scaler.data_ptr(), g.workspace.data_ptr(), g.sptr
        Z.zero_reduce_scatter(g.plan, -1, lo, hi, g.rep_ptrs(), g.wbase, g.ghat_ptrs(), d_sc, 0,
                              ws, st)
        got_ghat = g.ghat[:, :g.S].reshape(-1).cpu().numpy()
        assert np.array_equal(got_ghat.view(np.uint32), ghat_host.view(np.uint32))

        def check(what):
            d = g.read_scaler()
            assert d.norm_step == 1 and d.error == 0, what
            tol = norm_tol(n, g.info.n_tiles, wl.n_ranks)
            assert abs(d.norm_sq - sc.norm_sq) <= tol * sc.norm_sq, (
                what, d.norm_sq, sc.norm_sq)
            assert d.clip_apply == (1 if sc.clip_coef < 1.0 else 0), what
            assert abs(float(d.clip_coef) - float(sc.clip_coef)) <= \
                2.0 ** -23 * float(sc.clip_coef), what
            return d

        poison_norm_fields(g)
        Z.zero_grad_norm(g.plan, lo, hi, None, g.hp, d_sc, ws, st)
        from_records = check("records of the reduce pass")
        poison_norm_fields(g)
        Z.zero_grad_norm(g.plan, lo, hi, g.ghat_ptrs(), g.hp, d_sc, ws, st)
        check("records recomputed from the reduced gradients")
        poison_norm_fields(g)
        Z.zero_grad_norm_noalloc(g.plan, lo, hi, g.ghat_ptrs(), g.hp, d_sc, st)
        check("no-allocation entry")
        # export + import in one process: the same total, bit for bit
        Z.zero_reduce_scatter(g.plan, -1, lo, hi, g.rep_ptrs(), g.wbase, g.ghat_ptrs(), d_sc, 0,
                              ws, st)
        poison_norm_fields(g)
        ex = g.exchange.data_ptr()
        Z.zero_grad_norm_local(g.plan, lo, hi, None, g.hp, d_sc, ws, ex, st)
        Z.zero_grad_norm_apply(g.plan, ex, g.hp, d_sc, st)
        d = check("export and import")
        assert (d.norm_sq, d.clip_coef) == (from_records.norm_sq, from_records.clip_coef)
        blob = Z.ZeroExchange.from_buffer_copy(bytes(g.exchange.cpu().numpy().tobytes()))
        assert blob.overflow == 0 and tuple(blob.reserved) == (0, 0, 0)
        for o in range(Z.ZERO_MAX_RANKS):
            rec = blob.owner[o]
            nonzero = any((rec.hi, rec.lo, rec.big_hi, rec.big_lo))
            assert nonzero == (lo <= o < hi), o
    finally:
        g.close()


def test_export_without_clip_carries_only_the_overflow_word():
    """Without clipping the export needs no workspace and writes zero
    records; its overflow word follows the scaler's pending word."""
    wl = W.Workload("ex_noclip", [4 * 10_001], 4, 0, False, 45, 1e-4, init_scale=1024.0,
                    dynamic_scale=True, steps=1, inject=(1, 1, 30_000, W.FP16_POS_INF))
    g = harness.Group(wl, two_pass=True)
    try:
        g.init_state()
        g.gen_grads(1)
        d_sc, st = g.scaler.data_ptr(), g.sptr
        Z.zero_reduce_scatter(g.plan, -1, 0, 2, g.rep_ptrs(), 0, g.ghat_ptrs(), d_sc, 0, 0, st)
        ex = g.exchange.data_ptr()
        g.exchange.fill_(0xAB)
        Z.zero_grad_norm_local(g.plan, 0, 2, None, g.hp, d_sc, 0, ex, st)
        blob = Z.ZeroExchange.from_buffer_copy(bytes(g.exchange.cpu().numpy().tobytes()))
        assert blob.overflow == 0  # element 30,000 belongs to owner 2
        assert all(not any((r.hi, r.lo, r.big_hi, r.big_lo)) for r in blob.owner)
        Z.zero_reduce_scatter(g.plan, -1, 2, 4, g.rep_ptrs(), 0, g.ghat_ptrs(), d_sc, 0, 0, st)
        Z.zero_grad_norm_local(g.plan, 2, 4, None, g.hp, d_sc, 0, ex, st)
        blob = Z.ZeroExchange.from_buffer_copy(bytes(g.exchange.cpu().numpy().tobytes()))
        assert blob.overflow == 1
        assert C.sizeof(blob) == g.exchange.numel()
    finally:
        g.close()
