"""GPU parity: libzero's kernels against the CPU checker, element by element,
on the same seeded inputs (sizes the checker finishes in seconds, spanning
many tiles and ragged tails), plus edge cases."""
import numpy as np
import pytest
import torch

import oracle
from fsdp_sharded_mixed_shard_gb300 import harness, workloads as W
from parity_util import run_small

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def tiny_transformer_numels(d=64, vocab=503, ctx=128, layers=3):
    out = [vocab * d, ctx * d]
    for _ in range(layers):
        out += [d, d, d * 3 * d, 3 * d, d * d, d, d, d, d * 4 * d, 4 * d, 4 * d * d, d]
    return out + [d, d]


def test_tiny_flat_full_size():
    """1,000,003 parameters, 4 ranks (odd shard: scalar path for ranks 1-3),
    fp16 gradients under a static loss scale of 1024, 3 steps, fused path."""
    stats, dev, orc = run_small(W.TINY_FLAT)
    assert dev.t == 3


def test_gpt2_shaped_small_fused():
    wl = W.GPT2_SMALL.scaled(numels=tiny_transformer_numels(), bucket_elems=50_000, steps=4)
    run_small(wl)


def test_gpt2_shaped_small_two_pass_per_bucket():
    wl = W.GPT2_SMALL.scaled(numels=tiny_transformer_numels(), bucket_elems=50_000, steps=3)
    run_small(wl, per_bucket=True, two_pass=True)


def test_flat_fp16_dynamic_clip_inject():
    """fp16 under a dynamic scale of 65536, clip 1.0, +inf injected at step 3
    in rank 5: the step is skipped and the scale halves."""
    psi = 1_000_003
    wl = W.FLAT_1P5B.scaled(numels=[psi], inject=(3, 5, psi // 3, W.FP16_POS_INF))
    stats, dev, orc = run_small(wl)
    assert dev.t == 4 and dev.scale == 32768.0 and dev.n_skipped == 1


@pytest.mark.parametrize("per_bucket", [False, True])
def test_two_pass_in_place_one_set(per_bucket):
    """The two-pass path with one optimizer state set, updated in place (the
    harness default is two sets, read one and write the other): clip, a
    dynamic fp16 scale and a skipped step, whole buckets or bucket by bucket."""
    psi = 600_011
    wl = W.FLAT_1P5B.scaled(numels=[psi], bucket_elems=100_000 if per_bucket else 0,
                            inject=(2, 3, psi // 2, W.FP16_POS_INF), steps=4)
    stats, dev, orc = run_small(wl, per_bucket=per_bucket, n_sets=1)
    assert dev.t == 3 and dev.n_skipped == 1 and dev.state_index == 0


def test_flat_fp16_inject_fused_skip_recast():
    """Same injection on the fused path: the speculative pass writes the other
    state set and the parameters; the skip re-casts them from the kept set."""
    psi = 1_000_003
    wl = W.FLAT_1P5B.scaled(numels=[psi], max_grad_norm=0.0,
                            inject=(2, 5, psi // 3, W.FP16_POS_INF), steps=3)
    stats, dev, orc = run_small(wl)
    assert dev.t == 2 and dev.scale == 32768.0


@pytest.mark.parametrize("n,n_micro", [(4, 1), (4, 2), (16, 1)])
def test_folded_finish_equals_two_launches(n, n_micro):
    """zero_step on a small fused step is one launch (the short-step kernel
    without micro-batches, the pipelined pass with them; the last CTA does
    the bookkeeping, and on an overflow re-casts the parameters alone);
    zero_step_update + zero_step_finish is two launches of the pipelined
    pass and the finish. Same state, parameters and scaler after every step,
    bit for bit, through a skipped step."""
    import fsdp_sharded_mixed_shard_gb300 as Z
    psi = n * 50_001 - 1
    wl = W.Workload("fold", [psi], n, 0, False, 24, 1e-4, init_scale=4096.0,
                    dynamic_scale=True, steps=4, n_micro=n_micro,
                    inject=(2, 1, psi // 2, W.FP16_POS_INF))
    a, b = harness.Group(wl), harness.Group(wl)
    try:
        for g in (a, b):
            g.init_state()
        for step in range(1, wl.steps + 1):
            for g in (a, b):
                for mb in range(1, n_micro):
                    g.gen_grads(step, micro=mb)
                    g.accumulate(first=(mb == 1))
                g.gen_grads(step)
            a.step()   # zero_step_accum: folded
            m, v, w = b._state_ptrs(0), b._state_ptrs(1), b._state_ptrs(2)
            acc = b.accum_ptrs() if n_micro > 1 else None
            b.flags.zero_()
            Z.zero_step_update_accum(b.plan, 0, n, m, v, w, 2, None, b.rep_ptrs(), acc, n_micro,
                                     0, b.flat.data_ptr(), b.hp, b.scaler.data_ptr(),
                                     b.flags.data_ptr(), b.sptr)
            Z.zero_step_finish(b.plan, 0, n, m, 2, None, 0, b.flat.data_ptr(), b.hp,
                               b.scaler.data_ptr(), b.sptr)
            torch.cuda.synchronize()
            assert bytes(a.scaler.cpu().numpy()) == bytes(b.scaler.cpu().numpy()), step
            assert torch.equal(a.flat, b.flat), step
            sa, sb = a.current_state(), b.current_state()
            for x, y in zip(sa, sb):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32)), step
        s = a.read_scaler()
        assert s.t == 3 and s.n_skipped == 1 and s.finish_count == 0
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("rank", [0, 5])
def test_stage3_slice_small(rank):
    S = 20011  # odd: rank 5's window starts off the 16-byte grid
    wl = W.STAGE3_SLICE.scaled(numels=[64 * S], rank_lo=rank, rank_hi=rank + 1, steps=3)
    run_small(wl)


def test_llama_shaped_small_outliers_clip():
    d, f, v = 128, 512, 1000
    numels = [v * d]
    for _ in range(2):
        numels += [d, d * d, d * d, d * d, d * d, d, d * f, d * f, f * d]
    numels += [d]
    wl = W.LLAMA_2B.scaled(numels=numels, bucket_elems=100_000, steps=3)
    run_small(wl, per_bucket=True)


@pytest.mark.parametrize("n,numels,bucket,bf16,two_pass", [
    (1, [4099], 0, True, False),             # one rank: identity reduction
    (3, [1001, 7], 0, False, True),          # non power-of-two N, two-pass, no clip
    (3, [2], 0, True, False),                # psi < N: mostly padding
    (4, [0, 5, 0, 3], 0, True, False),       # empty tensors in the list
    (4, [300], 1, True, True),               # 300 one-element buckets: > 128 segments
    (5, [12345], 7, False, False),           # odd bucket size, misaligned segments
    (8, [8 * 4096 * 3 + 17], 0, True, False),  # several tiles per rank plus a tail
    (16, [16 * 4096 - 3], 50_000, True, True),
])
def test_edge_shapes(n, numels, bucket, bf16, two_pass):
    wl = W.Workload("edge", numels, n, bucket, bf16, 11, 1e-3,
                    init_scale=1.0 if bf16 else 1024.0, steps=3)
    run_small(wl, two_pass=two_pass)


@pytest.mark.parametrize("bits", [0x7C00, 0xFC00, 0x7E00])
@pytest.mark.parametrize("where", ["first", "last", "pad", "bucket_edge"])
@pytest.mark.parametrize("two_pass", [False, True])
def test_nonfinite_injection(bits, where, two_pass):
    n, psi, bsz = 4, 40_001, 8192
    psip = psi + (-psi) % n
    e = {"first": 0, "last": psi - 1, "pad": psip - 1, "bucket_edge": 2 * bsz}[where]
    wl = W.Workload("inject", [psi], n, bsz, False, 13, 1e-4, init_scale=4096.0,
                    dynamic_scale=True, steps=3, inject=(2, 1, e, bits))
    stats, dev, orc = run_small(wl, two_pass=two_pass)
    assert dev.t == 2 and dev.scale == 2048.0 and dev.overflow == 0


def test_clip_inactive_equals_no_clip():
    wl = W.Workload("clipbig", [70_001], 4, 0, True, 21, 1e-3, max_grad_norm=1e9, steps=2)
    stats, dev, orc = run_small(wl)
    assert dev.clip_apply == 0


def test_clip_active_two_pass_recomputed_norm():
    """zero_grad_norm recomputing the partials from the reduced gradients
    agrees with the partials left by zero_reduce_scatter (both fixed-order,
    with different per-thread groupings: equal within the norm tolerance)."""
    import fsdp_sharded_mixed_shard_gb300 as Z
    wl = W.Workload("clipnorm", [200_003], 4, 30_000, True, 22, 1e-2, max_grad_norm=0.5,
                    steps=1)
    g = harness.Group(wl)
    g.init_state()
    g.gen_grads(1)
    sc, ws, st = g.scaler.data_ptr(), g.workspace.data_ptr(), g.sptr
    Z.zero_reduce_scatter(g.plan, -1, 0, 4, g.rep_ptrs(), 0, g.ghat_ptrs(), sc, 0, ws, st)
    Z.zero_grad_norm(g.plan, 0, 4, None, g.hp, sc, ws, st)
    a = g.read_scaler()
    Z.zero_grad_norm(g.plan, 0, 4, g.ghat_ptrs(), g.hp, sc, ws, st)
    b = g.read_scaler()
    from parity_util import norm_tol
    assert abs(a.norm_sq - b.norm_sq) <= \
        2 * norm_tol(g.info.psi_pad, g.info.n_tiles, wl.n_ranks) * b.norm_sq
    assert abs(float(a.clip_coef) - float(b.clip_coef)) <= 2.0 ** -23 * float(b.clip_coef)
    assert a.clip_apply == 1 and b.clip_apply == 1
    g.close()


def test_abi_rejects_bad_arguments():
    import fsdp_sharded_mixed_shard_gb300 as Z
    wl = W.Workload("bad", [1000], 4, 0, True, 1, 1e-3, steps=1)
    g = harness.Group(wl)
    g.init_state()
    m, v, w = g._state_ptrs(0), g._state_ptrs(1), g._state_ptrs(2)
    sc = g.scaler.data_ptr()
    with pytest.raises(Z.ZeroError) as e:   # fused with clip
        hp = harness.hparams_of(wl.scaled(max_grad_norm=1.0))
        Z.zero_step(g.plan, 0, 4, m, v, w, 2, None, g.rep_ptrs(), 0, g.flat.data_ptr(), hp, sc)
    assert e.value.status == -1
    with pytest.raises(Z.ZeroError) as e:   # misaligned replica
        reps = g.rep_ptrs()
        reps[1] += 2
        Z.zero_step(g.plan, 0, 4, m, v, w, 2, None, reps, 0, g.flat.data_ptr(), g.hp, sc)
    assert e.value.status == -2
    with pytest.raises(Z.ZeroError):        # bad rank range
        Z.zero_step(g.plan, 2, 1, m, v, w, 2, None, g.rep_ptrs(), 0, g.flat.data_ptr(), g.hp, sc)
    g.close()


def test_missing_norm_sets_device_error():
    """Two-pass step with clip but no zero_grad_norm in this step: the kernel
    writes nothing and records ZERO_DEVERR_NO_NORM."""
    import fsdp_sharded_mixed_shard_gb300 as Z
    wl = W.Workload("nonorm", [5000], 2, 0, True, 1, 1e-3, max_grad_norm=1.0, steps=1)
    g = harness.Group(wl)
    g.init_state()
    g.gen_grads(1)
    before = g.state.clone()
    sc = g.scaler.data_ptr()
    Z.zero_reduce_scatter(g.plan, -1, 0, 2, g.rep_ptrs(), 0, g.ghat_ptrs(), sc, 0, 0, g.sptr)
    Z.zero_step(g.plan, 0, 2, g._state_ptrs(0), g._state_ptrs(1), g._state_ptrs(2), 1,
                g.ghat_ptrs(), None, 0, g.flat.data_ptr(), g.hp, sc, 0, g.sptr)
    s = g.read_scaler()
    assert s.error == 2
    assert torch.equal(before, g.state)
    g.close()


@pytest.mark.parametrize("bf16", [False, True])
def test_widening_all_16bit_patterns(bf16):
    """One rank, loss scale 1: the reduced gradient is the replica value
    widened exactly, for every one of the 65536 bit patterns (NaNs compared
    as NaN), and every non-finite pattern raises the flag."""
    import fsdp_sharded_mixed_shard_gb300 as Z
    n = 65536
    wl = W.Workload("widen", [n], 1, 4096, bf16, 1, 1e-3, steps=1, max_grad_norm=1.0)
    g = harness.Group(wl)
    g.init_state()
    pats = torch.arange(n, dtype=torch.int32).to(torch.int16)
    g.replicas[0, :n].copy_(pats.to(g.device))
    g.flags.zero_()
    sc = g.scaler.data_ptr()
    Z.zero_reduce_scatter(g.plan, -1, 0, 1, g.rep_ptrs(), 0, g.ghat_ptrs(), sc,
                          g.flags.data_ptr(), g.workspace.data_ptr(), g.sptr)
    got = g.ghat[0, :n].cpu().numpy()
    want = oracle.widen16(np.arange(n, dtype=np.uint16), bf16)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
    bad_bucket = ~np.isfinite(want).reshape(-1, 4096).all(axis=1)
    assert np.array_equal(g.flags_u32() != 0, bad_bucket)
    assert g.read_scaler().pending == 1
    g.close()


def test_bounded_wait_times_out_without_fault():
    """The pipeline's bounded barrier wait, driven to expiry on purpose (a
    barrier nobody completes, 5 ms limit): the kernel records
    ZERO_DEVERR_TIMEOUT and returns; the context stays usable for a normal
    step afterwards."""
    import fsdp_sharded_mixed_shard_gb300 as Z
    wl = W.Workload("timeout", [10_000], 2, 0, True, 1, 1e-3, steps=1)
    g = harness.Group(wl)
    g.init_state()
    Z.zero_selftest_wait_timeout(g.scaler.data_ptr(), 5_000_000, g.sptr)
    assert g.read_scaler().error == 3
    g.init_state()  # fresh scaler
    g.gen_grads(1)
    g.step()
    s = g.read_scaler()
    assert s.error == 0 and s.t == 1
    g.close()


@pytest.mark.parametrize("k,two_pass,bf16,n", [(2, False, True, 8), (3, False, False, 4),
                                              (2, True, True, 16), (4, True, False, 8),
                                              (3, False, True, 64)])
def test_micro_batch_accumulation(k, two_pass, bf16, n):
    """k micro-batches accumulated in fp32 (zero_accumulate), the last one
    added inside the reduce (zero_step_accum / zero_reduce_scatter_accum),
    unscale 1/(S N k); fused and two-pass paths, against the checker."""
    psi = n * 4096 * 2 + 77
    wl = W.Workload("accum", [psi], n, 30_000, bf16, 41, 1e-3,
                    init_scale=1.0 if bf16 else 1024.0, steps=3, n_micro=k,
                    max_grad_norm=0.5 if two_pass else 0.0)
    run_small(wl, two_pass=two_pass)


def test_micro_batch_accumulation_overflow_in_last_micro_batch():
    psi = 8 * 4096 + 5
    wl = W.Workload("accum_inf", [psi], 8, 0, False, 42, 1e-4, init_scale=2048.0,
                    dynamic_scale=True, steps=3, n_micro=3, inject=(2, 3, psi // 2, 0x7C00))
    stats, dev, orc = run_small(wl)
    assert dev.t == 2 and dev.scale == 1024.0


@pytest.mark.parametrize("n", [4, 8, 16])
def test_clip_with_big_squares_in_some_warps(n):
    """Gradients with |g| >= 2^56 (their squares go through the scaled
    accumulator pair) in a few tiles and warps only, clip active: the
    two-pass norm and the whole state match the checker."""
    from parity_util import assert_params, assert_state, norm_tol, oracle_hp
    psi = 3 * 4096 * n + 1001
    wl = W.Workload("bigsq", [psi], n, 0, True, 31, 1e-3, max_grad_norm=1.0, steps=1)
    g = harness.Group(wl)
    g.init_state()
    g.gen_grads(1)
    torch.cuda.synchronize()
    # bf16 patterns of 2^60, -2^100 and 2^75 planted in one replica each
    plant = [(1, 5, 0x5D80), (0, 4096 + 600, 0xF180), (n - 1, g.S + 7, 0x6500),
             (2 % n, 2 * g.S + 4096 + 3000, 0x5D80)]
    for r, e, bits in plant:
        g.replicas[r, e] = bits - 65536 if bits >= 32768 else bits
    torch.cuda.synchronize()
    reps_host = [np.ascontiguousarray(x) for x in g.replicas_u16()]
    g.step()
    torch.cuda.synchronize()
    dev = g.read_scaler()
    p, _, _ = oracle.make_plan(wl.numels, n, 0)
    hp = oracle_hp(wl)
    sc = oracle.scaler(wl.init_scale)
    from fsdp_sharded_mixed_shard_gb300 import synth
    master = synth.master_f32(p.psi_pad, 0, wl.seed, psi)
    m = np.zeros(p.psi_pad, np.float32)
    v = np.zeros(p.psi_pad, np.float32)
    params = oracle.cast16(master, True)
    oracle.step_arrays(p, 0, n, True, reps_host, 0, master, m, v, params, hp, sc)
    assert sc.norm_sq > 2.0 ** 190 and dev.clip_apply == 1 and dev.overflow == 0
    assert abs(dev.norm_sq - sc.norm_sq) <= \
        norm_tol(p.psi_pad, g.info.n_tiles, wl.n_ranks) * sc.norm_sq
    got_master, got_m, got_v = (x.numpy() for x in g.current_state())
    assert_state(got_master[:psi], master[:psi], "master")
    assert_state(got_m[:psi], m[:psi], "exp_avg")
    assert_state(got_v[:psi], v[:psi], "exp_avg_sq")
    assert_params(g.params_u16()[:psi], params[:psi])
    g.close()


@pytest.mark.parametrize("clip,n_micro", [(0.0, 1), (0.5, 1), (0.0, 2)])
def test_checkpoint_resume_is_bit_exact(tmp_path, clip, n_micro):
    """Run 2 steps, save through torch, keep going 2 more steps; a fresh group
    that loads the checkpoint and runs the same 2 steps ends bit-identical
    (state, parameters and every scaler field), on both ping-pong parities."""
    wl = W.GPT2_SMALL.scaled(name="resume", numels=tiny_transformer_numels(), bucket_elems=60_000,
                             max_grad_norm=clip, n_micro=n_micro, steps=4, dynamic_scale=True,
                             init_scale=1024.0)

    def run(g, steps):
        for step in steps:
            if n_micro > 1:
                g.step_micro(step)
            else:
                g.gen_grads(step)
                g.step()
        torch.cuda.synchronize()

    a = harness.Group(wl)
    a.init_state()
    run(a, (1, 2))
    path = tmp_path / "ckpt.pt"
    torch.save(a.state_dict(), path)
    run(a, (3, 4))
    b = harness.Group(wl)
    b.init_state()
    run(b, (1,))            # leave b on the other ping-pong set and other values first
    b.load_state_dict(torch.load(path))
    run(b, (3, 4))
    for x, y in zip(a.current_state(), b.current_state()):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert np.array_equal(a.params_u16(), b.params_u16())
    assert bytes(a.read_scaler()) == bytes(b.read_scaler())
    assert a.read_scaler().t == 4
    other = harness.Group(wl.scaled(name="other"))
    with pytest.raises(ValueError):
        other.load_state_dict(torch.load(path))
    other.close()
    a.close()
    b.close()


@pytest.mark.parametrize("clip", [0.0, 0.5])
def test_cuda_graph_replay_equals_eager_steps(clip):
    """One whole step (fused, or two-pass with the norm) captured into a CUDA
    graph and replayed 4 times ends bit-identical to 4 eager steps on the
    same inputs, including every scaler byte (ping-pong sets alternate
    through the device-resident state, so replay needs no host logic)."""
    wl = W.GPT2_SMALL.scaled(name="graph", numels=tiny_transformer_numels(), bucket_elems=60_000,
                             max_grad_norm=clip, steps=4)
    eager = harness.Group(wl)
    eager.init_state()
    eager.gen_grads(1)
    for _ in range(4):
        eager.step(clear_flags=False)
    torch.cuda.synchronize()
    g = harness.Group(wl, stream=torch.cuda.Stream())  # capture needs a non-default stream
    g.init_state()
    g.gen_grads(1)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=g.stream):
        g.step(clear_flags=False)
    with torch.cuda.stream(g.stream):  # replay() launches on the current stream
        for _ in range(4):
            graph.replay()
    torch.cuda.synchronize()
    for x, y in zip(eager.current_state(), g.current_state()):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert np.array_equal(eager.params_u16(), g.params_u16())
    assert bytes(eager.read_scaler()) == bytes(g.read_scaler())
    assert g.read_scaler().t == 4
    eager.close()
    g.close()


@pytest.mark.parametrize("n,psi,two_pass,micro", [(8, 99_997, False, 1), (8, 99_997, True, 1),
                                                  (64, 64_250, False, 1), (64, 64_250, False, 2)])
def test_slices_off_the_8_element_grid(n, psi, two_pass, micro):
    """Shards of S = 4 (mod 8) elements: odd owners start 4 elements off the
    windows' 8-element grid. The fused step and the reduce pass give their
    tiles a shifted body (copies from 4 elements early); with micro-batch
    accumulators every tile has a few edge elements outside its aligned body
    (the warp-cooperative path). Against the checker element by element."""
    wl = W.Workload("offgrid", [psi], n, 0, True, 51, 1e-3, steps=2, n_micro=micro,
                    max_grad_norm=0.5 if two_pass else 0.0)
    p, _, _ = oracle.make_plan(wl.numels, n, 0)
    assert p.shard % 8 == 4
    run_small(wl, two_pass=two_pass)


@pytest.mark.parametrize("n,psi,mod4,bf16,two_pass,micro", [
    (8, 8 * 25_001 - 5, 1, True, False, 1),     # S odd
    (8, 8 * 25_001 - 5, 1, False, True, 1),     # S odd, fp16, clipped in two passes
    (8, 8 * 25_002, 2, True, False, 1),         # S = 2 (mod 4)
    (8, 8 * 25_002, 2, True, True, 1),
    (8, 8 * 25_003, 3, False, False, 1),        # S = 3 (mod 4)
    (8, 8 * 25_003, 3, True, True, 1),
    (64, 64 * 3_001 - 7, 1, True, False, 1),
    (64, 64 * 3_001 - 7, 1, True, True, 1),
    (64, 64 * 3_002, 2, True, False, 2),        # micro-batches: shifted accumulator copies
    (8, 8 * 25_001 - 5, 1, True, False, 3),
    (8, 8 * 25_003, 3, False, True, 2),
])
def test_slices_out_of_phase_with_the_window(n, psi, mod4, bf16, two_pass, micro):
    """Shards whose size is not a multiple of 4: the owners' slices start at
    every 16-bit phase of the 16-byte grid, so their tiles take the shifted
    body (replica and accumulator chunks copied from the 16-byte block below
    the first element, unaligned parameter stores), against the checker
    element by element."""
    wl = W.Workload("phase", [psi], n, 0, bf16, 53 + mod4, 1e-3, steps=2, n_micro=micro,
                    max_grad_norm=0.5 if two_pass else 0.0)
    p, _, _ = oracle.make_plan(wl.numels, n, 0)
    assert p.shard % 4 == mod4
    run_small(wl, two_pass=two_pass)


@pytest.mark.parametrize("rank_lo,rank_hi,bucket,per_bucket,micro", [
    (3, 6, 0, False, 1),          # a window that starts at an odd owner
    (0, 8, 30_001, True, 1),      # odd bucket size: segments start off every grid
    (5, 6, 0, False, 1),          # one odd owner alone (window base = 5 S)
    (0, 8, 30_001, True, 2),      # the same with micro-batch accumulators
    (2, 7, 0, False, 3),
])
def test_out_of_phase_windows_and_buckets(rank_lo, rank_hi, bucket, per_bucket, micro):
    """S odd with rank windows and odd bucket boundaries: the owners' phase
    against the 16-byte grid is taken relative to the window base, and a
    segment that starts at a bucket boundary starts its body at the next
    shard index that is a multiple of 4. Fused and two-pass clipped steps,
    against the checker element by element."""
    for clip in (0.0, 0.5):
        wl = W.Workload("window", [8 * 25_001 - 3], 8, bucket, True, 61, 1e-3, steps=2,
                        rank_lo=rank_lo, rank_hi=rank_hi, max_grad_norm=clip, n_micro=micro)
        p, _, _ = oracle.make_plan(wl.numels, 8, bucket)
        assert p.shard % 2 == 1
        run_small(wl, per_bucket=per_bucket and clip > 0, two_pass=clip > 0)


@pytest.mark.parametrize("n,psi,bf16,scale,dynamic,lo,hi,bucket,inject", [
    (4, 4 * 30_001 - 1, False, 1024.0, False, 0, 4, 0, None),   # S odd: every 16-bit phase
    (4, 4 * 30_001 - 1, False, 1000.0, False, 0, 4, 0, None),   # S_l not a power of two
    (3, 3 * 30_002, True, 1.0, False, 0, 3, 0, None),           # S_l N = 3
    (2, 2 * 30_003, True, 2.0 ** -20, False, 0, 2, 7, None),    # small S_l, odd buckets
    (4, 4 * 30_001 - 1, True, 1.0, False, 1, 3, 0, None),       # a window of two owners
    (1, 1_000_000, True, 1.0, False, 0, 1, 0, None),
    (4, 4 * 30_002, False, 3000.0, True, 0, 4, 0, (2, 2, 70_001, 0x7C00)),  # overflow, re-cast
    (8, 8 * 30_001 - 3, True, 1.0, False, 0, 8, 0, None),
    (16, 16 * 20_001 - 5, False, 1024.0, False, 0, 16, 30_001, None),
    (16, 16 * 20_003, True, 1.0, False, 3, 11, 0, None),          # owners 3..10 of 16
    (12, 12 * 20_002, False, 1000.0, True, 0, 12, 0, (3, 11, 12 * 20_002 - 1, 0xFC00)),
])
def test_short_steps(n, psi, bf16, scale, dynamic, lo, hi, bucket, inject):
    """Fused steps over at most 2^20 elements at N <= 16 without micro-batch
    accumulators run the short-step kernel (one wave of small CTAs, each CTA
    inside one owner's slice). Every shard phase against the 16-byte grid,
    loss scales whose product with N is and is not a power of two (two ways
    of forming 1 / (S_l N)), rank windows and an overflowed step, against the
    checker element by element."""
    wl = W.Workload("short", [psi], n, bucket, bf16, 71, 1e-3, init_scale=scale,
                    dynamic_scale=dynamic, steps=3, rank_lo=lo, rank_hi=hi, inject=inject)
    stats, dev, orc = run_small(wl, two_pass=False)
    if inject is not None:
        assert dev.n_skipped == 1 and dev.scale == scale / 2


@pytest.mark.parametrize("t0", [1000, 6800, 100_000, 720_000, 2_000_000])
@pytest.mark.parametrize("n,two_pass", [(4, False), (8, False), (4, True)])
def test_bias_corrections_late_in_training(t0, n, two_pass):
    """Steps t0 + 1 and t0 + 2, with the scaler's beta powers as t0 good
    steps leave them: the bias corrections come from the integer form of
    the fp64 product and difference while the powers are normal, from the
    fp64 pipe once beta1^t (t0 >= 6800) or beta2^t (t0 >= 720,000) has
    become subnormal or zero. Short-step kernel (N = 4, fused), pipelined
    fused pass (N = 8) and update pass (two-pass), against the checker
    element by element; the stored powers continue the fp64 product chain
    bit for bit."""
    wl = W.Workload("late", [70_001], n, 0, True, 81, 1e-3, steps=2,
                    max_grad_norm=0.5 if two_pass else 0.0)
    stats, dev, orc = run_small(wl, two_pass=two_pass, t0=t0)
    p1 = p2 = 1.0
    for _ in range(t0 + 2):
        p1 *= wl.beta1
        p2 *= wl.beta2
    assert dev.t == t0 + 2
    assert dev.beta1_pow == p1 and dev.beta2_pow == p2


@pytest.mark.parametrize("n,psi,two_pass", [(4, 90_001, False), (64, 64 * 3_001, False),
                                            (8, 120_007, True)])
def test_state_index_outside_the_sets_is_a_device_error(n, psi, two_pass):
    """A scaler whose state index names no state set (a caller's corrupted or
    hand-written scaler): the step sets ZERO_DEVERR_STATE_INDEX in the
    scaler's error word and writes neither state set nor the parameters.
    Short-step kernel (N = 4), pipelined fused pass (N = 64) and the
    two-pass update (N = 8, clip)."""
    wl = W.Workload("badidx", [psi], n, 0, True, 91, 1e-3, steps=1,
                    max_grad_norm=0.5 if two_pass else 0.0)
    g = harness.Group(wl)
    try:
        g.init_state()
        g.gen_grads(1)
        sc = g.read_scaler()
        sc.state_index = 5
        g.scaler.copy_(torch.frombuffer(bytearray(bytes(sc)), dtype=torch.uint8))
        torch.cuda.synchronize()
        state0, flat0 = g.state.clone(), g.flat.clone()
        g.step()
        torch.cuda.synchronize()
        dev = g.read_scaler()
        assert dev.error == 1  # ZERO_DEVERR_STATE_INDEX
        assert torch.equal(g.state.view(torch.int32), state0.view(torch.int32))
        assert torch.equal(g.flat, flat0)
    finally:
        g.close()


@pytest.mark.parametrize("beta1,beta2", [(0.95, 0.98), (0.5, 0.75), (0.8, 0.9999)])
@pytest.mark.parametrize("t0", [0, 37, 5000])
@pytest.mark.parametrize("n,two_pass", [(4, False), (8, True)])
def test_bias_corrections_other_betas(beta1, beta2, t0, n, two_pass):
    """Betas other than the workloads' 0.9 / 0.999, from several step counts:
    the bias corrections' integer form on the device (and its fp64 fallback
    once a power is subnormal: 0.5^5000) against the checker's fp64 products,
    element by element, and the stored powers against the fp64 chain."""
    wl = W.Workload("betas", [50_003], n, 0, False, 93, 1e-3, init_scale=256.0, steps=2,
                    beta1=beta1, beta2=beta2, max_grad_norm=0.5 if two_pass else 0.0)
    stats, dev, orc = run_small(wl, two_pass=two_pass, t0=t0)
    p1 = p2 = 1.0
    for _ in range(t0 + 2):
        p1 *= beta1
        p2 *= beta2
    assert dev.t == t0 + 2
    assert dev.beta1_pow == p1 and dev.beta2_pow == p2
