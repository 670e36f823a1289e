"""zero_grad_norm_noalloc: the global-norm call for callers that cannot
allocate device memory (a host framework's allocator owns the GPU's memory,
or a fixed budget leaves no room for a model-sized workspace). It keeps its
tile records in a fixed array inside the library instead of a caller
workspace; these tests check, through the C ABI, that it gives what the
workspace form (zero_grad_norm recomputing from the same gradients) gives,
bit for bit, on calls in a row, and that it refuses sizes beyond its array.
Before every call the scaler's norm fields are overwritten with values no
norm call produces, so a call that launched or wrote nothing fails.
Collected last on purpose (file name), so a run that stops at the first
failure has run every other test before it."""
import pytest
import torch

import fsdp_sharded_mixed_shard_gb300 as Z
from fsdp_sharded_mixed_shard_gb300 import harness, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _poison(g):
    s = g.read_scaler()
    s.norm_sq, s.norm, s.clip_coef, s.clip_apply, s.norm_step = -1.0, -1.0, -1.0, -7, -7
    g.scaler.copy_(torch.frombuffer(bytearray(bytes(s)), dtype=torch.uint8).to(g.device))
    torch.cuda.synchronize()


def _both(g, lo, hi):
    """(workspace form, no-allocation form) of the norm of the owners
    [lo, hi) from the reduced gradients in g.ghat."""
    sc, ws, st = g.scaler.data_ptr(), g.workspace.data_ptr(), g.sptr
    _poison(g)
    Z.zero_grad_norm(g.plan, lo, hi, g.ghat_ptrs(), g.hp, sc, ws, st)
    want = g.read_scaler()
    _poison(g)
    Z.zero_grad_norm_noalloc(g.plan, lo, hi, g.ghat_ptrs(), g.hp, sc, st)
    got = g.read_scaler()
    return want, got


def _assert_same(want, got):
    assert want.norm_step > 0 and want.norm_sq > 0
    assert (got.norm_sq, got.norm, got.clip_coef, got.clip_apply, got.norm_step) == \
        (want.norm_sq, want.norm, want.clip_coef, want.clip_apply, want.norm_step)
    assert got.error == 0


def test_noalloc_norm_matches_workspace_norm_two_calls():
    wl = W.Workload("noalloc", [300_007, 4096, 13], 4, 50_000, True, 31, 1e-2,
                    max_grad_norm=0.5, steps=2)
    g = harness.Group(wl)
    try:
        g.init_state()
        sc, st = g.scaler.data_ptr(), g.sptr
        for step in (1, 2):   # two calls in a row, on different gradients
            g.gen_grads(step)
            Z.zero_reduce_scatter(g.plan, -1, 0, 4, g.rep_ptrs(), 0, g.ghat_ptrs(), sc, 0, 0, st)
            want, got = _both(g, 0, 4)
            _assert_same(want, got)
            assert got.clip_apply == 1
            # the clipped update that follows works from the no-allocation result
            Z.zero_step(g.plan, 0, 4, g._state_ptrs(0), g._state_ptrs(1), g._state_ptrs(2), 1,
                        g.ghat_ptrs(), None, 0, g.flat.data_ptr(), g.hp, sc, 0, st)
            assert g.read_scaler().t == step
    finally:
        g.close()


def test_noalloc_rank_subset():
    wl = W.Workload("noalloc_sub", [64 * 9001], 64, 0, True, 32, 1e-3, max_grad_norm=1e-3,
                    steps=1, rank_lo=5, rank_hi=7)
    g = harness.Group(wl)
    try:
        g.init_state()
        g.gen_grads(1)
        sc, st = g.scaler.data_ptr(), g.sptr
        Z.zero_reduce_scatter(g.plan, -1, 5, 7, g.rep_ptrs(), g.wbase, g.ghat_ptrs(), sc, 0, 0,
                              st)
        want, got = _both(g, 5, 7)
        _assert_same(want, got)
    finally:
        g.close()


def test_noalloc_many_segments_then_a_smaller_call():
    """More segments than one launch takes (several launches, each numbering
    its records from the call's first tile), then a smaller call over fewer
    owners: the second call reads only records it rewrote."""
    numels = [97 + (k * 37) % 500 for k in range(400)]
    wl = W.Workload("noalloc_segs", numels, 8, 101, True, 33, 1e-2, max_grad_norm=0.1, steps=1)
    g = harness.Group(wl)
    try:
        assert g.info.n_segments > 3 * 128
        g.init_state()
        g.gen_grads(1)
        sc, st = g.scaler.data_ptr(), g.sptr
        Z.zero_reduce_scatter(g.plan, -1, 0, 8, g.rep_ptrs(), 0, g.ghat_ptrs(), sc, 0, 0, st)
        big_want, big_got = _both(g, 0, 8)
        _assert_same(big_want, big_got)
        small_want, small_got = _both(g, 6, 8)
        _assert_same(small_want, small_got)
        assert small_got.norm_sq < big_got.norm_sq
    finally:
        g.close()


def test_noalloc_rejects_more_tiles_than_its_array():
    big = Z.ZERO_TILE_ELEMS * ((1 << 19) + 1)
    p = Z.zero_plan_create([big], 1, 0, Z.ZERO_BF16)
    hp = harness.hparams_of(W.Workload("x", [1], 1, max_grad_norm=1.0))
    scaler = torch.zeros(80, dtype=torch.uint8, device="cuda")
    fake = torch.zeros(16, dtype=torch.float32, device="cuda")  # never read: rejected first
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_grad_norm_noalloc(p, 0, 1, [fake.data_ptr()], hp, scaler.data_ptr())
    assert e.value.status == -3
    Z.zero_plan_destroy(p)
