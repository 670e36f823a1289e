"""zero_grad_norm_noalloc: the global-norm call for callers that cannot
allocate device memory (a host framework's allocator owns the GPU's memory,
or a fixed budget leaves no room for a model-sized workspace). It keeps its
tile partials in a fixed array inside the library instead of a caller
workspace; these tests check, through the C ABI, that it gives what the
workspace form gives, on two calls in a row, and that it refuses sizes
beyond its array. Collected last on purpose (file name), so a run that stops
at the first failure has run every other test before it."""
import pytest
import torch

import fsdp_sharded_mixed_shard_gb300 as Z
from fsdp_sharded_mixed_shard_gb300 import harness, workloads as W
from parity_util import norm_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_noalloc_norm_matches_workspace_norm_two_calls():
    wl = W.Workload("noalloc", [300_007, 4096, 13], 4, 50_000, True, 31, 1e-2,
                    max_grad_norm=0.5, steps=2)
    g = harness.Group(wl)
    try:
        g.init_state()
        sc, ws, st = g.scaler.data_ptr(), g.workspace.data_ptr(), g.sptr
        n_elems = g.info.psi_pad
        for step in (1, 2):   # two calls in a row, on different gradients
            g.gen_grads(step)
            Z.zero_reduce_scatter(g.plan, -1, 0, 4, g.rep_ptrs(), 0, g.ghat_ptrs(), sc, 0, 0, st)
            Z.zero_grad_norm(g.plan, 0, 4, g.ghat_ptrs(), g.hp, sc, ws, st)
            want = g.read_scaler()
            Z.zero_grad_norm_noalloc(g.plan, 0, 4, g.ghat_ptrs(), g.hp, sc, st)
            got = g.read_scaler()
            assert abs(got.norm_sq - want.norm_sq) <= norm_tol(n_elems) * want.norm_sq
            assert got.clip_coef == want.clip_coef and got.clip_apply == want.clip_apply
            assert got.norm_step == want.norm_step and got.error == 0
            # the clipped update that follows works from either result
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
        sc, ws, st = g.scaler.data_ptr(), g.workspace.data_ptr(), g.sptr
        Z.zero_reduce_scatter(g.plan, -1, 5, 7, g.rep_ptrs(), g.wbase, g.ghat_ptrs(), sc, 0, 0,
                              st)
        Z.zero_grad_norm(g.plan, 5, 7, g.ghat_ptrs(), g.hp, sc, ws, st)
        want = g.read_scaler()
        Z.zero_grad_norm_noalloc(g.plan, 5, 7, g.ghat_ptrs(), g.hp, sc, st)
        got = g.read_scaler()
        assert abs(got.norm_sq - want.norm_sq) <= norm_tol(g.wlen) * want.norm_sq
        assert got.clip_coef == want.clip_coef
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
