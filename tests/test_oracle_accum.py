"""Pins of the checker's micro-batch accumulation ("How far does splitting
the batch get you?", "What does gradient accumulation actually buy?": run k
micro-batches, accumulate locally in fp32, reduce once)."""
import numpy as np
import pytest
import torch

import oracle
from fsdp_sharded_mixed_shard_gb300 import synth
from test_oracle_step import _np_cast, _np_widen, simulate_ring_reduce_scatter

F32 = np.float32


def test_identical_micro_batches_average_back_exactly():
    # every rank sees k identical micro-batches of x*S: the accumulated sum is
    # k*x*S exactly and the step's gradient is x exactly
    for n, k, S, bf in ((4, 2, 1024.0, False), (8, 3, 1.0, True), (3, 5, 256.0, False)):
        x = F32(3 * 2.0 ** -12)
        bits = oracle.cast16(np.full(16, x * F32(S), F32), bf)
        acc = np.empty(16, F32)
        for mb in range(k):
            oracle.accumulate(bits, acc, bf, first=(mb == 0))
        assert np.all(acc == F32(k) * x * F32(S))
        inv = oracle.unscale_factor_k(S, n, k)
        assert inv == F32(1.0 / (S * n * k))
        g = F32(oracle.ring_sum(np.full(n, acc[0], F32), 0) * inv)
        denom = S * n * k
        if denom == 2.0 ** round(np.log2(denom)):
            assert g == x                      # power of two: exact
        else:
            # one rounding of 1/(S N k) and one of the product
            assert abs(float(g) - float(x)) <= 2 * 2.0 ** -24 * float(x)


def test_accumulation_order_is_micro_batch_order():
    # micro-batches 1, 2^-24, -1: (1 + 2^-24) - 1 = 0 in fp32, 1 + (2^-24 - 1) = 2^-24
    vals = [1.0, 2.0 ** -24, -1.0]
    acc = np.empty(1, F32)
    for i, x in enumerate(vals):
        oracle.accumulate(oracle.cast16([x], True), acc, True, first=(i == 0))
    assert acc[0] == 0.0


def test_one_micro_batch_equals_plain_step():
    n, psi, bf = 4, 3001, True
    p, _, _ = oracle.make_plan([psi], n)
    spec = synth.grad_spec(seed=3, psi=psi)
    reps = [oracle.cast16(synth.grad_f32(p.psi_pad, 0, spec, 1, r), bf) for r in range(n)]
    out = []
    for accum in (False, True):
        hp = oracle.hparams()
        sc = oracle.scaler(1.0)
        master = synth.master_f32(p.psi_pad, 0, 1, psi)
        m = np.zeros(p.psi_pad, F32)
        v = np.zeros(p.psi_pad, F32)
        params = oracle.cast16(master, bf)
        if accum:
            acc = [np.empty(p.psi_pad, F32) for _ in range(n)]
            for r in range(n):
                oracle.accumulate(reps[r], acc[r], bf, first=True)
            oracle.step_arrays_f32(p, 0, n, bf, acc, 1, 0, master, m, v, params, hp, sc)
        else:
            oracle.step_arrays(p, 0, n, bf, reps, 0, master, m, v, params, hp, sc)
        out.append((master, m, v, params))
    for a, b in zip(*out):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("n,k", [(1, 2), (2, 3), (4, 2), (3, 4)])
def test_sharded_accumulated_equals_unsharded(n, k):
    """Independent numpy restatement: fp32 accumulation of each rank's k
    micro-batches, ring sum, fp32(1/(S*N*k)), unsharded AdamW."""
    bf, S = False, 512.0
    numels = [37, 5, 90]
    p, _, _ = oracle.make_plan(numels, n)
    psi, psip, shard = p.psi, p.psi_pad, p.shard
    hp = oracle.hparams()
    sc = oracle.scaler(S)
    master = synth.master_f32(psip, 0, 2, psi)
    m = np.zeros(psip, F32)
    v = np.zeros(psip, F32)
    params = oracle.cast16(master, bf)
    rm, rmm, rv = master.copy(), m.copy(), v.copy()
    for step in (1, 2):
        spec = synth.grad_spec(seed=k, sigma=1e-3, loss_scale=S, psi=psi)
        micro = [[oracle.cast16(synth.grad_f32(psip, 0, spec, step * 64 + mb, r), bf)
                  for r in range(n)] for mb in range(1, k + 1)]
        acc = [np.empty(psip, F32) for _ in range(n)]
        for mb in range(k):
            for r in range(n):
                oracle.accumulate(micro[mb][r], acc[r], bf, first=(mb == 0))
        oracle.step_arrays_f32(p, 0, n, bf, acc, k, 0, master, m, v, params, hp, sc)
        # numpy side
        nacc = [_np_widen(micro[0][r], bf) for r in range(n)]
        for mb in range(1, k):
            nacc = [(nacc[r] + _np_widen(micro[mb][r], bf)).astype(F32) for r in range(n)]
        vals = np.stack(nacc)
        g = np.empty(psip, F32)
        for j in range(psip):
            owner = j // shard
            chunk = np.zeros((n, n), F32)
            chunk[:, owner] = vals[:, j]
            g[j] = simulate_ring_reduce_scatter(chunk)[owner]
        g = (g * F32(1.0 / (S * n * k))).astype(F32)
        rmm = (F32(hp.beta1) * rmm + F32(1 - hp.beta1) * g).astype(F32)
        rv = (F32(hp.beta2) * rv + F32(1 - hp.beta2) * (g * g)).astype(F32)
        mh = rmm / F32(1 - hp.beta1 ** step)
        vh = rv / F32(1 - hp.beta2 ** step)
        u = mh / (np.sqrt(vh) + F32(hp.eps))
        rm = (rm * F32(1 - hp.lr * hp.weight_decay) - F32(hp.lr) * u).astype(F32)
        assert np.array_equal(master, rm) and np.array_equal(m, rmm) and np.array_equal(v, rv)
        assert np.array_equal(params, _np_cast(rm, bf))


@pytest.mark.parametrize("k", [2, 4])
def test_single_rank_accumulated_matches_torch(k):
    """N = 1, scale 1: torch accumulates p.grad over k micro-batches (fp32 +=),
    divides by k (exact for k a power of two) and steps AdamW."""
    psi, bf = 2049, True
    p, _, _ = oracle.make_plan([psi], 1)
    hp = oracle.hparams(lr=1e-3, weight_decay=0.01)
    sc = oracle.scaler(1.0)
    master = synth.master_f32(psi, 0, 4, psi)
    m = np.zeros(psi, F32)
    v = np.zeros(psi, F32)
    params = oracle.cast16(master, bf)
    w = torch.nn.Parameter(torch.from_numpy(master.copy()))
    opt = torch.optim.AdamW([w], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    for step in (1, 2, 3):
        spec = synth.grad_spec(seed=9, psi=psi)
        acc = np.empty(psi, F32)
        grad = None
        for mb in range(1, k + 1):
            h = oracle.cast16(synth.grad_f32(psi, 0, spec, step * 64 + mb, 0), bf)
            oracle.accumulate(h, acc, bf, first=(mb == 1))
            gt = torch.from_numpy(_np_widen(h, bf))
            grad = gt.clone() if grad is None else grad + gt
        oracle.step_arrays_f32(p, 0, 1, bf, [acc], k, 0, master, m, v, params, hp, sc)
        w.grad = grad / k
        opt.step()
        assert np.allclose(master, w.detach().numpy(), rtol=1e-6, atol=1e-9)
