"""Pins of the checker's step: ring-order reduction (simulated ring,
exact sums), unscale, AdamW (closed form at step 1, torch.optim.AdamW),
sharded == unsharded, clip, skip and loss-scale bookkeeping."""
import math

import numpy as np
import pytest
import torch

import oracle
from fsdp_sharded_mixed_shard_gb300 import synth

F32 = np.float32
U = 2.0 ** -24


# ----------------------------------------------------------- ring order ----

def simulate_ring_reduce_scatter(vals):
    """Literal ring reduce-scatter of one element per chunk: at hop s every
    rank r passes its running partial of chunk (r - 1 - s) mod d to rank r+1,
    which adds its own contribution (fp32). After d-1 hops rank i holds the
    full sum of chunk i. vals[r][c] = rank r's value of chunk c."""
    d = len(vals)
    buf = [[F32(vals[r][c]) for c in range(d)] for r in range(d)]
    for s in range(d - 1):
        sent = [(r, (r - 1 - s) % d, buf[r][(r - 1 - s) % d]) for r in range(d)]
        for r, c, part in sent:
            dst = (r + 1) % d
            buf[dst][c] = F32(part + buf[dst][c])
    return [buf[i][i] for i in range(d)]


def test_ring_order_matches_simulated_ring():
    rng = np.random.default_rng(0)
    for d in (1, 2, 3, 5, 8, 16):
        for _ in range(20):
            vals = rng.standard_normal((d, d)).astype(F32) * F32(10.0) ** rng.integers(-6, 6, (d, d)).astype(F32)
            want = simulate_ring_reduce_scatter(vals)
            for i in range(d):
                got = oracle.ring_sum(vals[:, i], i)
                assert got == want[i] or (np.isnan(got) and np.isnan(want[i]))


def test_ring_order_crafted_cancellation():
    # ranks hold 1, 2^-24, -1: only the ring order gives (2^-24, 2^-24, 0)
    vals = np.array([1.0, U, -1.0], dtype=F32)
    got = [oracle.ring_sum(vals, i) for i in range(3)]
    assert got == [F32(U), F32(U), F32(0.0)]


def test_ring_sum_error_bound_against_exact_sum():
    rng = np.random.default_rng(1)
    for n in (2, 3, 8, 16, 64):
        g = n * U / (1 - n * U)
        for _ in range(50):
            vals = (rng.standard_normal(n) * 1e-3).astype(F32)
            for owner in (0, n - 1):
                s = float(oracle.ring_sum(vals, owner))
                exact = math.fsum(float(x) for x in vals)
                assert abs(s - exact) <= g * sum(abs(float(x)) for x in vals)


def test_single_rank_is_identity():
    for x in (0.0, 1.5, -3.25e-5, float("inf")):
        assert oracle.ring_sum(np.array([x], F32), 0) == F32(x)


def test_unscale_exact_average():
    # N identical replicas holding x*S average back to x exactly (x with few
    # significant bits, so every partial sum is exact)
    for n, S in ((4, 1024.0), (8, 65536.0), (16, 1.0), (64, 1.0)):
        inv = oracle.unscale_factor(S, n)
        assert inv == F32(1.0 / (S * n))
        for x in (F32(3 * 2.0 ** -12), F32(-5 * 2.0 ** -14), F32(0.125)):
            vals = np.full(n, F32(x) * F32(S), dtype=F32)
            assert F32(oracle.ring_sum(vals, 0) * inv) == x
    assert oracle.unscale_factor(1.0, 3) == F32(1.0 / 3.0)


# ----------------------------------------------------------------- adamw ----

def test_adamw_step1_closed_form():
    """At t = 1, m_hat = g and v_hat = g^2, so
    theta_1 = theta_0 (1 - lr wd) - lr g / (|g| + eps) (up to fp32 rounding)."""
    hp = oracle.hparams(lr=1e-3, weight_decay=0.01, eps=1e-8)
    a = oracle.adam_scalars(hp, 1)
    rng = np.random.default_rng(2)
    for _ in range(200):
        th0 = F32(rng.uniform(-0.05, 0.05))
        g = F32(rng.standard_normal() * 10.0 ** rng.integers(-6, 0))
        th, m, v = oracle.adamw_elem(th0, 0.0, 0.0, g, a)
        want = float(th0) * (1 - 1e-3 * 0.01) - 1e-3 * float(g) / (abs(float(g)) + 1e-8)
        assert abs(float(th) - want) <= 4e-7 * abs(want) + 1e-9
        assert m == pytest.approx(0.1 * float(g), rel=1e-6)
        assert v == pytest.approx(0.001 * float(g) ** 2, rel=1e-6)


def test_adamw_zero_gradient_keeps_decay_only():
    hp = oracle.hparams(lr=1e-2, weight_decay=0.1)
    a = oracle.adam_scalars(hp, 3)
    th, m, v = oracle.adamw_elem(0.5, 0.0, 0.0, 0.0, a)
    assert th == F32(F32(0.5) * F32(1 - 1e-3)) and m == 0 and v == 0


def test_bias_correction_scalars():
    hp = oracle.hparams(beta1=0.9, beta2=0.999)
    for t in (1, 2, 10, 1000):
        a = oracle.adam_scalars(hp, t)
        assert a.bc1 == pytest.approx(1 - 0.9 ** t, rel=1e-6)
        assert a.bc2 == pytest.approx(1 - 0.999 ** t, rel=1e-6)
    a = oracle.adam_scalars(hp, 1)
    assert a.bc1 == a.omb1 and a.bc2 == a.omb2


def _gen_replicas(n_ranks, psip, psi, is_bf16, step, seed=0, sigma=1e-3, scale=1.0):
    spec = synth.grad_spec(seed=seed, sigma=sigma, loss_scale=scale, psi=psi)
    return [oracle.cast16(synth.grad_f32(psip, 0, spec, step, r), is_bf16)
            for r in range(n_ranks)]


@pytest.mark.parametrize("is_bf16", [False, True])
def test_single_rank_matches_torch_adamw(is_bf16):
    """N = 1 and loss scale 1: the step is plain AdamW on the fp32 master
    (torch.optim.AdamW, CPU, fp32)."""
    psi = 4099
    p, _, _ = oracle.make_plan([psi], 1)
    hp = oracle.hparams(lr=1e-3, weight_decay=0.01)
    sc = oracle.scaler(1.0)
    master = synth.master_f32(psi, 0, 7, psi)
    m = np.zeros(psi, F32)
    v = np.zeros(psi, F32)
    params = oracle.cast16(master, is_bf16)
    w = torch.nn.Parameter(torch.from_numpy(master.copy()))
    opt = torch.optim.AdamW([w], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    for step in range(1, 6):
        reps = _gen_replicas(1, psi, psi, is_bf16, step)
        oracle.step_arrays(p, 0, 1, is_bf16, reps, 0, master, m, v, params, hp, sc)
        w.grad = torch.from_numpy(oracle.widen16(reps[0], is_bf16))
        opt.step()
        ref = w.detach().numpy()
        assert np.allclose(master, ref, rtol=1e-6, atol=1e-9)
        st = opt.state[w]
        assert np.allclose(m, st["exp_avg"].numpy(), rtol=1e-5, atol=1e-6 * np.abs(m).max())
        assert np.allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-5, atol=1e-6 * np.abs(v).max())
    assert sc.t == 5
    assert np.array_equal(params, oracle.cast16(master, is_bf16))


def _np_cast(x, is_bf16):
    if is_bf16:
        return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return x.astype(np.float16).view(np.uint16)


def _np_widen(h, is_bf16):
    if is_bf16:
        return torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    return h.view(np.float16).astype(F32)


def unsharded_reference_step(reps, is_bf16, scale, master, m, v, hp, t, shard):
    """Independent numpy restatement: average the gradient with the simulated
    ring, then one AdamW step over the whole (unsharded) vector."""
    n = len(reps)
    vals = np.stack([_np_widen(r, is_bf16) for r in reps])      # [rank, elem]
    psip = vals.shape[1]
    g = np.empty(psip, F32)
    for j in range(psip):
        owner = j // shard
        chunk = np.zeros((n, n), F32)
        chunk[:, owner] = vals[:, j]
        g[j] = simulate_ring_reduce_scatter(chunk)[owner]
    g = (g * F32(1.0 / (scale * n))).astype(F32)
    b1, b2 = F32(hp.beta1), F32(hp.beta2)
    m = (b1 * m + F32(1 - hp.beta1) * g).astype(F32)
    v = (b2 * v + F32(1 - hp.beta2) * (g * g)).astype(F32)
    mh = m / F32(1 - hp.beta1 ** t)
    vh = v / F32(1 - hp.beta2 ** t)
    u = mh / (np.sqrt(vh) + F32(hp.eps))
    th = master * F32(1 - hp.lr * hp.weight_decay)
    th = (th - F32(hp.lr) * u).astype(F32)
    return th, m, v, _np_cast(th, is_bf16)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 7])
@pytest.mark.parametrize("is_bf16", [False, True])
def test_sharded_equals_unsharded(n, is_bf16):
    rng = np.random.default_rng(n)
    for trial in range(4):
        numels = [int(x) for x in rng.integers(0, 20, rng.integers(1, 5))]
        psi = sum(numels)
        p, _, _ = oracle.make_plan(numels, n)
        psip, S = p.psi_pad, p.shard
        scale = 1024.0 if not is_bf16 else 1.0
        hp = oracle.hparams()
        sc = oracle.scaler(scale)
        master = synth.master_f32(psip, 0, trial, psi)
        m = np.zeros(psip, F32)
        v = np.zeros(psip, F32)
        params = oracle.cast16(master, is_bf16)
        rm, rmm, rv = master.copy(), m.copy(), v.copy()
        for step in range(1, 4):
            reps = _gen_replicas(n, psip, psi, is_bf16, step, seed=trial, scale=scale)
            oracle.step_arrays(p, 0, n, is_bf16, reps, 0, master, m, v, params, hp, sc)
            if psip == 0:
                continue
            rm, rmm, rv, rp = unsharded_reference_step(reps, is_bf16, scale, rm, rmm, rv, hp,
                                                       step, S)
            assert np.array_equal(master, rm) and np.array_equal(m, rmm)
            assert np.array_equal(v, rv) and np.array_equal(params, rp)


# ----------------------------------------------------------- clip / norm ----

def _const_replicas(n, psip, value, is_bf16=True):
    return [oracle.cast16(np.full(psip, value, F32), is_bf16) for _ in range(n)]


def test_clip_all_ones_norm_is_sqrt_psi():
    n, psi = 2, 4096
    p, _, _ = oracle.make_plan([psi], n)
    hp = oracle.hparams(max_grad_norm=1.0)
    sc = oracle.scaler(1.0)
    master = np.zeros(psi, F32)
    m = np.zeros(psi, F32)
    v = np.zeros(psi, F32)
    params = np.zeros(psi, np.uint16)
    oracle.step_arrays(p, 0, n, True, _const_replicas(n, psi, 1.0), 0, master, m, v, params,
                       hp, sc)
    assert sc.norm_sq == psi and sc.norm == 64.0
    assert sc.clip_coef == F32(1.0 / (64.0 + 1e-6))
    # m after step 1 = (1 - b1) * g * c
    assert m[0] == F32(F32(0.1) * F32(1.0 * sc.clip_coef))


def test_clip_inactive_is_bit_identical_to_no_clip():
    n, psi = 4, 1000
    p, _, _ = oracle.make_plan([psi], n)
    states = []
    for mx in (0.0, 1e9):
        hp = oracle.hparams(max_grad_norm=mx)
        sc = oracle.scaler(1.0)
        master = synth.master_f32(psi, 0, 1, psi)
        m = np.zeros(psi, F32)
        v = np.zeros(psi, F32)
        params = oracle.cast16(master, True)
        for step in (1, 2):
            oracle.step_arrays(p, 0, n, True, _gen_replicas(n, psi, psi, True, step), 0,
                               master, m, v, params, hp, sc)
        states.append((master, m, v, params))
    for a, b in zip(*states):
        assert np.array_equal(a, b)


def test_norm_chunked_sum_within_fp64_bound():
    n, psi = 1, (1 << 20) * 2 + 12345
    p, _, _ = oracle.make_plan([psi], n)
    hp = oracle.hparams(max_grad_norm=1.0)
    sc = oracle.scaler(1.0)
    reps = _gen_replicas(n, psi, psi, True, 1)
    g = oracle.widen16(reps[0], True).astype(np.float64)
    exact = math.fsum((g * g).tolist())
    master = np.zeros(psi, F32)
    oracle.step_arrays(p, 0, n, True, reps, 0, master, np.zeros(psi, F32), np.zeros(psi, F32),
                       np.zeros(psi, np.uint16), hp, sc)
    assert abs(sc.norm_sq - exact) <= psi * 2.0 ** -53 * exact


def _torch_clip(grads, max_norm):
    """torch.nn.utils.clip_grad_norm_ on fp64 CPU tensors: an outside
    implementation of the same convention (total L2 norm over all tensors,
    coefficient max_norm / (norm + 1e-6), clamped at 1). Returns (norm, the
    multiplier it applied, the clipped gradients)."""
    import torch
    ps = []
    for g in grads:
        t = torch.zeros(len(g), dtype=torch.float64, requires_grad=True)
        t.grad = torch.tensor(g, dtype=torch.float64)
        ps.append(t)
    before = [p.grad.clone() for p in ps]
    total = float(torch.nn.utils.clip_grad_norm_(ps, max_norm, norm_type=2.0))
    after = [p.grad.numpy().copy() for p in ps]
    k = int(np.argmax(np.abs(before[0].numpy())))
    mult = float(after[0][k] / before[0][k].item())
    return total, mult, after


@pytest.mark.parametrize("case", range(12))
def test_clip_coef_matches_torch_clip_grad_norm(case):
    """orc_clip_coef against torch's clip_grad_norm_ on fp64 gradients,
    norms on both sides of max_norm: the same apply decision, the same
    norm (to fp64 rounding) and, when it clips, the same coefficient after
    rounding to fp32 (one ulp when torch's norm and the checker's sit on
    either side of an fp32 rounding boundary). A misplaced eps
    (max/norm + eps) moves c by ~eps/c, i.e. many fp32 ulps at these norms."""
    rng = np.random.default_rng(1000 + case)
    sizes = [int(x) for x in rng.integers(1, 5000, size=int(rng.integers(1, 5)))]
    scale = float(10.0 ** rng.uniform(-4, 2))
    grads = [rng.standard_normal(n) * scale for n in sizes]
    max_norm = float(rng.choice([0.05, 0.5, 1.0, 3.0, 1e3]))
    nsq = math.fsum(float(x) * float(x) for g in grads for x in g)
    apply, c, nrm = oracle.clip_coef(nsq, max_norm)
    total, mult, after = _torch_clip(grads, max_norm)
    assert nrm == pytest.approx(total, rel=4e-16)
    assert apply == (mult < 1.0)
    if apply:
        assert abs(float(c) - float(F32(mult))) <= 2.0 ** -23 * float(c)
        for g, a in zip(grads, after):
            want = np.asarray(g) * float(c)
            assert np.allclose(a, want, rtol=2.0 ** -22, atol=0.0)
    else:
        assert c == 1.0 and mult == 1.0
        for g, a in zip(grads, after):
            assert np.array_equal(a, np.asarray(g))


def test_clip_coef_at_and_near_the_limit():
    """Norms just below, at and above the point where c reaches 1, against
    torch. Within an ulp of that point the fp64 test c < 1 follows the norm's
    last bit (torch's norm and sqrt of the checker's sum may differ there),
    but the fp32 multiplier that reaches the gradient is 1.0 on both sides;
    further out the decisions agree."""
    for max_norm in (1.0, 0.25, 7.0):
        x = max_norm - 1e-6
        for nrm in (np.nextafter(x, 0.0), x, np.nextafter(x, 2 * x), 0.5 * max_norm,
                    2 * max_norm):
            g = [[float(nrm)]]
            apply, c, got = oracle.clip_coef(float(nrm) * float(nrm), max_norm)
            total, mult, _ = _torch_clip(g, max_norm)
            effective = float(c) if apply else 1.0
            assert effective == float(F32(mult)), (max_norm, nrm, c, mult)
            if nrm in (0.5 * max_norm, 2 * max_norm):
                assert apply == (mult < 1.0)


# ------------------------------------------------------- skip and scaler ----

@pytest.mark.parametrize("bad", [0x7C00, 0xFC00, 0x7E00])
@pytest.mark.parametrize("where", ["first", "last", "pad", "bucket_edge"])
def test_overflow_skips_whole_step(bad, where):
    n, psi, bsz = 4, 1001, 128
    p, _, _ = oracle.make_plan([psi], n, bsz)
    psip = p.psi_pad
    j = {"first": 0, "last": psi - 1, "pad": psip - 1, "bucket_edge": 2 * bsz}[where]
    hp = oracle.hparams(dynamic_scale=1)
    sc = oracle.scaler(65536.0)
    master = synth.master_f32(psip, 0, 3, psi)
    m = np.full(psip, 1e-4, F32)
    v = np.full(psip, 1e-8, F32)
    params = oracle.cast16(master, False)
    before = [a.copy() for a in (master, m, v, params)]
    sc.t = 2
    reps = _gen_replicas(n, psip, psi, False, 3, sigma=1e-4, scale=65536.0)
    reps[1][j] = bad
    flags = np.zeros(p.n_buckets, np.uint32)
    oracle.step_arrays(p, 0, n, False, reps, 0, master, m, v, params, hp, sc, flags)
    for a, b in zip((master, m, v, params), before):
        assert np.array_equal(a, b)
    assert sc.overflow == 1 and sc.t == 2 and sc.scale == 32768.0 and sc.good_steps == 0
    want = np.zeros(p.n_buckets, np.uint32)
    want[j // bsz] = 1
    assert np.array_equal(flags, want)


def test_scaler_bookkeeping():
    hp = oracle.hparams(dynamic_scale=1, growth_interval=3)
    sc = oracle.scaler(4.0)
    for _ in range(3):
        oracle.scaler_finish(sc, hp, 0)
    assert sc.scale == 8.0 and sc.t == 3 and sc.good_steps == 0
    for _ in range(5):
        oracle.scaler_finish(sc, hp, 1)
    assert sc.scale == 1.0 and sc.t == 3          # halved, floor 1
    static = oracle.hparams(dynamic_scale=0)
    sc = oracle.scaler(1024.0)
    oracle.scaler_finish(sc, static, 1)
    assert sc.scale == 1024.0 and sc.overflow == 1 and sc.t == 0


# ------------------------------------------- generator-driven == arrays ----

@pytest.mark.parametrize("case", ["plain", "clip", "inject", "bias_outliers", "subset"])
def test_gen_driver_matches_array_driver(case):
    n, numels, bsz, bf16 = 8, [300, 7000, 5], 1000, True
    spec = dict(seed=5, sigma=1e-3, psi=sum(numels))
    hp = oracle.hparams()
    inject = None
    rlo, rhi = 0, n
    scale = 1.0
    if case == "clip":
        hp = oracle.hparams(max_grad_norm=0.05)
    if case == "inject":
        bf16, scale = False, 512.0
        hp = oracle.hparams(dynamic_scale=1, max_grad_norm=1.0)
        inject = (2, 5, 4000, 0x7C00)
    if case == "bias_outliers":
        spec.update(bias_sigma=1e-5, outliers=True)
    if case == "subset":
        rlo, rhi = 2, 5
    p, _, _ = oracle.make_plan(numels, n, bsz)
    psip, S = p.psi_pad, p.shard
    lo, hi = rlo * S, rhi * S
    sp = synth.grad_spec(**spec)
    g = oracle.gen(sp, bf16, inject)
    sc_a, sc_g = oracle.scaler(scale), oracle.scaler(scale)
    master = synth.master_f32(psip, 0, 9, sp.psi)
    m = np.zeros(psip, F32)
    v = np.zeros(psip, F32)
    params = oracle.cast16(master, bf16)
    elems = np.array(sorted({lo, hi - 1, (lo + hi) // 2, lo + 999, lo + 1000}), np.int64)
    gm, gmm, gv, gp = master[elems].copy(), m[elems].copy(), v[elems].copy(), params[elems].copy()
    for step in (1, 2, 3):
        sp_step = synth.grad_spec(**spec, loss_scale=sc_a.scale)
        reps = [oracle.cast16(synth.grad_f32(psip, 0, sp_step, step, r), bf16) for r in range(n)]
        if inject and inject[0] == step:
            reps[inject[1]][inject[2]] = inject[3]
        fa = np.zeros(p.n_buckets, np.uint32)
        fg = np.zeros(p.n_buckets, np.uint32)
        oracle.step_arrays(p, rlo, rhi, bf16, reps, 0, master, m, v, params, hp, sc_a, fa)
        oracle.gen_step(p, rlo, rhi, g, step, elems, gm, gmm, gv, gp, hp, sc_g, fg, n_threads=3)
        assert np.array_equal(fa, fg)
        assert (sc_a.t, sc_a.scale, sc_a.overflow) == (sc_g.t, sc_g.scale, sc_g.overflow)
        assert sc_a.norm_sq == sc_g.norm_sq
        for a, b in ((master, gm), (m, gmm), (v, gv), (params, gp)):
            assert np.array_equal(a[elems], b)
    if case == "inject":
        assert sc_a.t == 2 and sc_a.scale == 256.0
