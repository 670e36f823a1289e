"""Shared helpers of the GPU parity tests: run a workload through libzero and
through the CPU checker on the same seeded inputs and compare."""
import json
import os

import numpy as np
import torch

import oracle
from fsdp_sharded_mixed_shard_gb300 import harness, synth

F32 = np.float32

# acceptance bars
MASTER_REL = 1e-6        # fp32 master / exp_avg / exp_avg_sq: max relative error
PARAM_EXACT_FRAC = 0.9999
PARAM_MAX_ULP = 1


def oracle_hp(wl):
    return oracle.hparams(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps,
                          weight_decay=wl.weight_decay, max_grad_norm=wl.max_grad_norm,
                          dynamic_scale=int(wl.dynamic_scale),
                          growth_interval=wl.growth_interval)


def rel_err(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    d = np.abs(got - want) / np.maximum(np.abs(want), np.finfo(np.float64).tiny)
    d[same] = 0.0
    return float(d.max()) if d.size else 0.0


def ulp_diff16(a, b):
    """Distance in representable 16-bit values (same-sign encodings)."""
    a = np.asarray(a, np.int64)
    b = np.asarray(b, np.int64)

    def ordered(x):
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)

    return np.abs(ordered(a) - ordered(b))


def assert_params(got, want):
    got = np.asarray(got, np.uint16)
    want = np.asarray(want, np.uint16)
    if got.size == 0:
        return
    exact = (got == want).mean()
    assert exact >= PARAM_EXACT_FRAC, "params exact fraction %.6f" % exact
    assert ulp_diff16(got, want).max() <= PARAM_MAX_ULP


def assert_state(got, want, what):
    e = rel_err(got, want)
    assert e <= MASTER_REL, "%s max rel err %.3g" % (what, e)


def norm_tol(n_elems, n_tiles, n_ranks):
    """Relative tolerance on norm^2 between the device and the checker, the
    sum of two bounds (every square is exact on both sides, all terms are
    non-negative, so every partial sum is at most the total):
      checker: fp64 recursive sums, in chunks of 2^20 elements, chunk sums
        added in order: at most (min(n, 2^20) + ceil(n / 2^20)) * 2^-53;
      device: fp32 float-float (hi, lo) additions and merges, the total kept
        as hi + lo in fp64; along a chain of k of them lo holds at most
        k * 2^-23 of the partial sum and each rounding of lo errs by 2^-24 of
        that, so a chain of at most L additions errs by at most L^2 * 2^-47.
        L = 16 (a thread's elements of one tile) + 21 (the tile record: 16
        per lane, 5 shuffle levels) + ceil(T / 4096) (a finish thread's
        share of one owner's at most T tiles) + 8 (the CTA tree) + 4 (the 16
        shares of an owner) + N (owner records merged in order).
    """
    oracle = (min(n_elems, 1 << 20) + -(-n_elems // (1 << 20))) * 2.0 ** -53
    chain = 16 + 21 + -(-n_tiles // 4096) + 8 + 4 + n_ranks
    return oracle + chain * chain * 2.0 ** -47


def compare_scaler(dev, orc, n_elems, clip, n_tiles, n_ranks):
    assert dev.t == orc.t, (dev.t, orc.t)
    assert dev.scale == orc.scale, (dev.scale, orc.scale)
    assert dev.overflow == orc.overflow
    assert dev.good_steps == orc.good_steps
    assert dev.error == 0
    if clip and not orc.overflow:
        assert abs(dev.norm_sq - orc.norm_sq) <= norm_tol(n_elems, n_tiles, n_ranks) * orc.norm_sq
        if dev.clip_coef != orc.clip_coef:
            # only a norm at an fp32 rounding boundary may move c by one ulp
            assert abs(float(dev.clip_coef) - float(orc.clip_coef)) <= \
                2.0 ** -23 * abs(float(orc.clip_coef))


def report(wl, step, mode, n_compared, dev, orc, got, want, flags_equal):
    """One JSON line of parity statistics per workload and step, appended to
    the file named by PARITY_REPORT (no-op when unset)."""
    path = os.environ.get("PARITY_REPORT")
    if not path:
        return
    gm, gmm, gv, gp = got
    m, mm, v, p = want
    gp = np.asarray(gp, np.uint16)
    p = np.asarray(p, np.uint16)
    rec = {"workload": wl.name, "step": step, "mode": mode, "elements": int(n_compared),
           "master_max_rel": rel_err(gm, m), "exp_avg_max_rel": rel_err(gmm, mm),
           "exp_avg_sq_max_rel": rel_err(gv, v),
           "master_bit_exact": bool(np.array_equal(np.asarray(gm, np.float32).view(np.uint32),
                                                   np.asarray(m, np.float32).view(np.uint32))),
           "params_exact_frac": float((gp == p).mean()) if gp.size else 1.0,
           "params_max_ulp": int(ulp_diff16(gp, p).max()) if gp.size else 0,
           "flags_equal": bool(flags_equal), "t": dev.t, "t_checker": orc.t,
           "scale": dev.scale, "scale_checker": orc.scale, "overflow": dev.overflow,
           "norm_rel_diff": (abs(dev.norm_sq - orc.norm_sq) / orc.norm_sq
                             if orc.norm_sq > 0 else 0.0)}
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def set_step_count(g, t0):
    """Put the group's scaler at step t0, as t0 good steps would leave it:
    the beta powers formed by t0 successive fp64 products."""
    dev = g.read_scaler()
    p1 = p2 = 1.0
    for _ in range(t0):
        p1 *= g.wl.beta1
        p2 *= g.wl.beta2
    dev.t, dev.beta1_pow, dev.beta2_pow = t0, p1, p2
    g.scaler.copy_(torch.frombuffer(bytearray(bytes(dev)), dtype=torch.uint8))
    return p1, p2


def run_small(wl, per_bucket=False, two_pass=None, check_replicas=True, n_sets=None, t0=0):
    """Full element-wise comparison over every step of `wl` (from step t0 + 1
    when t0 > 0). Returns the per-step max relative errors for reporting."""
    g = harness.Group(wl, two_pass=two_pass, n_sets=n_sets)
    try:
        g.init_state()
        p, _, _ = oracle.make_plan(wl.numels, wl.n_ranks, wl.bucket_elems)
        lo, hi = wl.ranks
        S = p.shard
        wbase, wlen = lo * S, (hi - lo) * S
        bf = wl.is_bf16
        hp = oracle_hp(wl)
        sc = oracle.scaler(wl.init_scale)
        if t0:
            set_step_count(g, t0)
            sc.t = t0
        master = synth.master_f32(wlen, wbase, wl.seed, wl.psi)
        m = np.zeros(wlen, F32)
        v = np.zeros(wlen, F32)
        params = oracle.cast16(master, bf)
        assert np.array_equal(g.params_u16(), params), "initial working copy"
        stats = []
        k_micro = wl.n_micro
        for step in range(1, wl.steps + 1):
            spec = synth.grad_spec(seed=wl.seed, sigma=wl.sigma, bias_sigma=wl.bias_sigma,
                                   loss_scale=sc.scale, outliers=wl.outliers, psi=wl.psi)
            # checker side: every micro-batch generated on the host, accumulated in fp32
            acc = [np.empty(wlen, np.float32) for _ in range(wl.n_ranks)]
            for mb in range(1, k_micro + 1):
                key = wl.gen_step(step, mb)
                reps = [oracle.cast16(synth.grad_f32(wlen, wbase, spec, key, r), bf)
                        for r in range(wl.n_ranks)]
                if mb == k_micro and wl.inject is not None and wl.inject[0] == step:
                    _, r, e, bits = wl.inject
                    if wbase <= e < wbase + wlen:
                        reps[r][e - wbase] = bits
                if k_micro > 1:
                    for r in range(wl.n_ranks):
                        oracle.accumulate(reps[r], acc[r], bf, first=(mb == 1))
            # device side: the same micro-batches, the last one fused into the reduce
            if k_micro > 1:
                g.step_micro(step, per_bucket=per_bucket)
            else:
                g.gen_grads(step)
                g.step(per_bucket=per_bucket)
            flags = np.zeros(max(p.n_buckets, 1), np.uint32)
            if k_micro > 1:
                oracle.step_arrays_f32(p, lo, hi, bf, acc, k_micro, wbase, master, m, v, params,
                                       hp, sc, flags)
            else:
                oracle.step_arrays(p, lo, hi, bf, reps, wbase, master, m, v, params, hp, sc,
                                   flags)
            if check_replicas and wlen:
                assert np.array_equal(g.replicas_u16(), np.stack(reps)), "generator parity"
            dev = g.read_scaler()
            gm, gmm, gv = (t.numpy() for t in g.current_state())
            report(wl, step, "full", wlen, dev, sc, (gm, gmm, gv, g.params_u16()),
                   (master, m, v, params), np.array_equal(g.flags_u32(), flags[:p.n_buckets]))
            compare_scaler(dev, sc, wlen, wl.max_grad_norm > 0, g.info.n_tiles, wl.n_ranks)
            assert np.array_equal(g.flags_u32(), flags[:p.n_buckets])
            assert_state(gm, master, "master")
            assert_state(gmm, m, "exp_avg")
            assert_state(gv, v, "exp_avg_sq")
            assert_params(g.params_u16(), params)
            stats.append((rel_err(gm, master), rel_err(gmm, m), rel_err(gv, v),
                          float((g.params_u16() == params).mean()) if wlen else 1.0))
        return stats, g.read_scaler(), sc
    finally:
        g.close()
        del g
        torch.cuda.empty_cache()


def sample_elems(wl, p, n_random=2048, seed=0):
    """Sampled flat indices inside the processed owners' slices: slice and
    bucket edges, padding, the injected element, and random ones."""
    lo, hi = wl.ranks
    a, b = lo * p.shard, hi * p.shard
    pts = set()
    for i in range(lo, hi + 1):
        for d in (-9, -8, -1, 0, 1, 7, 8):
            pts.add(i * p.shard + d)
    if p.bucket_elems:
        for k in range(1, p.n_buckets):
            for d in (-1, 0, 1):
                pts.add(k * p.bucket_elems + d)
    for d in (-2, -1, 0, 1):
        pts.add(p.psi + d)
    if wl.inject is not None:
        pts.add(wl.inject[2])
    for edge in (2 ** 31, 2 ** 32):  # where 32-bit index arithmetic would wrap
        for d in (-2, -1, 0, 1, 2):
            pts.add(edge + d)
    rng = np.random.default_rng(seed)
    if b > a:
        pts.update(rng.integers(a, b, n_random).tolist())
    e = np.array(sorted(x for x in pts if a <= x < b), dtype=np.int64)
    return e


def gather_state(g, elems):
    idx_set = g.read_scaler().state_index if g.n_sets == 2 else 0
    i = elems // g.S
    k = elems - i * g.S
    flat_idx = torch.from_numpy((i - g.lo) * g.srow + k).to(g.device)
    out = []
    for which in range(3):
        t = g.state[idx_set, which].reshape(-1)
        out.append(t.index_select(0, flat_idx).cpu().numpy())
    w = torch.from_numpy(elems - g.wbase).to(g.device)
    params = g.flat.index_select(0, w).cpu().numpy().view(np.uint16)
    return out[0], out[1], out[2], params


def run_sampled(wl, steps=None, n_random=2048, n_threads=None, n_sets=None):
    """Full-size run on the device; the checker regenerates every input on
    the host, computes the global quantities (flags, overflow, norm) over all
    elements and the updates of the sampled elements."""
    steps = wl.steps if steps is None else steps
    g = harness.Group(wl, n_sets=n_sets)
    try:
        g.init_state()
        p, _, _ = oracle.make_plan(wl.numels, wl.n_ranks, wl.bucket_elems)
        elems = sample_elems(wl, p, n_random)
        bf = wl.is_bf16
        hp = oracle_hp(wl)
        sc = oracle.scaler(wl.init_scale)
        master = synth.master_f32_at(elems, wl.seed, wl.psi)
        m = np.zeros(len(elems), F32)
        v = np.zeros(len(elems), F32)
        params = oracle.cast16(master, bf)
        spec = synth.grad_spec(seed=wl.seed, sigma=wl.sigma, bias_sigma=wl.bias_sigma,
                               loss_scale=1.0, outliers=wl.outliers, psi=wl.psi)
        gen = oracle.gen(spec, bf, wl.inject)
        lo, hi = wl.ranks
        for step in range(1, steps + 1):
            g.gen_grads(step)
            g.step()
            flags = np.zeros(max(p.n_buckets, 1), np.uint32)
            oracle.gen_step(p, lo, hi, gen, step, elems, master, m, v, params, hp, sc, flags,
                            n_threads=n_threads)
            dev = g.read_scaler()
            gm, gmm, gv, gp = gather_state(g, elems)
            report(wl, step, "sampled", len(elems), dev, sc, (gm, gmm, gv, gp),
                   (master, m, v, params), np.array_equal(g.flags_u32(), flags[:p.n_buckets]))
            compare_scaler(dev, sc, (hi - lo) * p.shard, wl.max_grad_norm > 0, g.info.n_tiles,
                           wl.n_ranks)
            assert np.array_equal(g.flags_u32(), flags[:p.n_buckets])
            assert_state(gm, master, "master")
            assert_state(gmm, m, "exp_avg")
            assert_state(gv, v, "exp_avg_sq")
            assert_params(gp, params)
        return g.read_scaler(), sc
    finally:
        g.close()
        del g
        torch.cuda.empty_cache()


def random_case(i):
    """Random-shape case i (seeded): N, tensor list, bucket, rank window,
    micro-batches, gradient format, clip and per-bucket calls."""
    rng = np.random.default_rng(20_261_202 + i)
    n = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 13, 16, 31, 64]))
    n_tensors = int(rng.integers(1, 5))
    numels = [int(x) for x in rng.integers(0, 60_000, size=n_tensors)]
    if sum(numels) == 0:
        numels[0] = 1
    bucket = int(rng.choice([0, 0, 7, 4096, 10_001, 32_768]))
    lo = int(rng.integers(0, n))
    hi = int(rng.integers(lo + 1, n + 1))
    micro = int(rng.choice([1, 1, 2, 3]))
    bf16 = bool(rng.integers(0, 2))
    clip = float(rng.choice([0.0, 0.0, 0.3]))
    per_bucket = clip > 0 and bucket > 0 and bool(rng.integers(0, 2))
    return dict(n=n, numels=numels, bucket=bucket, lo=lo, hi=hi, micro=micro, bf16=bf16,
                clip=clip, per_bucket=per_bucket)


def random_workload(i):
    """(workload, per_bucket, two_pass) of random-shape case i."""
    from fsdp_sharded_mixed_shard_gb300 import workloads as W
    c = random_case(i)
    wl = W.Workload("random%d" % i, c["numels"], c["n"], c["bucket"], c["bf16"], 100 + i, 1e-3,
                    init_scale=1.0 if c["bf16"] else 1024.0, steps=2, rank_lo=c["lo"],
                    rank_hi=c["hi"], n_micro=c["micro"], max_grad_norm=c["clip"])
    return wl, c["per_bucket"], c["clip"] > 0
