#!/usr/bin/env python3
"""Benchmark of the per-shard ZeRO step of mixed-precision AdamW on GB300.

One step = the whole hot path over one batch of synthetic gradients:
reduce-scatter of N resident replicas in ring order with fp32 accumulation,
unscale, non-finite vote, (clip for clip workloads), AdamW on the fp32
master/m/v shard, cast to the 16-bit working copy, loss-scale bookkeeping.

Default workload: one flat tensor of 1.5e9 parameters, N = 8 simulated ranks,
fp16 gradients with a dynamic loss scale, global-norm clip at 1.0: the
largest parameter count of the five workloads on one GPU, on the two-pass
path (reduce-scatter with norm records, norm finish, update, bookkeeping).

Prints ONE JSON line (rank 0). `value` is Gparams/s of the whole job with
inputs resident in HBM; `e2e` is the same metric through the C ABI with the
replicas copied from pinned host memory and the updated parameters read
back every step; `roofline` is the dominant kernel's algorithmic HBM bytes
per launch over its CUDA-event duration against the measured copy
bandwidth; `cpu_baseline` is the CPU checker timed on a bounded sample.

`--impl reference` times the CPU checker (the only reference that exists
for this path) on the host cores, same workload, metric and unit.
Multi-GPU (torchrun): every rank runs an independent replica group on its
own GPU (no collective on the data path), timing is max over ranks and
`value` sums the ranks' work ("scaling": "weak").
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sharded AdamW step Gparams/s; achieved HBM GB/s as % of GB300 peak"
UNIT = "Gparams/s"
PHASE_SAMPLE = 8   # short steps: one timed step in PHASE_SAMPLE carries per-phase events
LONG_STEP_MS = 2.0  # steps at least this long carry per-phase events on every timed step
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="libzero", choices=["libzero", "reference"])
    ap.add_argument("--workload", default="flat_1p5b",
                    choices=["tiny_flat", "gpt2_small", "flat_1p5b", "stage3_slice", "llama_2b"])
    ap.add_argument("--e2e-steps", type=int, default=20,
                    help="steps of the end-to-end leg (0: leave it out, e.g. for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--micro", type=int, default=1,
                    help="micro-batches per optimizer step, accumulated in fp32 (>= 1)")
    ap.add_argument("--graph", action="store_true",
                    help="capture one whole step into a CUDA graph and replay it in the timed loop")
    ap.add_argument("--gather", action="store_true",
                    help="time the stage-3 unit all-gather (forward and backward gathers of "
                         "every unit) on the 8.81B-parameter layout at 64 ranks instead")
    ap.add_argument("--units-align", type=int, default=1,
                    help="unit padding grain in elements for --gather (1: multiple of N)")
    ap.add_argument("--units-per-call", type=int, default=1,
                    help="--gather: units gathered per call (a prefetch window), 1 or more")
    ap.add_argument("--numel-cap", type=int, default=0,
                    help="run the workload's first N flat parameters only (small profiling case)")
    ap.add_argument("--flat", type=int, default=0,
                    help="instead of --workload: one flat bf16 tensor of this many parameters "
                         "(shape studies, e.g. shards that start off the 16-byte grid)")
    ap.add_argument("--ranks", type=int, default=8, help="simulated ranks N for --flat")
    ap.add_argument("--clip", type=float, default=0.0,
                    help="max grad norm for --flat (> 0: the two-pass clipped step)")
    return ap.parse_args()


def selected_workload(args):
    """The workload a run times: --flat PSI --ranks N [--clip C] (seeded
    N(0, 1e-3) bf16 gradients, the GPT-2 workload's hyperparameters), else
    the named --workload."""
    if args.flat:
        from fsdp_sharded_mixed_shard_gb300 import workloads as W
        name = "flat_%d_n%d_bf16%s" % (args.flat, args.ranks, "_clip" if args.clip > 0 else "")
        return W.Workload(name, [args.flat], args.ranks, 0, True, 3, 1e-3,
                          max_grad_norm=args.clip)
    return workload(args.workload)


def workload(name):
    from fsdp_sharded_mixed_shard_gb300 import workloads as W
    return {"tiny_flat": W.TINY_FLAT, "gpt2_small": W.GPT2_SMALL, "flat_1p5b": W.FLAT_1P5B,
            "stage3_slice": W.STAGE3_SLICE, "llama_2b": W.LLAMA_2B}[name]


def psi_step(wl):
    """Parameters one step updates: the whole psi, or the owned slices."""
    from fsdp_sharded_mixed_shard_gb300 import workloads as W  # noqa: F401
    lo, hi = wl.ranks
    if (lo, hi) == (0, wl.n_ranks):
        return wl.psi
    n = wl.n_ranks
    S = (wl.psi + (-wl.psi) % n) // n
    return min(hi * S, wl.psi) - min(lo * S, wl.psi)


L2_BYTES = 129e6   # GB300 L2
FOLD_MAX_ELEMS = 1 << 22  # zero_step: largest single-launch fused window that folds its finish
SHORT_MAX_ELEMS = 1 << 20  # zero_step: largest fused window (N <= 16, one micro-batch) taken by the short-step kernel
SHORT_MAX_RANKS = 16
FLUSH_BYTES = 256 << 20


def step_bytes(wl, path):
    return (2 * wl.n_ranks + (34 if path == "two_pass" else 26)) * psi_step(wl)


def needs_flush(wl, path):
    """A step that moves less than twice the L2 would run from L2 when
    repeated back to back: such workloads flush L2 before every timed step."""
    return step_bytes(wl, path) < 2 * L2_BYTES


def run_config(wl, path, world):
    """The line's `config`: the workload and how its ranks are placed (the
    same for both arms)."""
    return dict(config_of(wl, path), parallelism="%d simulated ranks per GPU x %d GPUs"
                % (wl.n_ranks, world))


def config_of(wl, path):
    psip = wl.psi + (-wl.psi) % wl.n_ranks
    lo, hi = wl.ranks
    S = psip // wl.n_ranks
    step_gb = step_bytes(wl, path) / 1e9
    if needs_flush(wl, path):
        l2 = ("L2 flushed before every timed step (%d MB written outside the step's events; "
              "per-step events summed; %.3f GB of HBM traffic per step, L2 129 MB)"
              % (FLUSH_BYTES >> 20, step_gb))
    else:
        l2 = "inputs larger than L2 (%.1f GB of HBM traffic per step, L2 129 MB)" % step_gb
    return {"workload": wl.name, "psi": wl.psi, "psi_step": psi_step(wl),
            "n_ranks": wl.n_ranks, "owners": [lo, hi], "shard_elems": S,
            "bucket_elems": wl.bucket_elems, "grad_dtype": "bf16" if wl.is_bf16 else "fp16",
            "path": path, "clip": wl.max_grad_norm, "l2": l2}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha(source="zero_kernels.cu"):
    """Hash of a kernel source's code, with comments and whitespace removed:
    a comment edit keeps the committed traffic figures valid, any code edit
    voids them."""
    p = os.path.join(ROOT, "fsdp_sharded_mixed_shard_gb300", "csrc", source)
    return code_sha(open(p, encoding="utf-8").read())


def code_sha(txt):
    txt = re.sub(r"/\*.*?\*/", " ", txt, flags=re.S)
    txt = re.sub(r"//[^\n]*", " ", txt)
    return hashlib.sha256(" ".join(txt.split()).encode()).hexdigest()[:16]


def profiled_traffic(kernel, wl_name, source="zero_kernels.cu"):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source (line: `traffic: kernel=<k> workload=<w>
    bytes_per_launch=<b> source_sha=<sha>`); otherwise None."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    sha = kernel_source_sha(source)
    pat = re.compile(r"traffic:\s+kernel=(\S+)\s+workload=(\S+)\s+bytes_per_launch=([0-9.eE+]+)"
                     r"\s+source_sha=(\w+)")
    for f in sorted(os.listdir(d)):
        if not f.endswith((".md", ".txt")):
            continue
        for m in pat.finditer(open(os.path.join(d, f)).read()):
            if m.group(1) == kernel and m.group(2) == wl_name and m.group(4) == sha:
                return float(m.group(3))
    return None


# --------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((float(parts[2]), float(parts[3]), float(parts[4]), parts[5:10]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[3][1:]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows),
                "reasons": sorted(reasons)}


def device_uuid(dev):
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        return uuid if not uuid or uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        return None


# --------------------------------------------------------- multi-GPU glue ----

def max_over_ranks(dist, ms):
    """Slowest rank's time for the timed region (identity on one process)."""
    if not dist:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(psi_per_rank_step, steps, world, total_ms):
    """Whole-job Gparams/s: every rank updates psi_per_rank_step parameters
    per step (weak scaling), over the slowest rank's time."""
    return psi_per_rank_step * steps * world / (total_ms / 1e3) / 1e9


# ------------------------------------------------------------ libzero arm ----

def run_libzero(args, rank, world, dist):
    import numpy as np
    import torch
    import fsdp_sharded_mixed_shard_gb300 as Z
    from fsdp_sharded_mixed_shard_gb300 import harness

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = selected_workload(args)
    if args.numel_cap:
        wl = truncated(wl, args.numel_cap)
    if args.micro > 1:
        wl = wl.scaled(name="%s_micro%d" % (wl.name, args.micro), n_micro=args.micro)
    # a graph is captured on a stream of its own (the legacy default stream cannot be captured)
    g = harness.Group(wl, device=dev, stream=torch.cuda.Stream(device=dev) if args.graph else None)
    path = "two_pass" if g.two_pass else "fused"
    g.init_state()
    g.gen_grads(1)
    torch.cuda.synchronize()
    st = g.sptr
    N = wl.n_ranks
    lo, hi = wl.ranks
    # per-rank pointer tables built once as uint64 arrays, which the binding
    # passes through unchanged (lists are marshalled on every call)
    table = lambda ptrs: None if ptrs is None else np.array(  # noqa: E731
        [0 if q is None else q for q in ptrs], dtype=np.uint64)
    reps = table(g.rep_ptrs())
    m, v, w = table(g._state_ptrs(0)), table(g._state_ptrs(1)), table(g._state_ptrs(2))
    sc, fl, flat = g.scaler.data_ptr(), g.flags.data_ptr(), g.flat.data_ptr()
    ws = g.workspace.data_ptr()
    clip = wl.max_grad_norm > 0
    gp = table(g.ghat_ptrs()) if g.two_pass else None

    # phases of one step (each a C-ABI call on stream st); for the fused path
    # the update is one kernel launch per 128 segments. With k micro-batches
    # the first k - 1 are accumulated in fp32 and the last is added inside
    # the reduce (the same replica buffer stands for every micro-batch).
    k_micro = wl.n_micro
    acc = table(g.accum_ptrs()) if k_micro > 1 else None

    def phases():
        pre = []
        for mb in range(1, k_micro):
            name = "accumulate_first" if mb == 1 else "accumulate"
            pre.append((name, (lambda first: lambda: Z.zero_accumulate(
                g.plan, lo, hi, reps, acc, g.wbase, first, st))(mb == 1)))
        if not g.two_pass and cold:
            # a step timed cold (L2 flushed first) is a short one: the single
            # zero_step call, which folds the finish into the fused pass
            # when the step fits one launch
            return pre + [("fused_step", lambda: Z.zero_step_accum(
                g.plan, lo, hi, m, v, w, 2, None, reps, acc, k_micro, g.wbase, flat, g.hp, sc,
                fl, st))]
        if not g.two_pass:
            return pre + [("fused_update", lambda: Z.zero_step_update_accum(
                        g.plan, lo, hi, m, v, w, 2, None, reps, acc, k_micro, g.wbase, flat, g.hp,
                        sc, fl, st)),
                    ("finish", lambda: Z.zero_step_finish(
                        g.plan, lo, hi, m, 2, None, g.wbase, flat, g.hp, sc, st))]
        out = pre + [("reduce_scatter", lambda: Z.zero_reduce_scatter_accum(
                    g.plan, -1, lo, hi, reps, acc, k_micro, g.wbase, gp, sc, fl,
                    ws if clip else 0, st))]
        if clip:
            out.append(("grad_norm", lambda: Z.zero_grad_norm(g.plan, lo, hi, None, g.hp, sc, ws,
                                                              st)))
        out += [("update", lambda: Z.zero_step_update(
                    g.plan, lo, hi, m, v, w, g.n_sets, gp, None, g.wbase, flat, g.hp, sc, fl,
                    st)),
                ("finish", lambda: Z.zero_step_finish(
                    g.plan, lo, hi, m, g.n_sets, gp, g.wbase, flat, g.hp, sc, st))]
        return out

    cold = needs_flush(wl, "two_pass" if g.two_pass else "fused")
    ph = phases()
    segs = g.info.n_segments if (lo, hi) == (0, N) else None
    if segs is None:
        segs = sum(1 for s in Z.zero_plan_segments(g.plan) if lo <= s[2] < hi)
    L = -(-segs // 128)
    # fused: update + (re-cast check merged with bookkeeping); two-pass:
    # reduce + norm finish (2) + update + bookkeeping
    launches_per_step = ((2 * L) if not g.two_pass else (L + (2 if clip else 0) + L + 1)) + \
        (k_micro - 1)
    if not g.two_pass and cold and L == 1 and (hi - lo) * g.S <= FOLD_MAX_ELEMS:
        launches_per_step = 1 + (k_micro - 1)  # zero_step folds the finish into the pass

    # the clock sampler starts before the warm-up, so that the timed region
    # follows the warm-up steps directly (no idle gap before the first step)
    clocks = ClockSampler(device_uuid(dev))
    clocks.start()
    time.sleep(0.3)
    # the last warm-up step's time decides how the phases are sampled below
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        if i == args.warmup - 1:
            w0.record(g.stream)
        for _, f in ph:
            f()
    w1.record(g.stream)
    torch.cuda.synchronize()
    warm_ms = w0.elapsed_time(w1)
    graph = None
    if args.graph:
        # one whole step as a CUDA graph: the device-resident scaler carries
        # the step count, loss scale and ping-pong set, so replays need no
        # host logic
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=g.stream):
            for _, f in ph:
                f()
        torch.cuda.synchronize()

    K = args.steps
    # A step smaller than twice the L2 is timed cold: L2 is flushed before
    # every step, outside that step's events, and every step carries events.
    flush_buf = None
    if needs_flush(wl, "two_pass" if g.two_pass else "fused"):
        flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    # Per-phase events. An event between two launches stops the next kernel
    # from starting early (programmatic dependent launch), which costs a few
    # microseconds per launch: steps of LONG_STEP_MS or more carry events on
    # every timed step (the cost is under 0.2 % of such a step, and the
    # per-kernel means then come from exactly the timed steps); shorter steps
    # carry them on one timed step in PHASE_SAMPLE, never the first, and run
    # the others back to back as a user's do.
    if flush_buf is not None or warm_ms >= LONG_STEP_MS:
        every, first_sampled = 1, 0
    else:
        every, first_sampled = PHASE_SAMPLE, min(PHASE_SAMPLE - 1, K - 1)
    sampled = [k for k in range(K) if k % every == first_sampled % every and k >= first_sampled]
    # cold steps: one event pair per step; with a single phase it is the
    # phase's own pair (an event pair costs the GPU a few microseconds, which
    # two nested pairs would count twice)
    nested = flush_buf is not None and len(ph) > 1
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(K if nested else 0)]
    evs = {name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(len(sampled) * max(1, k_micro))] for name, _ in ph}
    ev_i = {name: 0 for name, _ in ph}
    sampled_set = set(sampled)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if flush_buf is not None and hasattr(torch.cuda, "_sleep"):
        # cold steps are short: a GPU-side pause before the loop lets the host
        # enqueue ahead of the GPU, so no event pair waits for the host
        with torch.cuda.stream(g.stream):
            torch.cuda._sleep(int(2e7))
    wall0 = time.time()
    t0.record(g.stream)
    for k in range(K):
        if flush_buf is not None:
            with torch.cuda.stream(g.stream):
                flush_buf.fill_(k)
            if nested:
                step_evs[k][0].record(g.stream)
        if k not in sampled_set:
            if graph is not None:
                with torch.cuda.stream(g.stream):  # replay() launches on the current stream
                    graph.replay()
            else:
                for _, f in ph:
                    f()
            continue
        for name, f in ph:
            a, b = evs[name][ev_i[name]]
            ev_i[name] += 1
            a.record(g.stream)
            f()
            b.record(g.stream)
        if nested:
            step_evs[k][1].record(g.stream)
    t1.record(g.stream)
    torch.cuda.synchronize()
    wall = time.time() - wall0
    clk = clocks.stop()
    if dist:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    if nested:
        total_ms = sum(a.elapsed_time(b) for a, b in step_evs)
    elif flush_buf is not None:
        total_ms = sum(a.elapsed_time(b) for a, b in evs[ph[0][0]][:ev_i[ph[0][0]]])
    phase_ms = {name: statistics.mean(a.elapsed_time(b) for a, b in evs[name][:ev_i[name]])
                for name, _ in ph}

    total_ms = max_over_ranks(dist, total_ms)
    ms_per_step = total_ms / K
    pstep = psi_step(wl)
    value = job_throughput(pstep, K, world, total_ms)

    # roofline of the dominant kernel
    peak, peak_kind = peaks()
    extra = 4 * N if k_micro > 1 else 0  # fp32 accumulators read by the reduce
    bytes_per_param = {"fused_update": 2 * N + 26 + extra, "fused_step": 2 * N + 26 + extra,
                       "reduce_scatter": 2 * N + 4 + extra,
                       "update": 30, "grad_norm": 0, "finish": 0,
                       "accumulate_first": 6 * N, "accumulate": 10 * N}
    dom = max((n for n, _ in ph if bytes_per_param[n] > 0), key=lambda n: phase_ms[n])
    alg_bytes = bytes_per_param[dom] * pstep
    achieved = alg_bytes / (phase_ms[dom] / 1e3) / 1e9
    kernel_name = {"fused_update": "bulk_kernel<kFused>", "fused_step": "bulk_kernel<kFused>",
                   "reduce_scatter": "bulk_kernel<kReduce>",
                   "update": "bulk_kernel<kUpdate>", "accumulate": "accumulate_kernel:add",
                   "accumulate_first": "accumulate_kernel:first"}[dom]
    if (dom == "fused_step" and L == 1 and (hi - lo) * g.S <= SHORT_MAX_ELEMS
            and N <= SHORT_MAX_RANKS and k_micro == 1):
        kernel_name = "short_fused_kernel"
    if k_micro > 1 and dom in ("fused_update", "fused_step", "reduce_scatter"):
        kernel_name = (kernel_name[:-1] + ",acc>" if kernel_name.endswith(">")
                       else kernel_name + "<acc>")
    kernel_gbs = {n: round(bytes_per_param[n] * pstep / (phase_ms[n] / 1e3) / 1e9, 1)
                  for n, _ in ph if bytes_per_param[n] > 0}
    traffic = profiled_traffic(kernel_name, wl.name)
    step_bytes = (2 * N + (34 if g.two_pass else 26) + extra
                  + (6 * N + 10 * N * (k_micro - 2) if k_micro > 1 else 0)) * pstep
    roofline = {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_kind": peak_kind + " (copy bandwidth, burst)",
                "traffic": traffic, "algorithmic_bytes_per_launch": alg_bytes,
                "kernel_ms": round(phase_ms[dom], 4),
                "step_bytes_per_param": step_bytes / pstep,
                "step_achieved_gbs": round(step_bytes / (ms_per_step / 1e3) / 1e9, 1),
                "step_frac": round(step_bytes / (ms_per_step / 1e3) / 1e9 / peak, 4),
                "frac_of_2n26_bytes": round((2 * N + 26) * pstep / (ms_per_step / 1e3) / 1e9
                                              / peak, 4),
                "kernel_gbs": kernel_gbs}

    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, g, wl, K, world, dist, k_micro, acc, m, v, w, sc, fl, ws, clip, gp,
                      lo, hi, N, dev, pstep)
    sk = g.read_scaler()
    g.close()

    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic: seeded counter-based generator (SplitMix64 + Irwin-Hall normal), "
                    "same replicas every timed step",
            "config": run_config(wl, path, world),
            "roofline": roofline, "e2e": e2e, "gpu_launches": launches_per_step * K,
            "clocks": clk, "phase_ms": {k: round(v, 4) for k, v in phase_ms.items()},
            "phase_events": "per-kernel CUDA events on %d of %d timed steps (%s)"
                            % (len(sampled), K, "every step" if every == 1 else
                               "steps %d, %d, ... of the timed loop" % (sampled[0], sampled[0] + every)),
            "launch": "CUDA graph replay of one captured step (eager on event steps)"
                      if graph is not None else "eager C-ABI calls",
            "wall_s_timed": round(wall, 3), "scaler_t": sk.t, "device_error": sk.error}
    return line


def run_e2e(args, g, wl, K, world, dist, k_micro, acc, m, v, w, sc, fl, ws, clip, gp, lo, hi,
            N, dev, pstep):
    """End to end through the C ABI: every step copies that step's replicas
    from pinned host memory and reads the updated parameters and the scaler
    back. Steps are pipelined over two replica buffers and two parameter
    buffers: the host->device copy of step k+1 (split over two copy streams)
    runs while step k computes, and step k's read-back runs on a third
    stream."""
    import torch
    import fsdp_sharded_mixed_shard_gb300 as Z
    st = g.sptr
    E = max(1, min(args.e2e_steps, K))
    host_reps = torch.empty(g.replicas.shape, dtype=torch.int16, pin_memory=True)
    host_reps.copy_(g.replicas)
    host_params = [torch.empty(g.flat.shape, dtype=torch.int16, pin_memory=True) for _ in range(2)]
    host_scaler = [torch.empty(g.scaler.shape, dtype=torch.uint8, pin_memory=True)
                   for _ in range(2)]
    dev_reps = [g.replicas, torch.empty_like(g.replicas)]
    dev_flat = [g.flat, torch.empty_like(g.flat)]
    scaler_snap = [torch.empty_like(g.scaler) for _ in range(2)]
    rep_ptrs = [g.rep_ptrs(dev_reps[0]), g.rep_ptrs(dev_reps[1])]
    h2d = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    d2h = torch.cuda.Stream(device=dev)
    half = N // 2 if N > 1 else N
    ev = lambda: torch.cuda.Event()  # noqa: E731
    landed = [ev(), ev()]       # replicas of buffer b on the device
    computed = [ev(), ev()]     # step that used buffer b finished
    read_back = [ev(), ev()]    # parameters of buffer b copied to the host

    def copy_in(b):
        for i, (lo_r, hi_r) in enumerate(((0, half), (half, N))):
            if hi_r <= lo_r:
                continue
            with torch.cuda.stream(h2d[i]):
                h2d[i].wait_event(computed[b])
                dev_reps[b][lo_r:hi_r].copy_(host_reps[lo_r:hi_r], non_blocking=True)
        h2d[0].wait_stream(h2d[1])
        landed[b].record(h2d[0])

    def step_on(b, p):
        """Last micro-batch of a step: replicas in buffer b, parameters into buffer p."""
        rp, fp = rep_ptrs[b], dev_flat[p].data_ptr()
        if not g.two_pass:
            Z.zero_step_accum(g.plan, lo, hi, m, v, w, 2, None, rp, acc, k_micro, g.wbase, fp,
                              g.hp, sc, fl, st)
        else:
            Z.zero_reduce_scatter_accum(g.plan, -1, lo, hi, rp, acc, k_micro, g.wbase, gp, sc, fl,
                                        ws if clip else 0, st)
            if clip:
                Z.zero_grad_norm(g.plan, lo, hi, None, g.hp, sc, ws, st)
            Z.zero_step(g.plan, lo, hi, m, v, w, g.n_sets, gp, None, g.wbase, fp, g.hp, sc, fl,
                        st)

    for e in computed + read_back:
        e.record(g.stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    e0.record(g.stream)
    h2d[0].wait_event(e0)
    h2d[1].wait_event(e0)
    copy_in(0)
    # one slot per micro-batch: every micro-batch's replicas cross the host
    # link; the first k - 1 are accumulated, the last one completes the step
    slots = E * k_micro
    for j in range(slots):
        b = j % 2
        if j + 1 < slots:
            copy_in(1 - b)
        g.stream.wait_event(landed[b])
        mb = j % k_micro + 1
        if mb < k_micro:
            Z.zero_accumulate(g.plan, lo, hi, rep_ptrs[b], acc, g.wbase, 1 if mb == 1 else 0, st)
            computed[b].record(g.stream)
            continue
        p = (j // k_micro) % 2
        g.stream.wait_event(read_back[p])   # parameters buffer p free again
        step_on(b, p)
        with torch.cuda.stream(g.stream):
            scaler_snap[p].copy_(g.scaler, non_blocking=True)  # this step's scaler
        computed[b].record(g.stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(computed[b])
            host_params[p].copy_(dev_flat[p], non_blocking=True)
            host_scaler[p].copy_(scaler_snap[p], non_blocking=True)
        read_back[p].record(d2h)
    g.stream.wait_stream(d2h)
    e1.record(g.stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1))
    e2e = {"value": round(job_throughput(pstep, E, world, e2e_ms), 4), "unit": UNIT,
           "steps": E, "h2d_bytes_per_step": int(g.replicas.numel() * 2 * k_micro),
           "d2h_bytes_per_step": int(g.flat.numel() * 2 + g.scaler.numel()),
           "pipelined": "two replica and parameter buffers; H2D of step k+1 overlaps step k"}
    del dev_reps, host_reps
    return e2e


# ------------------------------------------------ stage-3 unit all-gather ----

GATHER_METRIC = "stage-3 unit all-gather Gparams/s (forward + backward gathers of every unit)"


def run_gather(args, rank, world, dist):
    """One step = the all-gathers of stage 3 on one rank's view: every unit
    gathered before its forward (units 0..U-1) and again before its backward
    (U-1..0), one call per unit into a ring of two unit buffers. Each
    gathered element moves 4 bytes (2 read from a shard, 2 written)."""
    import torch
    from fsdp_sharded_mixed_shard_gb300 import harness, workloads as W
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    uw = W.stage3_8p81b_units(64, args.units_align)
    if args.numel_cap:
        # a small case with the same unit sizes: the first units (root + blocks)
        # whose parameters fit the cap, at least two
        k, tot = 0, 0
        while k < uw.n_units and (k < 2 or tot + uw.numels[k] <= args.numel_cap):
            tot += uw.numels[k]
            k += 1
        uw = W.UnitWorkload(uw.name + "_first%d" % k, uw.numels[:k], list(range(k)), k,
                            uw.n_ranks, uw.align_elems, uw.seed)
    W_ = max(1, args.units_per_call)
    # two sets of W unit buffers: consecutive calls alternate between them
    g = harness.UnitGroup(uw, device=dev, window=2 * W_)
    g.fill_shards()
    U = uw.n_units
    # forward: windows of W units in order; backward: the same windows in reverse
    fwd = [(u, min(u + W_, U)) for u in range(0, U, W_)]
    calls = [(lo_u, hi_u, (i % 2) * W_) for i, (lo_u, hi_u) in
             enumerate(fwd + list(reversed(fwd)))]
    gathered = 2 * g.info.psi_pad
    for _ in range(args.warmup):
        for lo_u, hi_u, slot in calls:
            g.gather(lo_u, hi_u, slot)
    torch.cuda.synchronize()
    K = args.steps
    # per-call events on one timed step in PHASE_SAMPLE (never the first; the
    # last step when there are fewer): an event between two launches stops
    # the next one from starting early, so the other steps run back to back
    first = min(PHASE_SAMPLE - 1, K - 1)
    sampled = [k for k in range(first, K, PHASE_SAMPLE)]
    evs = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in calls] for k in sampled}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device_uuid(dev))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record(g.stream)
    for k in range(K):
        if k not in evs:
            for lo_u, hi_u, slot in calls:
                g.gather(lo_u, hi_u, slot)
            continue
        for (lo_u, hi_u, slot), (a, b) in zip(calls, evs[k]):
            a.record(g.stream)
            g.gather(lo_u, hi_u, slot)
            b.record(g.stream)
    t1.record(g.stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    total_ms = max_over_ranks(dist, t0.elapsed_time(t1))
    ms_per_step = total_ms / K
    # call durations of the calls made of block units only (the root unit
    # differs in size), per gathered block unit
    blk = g.info.max_unit_psi_pad
    block = [i for i, (lo_u, hi_u, _) in enumerate(calls)
             if all(g.units[u].psi_pad == blk for u in range(lo_u, hi_u))]
    per_unit = [evs[k][i][0].elapsed_time(evs[k][i][1]) / (calls[i][1] - calls[i][0])
                for k in sampled for i in block]
    blk_ms = statistics.mean(per_unit)
    peak, peak_kind = peaks()
    unit_bytes = 4 * blk
    achieved = unit_bytes / (blk_ms / 1e3) / 1e9
    # one launch per 256 slices of non-empty units in a call (N slices per unit)
    launches = sum(-(-sum(g.N for u in range(lo_u, hi_u) if g.units[u].shard_elems) // 256)
                   for lo_u, hi_u, _ in calls)
    traffic = profiled_traffic("copy_kernel", uw.name, "gather.cu")
    # per-rank accounting of the layout under each sharding strategy (host)
    import fsdp_sharded_mixed_shard_gb300 as Z
    accounting = {}
    for name, strat, reps in (("FULL_SHARD", Z.ZERO_FULL_SHARD, 1),
                              ("SHARD_GRAD_OP", Z.ZERO_SHARD_GRAD_OP, 1),
                              ("NO_SHARD", Z.ZERO_NO_SHARD, 1),
                              ("NO_RESHARD_AFTER_FORWARD", Z.ZERO_NO_RESHARD_AFTER_FORWARD, 1)):
        c = Z.zero_unit_plan_strategy_cost(g.plan, strat, reps)
        accounting[name] = {"persistent_gb": round(c.persistent_bytes / 1e9, 4),
                            "peak_gb": round(c.peak_bytes / 1e9, 4),
                            "wire_gb_per_step": round(2 * c.comm_elems / 1e9, 4)}
    line = {"metric": GATHER_METRIC, "value": round(gathered * K * world / (total_ms / 1e3) / 1e9, 4),
            "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u16", "data": "synthetic: seeded generator bf16 "
            "patterns in every shard",
            "config": {"workload": uw.name, "n_units": U, "n_ranks": 64,
                       "align_elems": uw.align_elems, "psi": g.info.psi,
                       "psi_pad": g.info.psi_pad, "block_unit_elems": g.info.max_unit_psi_pad,
                       "gathers_per_step": len(calls), "units_per_call": W_,
                       "l2": "inputs larger than L2 (%.1f GB of shards)" % (2 * g.info.psi_pad / 1e9)},
            "roofline": {"bound": "hbm", "kernel": "copy_kernel", "achieved": round(achieved, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_kind": peak_kind + " (copy bandwidth, burst)", "traffic": traffic,
                         "algorithmic_bytes_per_launch": unit_bytes,
                         "kernel_ms": round(blk_ms, 5),
                         "step_achieved_gbs": round(4 * gathered / (ms_per_step / 1e3) / 1e9, 1),
                         "step_frac": round(4 * gathered / (ms_per_step / 1e3) / 1e9 / peak, 4)},
            "accounting_per_rank": accounting,
            "phase_events": "per-call CUDA events on %d of %d timed steps" % (len(sampled), K),
            "e2e": None, "gpu_launches": launches * K, "clocks": clk}
    g.close()
    return line


# ---------------------------------------------------------- CPU checker ----

def truncated(wl, n_elems):
    """The workload's first n_elems flat elements (tensor list cut there),
    same N, buckets, gradient format and hyperparameters."""
    numels, left = [], n_elems
    for x in wl.numels:
        if left <= 0:
            break
        numels.append(min(x, left))
        left -= numels[-1]
    return wl.scaled(name="%s_first%d" % (wl.name, sum(numels)), numels=numels, rank_lo=0,
                     rank_hi=None, inject=None)


oracle_sample = truncated


def time_oracle_steps(wl_s, steps, threads=1):
    """Runs `steps` checker steps on wl_s; returns seconds of checker time
    (input generation excluded). With threads > 1 the owners are split into
    contiguous rank ranges, one host thread each (the C checker runs without
    the interpreter lock); every range has its own scaler and flags, so this
    is for workloads without a global clip (the fused path)."""
    import numpy as np
    import oracle
    from fsdp_sharded_mixed_shard_gb300 import synth
    p, _, _ = oracle.make_plan(wl_s.numels, wl_s.n_ranks, wl_s.bucket_elems)
    psip = p.psi_pad
    hp = oracle.hparams(lr=wl_s.lr, beta1=wl_s.beta1, beta2=wl_s.beta2, eps=wl_s.eps,
                        weight_decay=wl_s.weight_decay, max_grad_norm=wl_s.max_grad_norm,
                        dynamic_scale=int(wl_s.dynamic_scale),
                        growth_interval=wl_s.growth_interval)
    sc = oracle.scaler(wl_s.init_scale)
    master = synth.master_f32(psip, 0, wl_s.seed, wl_s.psi)
    m = np.zeros(psip, np.float32)
    v = np.zeros(psip, np.float32)
    params = oracle.cast16(master, wl_s.is_bf16)
    spec = synth.grad_spec(seed=wl_s.seed, sigma=wl_s.sigma, bias_sigma=wl_s.bias_sigma,
                           loss_scale=wl_s.init_scale, outliers=wl_s.outliers, psi=wl_s.psi)
    reps = [oracle.cast16(synth.grad_f32(psip, 0, spec, 1, r), wl_s.is_bf16)
            for r in range(wl_s.n_ranks)]
    flags = np.zeros(max(p.n_buckets, 1), np.uint32)
    t = 0.0
    if threads <= 1:
        for _ in range(steps):
            a = time.perf_counter()
            oracle.step_arrays(p, 0, wl_s.n_ranks, wl_s.is_bf16, reps, 0, master, m, v, params,
                               hp, sc, flags)
            t += time.perf_counter() - a
        return t
    import threading
    n = wl_s.n_ranks
    cuts = [n * k // threads for k in range(threads + 1)]
    ranges = [(cuts[k], cuts[k + 1]) for k in range(threads) if cuts[k + 1] > cuts[k]]
    scalers = [oracle.scaler(wl_s.init_scale) for _ in ranges]
    flag_sets = [np.zeros_like(flags) for _ in ranges]
    for _ in range(steps):
        work = [threading.Thread(target=oracle.step_arrays,
                                 args=(p, lo, hi, wl_s.is_bf16, reps, 0, master, m, v, params, hp,
                                       scalers[i], flag_sets[i]))
                for i, (lo, hi) in enumerate(ranges)]
        a = time.perf_counter()
        for w in work:
            w.start()
        for w in work:
            w.join()
        t += time.perf_counter() - a
    return t


def calibrate_oracle(wl, seconds_total, steps):
    probe = oracle_sample(wl, 1 << 17)
    t = time_oracle_steps(probe, 1)
    rate = probe.psi / max(t, 1e-6)                      # params/s
    n = int(rate * seconds_total / max(steps, 1))
    n = max(wl.n_ranks * 1024, min(n, 1 << 25, wl.psi))
    return n, rate


def cpu_baseline(wl, seconds):
    """The checker timed on a bounded sample: the first n parameters (at
    most 2^25, so the materialised replicas stay within host memory) for as
    many steps (at least 3) as fill about `seconds` of single-core time."""
    n, rate = calibrate_oracle(wl, seconds, 3)
    steps = max(3, int(round(seconds * rate / n)))
    s = oracle_sample(wl, n)
    t = time_oracle_steps(s, steps)
    out = {"value": round(s.psi * steps / t / 1e9, 6), "unit": UNIT, "cores": 1,
           "kind": "oracle",
           "sample": "first %d flat parameters of %s (same N=%d, buckets, format and "
                     "hyperparameters), %d steps, plain single-threaded C checker, inputs "
                     "materialised in host memory, generation untimed" % (
                         s.psi, wl.name, wl.n_ranks, steps),
           "seconds": round(t, 2)}
    # the same checker on every host core the ranks can use (one rank range
    # per thread; no global clip on this path)
    threads = min(os.cpu_count() or 1, wl.n_ranks)
    if threads > 1 and wl.max_grad_norm <= 0:
        t_all = time_oracle_steps(s, steps, threads)
        out["all_cores"] = {"value": round(s.psi * steps / t_all / 1e9, 6), "unit": UNIT,
                            "cores": threads, "seconds": round(t_all, 2),
                            "sample": "the same sample, ranks split over %d host threads"
                                      % threads}
    return out


def run_reference(args):
    """The CPU checker on the host cores: each of the warmup + steps steps is a
    bounded sample of the workload, sized so the run takes about two minutes."""
    wl = selected_workload(args)
    total = args.steps + args.warmup
    n, _ = calibrate_oracle(wl, 100.0, total)
    s = oracle_sample(wl, n)
    time_oracle_steps(s, min(args.warmup, 3))
    t = time_oracle_steps(s, args.steps)
    value = s.psi * args.steps / t / 1e9
    sample = ("first %d flat parameters of %s per step (same N=%d, buckets, format and "
              "hyperparameters), plain single-threaded C checker" % (s.psi, wl.name, wl.n_ranks))
    path = "two_pass" if wl.max_grad_norm > 0 else "fused"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic: seeded counter-based generator",
            "config": run_config(wl, path, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    if args.gather:
        line = run_gather(args, rank, world, dist)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return 0
    line = run_libzero(args, rank, world, dist)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(selected_workload(args), args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
