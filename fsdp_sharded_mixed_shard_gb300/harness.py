"""Device buffers and step driver for one synthetic workload (harness only).

Used by the GPU tests, the smoke check and the benchmark. PyTorch provides
device memory and streams; every step of the path runs in libzero's kernels
through the C ABI, and the inputs come from the seeded generator kernels.

Layout in HBM for a workload with N ranks processing owners [lo, hi):
  replicas   int16 [N, row]       rank r's 16-bit gradient window
                                  [lo*S, hi*S), rows padded to 16 bytes
  flat       int16 [row]          16-bit working parameters (same window)
  state      fp32 [n_sets, 3, n_own, srow]  master / exp_avg / exp_avg_sq
                                  shard of each owned rank, rows padded to 16 B;
                                  n_sets = 2 (ping-pong) unless the two-pass
                                  path is asked for one set
  ghat       fp32 [n_own, srow]   reduced gradients (two-pass path only)
  scaler     80 bytes             zero_scaler
  flags      uint32 [n_buckets]   per-bucket non-finite flags
  workspace  zero_workspace_bytes (norm tile records, clip path only)
  exchange   1040 bytes           zero_exchange (owners split over processes)
"""
import ctypes as C

import torch

from . import (ZERO_BF16, ZERO_FP16, ZeroExchange, ZeroHParams, ZeroScaler, zero_accumulate,
               zero_cast_params, zero_gather_units, zero_grad_norm, zero_grad_norm_apply,
               zero_grad_norm_local, zero_plan_create, zero_plan_destroy, zero_plan_get_info,
               zero_reduce_scatter_accum, zero_scaler_init, zero_shard_units, zero_step,
               zero_step_accum, zero_step_finish, zero_step_update_accum, zero_unit_plan_create,
               zero_unit_plan_destroy, zero_unit_plan_get_info, zero_unit_plan_units,
               zero_workspace_bytes)
from . import synth


def _round_up(x, m):
    return (x + m - 1) // m * m


def hparams_of(wl):
    return ZeroHParams(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.weight_decay, wl.max_grad_norm,
                       int(wl.dynamic_scale), wl.growth_interval, wl.init_scale)


class Group:
    """All device state of one simulated data-parallel group on one GPU."""

    def __init__(self, wl, device="cuda", two_pass=None, stream=None, alloc_replicas=True,
                 n_sets=None):
        self.wl = wl
        self.device = torch.device(device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.two_pass = (wl.max_grad_norm > 0) if two_pass is None else two_pass
        # optimizer state sets: two by default (ping-pong: each step reads
        # one set and writes the other); the two-pass path also takes one
        # (updated in place, 12 bytes per element less memory)
        self.n_sets = 2 if n_sets is None else n_sets
        self.is_bf16 = wl.is_bf16
        self.plan = zero_plan_create(wl.numels, wl.n_ranks, wl.bucket_elems,
                                     ZERO_BF16 if wl.is_bf16 else ZERO_FP16)
        self.info = zero_plan_get_info(self.plan)
        self.N = wl.n_ranks
        self.S = self.info.shard_elems
        self.lo, self.hi = wl.ranks
        self.wbase = self.lo * self.S
        self.wlen = (self.hi - self.lo) * self.S
        self.row = _round_up(max(self.wlen, 1), 8)
        self.srow = _round_up(max(self.S, 1), 4)
        self.hp = hparams_of(wl)
        n_own = self.hi - self.lo
        dev = self.device
        self.replicas = (torch.zeros((self.N, self.row), dtype=torch.int16, device=dev)
                         if alloc_replicas else None)
        self.flat = torch.zeros(self.row, dtype=torch.int16, device=dev)
        self.state = torch.zeros((self.n_sets, 3, n_own, self.srow), dtype=torch.float32,
                                 device=dev)
        self.ghat = (torch.zeros((n_own, self.srow), dtype=torch.float32, device=dev)
                     if self.two_pass else None)
        # fp32 accumulators of the earlier micro-batches (one per replica)
        self.n_micro = wl.n_micro
        self.accum = (torch.zeros((self.N, self.row), dtype=torch.float32, device=dev)
                      if wl.n_micro > 1 else None)
        self.scaler = torch.zeros(C.sizeof(ZeroScaler), dtype=torch.uint8, device=dev)
        self.flags = torch.zeros(max(self.info.n_buckets, 1), dtype=torch.int32, device=dev)
        ws = zero_workspace_bytes(self.plan, 1)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev)
        self.exchange = torch.zeros(C.sizeof(ZeroExchange), dtype=torch.uint8, device=dev)

    def close(self):
        if self.plan:
            zero_plan_destroy(self.plan)
            self.plan = None

    # -------------------------------------------------------------- pointers
    @property
    def sptr(self):
        return self.stream.cuda_stream

    def rep_ptrs(self, replicas=None):
        t = self.replicas if replicas is None else replicas
        base, rb = t.data_ptr(), self.row * 2
        return [base + r * rb for r in range(self.N)]

    def _state_ptrs(self, which):
        """Per-set, per-rank shard addresses of one optimizer array (computed
        arithmetically: indexing the tensor per rank costs microseconds each)."""
        out = [None] * (self.n_sets * self.N)
        base = self.state.data_ptr()
        sset = self.state.stride(0) * 4
        sarr = self.state.stride(1) * 4
        srank = self.state.stride(2) * 4
        for s in range(self.n_sets):
            for i in range(self.lo, self.hi):
                out[s * self.N + i] = base + s * sset + which * sarr + (i - self.lo) * srank
        return out

    def ghat_ptrs(self):
        out = [None] * self.N
        base, srank = self.ghat.data_ptr(), self.ghat.stride(0) * 4
        for i in range(self.lo, self.hi):
            out[i] = base + (i - self.lo) * srank
        return out

    # ----------------------------------------------------------------- init
    def init_state(self):
        wl = self.wl
        with torch.cuda.stream(self.stream):
            self.state.zero_()
            for i in range(self.lo, self.hi):
                synth.gpu_fill_master(self.state[0, 0, i - self.lo].data_ptr(), self.S,
                                      i * self.S, wl.seed, wl.psi, self.sptr)
            master0 = [None] * self.N
            for i in range(self.lo, self.hi):
                master0[i] = self.state[0, 0, i - self.lo].data_ptr()
            zero_cast_params(self.plan, self.lo, self.hi, master0, self.flat.data_ptr(),
                             self.wbase, self.sptr)
            sc = zero_scaler_init(self.hp)
            host = torch.frombuffer(bytearray(bytes(sc)), dtype=torch.uint8)
            self.scaler.copy_(host)

    def read_scaler(self):
        self.stream.synchronize()
        raw = bytes(self.scaler.cpu().numpy().tobytes())
        return ZeroScaler.from_buffer_copy(raw)

    def grad_spec(self, scale):
        wl = self.wl
        return synth.grad_spec(seed=wl.seed, sigma=wl.sigma, bias_sigma=wl.bias_sigma,
                               loss_scale=scale, outliers=wl.outliers, psi=wl.psi)

    def gen_grads(self, step, scale=None, replicas=None, micro=None):
        """Fill the replicas with step `step`'s gradients (micro-batch `micro`,
        default the last) at the device's current loss scale (read back from
        the scaler unless given)."""
        if scale is None:
            scale = self.read_scaler().scale
        micro = self.n_micro if micro is None else micro
        t = self.replicas if replicas is None else replicas
        spec = self.grad_spec(scale)
        ptrs = self.rep_ptrs(t)
        key = self.wl.gen_step(step, micro)
        for r in range(self.N):
            synth.gpu_fill_grad(ptrs[r], self.wlen, self.wbase, spec, key, r, self.is_bf16,
                                self.sptr)
        inj = self.wl.inject
        if inj is not None and inj[0] == step and micro == self.n_micro:
            _, r, e, bits = inj
            if self.wbase <= e < self.wbase + self.wlen:
                with torch.cuda.stream(self.stream):
                    t[r, e - self.wbase] = bits - 65536 if bits >= 32768 else bits

    # ----------------------------------------------------------------- step
    def accum_ptrs(self):
        base, rb = self.accum.data_ptr(), self.row * 4
        return [base + r * rb for r in range(self.N)]

    def accumulate(self, first):
        """Add the replicas (one micro-batch) into the fp32 accumulators."""
        zero_accumulate(self.plan, self.lo, self.hi, self.rep_ptrs(), self.accum_ptrs(),
                        self.wbase, first, self.sptr)

    def step_micro(self, step, per_bucket=False):
        """A whole optimizer step of n_micro micro-batches: generate and
        accumulate the first n_micro - 1, generate the last, then step (the
        last micro-batch is added inside the reduce)."""
        for mb in range(1, self.n_micro):
            self.gen_grads(step, micro=mb)
            self.accumulate(first=(mb == 1))
        self.gen_grads(step, micro=self.n_micro)
        self.step(per_bucket=per_bucket)

    def step(self, per_bucket=False, replicas=None, clear_flags=True, exchange=None):
        """One optimizer step through the C ABI (fused or two-pass), with the
        accumulators of the earlier micro-batches when n_micro > 1.
        exchange: None for a group that holds all its owners' decisions, or a
        callable that sums this process's zero_exchange blob (a uint8 device
        tensor) with the other processes' (see dist.sum_exchange), for owners
        split over processes."""
        st = self.sptr
        if clear_flags:
            with torch.cuda.stream(self.stream):
                self.flags.zero_()
        reps = self.rep_ptrs(replicas)
        acc = self.accum_ptrs() if self.n_micro > 1 else None
        k = self.n_micro
        m, v, w = self._state_ptrs(0), self._state_ptrs(1), self._state_ptrs(2)
        sc = self.scaler.data_ptr()
        fl = self.flags.data_ptr()
        ex = self.exchange.data_ptr()
        if not self.two_pass:
            if exchange is None:
                zero_step_accum(self.plan, self.lo, self.hi, m, v, w, self.n_sets, None, reps,
                                acc, k, self.wbase, self.flat.data_ptr(), self.hp, sc, fl, st)
                return
            zero_step_update_accum(self.plan, self.lo, self.hi, m, v, w, self.n_sets, None, reps,
                                   acc, k, self.wbase, self.flat.data_ptr(), self.hp, sc, fl, st)
            zero_grad_norm_local(self.plan, self.lo, self.hi, None, self.hp, sc, 0, ex, st)
            exchange(self.exchange)
            zero_grad_norm_apply(self.plan, ex, self.hp, sc, st)
            zero_step_finish(self.plan, self.lo, self.hi, m, self.n_sets, None, self.wbase,
                             self.flat.data_ptr(), self.hp, sc, st)
            return
        clip = self.hp.max_grad_norm > 0
        ws = self.workspace.data_ptr() if clip else 0
        gp = self.ghat_ptrs()
        buckets = range(self.info.n_buckets) if per_bucket else [-1]
        for b in buckets:
            zero_reduce_scatter_accum(self.plan, b, self.lo, self.hi, reps, acc, k, self.wbase,
                                      gp, sc, fl, ws, st)
        if exchange is not None:
            zero_grad_norm_local(self.plan, self.lo, self.hi, None, self.hp, sc, ws, ex, st)
            exchange(self.exchange)
            zero_grad_norm_apply(self.plan, ex, self.hp, sc, st)
        elif clip:
            zero_grad_norm(self.plan, self.lo, self.hi, None, self.hp, sc, ws, st)
        zero_step(self.plan, self.lo, self.hi, m, v, w, self.n_sets, gp, None, self.wbase,
                  self.flat.data_ptr(), self.hp, sc, fl, st)

    # ----------------------------------------------------------- checkpoint
    def state_dict(self):
        """Everything a later step depends on, as CPU tensors: the owned
        master/exp_avg/exp_avg_sq shards of the current state set, the
        16-bit working parameters and the 80-byte device scaler. The other
        ping-pong set and the replicas are scratch between steps."""
        self.stream.synchronize()
        idx = self.read_scaler().state_index if self.n_sets == 2 else 0
        return {"state": self.state[idx].cpu().clone(), "flat": self.flat.cpu().clone(),
                "scaler": self.scaler.cpu().clone(), "workload": self.wl.name,
                "layout": (self.N, self.lo, self.hi, self.S, self.srow, self.row)}

    def load_state_dict(self, sd):
        """Restore a state_dict() of the same workload and layout; the state
        goes back into the set the saved scaler names as current."""
        if sd["workload"] != self.wl.name or tuple(sd["layout"]) != (
                self.N, self.lo, self.hi, self.S, self.srow, self.row):
            raise ValueError("state_dict of another workload or layout")
        self.stream.synchronize()
        self.scaler.copy_(sd["scaler"])
        idx = self.read_scaler().state_index if self.n_sets == 2 else 0
        self.state[idx].copy_(sd["state"])
        self.flat.copy_(sd["flat"])
        torch.cuda.synchronize()

    # ------------------------------------------------------------- readback
    def current_state(self):
        """(master, exp_avg, exp_avg_sq) of the owned window as fp32 CPU
        tensors indexed by flat element - wbase."""
        idx = self.read_scaler().state_index if self.n_sets == 2 else 0
        st = self.state[idx, :, :, :self.S].reshape(3, -1).cpu()
        return st[0], st[1], st[2]

    def params_u16(self):
        self.stream.synchronize()
        return self.flat[:self.wlen].cpu().numpy().view("uint16")

    def replicas_u16(self):
        self.stream.synchronize()
        return self.replicas[:, :self.wlen].cpu().numpy().view("uint16")

    def flags_u32(self):
        self.stream.synchronize()
        return self.flags[:self.info.n_buckets].cpu().numpy().view("uint32")


class UnitGroup:
    """Device state of a stage-3 unit layout on one GPU: the N ranks' 16-bit
    shard buffers and a ring of `window` unit buffers, each large enough for
    the biggest gathered unit (only a window of units is ever resident).

      shards   int16 [N, row]            rank r's slices of every unit, row =
                                         shard elements rounded up to 8
      buffers  int16 [window, urow]      gathered units, urow = largest unit
                                         rounded up to 8
    """

    def __init__(self, uwl, device="cuda", window=2, stream=None):
        self.wl = uwl
        self.dev = torch.device(device)
        self.N = uwl.n_ranks
        self.plan = zero_unit_plan_create(uwl.numels, uwl.unit_of_tensor, uwl.n_units, self.N,
                                          uwl.align_elems)
        self.info = zero_unit_plan_get_info(self.plan)
        self.units = zero_unit_plan_units(self.plan)
        self.row = _round_up(max(self.info.shard_elems, 1), 8)
        self.urow = _round_up(max(self.info.max_unit_psi_pad, 1), 8)
        self.window = window
        self.stream = stream if stream is not None else torch.cuda.Stream(device=self.dev)
        self.sptr = self.stream.cuda_stream
        self.shards = torch.zeros((self.N, self.row), dtype=torch.int16, device=self.dev)
        self.buffers = torch.zeros((window, self.urow), dtype=torch.int16, device=self.dev)

    def close(self):
        if self.plan:
            zero_unit_plan_destroy(self.plan)
            self.plan = None

    def shard_ptrs(self):
        base, rb = self.shards.data_ptr(), self.row * 2
        return [base + r * rb for r in range(self.N)]

    def buffer_ptr(self, slot):
        return self.buffers.data_ptr() + (slot % self.window) * self.urow * 2

    def fill_shards(self, seed=None):
        """Seeded 16-bit patterns in every shard buffer (the generator's bf16
        normal stream, one stream per rank)."""
        spec = synth.grad_spec(seed=self.wl.seed if seed is None else seed, sigma=1.0,
                               psi=self.row)
        for r, ptr in enumerate(self.shard_ptrs()):
            synth.gpu_fill_grad(ptr, self.row, 0, spec, 1, r, True, self.sptr)

    def gather(self, unit_lo, unit_hi, slot0=0):
        """All-gather units [unit_lo, unit_hi) into buffer slots slot0, slot0 + 1, ..."""
        ptrs = [self.buffer_ptr(slot0 + i) for i in range(unit_hi - unit_lo)]
        zero_gather_units(self.plan, unit_lo, unit_hi, self.shard_ptrs(), ptrs, self.sptr)

    def shard(self, unit_lo, unit_hi, slot0=0):
        """Write buffer slots slot0, ... back into the units' slices."""
        ptrs = [self.buffer_ptr(slot0 + i) for i in range(unit_hi - unit_lo)]
        zero_shard_units(self.plan, unit_lo, unit_hi, ptrs, self.shard_ptrs(), self.sptr)


class RingRank:
    """Device state of one rank of a group whose N ranks are N processes
    (one gradient replica each; "How far does splitting the batch get you?",
    "Why does the all-reduce not get more expensive with more ranks?"):

      grad     int16 [row]            this rank's 16-bit gradient, all psi_pad
                                      elements (row rounded up to 8)
      flat     int16 [row]            16-bit working parameters, all slots
                                      (own slot written by the step, the
                                      others by the all-gather)
      state    fp32 [n_sets, 3, srow] master / exp_avg / exp_avg_sq of this
                                      rank's slice
      shard    fp32 [srow]            this rank's reduced gradient
      bufs     fp32 [2, srow]         partials sent to and received from the
                                      neighbours
    plus the scaler, bucket flags, norm workspace and exchange blob.
    """

    def __init__(self, wl, rank, device="cuda", stream=None, n_sets=2):
        self.wl = wl
        self.rank = rank
        self.device = torch.device(device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.plan = zero_plan_create(wl.numels, wl.n_ranks, wl.bucket_elems,
                                     ZERO_BF16 if wl.is_bf16 else ZERO_FP16)
        self.info = zero_plan_get_info(self.plan)
        self.N, self.S = wl.n_ranks, self.info.shard_elems
        self.n_sets = n_sets
        self.hp = hparams_of(wl)
        self.row = _round_up(max(self.info.psi_pad, 1), 8)
        self.srow = _round_up(max(self.S, 1), 4)
        dev = self.device
        self.grad = torch.zeros(self.row, dtype=torch.int16, device=dev)
        self.flat = torch.zeros(self.row, dtype=torch.int16, device=dev)
        self.state = torch.zeros((n_sets, 3, self.srow), dtype=torch.float32, device=dev)
        self.shard = torch.zeros(self.srow, dtype=torch.float32, device=dev)
        self.bufs = torch.zeros((2, self.srow), dtype=torch.float32, device=dev)
        self.scaler = torch.zeros(C.sizeof(ZeroScaler), dtype=torch.uint8, device=dev)
        self.flags = torch.zeros(max(self.info.n_buckets, 1), dtype=torch.int32, device=dev)
        ws = zero_workspace_bytes(self.plan, 1)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev)
        self.exchange = torch.zeros(C.sizeof(ZeroExchange), dtype=torch.uint8, device=dev)

    def close(self):
        if self.plan:
            zero_plan_destroy(self.plan)
            self.plan = None

    @property
    def sptr(self):
        return self.stream.cuda_stream

    def _per_rank(self, ptr):
        out = [None] * self.N
        out[self.rank] = ptr
        return out

    def _state_ptrs(self, which):
        out = [None] * (self.n_sets * self.N)
        for s in range(self.n_sets):
            out[s * self.N + self.rank] = self.state[s, which].data_ptr()
        return out

    def init_state(self):
        """Master slice from the seeded generator, m = v = 0, the own slot of
        the parameters cast from it, the others all-gathered by the caller."""
        wl, r, S = self.wl, self.rank, self.S
        with torch.cuda.stream(self.stream):
            self.state.zero_()
            synth.gpu_fill_master(self.state[0, 0].data_ptr(), S, r * S, wl.seed, wl.psi,
                                  self.sptr)
            zero_cast_params(self.plan, r, r + 1, self._per_rank(self.state[0, 0].data_ptr()),
                             self.flat.data_ptr(), 0, self.sptr)
            self.scaler.copy_(torch.frombuffer(bytearray(bytes(zero_scaler_init(self.hp))),
                                               dtype=torch.uint8))

    def read_scaler(self):
        self.stream.synchronize()
        return ZeroScaler.from_buffer_copy(bytes(self.scaler.cpu().numpy().tobytes()))

    def gen_grads(self, step, scale=None):
        """This rank's replica of step `step` (replica index = rank), with the
        workload's injection when it lands in this replica."""
        if scale is None:
            scale = self.read_scaler().scale
        wl = self.wl
        spec = synth.grad_spec(seed=wl.seed, sigma=wl.sigma, bias_sigma=wl.bias_sigma,
                               loss_scale=scale, outliers=wl.outliers, psi=wl.psi)
        synth.gpu_fill_grad(self.grad.data_ptr(), self.info.psi_pad, 0, spec,
                            wl.gen_step(step, wl.n_micro), self.rank, wl.is_bf16, self.sptr)
        inj = wl.inject
        if inj is not None and inj[0] == step and inj[1] == self.rank:
            with torch.cuda.stream(self.stream):
                self.grad[inj[2]] = inj[3] - 65536 if inj[3] >= 32768 else inj[3]

    def step(self, group=None):
        """One optimizer step: ring reduce-scatter, the global scalars across
        the processes, the update of this rank's slice, the all-gather."""
        from . import dist as zdist
        st, r = self.sptr, self.rank
        with torch.cuda.stream(self.stream):
            self.flags.zero_()
        sc, fl = self.scaler.data_ptr(), self.flags.data_ptr()
        zdist.ring_reduce_scatter(self.plan, r, self.N, self.grad.data_ptr(), self.shard,
                                  (self.bufs[0], self.bufs[1]), sc, fl, self.stream, group)
        gp = self._per_rank(self.shard.data_ptr())
        ex = self.exchange.data_ptr()
        clip = self.hp.max_grad_norm > 0
        zero_grad_norm_local(self.plan, r, r + 1, gp if clip else None, self.hp, sc,
                             self.workspace.data_ptr(), ex, st)
        zdist.sum_exchange(self.exchange, self.stream, group)
        zero_grad_norm_apply(self.plan, ex, self.hp, sc, st)
        zero_step(self.plan, r, r + 1, self._state_ptrs(0), self._state_ptrs(1),
                  self._state_ptrs(2), self.n_sets, gp, None, 0, self.flat.data_ptr(), self.hp,
                  sc, fl, st)
        zdist.all_gather_params(self.flat, r, self.N, self.S, self.stream, group)

    def current_state(self):
        idx = self.read_scaler().state_index if self.n_sets == 2 else 0
        st = self.state[idx, :, :self.S].cpu()
        return st[0], st[1], st[2]
