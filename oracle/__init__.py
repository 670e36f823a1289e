"""CPU checker (oracle) for the sharded mixed-precision AdamW step.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg call it; the product path never imports it. It shares no code
with the CUDA library; its inputs come from the shared seeded generator
(``fsdp_sharded_mixed_shard_gb300.synth``), which holds none of the step's
arithmetic.

This module is a ctypes binding of liboracle.so (oracle.c): all arithmetic is
in the C file, which cites the passages it follows.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


class Segment(C.Structure):
    _fields_ = [("lo", C.c_int64), ("hi", C.c_int64), ("rank", C.c_int32), ("bucket", C.c_int32)]


class Plan(C.Structure):
    _fields_ = [("psi", C.c_int64), ("pad", C.c_int64), ("psi_pad", C.c_int64),
                ("shard", C.c_int64), ("bucket_elems", C.c_int64), ("n_ranks", C.c_int32),
                ("n_buckets", C.c_int32), ("n_segments", C.c_int32), ("reserved", C.c_int32),
                ("bill_ddp", C.c_double), ("bill_z1", C.c_double), ("bill_z2", C.c_double),
                ("bill_z3", C.c_double), ("ring_bytes_per_rank", C.c_double),
                ("ring_hops", C.c_double), ("comm_ddp", C.c_double), ("comm_z1", C.c_double),
                ("comm_z2", C.c_double), ("comm_z3", C.c_double)]


class HParams(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double),
                ("max_grad_norm", C.c_double), ("dynamic_scale", C.c_int32),
                ("growth_interval", C.c_int32)]


class Scaler(C.Structure):
    _fields_ = [("scale", C.c_float), ("good_steps", C.c_int32), ("t", C.c_int32),
                ("overflow", C.c_int32), ("norm_sq", C.c_double), ("norm", C.c_double),
                ("clip_coef", C.c_float), ("reserved", C.c_int32)]


class AdamScalars(C.Structure):
    _fields_ = [(n, C.c_float) for n in ("b1", "omb1", "b2", "omb2", "bc1", "bc2", "lr",
                                         "decay", "eps")]


class GradSpec(C.Structure):
    """Mirror of synth.h's zs_grad_spec."""
    _fields_ = [("seed", C.c_uint64), ("sigma", C.c_float), ("bias_sigma", C.c_float),
                ("loss_scale", C.c_float), ("outliers", C.c_int32), ("psi", C.c_int64)]


class Unit(C.Structure):
    _fields_ = [("psi", C.c_int64), ("pad", C.c_int64), ("psi_pad", C.c_int64),
                ("shard", C.c_int64), ("shard_offset", C.c_int64), ("flat_offset", C.c_int64),
                ("n_tensors", C.c_int32), ("first_slot", C.c_int32)]


class UnitPlan(C.Structure):
    _fields_ = [("psi", C.c_int64), ("psi_pad", C.c_int64), ("shard", C.c_int64),
                ("max_unit_psi_pad", C.c_int64), ("n_units", C.c_int32),
                ("n_ranks", C.c_int32), ("n_tensors", C.c_int32), ("align_elems", C.c_int32),
                ("persistent_bytes", C.c_double), ("peak_one_bytes", C.c_double),
                ("peak_two_bytes", C.c_double), ("peak_backward_bytes", C.c_double),
                ("max_unit_fraction", C.c_double), ("comm_elems", C.c_double),
                ("comm_bytes", C.c_double), ("ring_bytes", C.c_double),
                ("n_gathers", C.c_int32), ("reserved", C.c_int32)]


class StrategyCost(C.Structure):
    _fields_ = [("persistent_bytes", C.c_double), ("peak_bytes", C.c_double),
                ("comm_elems", C.c_double), ("comm_elems_inter", C.c_double),
                ("ring_bytes", C.c_double), ("ring_bytes_inter", C.c_double),
                ("shard_ranks", C.c_int32), ("gathers_per_unit", C.c_int32)]


FULL_SHARD, SHARD_GRAD_OP, NO_SHARD, HYBRID_SHARD, NO_RESHARD_AFTER_FORWARD = range(5)


class Gen(C.Structure):
    _fields_ = [("spec", GradSpec), ("is_bf16", C.c_int32), ("inject_step", C.c_int32),
                ("inject_rank", C.c_int32), ("inject_bits", C.c_uint32),
                ("inject_elem", C.c_int64)]


def lib():
    """Load (building if needed) liboracle.so."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.POINTER
        L.orc_plan_make.argtypes = [P(C.c_int64), C.c_int32, C.c_int32, C.c_int64, P(Plan),
                                    P(C.c_int64), P(Segment), C.c_int32]
        L.orc_plan_make.restype = C.c_int
        L.orc_bills.argtypes = [C.c_double, C.c_int32, P(C.c_double)]
        L.orc_ring_bytes.argtypes = [C.c_double, C.c_int32]
        L.orc_ring_bytes.restype = C.c_double
        L.orc_f32_to_f16.argtypes = [C.c_float]
        L.orc_f32_to_f16.restype = C.c_uint16
        L.orc_f32_to_bf16.argtypes = [C.c_float]
        L.orc_f32_to_bf16.restype = C.c_uint16
        L.orc_f16_to_f32.argtypes = [C.c_uint16]
        L.orc_f16_to_f32.restype = C.c_float
        L.orc_bf16_to_f32.argtypes = [C.c_uint16]
        L.orc_bf16_to_f32.restype = C.c_float
        L.orc_cast_array.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int32]
        L.orc_widen_array.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int32]
        L.orc_ring_sum.argtypes = [C.c_void_p, C.c_int32, C.c_int32]
        L.orc_ring_sum.restype = C.c_float
        L.orc_unscale_factor.argtypes = [C.c_float, C.c_int32]
        L.orc_unscale_factor.restype = C.c_float
        L.orc_adam_scalars_make.argtypes = [P(HParams), C.c_int32]
        L.orc_adam_scalars_make.restype = AdamScalars
        L.orc_adamw_elem.argtypes = [P(C.c_float), P(C.c_float), P(C.c_float), C.c_float,
                                     P(AdamScalars)]
        L.orc_clip_coef.argtypes = [C.c_double, C.c_double, P(C.c_float), P(C.c_double)]
        L.orc_clip_coef.restype = C.c_int32
        L.orc_scaler_finish.argtypes = [P(Scaler), P(HParams), C.c_int32]
        L.orc_step_arrays.argtypes = [P(Plan), C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                      C.c_int64, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_void_p, C.c_void_p, P(HParams),
                                      P(Scaler)]
        L.orc_step_arrays.restype = C.c_int
        L.orc_step_arrays_f32.argtypes = [P(Plan), C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                          C.c_int32, C.c_int64, C.c_void_p, C.c_void_p,
                                          C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                          P(HParams), P(Scaler)]
        L.orc_step_arrays_f32.restype = C.c_int
        L.orc_unscale_factor_k.argtypes = [C.c_float, C.c_int32, C.c_int32]
        L.orc_unscale_factor_k.restype = C.c_float
        L.orc_accumulate.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int32, C.c_int32]
        L.orc_gen_step.argtypes = [P(Plan), C.c_int32, C.c_int32, P(Gen), C.c_uint32,
                                   C.c_int32, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                                   C.c_void_p, C.c_void_p, C.c_void_p, P(HParams), P(Scaler)]
        L.orc_gen_step.restype = C.c_int
        L.orc_gen_ghat.argtypes = [P(Plan), P(Gen), C.c_uint32, C.c_float, C.c_void_p,
                                   C.c_int64, C.c_void_p]
        L.orc_gen_ghat.restype = C.c_int
        L.orc_unit_plan_make.argtypes = [P(C.c_int64), C.c_int32, P(C.c_int32), C.c_int32,
                                         C.c_int32, C.c_int32, P(UnitPlan), P(Unit),
                                         P(C.c_int32), P(C.c_int64)]
        L.orc_unit_plan_make.restype = C.c_int
        L.orc_gather_unit.argtypes = [P(Unit), C.c_int32, C.c_void_p, C.c_void_p]
        L.orc_shard_unit.argtypes = [P(Unit), C.c_int32, C.c_void_p, C.c_void_p]
        L.orc_strategy_cost_make.argtypes = [P(UnitPlan), C.c_int32, C.c_int32,
                                             P(StrategyCost)]
        L.orc_strategy_cost_make.restype = C.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


# ------------------------------------------------------------------ plan ----

def make_plan(numels, n_ranks, bucket_elems=0):
    """Returns (Plan, offsets ndarray, list of (lo, hi, rank, bucket))."""
    L = lib()
    arr = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    offs = np.zeros(max(len(arr), 1), dtype=np.int64)
    p = Plan()
    rc = L.orc_plan_make(arr.ctypes.data_as(C.POINTER(C.c_int64)), len(arr), n_ranks,
                         bucket_elems, C.byref(p), offs.ctypes.data_as(C.POINTER(C.c_int64)),
                         None, 0)
    if rc != 0:
        raise ValueError("orc_plan_make failed: %d" % rc)
    segs = (Segment * max(p.n_segments, 1))()
    rc = L.orc_plan_make(arr.ctypes.data_as(C.POINTER(C.c_int64)), len(arr), n_ranks,
                         bucket_elems, C.byref(p), offs.ctypes.data_as(C.POINTER(C.c_int64)),
                         segs, p.n_segments)
    if rc != 0:
        raise ValueError("orc_plan_make failed: %d" % rc)
    seglist = [(s.lo, s.hi, s.rank, s.bucket) for s in segs[:p.n_segments]]
    return p, offs[:len(arr)].copy(), seglist


def bills(psi, n_ranks):
    out = (C.c_double * 4)()
    lib().orc_bills(float(psi), n_ranks, out)
    return list(out)


def ring_bytes(m_bytes, d):
    return lib().orc_ring_bytes(float(m_bytes), d)


# ----------------------------------------------------------------- casts ----

def cast16(x, is_bf16):
    """fp32 array -> uint16 bit patterns (RNE)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_cast_array(_ptr(x), _ptr(out), x.size, int(bool(is_bf16)))
    return out


def widen16(h, is_bf16):
    h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16))
    out = np.empty(h.shape, dtype=np.float32)
    lib().orc_widen_array(_ptr(h), _ptr(out), h.size, int(bool(is_bf16)))
    return out


# --------------------------------------------------------- building blocks ----

def ring_sum(vals, owner):
    v = np.ascontiguousarray(np.asarray(vals, dtype=np.float32))
    return np.float32(lib().orc_ring_sum(_ptr(v), len(v), owner))


def unscale_factor(scale, n_ranks):
    return np.float32(lib().orc_unscale_factor(scale, n_ranks))


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
            max_grad_norm=0.0, dynamic_scale=0, growth_interval=2000):
    return HParams(lr, beta1, beta2, eps, weight_decay, max_grad_norm, dynamic_scale,
                   growth_interval)


def scaler(scale=1.0):
    return Scaler(scale, 0, 0, 0, 0.0, 0.0, 1.0, 0)


def adam_scalars(hp, t):
    return lib().orc_adam_scalars_make(C.byref(hp), t)


def adamw_elem(theta, m, v, g, scal):
    th, mm, vv = C.c_float(theta), C.c_float(m), C.c_float(v)
    lib().orc_adamw_elem(C.byref(th), C.byref(mm), C.byref(vv), float(g), C.byref(scal))
    return np.float32(th.value), np.float32(mm.value), np.float32(vv.value)


def clip_coef(norm_sq, max_norm):
    c = C.c_float()
    n = C.c_double()
    apply = lib().orc_clip_coef(norm_sq, max_norm, C.byref(c), C.byref(n))
    return bool(apply), np.float32(c.value), n.value


def scaler_finish(sc, hp, overflow):
    lib().orc_scaler_finish(C.byref(sc), C.byref(hp), int(bool(overflow)))


# ---------------------------------------------------------------- drivers ----

def step_arrays(plan, rank_lo, rank_hi, is_bf16, replicas, wbase, master, m, v, params,
                hp, sc, bucket_flags=None, ghat=None):
    """One step on host arrays (modified in place). replicas: list of uint16
    arrays indexed by flat element - wbase."""
    reps = [np.ascontiguousarray(r, dtype=np.uint16) for r in replicas]
    ptrs = (C.c_void_p * len(reps))(*[r.ctypes.data for r in reps])
    for a, dt in ((master, np.float32), (m, np.float32), (v, np.float32), (params, np.uint16)):
        assert a.dtype == dt and a.flags.c_contiguous
    rc = lib().orc_step_arrays(C.byref(plan), rank_lo, rank_hi, int(bool(is_bf16)), ptrs,
                               wbase, _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                               _ptr(ghat), _ptr(bucket_flags), C.byref(hp), C.byref(sc))
    if rc != 0:
        raise ValueError("orc_step_arrays failed")


def unscale_factor_k(scale, n_ranks, n_micro):
    return np.float32(lib().orc_unscale_factor_k(scale, n_ranks, n_micro))


def accumulate(micro, acc, is_bf16, first):
    """acc (fp32, modified in place) += widen(micro); first: acc = widen(micro)."""
    micro = np.ascontiguousarray(micro, dtype=np.uint16)
    assert acc.dtype == np.float32 and acc.flags.c_contiguous and acc.size == micro.size
    lib().orc_accumulate(_ptr(micro), _ptr(acc), micro.size, int(bool(is_bf16)),
                         int(bool(first)))


def step_arrays_f32(plan, rank_lo, rank_hi, is_bf16, replicas_f32, n_micro, wbase, master, m, v,
                    params, hp, sc, bucket_flags=None, ghat=None):
    """One step whose replica values are fp32 accumulated gradients of
    n_micro micro-batches."""
    reps = [np.ascontiguousarray(r, dtype=np.float32) for r in replicas_f32]
    ptrs = (C.c_void_p * len(reps))(*[r.ctypes.data for r in reps])
    rc = lib().orc_step_arrays_f32(C.byref(plan), rank_lo, rank_hi, int(bool(is_bf16)), ptrs,
                                   n_micro, wbase, _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                                   _ptr(ghat), _ptr(bucket_flags), C.byref(hp), C.byref(sc))
    if rc != 0:
        raise ValueError("orc_step_arrays_f32 failed")


def gen(spec, is_bf16, inject=None):
    """inject = (step, rank, elem, bits16) or None."""
    g = Gen()
    g.spec = GradSpec(spec.seed, spec.sigma, spec.bias_sigma, spec.loss_scale, spec.outliers,
                      spec.psi)
    g.is_bf16 = int(bool(is_bf16))
    if inject is None:
        g.inject_step, g.inject_rank, g.inject_elem, g.inject_bits = -1, 0, 0, 0
    else:
        g.inject_step, g.inject_rank, g.inject_elem, g.inject_bits = inject
    return g


def gen_step(plan, rank_lo, rank_hi, g, step, elems, master, m, v, params, hp, sc,
             bucket_flags=None, n_threads=None):
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    elems = np.ascontiguousarray(elems, dtype=np.int64)
    rc = lib().orc_gen_step(C.byref(plan), rank_lo, rank_hi, C.byref(g), step, n_threads,
                            _ptr(elems), len(elems), _ptr(master), _ptr(m), _ptr(v),
                            _ptr(params), _ptr(bucket_flags), C.byref(hp), C.byref(sc))
    if rc != 0:
        raise ValueError("orc_gen_step failed")


def gen_ghat(plan, g, step, scale, elems):
    elems = np.ascontiguousarray(elems, dtype=np.int64)
    out = np.empty(len(elems), dtype=np.float32)
    rc = lib().orc_gen_ghat(C.byref(plan), C.byref(g), step, scale, _ptr(elems), len(elems),
                            _ptr(out))
    if rc != 0:
        raise ValueError("orc_gen_ghat failed")
    return out


# ------------------------------------------------------ stage-3 FSDP units ----

def make_unit_plan(numels, unit_of_tensor, n_units, n_ranks, align_elems=1):
    """Returns (UnitPlan, [Unit], slot_tensor ndarray, tensor_offset ndarray)."""
    L = lib()
    arr = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    uot = np.ascontiguousarray(np.asarray(unit_of_tensor, dtype=np.int32))
    if len(arr) != len(uot):
        raise ValueError("numels and unit_of_tensor differ in length")
    units = (Unit * max(n_units, 1))()
    slots = np.zeros(max(len(arr), 1), dtype=np.int32)
    offs = np.zeros(max(len(arr), 1), dtype=np.int64)
    p = UnitPlan()
    rc = L.orc_unit_plan_make(arr.ctypes.data_as(C.POINTER(C.c_int64)), len(arr),
                              uot.ctypes.data_as(C.POINTER(C.c_int32)), n_units, n_ranks,
                              align_elems, C.byref(p), units,
                              slots.ctypes.data_as(C.POINTER(C.c_int32)),
                              offs.ctypes.data_as(C.POINTER(C.c_int64)))
    if rc != 0:
        raise ValueError("orc_unit_plan_make failed: %d" % rc)
    return p, list(units)[:n_units], slots[:len(arr)], offs[:len(arr)]


def _ptr_array(arrays):
    ptrs = (C.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])
    return ptrs


def gather_unit(unit, shards):
    """All-gather of one unit from the N ranks' 16-bit shard buffers."""
    for a in shards:
        assert a.dtype == np.uint16 and a.flags.c_contiguous
        assert a.size >= unit.shard_offset + unit.shard
    full = np.empty(unit.psi_pad, dtype=np.uint16)
    lib().orc_gather_unit(C.byref(unit), len(shards), _ptr_array(shards), _ptr(full))
    return full


def shard_unit(unit, full, shards):
    """Write one gathered unit's slices into the N ranks' shard buffers."""
    full = np.ascontiguousarray(full, dtype=np.uint16)
    assert full.size == unit.psi_pad
    for a in shards:
        assert a.dtype == np.uint16 and a.flags.c_contiguous
        assert a.size >= unit.shard_offset + unit.shard
    lib().orc_shard_unit(C.byref(unit), len(shards), _ptr(full), _ptr_array(shards))


def strategy_cost(unit_plan, strategy, n_replicas=1):
    out = StrategyCost()
    rc = lib().orc_strategy_cost_make(C.byref(unit_plan), strategy, n_replicas, C.byref(out))
    if rc != 0:
        raise ValueError("orc_strategy_cost_make failed: %d" % rc)
    return out
