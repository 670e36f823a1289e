"""libzero Python binding: the per-shard ZeRO step of mixed-precision AdamW on
one GB300.

A thin ctypes layer over the C ABI in include/zero.h: every function below
has the C function's name and only marshals arguments (device pointers are
plain Python ints, host arrays become C arrays); all computation happens in
the sm_103a kernels of _lib/libzero.so. Loading fails loudly when the library
has not been built (run ``__graft_entry__.build()``); there is no fallback.
"""
import ctypes as C

import numpy as np
import os

from . import _build

__all__ = [
    "ZeroError", "ZeroPlanInfo", "ZeroSegment", "ZeroBucket", "ZeroHParams", "ZeroScaler",
    "ZeroNormRecord", "ZeroExchange",
    "ZERO_BF16", "ZERO_FP16", "ZERO_MAX_RANKS", "ZERO_TILE_ELEMS", "ZERO_NORM_OWNER_BLOCKS",
    "zero_plan_create", "zero_plan_destroy", "zero_plan_get_info", "zero_plan_info_get",
    "zero_plan_tensor_offsets", "zero_plan_segments", "zero_plan_buckets",
    "zero_plan_bucket_range", "zero_workspace_bytes", "zero_scaler_init",
    "zero_reduce_scatter", "zero_grad_norm", "zero_grad_norm_local", "zero_grad_norm_apply",
    "zero_ring_hop",
    "zero_step", "zero_step_update", "zero_step_finish",
    "zero_cast_params", "zero_accumulate", "zero_reduce_scatter_accum", "zero_step_accum",
    "zero_step_update_accum", "zero_grad_norm_noalloc", "zero_selftest_wait_timeout", "zero_strerror",
    "zero_checked_status", "zero_selftest_check", "use_checked_library",
    "zero_version", "lib",
    "ZeroUnit", "ZeroUnitPlanInfo", "ZERO_UNIT_MAX_ALIGN", "zero_unit_plan_create",
    "zero_unit_plan_destroy", "zero_unit_plan_get_info", "zero_unit_plan_units",
    "zero_unit_plan_tensors", "zero_gather_units", "zero_shard_units",
    "ZeroStrategyCost", "zero_unit_plan_strategy_cost", "ZERO_FULL_SHARD", "ZERO_SHARD_GRAD_OP",
    "ZERO_NO_SHARD", "ZERO_HYBRID_SHARD", "ZERO_NO_RESHARD_AFTER_FORWARD",
]

ZERO_BF16 = 0
ZERO_FP16 = 1
ZERO_MAX_RANKS = 64
ZERO_TILE_ELEMS = 4096
ZERO_NORM_OWNER_BLOCKS = 16
ZERO_UNIT_MAX_ALIGN = 4096
(ZERO_FULL_SHARD, ZERO_SHARD_GRAD_OP, ZERO_NO_SHARD, ZERO_HYBRID_SHARD,
 ZERO_NO_RESHARD_AFTER_FORWARD) = range(5)


class ZeroError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__("%s failed: %s (%d)" % (fn, zero_strerror(status), status))
        self.status = status


class ZeroPlanInfo(C.Structure):
    _fields_ = [("psi", C.c_int64), ("pad", C.c_int64), ("psi_pad", C.c_int64),
                ("shard_elems", C.c_int64), ("bucket_elems", C.c_int64), ("n_tiles", C.c_int64),
                ("n_ranks", C.c_int32), ("n_buckets", C.c_int32), ("n_segments", C.c_int32),
                ("n_tensors", C.c_int32), ("grad_dtype", C.c_int32), ("reserved", C.c_int32),
                ("bill_ddp", C.c_double), ("bill_z1", C.c_double), ("bill_z2", C.c_double),
                ("bill_z3", C.c_double), ("ring_bytes_per_rank", C.c_double),
                ("ring_hops", C.c_double), ("comm_elems_ddp", C.c_double),
                ("comm_elems_z1", C.c_double), ("comm_elems_z2", C.c_double),
                ("comm_elems_z3", C.c_double), ("step_bytes_fused", C.c_double),
                ("step_bytes_two_pass", C.c_double)]


class ZeroSegment(C.Structure):
    _fields_ = [("lo", C.c_int64), ("hi", C.c_int64), ("rank", C.c_int32), ("bucket", C.c_int32)]


class ZeroBucket(C.Structure):
    _fields_ = [("lo", C.c_int64), ("hi", C.c_int64), ("seg_first", C.c_int32),
                ("seg_count", C.c_int32)]


class ZeroNormRecord(C.Structure):
    _fields_ = [("hi", C.c_float), ("lo", C.c_float), ("big_hi", C.c_float),
                ("big_lo", C.c_float)]


class ZeroExchange(C.Structure):
    """zero.h zero_exchange: one process's share of a step's global scalars."""
    _fields_ = [("overflow", C.c_uint32), ("reserved", C.c_uint32 * 3),
                ("owner", ZeroNormRecord * ZERO_MAX_RANKS)]


class ZeroHParams(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double),
                ("max_grad_norm", C.c_double), ("dynamic_scale", C.c_int32),
                ("growth_interval", C.c_int32), ("init_scale", C.c_double)]


class ZeroScaler(C.Structure):
    _fields_ = [("scale", C.c_float), ("good_steps", C.c_int32), ("t", C.c_int32),
                ("pending", C.c_uint32), ("overflow", C.c_uint32), ("state_index", C.c_int32),
                ("beta1_pow", C.c_double), ("beta2_pow", C.c_double), ("norm_sq", C.c_double),
                ("norm", C.c_double), ("clip_coef", C.c_float), ("clip_apply", C.c_int32),
                ("norm_step", C.c_int32), ("n_skipped", C.c_int32), ("error", C.c_int32),
                ("finish_count", C.c_uint32)]


class ZeroUnit(C.Structure):
    """zero_units.h zero_unit: one stage-3 FSDP unit of a unit plan."""
    _fields_ = [("psi", C.c_int64), ("pad", C.c_int64), ("psi_pad", C.c_int64),
                ("shard_elems", C.c_int64), ("shard_offset", C.c_int64),
                ("flat_offset", C.c_int64), ("n_tensors", C.c_int32), ("first_slot", C.c_int32)]


class ZeroUnitPlanInfo(C.Structure):
    _fields_ = [("psi", C.c_int64), ("psi_pad", C.c_int64), ("shard_elems", C.c_int64),
                ("max_unit_psi_pad", C.c_int64), ("n_units", C.c_int32), ("n_ranks", C.c_int32),
                ("n_tensors", C.c_int32), ("align_elems", C.c_int32),
                ("persistent_bytes", C.c_double), ("peak_one_bytes", C.c_double),
                ("peak_two_bytes", C.c_double), ("peak_backward_bytes", C.c_double),
                ("max_unit_fraction", C.c_double), ("comm_elems", C.c_double),
                ("comm_bytes", C.c_double), ("ring_bytes", C.c_double),
                ("n_gathers", C.c_int32), ("reserved", C.c_int32)]


class ZeroStrategyCost(C.Structure):
    _fields_ = [("persistent_bytes", C.c_double), ("peak_bytes", C.c_double),
                ("comm_elems", C.c_double), ("comm_elems_inter", C.c_double),
                ("ring_bytes", C.c_double), ("ring_bytes_inter", C.c_double),
                ("shard_ranks", C.c_int32), ("gathers_per_unit", C.c_int32)]


_lib = None
_variant = "release"
_VP = C.c_void_p
_P = C.POINTER


def use_checked_library():
    """Make this process load libzero_checked.so, the build whose kernels test
    every memory range they touch (see zero_checked_status), instead of
    libzero.so. Call it before the first library call."""
    global _variant
    if _lib is not None and _variant != "checked":
        raise RuntimeError("libzero.so is already loaded in this process")
    _variant = "checked"


def lib():
    """The loaded libzero.so, or libzero_checked.so after use_checked_library()
    (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.ZERO_CHECKED_LIB if _variant == "checked" else _build.ZERO_LIB
        if not os.path.exists(path):
            raise RuntimeError("libzero.so is not built (%s); run __graft_entry__.build()" % path)
        L = C.CDLL(path)
        L.zero_plan_create.argtypes = [_P(C.c_int64), C.c_int32, C.c_int32, C.c_int64, C.c_int,
                                       _P(_VP)]
        L.zero_plan_destroy.argtypes = [_VP]
        L.zero_plan_destroy.restype = None
        L.zero_plan_get_info.argtypes = [_VP, _P(ZeroPlanInfo)]
        L.zero_plan_info_get.argtypes = [_VP, _P(ZeroPlanInfo)]
        L.zero_plan_buckets.argtypes = [_VP, _P(ZeroBucket), _P(ZeroSegment)]
        L.zero_plan_tensor_offsets.argtypes = [_VP, _P(C.c_int64)]
        L.zero_plan_segments.argtypes = [_VP, _P(ZeroSegment), C.c_int32]
        L.zero_plan_bucket_range.argtypes = [_VP, C.c_int32, _P(C.c_int64), _P(C.c_int64)]
        L.zero_workspace_bytes.argtypes = [_VP, C.c_int32]
        L.zero_workspace_bytes.restype = C.c_size_t
        L.zero_scaler_init.argtypes = [_P(ZeroHParams), _P(ZeroScaler)]
        L.zero_reduce_scatter.argtypes = [_VP, C.c_int32, C.c_int32, C.c_int32, _P(_VP),
                                          C.c_int64, _P(_VP), _VP, _VP, _VP, _VP]
        L.zero_grad_norm.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP), _P(ZeroHParams), _VP,
                                     _VP, _VP]
        L.zero_grad_norm_local.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP),
                                           _P(ZeroHParams), _VP, _VP, _VP, _VP]
        L.zero_grad_norm_apply.argtypes = [_VP, _VP, _P(ZeroHParams), _VP, _VP]
        L.zero_ring_hop.argtypes = [_VP, C.c_int32, C.c_int32, _VP, _VP, _VP, _VP, _VP, _VP]
        L.zero_step.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP), _P(_VP), _P(_VP), C.c_int32,
                                _P(_VP), _P(_VP), C.c_int64, _VP, _P(ZeroHParams), _VP, _VP, _VP]
        L.zero_step_update.argtypes = L.zero_step.argtypes
        L.zero_step_finish.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP), C.c_int32, _P(_VP),
                                       C.c_int64, _VP, _P(ZeroHParams), _VP, _VP]
        L.zero_cast_params.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP), _VP, C.c_int64, _VP]
        L.zero_accumulate.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP), _P(_VP), C.c_int64,
                                      C.c_int32, _VP]
        L.zero_reduce_scatter_accum.argtypes = [_VP, C.c_int32, C.c_int32, C.c_int32, _P(_VP),
                                                _P(_VP), C.c_int32, C.c_int64, _P(_VP), _VP,
                                                _VP, _VP, _VP]
        L.zero_step_accum.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP), _P(_VP), _P(_VP),
                                      C.c_int32, _P(_VP), _P(_VP), _P(_VP), C.c_int32,
                                      C.c_int64, _VP, _P(ZeroHParams), _VP, _VP, _VP]
        L.zero_step_update_accum.argtypes = L.zero_step_accum.argtypes
        L.zero_grad_norm_noalloc.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP),
                                             _P(ZeroHParams), _VP, _VP]
        L.zero_selftest_wait_timeout.argtypes = [_VP, C.c_int64, _VP]
        L.zero_checked_status.argtypes = [_P(C.c_int64), _P(C.c_int64), _VP]
        L.zero_selftest_check.argtypes = [_VP]
        L.zero_strerror.argtypes = [C.c_int]
        L.zero_strerror.restype = C.c_char_p
        L.zero_version.argtypes = []
        L.zero_unit_plan_create.argtypes = [_P(C.c_int64), C.c_int32, _P(C.c_int32), C.c_int32,
                                            C.c_int32, C.c_int32, _P(_VP)]
        L.zero_unit_plan_destroy.argtypes = [_VP]
        L.zero_unit_plan_destroy.restype = None
        L.zero_unit_plan_get_info.argtypes = [_VP, _P(ZeroUnitPlanInfo)]
        L.zero_unit_plan_units.argtypes = [_VP, _P(ZeroUnit), C.c_int32]
        L.zero_unit_plan_tensors.argtypes = [_VP, _P(C.c_int32), _P(C.c_int64), C.c_int32]
        L.zero_unit_plan_strategy_cost.argtypes = [_VP, C.c_int32, C.c_int32,
                                                   _P(ZeroStrategyCost)]
        L.zero_gather_units.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP), _P(_VP), _VP]
        L.zero_shard_units.argtypes = [_VP, C.c_int32, C.c_int32, _P(_VP), _P(_VP), _VP]
        _lib = L
    return _lib


def _check(fn, rc):
    if rc != 0:
        raise ZeroError(fn, rc)


def _ptrs(seq, need=0, what="pointer array"):
    """Device addresses (a list of int or None, or a uint64 numpy array built
    once by the caller) -> void** for the call. The library reads `need`
    entries (it cannot see the length), so a shorter list is refused here.
    The returned pointer keeps its array alive for the call."""
    if seq is None:
        return None
    if isinstance(seq, np.ndarray):
        arr = np.ascontiguousarray(seq, dtype=np.uint64)
    else:
        arr = np.fromiter((0 if q is None else q for q in seq), dtype=np.uint64, count=len(seq))
    if arr.size < need:
        raise ValueError(f"{what}: {arr.size} entries, the call reads {need}")
    return arr.ctypes.data_as(_P(_VP))


def _ranks(plan):
    """N of a plan (the pointer arrays hold N or n_sets * N entries); 0 for
    an invalid plan, which the call itself then reports."""
    info = ZeroPlanInfo()
    if not plan or lib().zero_plan_get_info(plan, C.byref(info)) != 0:
        return 0
    return info.n_ranks


def _unit_ranks(plan):
    info = ZeroUnitPlanInfo()
    if not plan or lib().zero_unit_plan_get_info(plan, C.byref(info)) != 0:
        return 0
    return info.n_ranks


def _vp(x):
    return None if not x else _VP(int(x))


# ------------------------------------------------------------------ plan ----

def zero_plan_create(numels, n_ranks, bucket_elems=0, grad_dtype=ZERO_BF16):
    arr = (C.c_int64 * max(len(numels), 1))(*[int(n) for n in numels])
    out = _VP()
    _check("zero_plan_create", lib().zero_plan_create(arr, len(numels), n_ranks, bucket_elems,
                                                      grad_dtype, C.byref(out)))
    return out


def zero_plan_destroy(plan):
    lib().zero_plan_destroy(plan)


def zero_plan_get_info(plan):
    info = ZeroPlanInfo()
    _check("zero_plan_get_info", lib().zero_plan_get_info(plan, C.byref(info)))
    return info


def zero_plan_info_get(plan):
    info = ZeroPlanInfo()
    _check("zero_plan_info_get", lib().zero_plan_info_get(plan, C.byref(info)))
    return info


def zero_plan_tensor_offsets(plan):
    n = zero_plan_get_info(plan).n_tensors
    out = (C.c_int64 * max(n, 1))()
    _check("zero_plan_tensor_offsets", lib().zero_plan_tensor_offsets(plan, out))
    return list(out)[:n]


def zero_plan_segments(plan):
    n = zero_plan_get_info(plan).n_segments
    out = (ZeroSegment * max(n, 1))()
    _check("zero_plan_segments", lib().zero_plan_segments(plan, out, n))
    return [(s.lo, s.hi, s.rank, s.bucket) for s in out[:n]]


def zero_plan_buckets(plan):
    """(buckets, segments): lists of (lo, hi, seg_first, seg_count) and of
    (lo, hi, rank, bucket)."""
    info = zero_plan_get_info(plan)
    bk = (ZeroBucket * max(info.n_buckets, 1))()
    sg = (ZeroSegment * max(info.n_segments, 1))()
    _check("zero_plan_buckets", lib().zero_plan_buckets(plan, bk, sg))
    return ([(b.lo, b.hi, b.seg_first, b.seg_count) for b in bk[:info.n_buckets]],
            [(s.lo, s.hi, s.rank, s.bucket) for s in sg[:info.n_segments]])


def zero_plan_bucket_range(plan, bucket):
    lo, hi = C.c_int64(), C.c_int64()
    _check("zero_plan_bucket_range", lib().zero_plan_bucket_range(plan, bucket, C.byref(lo),
                                                                  C.byref(hi)))
    return lo.value, hi.value


def zero_workspace_bytes(plan, two_pass=1):
    return int(lib().zero_workspace_bytes(plan, int(bool(two_pass))))


def zero_scaler_init(hp):
    out = ZeroScaler()
    _check("zero_scaler_init", lib().zero_scaler_init(C.byref(hp), C.byref(out)))
    return out


# ------------------------------------------------------------------ step ----

def _rank_arrays(plan, n_sets=1, **lists):
    """C arrays of the per-rank pointer lists of one call: replicas, accum,
    micro and grad_shards hold N entries, optimizer arrays n_sets * N."""
    n = _ranks(plan)
    per_set = {"master", "exp_avg", "exp_avg_sq"}
    return {k: _ptrs(v, (n_sets * n) if k in per_set else n, k) for k, v in lists.items()}


def zero_reduce_scatter(plan, bucket, rank_lo, rank_hi, replicas, window_base, grad_shards,
                        d_scaler, d_bucket_flags=0, d_workspace=0, stream=0):
    q = _rank_arrays(plan, replicas=replicas, grad_shards=grad_shards)
    _check("zero_reduce_scatter", lib().zero_reduce_scatter(
        plan, bucket, rank_lo, rank_hi, q["replicas"], window_base, q["grad_shards"],
        _vp(d_scaler), _vp(d_bucket_flags), _vp(d_workspace), _vp(stream)))


def zero_grad_norm(plan, rank_lo, rank_hi, grad_shards, hp, d_scaler, d_workspace, stream=0):
    q = _rank_arrays(plan, grad_shards=grad_shards)
    _check("zero_grad_norm", lib().zero_grad_norm(
        plan, rank_lo, rank_hi, q["grad_shards"], C.byref(hp), _vp(d_scaler),
        _vp(d_workspace), _vp(stream)))


def zero_grad_norm_local(plan, rank_lo, rank_hi, grad_shards, hp, d_scaler, d_workspace,
                         d_exchange, stream=0):
    q = _rank_arrays(plan, grad_shards=grad_shards)
    _check("zero_grad_norm_local", lib().zero_grad_norm_local(
        plan, rank_lo, rank_hi, q["grad_shards"], C.byref(hp), _vp(d_scaler), _vp(d_workspace),
        _vp(d_exchange), _vp(stream)))


def zero_grad_norm_apply(plan, d_exchange, hp, d_scaler, stream=0):
    _check("zero_grad_norm_apply", lib().zero_grad_norm_apply(
        plan, _vp(d_exchange), C.byref(hp), _vp(d_scaler), _vp(stream)))


def zero_ring_hop(plan, rank, hop, grad, recv, out, d_scaler, d_bucket_flags=0, stream=0):
    _check("zero_ring_hop", lib().zero_ring_hop(
        plan, rank, hop, _vp(grad), _vp(recv), _vp(out), _vp(d_scaler), _vp(d_bucket_flags),
        _vp(stream)))


def zero_step(plan, rank_lo, rank_hi, master, exp_avg, exp_avg_sq, n_sets, grad_shards,
              replicas, window_base, flat_params, hp, d_scaler, d_bucket_flags=0, stream=0):
    q = _rank_arrays(plan, n_sets, master=master, exp_avg=exp_avg, exp_avg_sq=exp_avg_sq,
                     grad_shards=grad_shards, replicas=replicas)
    _check("zero_step", lib().zero_step(
        plan, rank_lo, rank_hi, q["master"], q["exp_avg"], q["exp_avg_sq"], n_sets,
        q["grad_shards"], q["replicas"], window_base, _vp(flat_params), C.byref(hp),
        _vp(d_scaler), _vp(d_bucket_flags), _vp(stream)))


def zero_step_update(plan, rank_lo, rank_hi, master, exp_avg, exp_avg_sq, n_sets, grad_shards,
                     replicas, window_base, flat_params, hp, d_scaler, d_bucket_flags=0,
                     stream=0):
    q = _rank_arrays(plan, n_sets, master=master, exp_avg=exp_avg, exp_avg_sq=exp_avg_sq,
                     grad_shards=grad_shards, replicas=replicas)
    _check("zero_step_update", lib().zero_step_update(
        plan, rank_lo, rank_hi, q["master"], q["exp_avg"], q["exp_avg_sq"], n_sets,
        q["grad_shards"], q["replicas"], window_base, _vp(flat_params), C.byref(hp),
        _vp(d_scaler), _vp(d_bucket_flags), _vp(stream)))


def zero_step_finish(plan, rank_lo, rank_hi, master, n_sets, grad_shards, window_base,
                     flat_params, hp, d_scaler, stream=0):
    q = _rank_arrays(plan, n_sets, master=master, grad_shards=grad_shards)
    _check("zero_step_finish", lib().zero_step_finish(
        plan, rank_lo, rank_hi, q["master"], n_sets, q["grad_shards"], window_base,
        _vp(flat_params), C.byref(hp), _vp(d_scaler), _vp(stream)))


def zero_cast_params(plan, rank_lo, rank_hi, master, flat_params, window_base, stream=0):
    q = _rank_arrays(plan, 1, master=master)
    _check("zero_cast_params", lib().zero_cast_params(
        plan, rank_lo, rank_hi, q["master"], _vp(flat_params), window_base, _vp(stream)))


def zero_accumulate(plan, rank_lo, rank_hi, micro, accum, window_base, first, stream=0):
    q = _rank_arrays(plan, micro=micro, accum=accum)
    _check("zero_accumulate", lib().zero_accumulate(
        plan, rank_lo, rank_hi, q["micro"], q["accum"], window_base, int(bool(first)),
        _vp(stream)))


def zero_reduce_scatter_accum(plan, bucket, rank_lo, rank_hi, replicas, accum, n_micro,
                              window_base, grad_shards, d_scaler, d_bucket_flags=0,
                              d_workspace=0, stream=0):
    q = _rank_arrays(plan, replicas=replicas, accum=accum, grad_shards=grad_shards)
    _check("zero_reduce_scatter_accum", lib().zero_reduce_scatter_accum(
        plan, bucket, rank_lo, rank_hi, q["replicas"], q["accum"], n_micro, window_base,
        q["grad_shards"], _vp(d_scaler), _vp(d_bucket_flags), _vp(d_workspace), _vp(stream)))


def zero_step_accum(plan, rank_lo, rank_hi, master, exp_avg, exp_avg_sq, n_sets, grad_shards,
                    replicas, accum, n_micro, window_base, flat_params, hp, d_scaler,
                    d_bucket_flags=0, stream=0):
    q = _rank_arrays(plan, n_sets, master=master, exp_avg=exp_avg, exp_avg_sq=exp_avg_sq,
                     grad_shards=grad_shards, replicas=replicas, accum=accum)
    _check("zero_step_accum", lib().zero_step_accum(
        plan, rank_lo, rank_hi, q["master"], q["exp_avg"], q["exp_avg_sq"], n_sets,
        q["grad_shards"], q["replicas"], q["accum"], n_micro, window_base, _vp(flat_params),
        C.byref(hp), _vp(d_scaler), _vp(d_bucket_flags), _vp(stream)))


def zero_step_update_accum(plan, rank_lo, rank_hi, master, exp_avg, exp_avg_sq, n_sets,
                           grad_shards, replicas, accum, n_micro, window_base, flat_params, hp,
                           d_scaler, d_bucket_flags=0, stream=0):
    q = _rank_arrays(plan, n_sets, master=master, exp_avg=exp_avg, exp_avg_sq=exp_avg_sq,
                     grad_shards=grad_shards, replicas=replicas, accum=accum)
    _check("zero_step_update_accum", lib().zero_step_update_accum(
        plan, rank_lo, rank_hi, q["master"], q["exp_avg"], q["exp_avg_sq"], n_sets,
        q["grad_shards"], q["replicas"], q["accum"], n_micro, window_base, _vp(flat_params),
        C.byref(hp), _vp(d_scaler), _vp(d_bucket_flags), _vp(stream)))


def zero_grad_norm_noalloc(plan, rank_lo, rank_hi, grad_shards, hp, d_scaler, stream=0):
    """zero_grad_norm without a workspace: for callers that cannot allocate
    device memory (see include/zero.h)."""
    q = _rank_arrays(plan, grad_shards=grad_shards)
    _check("zero_grad_norm_noalloc", lib().zero_grad_norm_noalloc(
        plan, rank_lo, rank_hi, q["grad_shards"], C.byref(hp), _vp(d_scaler), _vp(stream)))


def zero_selftest_wait_timeout(d_scaler, limit_ns, stream=0):
    _check("zero_selftest_wait_timeout", lib().zero_selftest_wait_timeout(
        _vp(d_scaler), int(limit_ns), _vp(stream)))


def zero_strerror(status):
    return lib().zero_strerror(status).decode()


def zero_version():
    return lib().zero_version()


# ------------------------------------------------------ stage-3 FSDP units ----

def zero_unit_plan_create(numels, unit_of_tensor, n_units, n_ranks, align_elems=1):
    if len(numels) != len(unit_of_tensor):
        raise ValueError("numels and unit_of_tensor differ in length")
    n = len(numels)
    arr = (C.c_int64 * max(n, 1))(*[int(x) for x in numels])
    uot = (C.c_int32 * max(n, 1))(*[int(x) for x in unit_of_tensor])
    out = _VP()
    _check("zero_unit_plan_create", lib().zero_unit_plan_create(
        arr, n, uot, n_units, n_ranks, align_elems, C.byref(out)))
    return out


def zero_unit_plan_destroy(plan):
    lib().zero_unit_plan_destroy(plan)


def zero_unit_plan_get_info(plan):
    info = ZeroUnitPlanInfo()
    _check("zero_unit_plan_get_info", lib().zero_unit_plan_get_info(plan, C.byref(info)))
    return info


def zero_unit_plan_units(plan):
    n = zero_unit_plan_get_info(plan).n_units
    out = (ZeroUnit * n)()
    _check("zero_unit_plan_units", lib().zero_unit_plan_units(plan, out, n))
    return list(out)


def zero_unit_plan_tensors(plan):
    """(slot_tensor, tensor_offset) as lists."""
    n = zero_unit_plan_get_info(plan).n_tensors
    slots = (C.c_int32 * n)()
    offs = (C.c_int64 * n)()
    _check("zero_unit_plan_tensors", lib().zero_unit_plan_tensors(plan, slots, offs, n))
    return list(slots), list(offs)


def zero_gather_units(plan, unit_lo, unit_hi, shards, unit_buffers, stream=0):
    N = _unit_ranks(plan)
    _check("zero_gather_units", lib().zero_gather_units(
        plan, unit_lo, unit_hi, _ptrs(shards, N, "shards"), _ptrs(unit_buffers, unit_hi - unit_lo,
        "unit_buffers"), _vp(stream)))


def zero_shard_units(plan, unit_lo, unit_hi, unit_buffers, shards, stream=0):
    N = _unit_ranks(plan)
    _check("zero_shard_units", lib().zero_shard_units(
        plan, unit_lo, unit_hi, _ptrs(unit_buffers, unit_hi - unit_lo, "unit_buffers"),
        _ptrs(shards, N, "shards"), _vp(stream)))


def zero_unit_plan_strategy_cost(plan, strategy, n_replicas=1):
    out = ZeroStrategyCost()
    _check("zero_unit_plan_strategy_cost", lib().zero_unit_plan_strategy_cost(
        plan, strategy, n_replicas, C.byref(out)))
    return out


# ------------------------------------------------------------ checked build --

def zero_checked_status(stream=0):
    """(violations, first) recorded by a checked build since the last call;
    first = site << 48 | low 48 bits of the index. Raises ZeroError (status
    ZERO_ESTATE) in the release build."""
    n, first = C.c_int64(), C.c_int64()
    _check("zero_checked_status", lib().zero_checked_status(C.byref(n), C.byref(first),
                                                            _vp(stream)))
    return n.value, first.value


def zero_selftest_check(stream=0):
    _check("zero_selftest_check", lib().zero_selftest_check(_vp(stream)))
