"""Seeded synthetic inputs for the sharded AdamW step (harness only).

Thin ctypes binding of the generator in synth.h: a host build
(libzsynth_host.so, fp32 values) and a device build (libzsynth_gpu.so, writes
bf16/fp16 replicas and fp32 master weights straight into HBM). The generator
holds none of the step's arithmetic; see synth.h for its definition.
"""
import ctypes as C
import os

import numpy as np

from .. import _build

_host = None
_gpu = None


class GradSpec(C.Structure):
    """Mirror of zs_grad_spec."""
    _fields_ = [("seed", C.c_uint64), ("sigma", C.c_float), ("bias_sigma", C.c_float),
                ("loss_scale", C.c_float), ("outliers", C.c_int32), ("psi", C.c_int64)]


def grad_spec(seed=0, sigma=1e-3, bias_sigma=0.0, loss_scale=1.0, outliers=False, psi=0):
    return GradSpec(seed, sigma, bias_sigma, loss_scale, int(bool(outliers)), psi)


def _load(path):
    if not os.path.exists(path):
        raise RuntimeError("%s is not built; run __graft_entry__.build()" % path)
    return C.CDLL(path)


def host():
    global _host
    if _host is None:
        L = _load(_build.SYNTH_HOST_LIB)
        P = C.POINTER
        L.zs_host_u64.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint64]
        L.zs_host_u64.restype = C.c_uint64
        L.zs_host_mix64.argtypes = [C.c_uint64]
        L.zs_host_mix64.restype = C.c_uint64
        L.zs_host_normal.argtypes = [C.c_uint64]
        L.zs_host_normal.restype = C.c_float
        L.zs_host_fill_grad.argtypes = [C.c_void_p, C.c_int64, C.c_int64, P(GradSpec),
                                        C.c_uint32, C.c_uint32]
        L.zs_host_fill_master.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_uint64,
                                          C.c_int64]
        L.zs_host_grad_at.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, P(GradSpec),
                                      C.c_uint32, C.c_uint32]
        L.zs_host_master_at.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_uint64,
                                        C.c_int64]
        L.zs_host_spec_size.restype = C.c_int64
        assert L.zs_host_spec_size() == C.sizeof(GradSpec)
        _host = L
    return _host


def gpu():
    global _gpu
    if _gpu is None:
        L = _load(_build.SYNTH_GPU_LIB)
        L.zs_gpu_fill_grad.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.POINTER(GradSpec),
                                       C.c_uint32, C.c_uint32, C.c_int32, C.c_void_p]
        L.zs_gpu_fill_grad.restype = C.c_int
        L.zs_gpu_fill_master.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_uint64,
                                         C.c_int64, C.c_void_p]
        L.zs_gpu_fill_master.restype = C.c_int
        L.zs_gpu_spec_size.restype = C.c_int64
        assert L.zs_gpu_spec_size() == C.sizeof(GradSpec)
        _gpu = L
    return _gpu


# ------------------------------------------------------------------ host ----

def u64(seed, tag, step, rank, elem):
    return host().zs_host_u64(seed, tag, step, rank, elem)


def mix64(z):
    return host().zs_host_mix64(z)


def normal_from_hash(h):
    return np.float32(host().zs_host_normal(h))


def grad_f32(n, elem0, spec, step, rank):
    out = np.empty(n, dtype=np.float32)
    host().zs_host_fill_grad(out.ctypes.data, n, elem0, C.byref(spec), step, rank)
    return out


def grad_f32_at(elems, spec, step, rank):
    elems = np.ascontiguousarray(elems, dtype=np.int64)
    out = np.empty(len(elems), dtype=np.float32)
    host().zs_host_grad_at(out.ctypes.data, elems.ctypes.data, len(elems), C.byref(spec),
                           step, rank)
    return out


def master_f32(n, elem0, seed, psi):
    out = np.empty(n, dtype=np.float32)
    host().zs_host_fill_master(out.ctypes.data, n, elem0, seed, psi)
    return out


def master_f32_at(elems, seed, psi):
    elems = np.ascontiguousarray(elems, dtype=np.int64)
    out = np.empty(len(elems), dtype=np.float32)
    host().zs_host_master_at(out.ctypes.data, elems.ctypes.data, len(elems), seed, psi)
    return out


# ------------------------------------------------------------------- gpu ----

def gpu_fill_grad(ptr, n, elem0, spec, step, rank, is_bf16, stream=0):
    rc = gpu().zs_gpu_fill_grad(C.c_void_p(ptr), n, elem0, C.byref(spec), step, rank,
                                int(bool(is_bf16)), C.c_void_p(stream))
    if rc != 0:
        raise RuntimeError("zs_gpu_fill_grad: CUDA error %d" % rc)


def gpu_fill_master(ptr, n, elem0, seed, psi, stream=0):
    rc = gpu().zs_gpu_fill_master(C.c_void_p(ptr), n, elem0, seed, psi, C.c_void_p(stream))
    if rc != 0:
        raise RuntimeError("zs_gpu_fill_master: CUDA error %d" % rc)
