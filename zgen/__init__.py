"""Seeded synthetic inputs for the ZeRO AdamW step (host and device fills).

This module is shared by the CUDA path's tests/benchmark and by the oracle's
callers, and holds none of the optimizer step's arithmetic (see zgen.h for
the generator's definition).  The workload recipes - parameter-set shapes,
value distributions, seeds - live in ``zgen.workloads``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libzgen_host.so")
DEV_LIB = os.path.join(_HERE, "libzgen_dev.so")
_HOST_SRC = os.path.join(_HERE, "zgen_host.c")
_DEV_SRC = os.path.join(_HERE, "zgen_dev.cu")
_HDR = os.path.join(_HERE, "zgen.h")

IH_STD = 107019.57184877197          # must equal ZGEN_IH_STD in zgen.h
GAMMA = 0x9E3779B97F4A7C15

_lock = threading.Lock()
_host = None
_dev = None


def _stale(out, *srcs):
    return (not os.path.exists(out)
            or os.path.getmtime(out) < max(os.path.getmtime(s) for s in srcs))


def host_build_cmd():
    return ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
            "-Wall", "-o", HOST_LIB, _HOST_SRC]


def dev_build_cmd(nvcc="nvcc"):
    return [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
            "-Xcompiler", "-fPIC", "-shared", "-o", DEV_LIB, _DEV_SRC]


def build(device: bool = True) -> None:
    if _stale(HOST_LIB, _HOST_SRC, _HDR):
        subprocess.run(host_build_cmd(), check=True)
    if device and _stale(DEV_LIB, _DEV_SRC, _HDR):
        subprocess.run(dev_build_cmd(), check=True)


def host():
    global _host
    with _lock:
        if _host is None:
            if _stale(HOST_LIB, _HOST_SRC, _HDR):
                subprocess.run(host_build_cmd(), check=True)
            L = ctypes.CDLL(HOST_LIB)
            vp, i32, i64, u32, u64, f = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                         ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float)
            L.zgen_fill_grad_bf16.argtypes = [vp, i64, i64, u64, u64, f, f, u32]
            L.zgen_gather_grad_bf16.argtypes = [vp, vp, i64, u64, u64, f, f, u32]
            L.zgen_fill_state_f32.argtypes = [vp, i64, i64, u64, u64, f, i32]
            L.zgen_gather_state_f32.argtypes = [vp, vp, i64, u64, u64, f, i32]
            for fn in (L.zgen_fill_grad_bf16, L.zgen_gather_grad_bf16,
                       L.zgen_fill_state_f32, L.zgen_gather_state_f32):
                fn.restype = None
            L.zgen_draw_u64.argtypes = [u64, u64, i64]
            L.zgen_draw_u64.restype = u64
            _host = L
    return _host


def dev():
    """The device fill library (needs a CUDA device at call time)."""
    global _dev
    with _lock:
        if _dev is None:
            if not os.path.exists(DEV_LIB):
                raise RuntimeError(f"{DEV_LIB} is missing: run __graft_entry__.build()")
            L = ctypes.CDLL(DEV_LIB)
            vp, i32, i64, u32, u64, f = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                         ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float)
            L.zgen_dev_fill_grad_bf16.argtypes = [vp, i64, i64, u64, u64, f, f, u32, vp]
            L.zgen_dev_fill_state_f32.argtypes = [vp, i64, i64, u64, u64, f, i32, vp]
            L.zgen_dev_fill_const_f32.argtypes = [vp, i64, f, vp]
            for fn in (L.zgen_dev_fill_grad_bf16, L.zgen_dev_fill_state_f32,
                       L.zgen_dev_fill_const_f32):
                fn.restype = ctypes.c_int
            _dev = L
    return _dev


def scale_for(sigma: float) -> float:
    """The float multiplier that turns the Irwin-Hall integer into a value of
    standard deviation sigma (rounded once to float32)."""
    return float(np.float32(sigma / IH_STD))


# ----------------------------------------------------------- host fills --

def host_grad(seed, stream, lo, n, sigma, outlier=0.0, outlier_pct=0):
    out = np.empty(n, np.uint16)
    host().zgen_fill_grad_bf16(out.ctypes.data, lo, n, seed, stream, scale_for(sigma),
                               outlier, outlier_pct)
    return out


def host_grad_at(seed, stream, idx, sigma, outlier=0.0, outlier_pct=0):
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.uint16)
    host().zgen_gather_grad_bf16(out.ctypes.data, idx.ctypes.data, idx.size, seed, stream,
                                 scale_for(sigma), outlier, outlier_pct)
    return out


def host_state(seed, stream, lo, n, sigma, square=False):
    out = np.empty(n, np.float32)
    host().zgen_fill_state_f32(out.ctypes.data, lo, n, seed, stream, scale_for(sigma),
                               int(square))
    return out


def host_state_at(seed, stream, idx, sigma, square=False):
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.float32)
    host().zgen_gather_state_f32(out.ctypes.data, idx.ctypes.data, idx.size, seed, stream,
                                 scale_for(sigma), int(square))
    return out


def draw_u64(seed, stream, k):
    return int(host().zgen_draw_u64(seed, stream, k))


# --------------------------------------------------------- device fills --

def _chk(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with CUDA error {rc}")


def dev_grad(ptr, seed, stream, lo, n, sigma, outlier=0.0, outlier_pct=0, cuda_stream=0):
    _chk(dev().zgen_dev_fill_grad_bf16(ptr, lo, n, seed, stream, scale_for(sigma), outlier,
                                       outlier_pct, cuda_stream), "zgen_dev_fill_grad_bf16")


def dev_state(ptr, seed, stream, lo, n, sigma, square=False, cuda_stream=0):
    _chk(dev().zgen_dev_fill_state_f32(ptr, lo, n, seed, stream, scale_for(sigma),
                                       int(square), cuda_stream), "zgen_dev_fill_state_f32")


def dev_const(ptr, n, value, cuda_stream=0):
    _chk(dev().zgen_dev_fill_const_f32(ptr, n, value, cuda_stream), "zgen_dev_fill_const_f32")
