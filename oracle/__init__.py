"""CPU oracle for the ZeRO-1/2 mixed-precision AdamW step (ctypes binding).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite,
``__graft_entry__.smoke()`` and the cpu_baseline / reference leg of
``bench.py`` may import this package.  The product package
``zero_optimizer_step_rs_gb300`` never imports it and shares no source with
it; the seeded input generator ``zgen`` is the only module both sides use.

The arithmetic lives in ``zero_oracle.c`` (plain C11, one float operation at
a time, no FMA contraction); this file only builds it with gcc and marshals
numpy arrays.  See ``zero_oracle.h`` for the passages each function follows
and for the readings R1-R16 taken where the pages leave a step open.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.c")
_HDR = os.path.join(_HERE, "zero_oracle.h")
LIB_PATH = os.path.join(_HERE, "liboracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (idempotent)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= newest):
        return LIB_PATH
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class HParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float)]


class Scalars(ctypes.Structure):
    _fields_ = [("step_size", ctypes.c_float), ("bc2_sqrt", ctypes.c_float),
                ("decay", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("one_minus_beta1", ctypes.c_float),
                ("one_minus_beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("denom_rm", ctypes.c_float)]


def lib():
    """Load the oracle library.  ZERO_ORACLE_LIB names another build of the same
    source (the mutation tests use it to load an oracle with a planted
    mistake); by default the in-tree liboracle.so is built and loaded."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("ZERO_ORACLE_LIB")
            if not path:
                path = build()
            L = ctypes.CDLL(path)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            L.oracle_bf16_rne.argtypes = [ctypes.c_float]
            L.oracle_bf16_rne.restype = ctypes.c_uint16
            L.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_float.restype = ctypes.c_float
            L.oracle_make_scalars.argtypes = [ctypes.POINTER(HParams), i64, i32, i32,
                                              ctypes.POINTER(Scalars)]
            L.oracle_make_scalars.restype = None
            L.oracle_adamw_elem.argtypes = [ctypes.POINTER(Scalars), ctypes.c_float,
                                            ctypes.POINTER(ctypes.c_float),
                                            ctypes.POINTER(ctypes.c_float),
                                            ctypes.POINTER(ctypes.c_float)]
            L.oracle_adamw_elem.restype = None
            L.oracle_avg_grad.argtypes = [vp, i32, i32, i64, ctypes.c_float]
            L.oracle_avg_grad.restype = ctypes.c_float
            L.oracle_dp_step.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp,
                                         ctypes.POINTER(HParams), i64]
            L.oracle_dp_step.restype = ctypes.c_int
            L.oracle_dp_step_mt.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp,
                                            ctypes.POINTER(HParams), i64, i32]
            L.oracle_dp_step_mt.restype = ctypes.c_int
            L.oracle_shard_len.argtypes = [i64, i32, i32]
            L.oracle_shard_len.restype = i64
            L.oracle_zero_step.argtypes = [i64, i32, i32, i64, vp, vp, vp, vp, vp,
                                           ctypes.POINTER(HParams), i64]
            L.oracle_zero_step.restype = ctypes.c_int
            L.oracle_reduce_scatter_sum.argtypes = [i64, i32, i64, vp, vp]
            L.oracle_reduce_scatter_sum.restype = ctypes.c_int
            L.oracle_ring_allreduce.argtypes = [vp, i32, i64, vp]
            L.oracle_ring_allreduce.restype = ctypes.c_int
            L.oracle_zero_bytes.argtypes = [ctypes.c_double, i32, ctypes.c_double,
                                            ctypes.c_double, ctypes.c_double, vp]
            L.oracle_zero_bytes.restype = None
            L.oracle_grad_sumsq.argtypes = [vp, i64]
            L.oracle_grad_sumsq.restype = ctypes.c_double
            L.oracle_clip_coef.argtypes = [ctypes.c_double, ctypes.c_float,
                                           ctypes.POINTER(ctypes.c_int32)]
            L.oracle_clip_coef.restype = ctypes.c_float
            L.oracle_dp_step_clipped.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp,
                                                 ctypes.POINTER(HParams), i64, ctypes.c_float,
                                                 i32, ctypes.POINTER(ctypes.c_double),
                                                 ctypes.POINTER(ctypes.c_int32)]
            L.oracle_dp_step_clipped.restype = ctypes.c_int
            L.oracle_zero3_step.argtypes = [i64, i32, i32, i64, vp, vp, vp, vp, vp,
                                            ctypes.POINTER(HParams), i64, vp]
            L.oracle_zero3_step.restype = ctypes.c_int
            L.oracle_zero3_gather.argtypes = [i64, i32, i64, vp, i64, i64, i32, vp,
                                              ctypes.POINTER(ctypes.c_int64)]
            L.oracle_zero3_gather.restype = ctypes.c_int
            L.oracle_fp16_rne.argtypes = [ctypes.c_float]
            L.oracle_fp16_rne.restype = ctypes.c_uint16
            L.oracle_fp16_to_float.argtypes = [ctypes.c_uint16]
            L.oracle_fp16_to_float.restype = ctypes.c_float
            L.oracle_compress.argtypes = [i32, vp, i64, vp]
            L.oracle_compress.restype = None
            L.oracle_dp_step_compressed.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp,
                                                    ctypes.POINTER(HParams), i64, i32, vp]
            L.oracle_dp_step_compressed.restype = ctypes.c_int
            L.oracle_onebit_step.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, vp,
                                             ctypes.POINTER(HParams), i64, i64, vp, vp]
            L.oracle_onebit_step.restype = ctypes.c_int
            L.oracle_zero3_rs_unit.argtypes = [i64, i32, i32, i64, vp, i64, i64, vp, vp]
            L.oracle_zero3_rs_unit.restype = ctypes.c_int
            L.oracle_zero3_update.argtypes = [i64, i32, i32, i64, vp, vp, vp, vp, vp,
                                              ctypes.POINTER(HParams), i64]
            L.oracle_zero3_update.restype = ctypes.c_int
            _lib = L
    return _lib


# ----------------------------------------------------------------- helpers --

def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _ptr_array(arrs) -> ctypes.Array:
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def _check(a: np.ndarray, dtype, n=None, name="array"):
    if a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError(f"{name}: need a contiguous {np.dtype(dtype)} array")
    if n is not None and a.size < n:
        raise ValueError(f"{name}: need at least {n} elements, got {a.size}")


def hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1) -> HParams:
    return HParams(lr, beta1, beta2, eps, weight_decay)


def bf16_rne(x: float) -> int:
    return int(lib().oracle_bf16_rne(ctypes.c_float(x)))


def bf16_to_float(h: int) -> float:
    return float(lib().oracle_bf16_to_float(ctypes.c_uint16(h)))


def make_scalars(hp: HParams, step: int, R: int = 1, M: int = 1) -> Scalars:
    s = Scalars()
    lib().oracle_make_scalars(ctypes.byref(hp), step, R, M, ctypes.byref(s))
    return s


def adamw_elem(s: Scalars, g: float, w: float, m: float, v: float):
    cw, cm, cv = ctypes.c_float(w), ctypes.c_float(m), ctypes.c_float(v)
    lib().oracle_adamw_elem(ctypes.byref(s), ctypes.c_float(g), ctypes.byref(cw),
                            ctypes.byref(cm), ctypes.byref(cv))
    return cw.value, cm.value, cv.value


def shard_len(n: int, R: int, align: int = 64) -> int:
    return int(lib().oracle_shard_len(n, R, align))


def dp_step(G, W, m, v, P, hp: HParams, step: int, R: int, M: int,
            nthreads: int = 1) -> None:
    """Unsharded DP + AdamW, in place.  G: list of R*M uint16 (bf16 bit) arrays,
    W/m/v: float32 arrays of n, P: list of R uint16 arrays of n."""
    n = W.size
    if len(G) != R * M or len(P) != R:
        raise ValueError("need R*M gradient buffers and R replicas")
    for k, g in enumerate(G):
        _check(g, np.uint16, n, f"G[{k}]")
    for k, p in enumerate(P):
        _check(p, np.uint16, n, f"P[{k}]")
    for nm, a in (("W", W), ("m", m), ("v", v)):
        _check(a, np.float32, n, nm)
    ga, pa = _ptr_array(G), _ptr_array(P)
    if nthreads > 1:
        rc = lib().oracle_dp_step_mt(n, R, M, ctypes.addressof(ga), _ptr(W), _ptr(m),
                                     _ptr(v), ctypes.addressof(pa), ctypes.byref(hp),
                                     step, nthreads)
    else:
        rc = lib().oracle_dp_step(n, R, M, ctypes.addressof(ga), _ptr(W), _ptr(m),
                                  _ptr(v), ctypes.addressof(pa), ctypes.byref(hp), step)
    if rc != 0:
        raise RuntimeError(f"oracle_dp_step failed: {rc}")


def zero_step(G, W, m, v, P, hp: HParams, step: int, R: int, M: int, n: int,
              S: int) -> None:
    """ZeRO-1/2 step emulated card by card.  W/m/v hold R*S floats (shard r at
    r*S); G holds R*M uint16 arrays of n; P holds R uint16 arrays of n."""
    if len(G) != R * M or len(P) != R:
        raise ValueError("need R*M gradient buffers and R replicas")
    for k, g in enumerate(G):
        _check(g, np.uint16, n, f"G[{k}]")
    for k, p in enumerate(P):
        _check(p, np.uint16, n, f"P[{k}]")
    for nm, a in (("W", W), ("m", m), ("v", v)):
        _check(a, np.float32, R * S, nm)
    ga, pa = _ptr_array(G), _ptr_array(P)
    rc = lib().oracle_zero_step(n, R, M, S, ctypes.addressof(ga), _ptr(W), _ptr(m),
                                _ptr(v), ctypes.addressof(pa), ctypes.byref(hp), step)
    if rc != 0:
        raise RuntimeError(f"oracle_zero_step failed: {rc}")


def reduce_scatter_sum(inputs, S: int):
    """inputs: list of R float32 arrays of n.  Returns R float32 arrays of the
    shard lengths (rank r's chunk of the element-wise sum)."""
    R, n = len(inputs), inputs[0].size
    for k, a in enumerate(inputs):
        _check(a, np.float32, n, f"in[{k}]")
    outs = [np.zeros(S, np.float32) for _ in range(R)]
    ia, oa = _ptr_array(inputs), _ptr_array(outs)
    rc = lib().oracle_reduce_scatter_sum(n, R, S, ctypes.addressof(ia), ctypes.addressof(oa))
    if rc != 0:
        raise RuntimeError(f"oracle_reduce_scatter_sum failed: {rc}")
    return [o[:max(0, min(S, n - r * S))] for r, o in enumerate(outs)]


def ring_allreduce(cards):
    """Ring all-reduce of p float32 arrays in place; returns numbers sent per
    card (int64 array)."""
    p, n = len(cards), cards[0].size
    for k, a in enumerate(cards):
        _check(a, np.float32, n, f"card[{k}]")
    sent = np.zeros(p, np.int64)
    ca = _ptr_array(cards)
    rc = lib().oracle_ring_allreduce(ctypes.addressof(ca), p, n, _ptr(sent))
    if rc != 0:
        raise RuntimeError(f"oracle_ring_allreduce failed: {rc}")
    return sent


def zero_bytes(N: float, P: int, bp: float, bg: float, bo: float):
    out = np.zeros(4, np.float64)
    lib().oracle_zero_bytes(float(N), P, float(bp), float(bg), float(bo), _ptr(out))
    return out


def grad_sumsq(g: np.ndarray) -> float:
    """Pairwise sum of squares of a float32 vector: fp32 leaves g*g and fp32
    nodes over the leaves padded with zeros to a power of two, returned
    widened to double (reading R10)."""
    _check(g, np.float32, None, "g")
    return float(lib().oracle_grad_sumsq(_ptr(g), g.size))


def clip_coef(sumsq: float, max_norm: float):
    clip = ctypes.c_int32(0)
    c = lib().oracle_clip_coef(sumsq, max_norm, ctypes.byref(clip))
    return float(c), bool(clip.value)


def dp_step_clipped(G, W, m, v, P, hp: HParams, step: int, R: int, M: int,
                    max_norm: float, skip_nonfinite: bool = False):
    """DP step with global-norm clipping, in place; returns (sumsq, skipped)."""
    n = W.size
    if len(G) != R * M or len(P) != R:
        raise ValueError("need R*M gradient buffers and R replicas")
    for k, g in enumerate(G):
        _check(g, np.uint16, n, f"G[{k}]")
    for k, p in enumerate(P):
        _check(p, np.uint16, n, f"P[{k}]")
    for nm, a in (("W", W), ("m", m), ("v", v)):
        _check(a, np.float32, n, nm)
    ga, pa = _ptr_array(G), _ptr_array(P)
    ss = ctypes.c_double(0.0)
    sk = ctypes.c_int32(0)
    rc = lib().oracle_dp_step_clipped(n, R, M, ctypes.addressof(ga), _ptr(W), _ptr(m), _ptr(v),
                                      ctypes.addressof(pa), ctypes.byref(hp), step, max_norm,
                                      int(skip_nonfinite), ctypes.byref(ss), ctypes.byref(sk))
    if rc != 0:
        raise RuntimeError(f"oracle_dp_step_clipped failed: {rc}")
    return ss.value, bool(sk.value)


def zero3_step(G, W, m, v, Pshard, hp: HParams, step: int, R: int, M: int, n: int, S: int):
    """ZeRO-3 step card by card, in place; returns the per-card count of
    gradient numbers received from other cards."""
    for k, g in enumerate(G):
        _check(g, np.uint16, n, f"G[{k}]")
    for nm, a in (("W", W), ("m", m), ("v", v)):
        _check(a, np.float32, R * S, nm)
    _check(Pshard, np.uint16, R * S, "Pshard")
    ga = _ptr_array(G)
    recv = np.zeros(R, np.int64)
    rc = lib().oracle_zero3_step(n, R, M, S, ctypes.addressof(ga), _ptr(W), _ptr(m), _ptr(v),
                                 _ptr(Pshard), ctypes.byref(hp), step, _ptr(recv))
    if rc != 0:
        raise RuntimeError(f"oracle_zero3_step failed: {rc}")
    return recv


def zero3_gather(Pshard, n: int, R: int, S: int, lo: int, hi: int, card: int = 0):
    """All-gather of unit [lo, hi) for `card`; returns (values, numbers
    received from other cards)."""
    _check(Pshard, np.uint16, R * S, "Pshard")
    out = np.zeros(max(1, hi - lo), np.uint16)
    recv = ctypes.c_int64(0)
    rc = lib().oracle_zero3_gather(n, R, S, _ptr(Pshard), lo, hi, card, _ptr(out),
                                   ctypes.byref(recv))
    if rc != 0:
        raise RuntimeError(f"oracle_zero3_gather failed: {rc}")
    return out[:hi - lo], recv.value


COMP_NONE, COMP_FP16, COMP_INT8, COMP_SIGN = 0, 1, 2, 3


def fp16_rne(x: float) -> int:
    return int(lib().oracle_fp16_rne(ctypes.c_float(x)))


def fp16_to_float(h: int) -> float:
    return float(lib().oracle_fp16_to_float(ctypes.c_uint16(h)))


def compress(kind: int, x: np.ndarray) -> np.ndarray:
    _check(x, np.float32, None, "x")
    d = np.empty(max(1, x.size), np.float32)
    lib().oracle_compress(kind, _ptr(x), x.size, _ptr(d))
    return d[:x.size]


def dp_step_compressed(G, W, m, v, P, hp: HParams, step: int, R: int, M: int, kind: int,
                       E=None) -> None:
    n = W.size
    for k, g in enumerate(G):
        _check(g, np.uint16, n, f"G[{k}]")
    for k, p in enumerate(P):
        _check(p, np.uint16, n, f"P[{k}]")
    for nm, a in (("W", W), ("m", m), ("v", v)):
        _check(a, np.float32, n, nm)
    ga, pa = _ptr_array(G), _ptr_array(P)
    ea = None
    if E is not None:
        for k, e in enumerate(E):
            _check(e, np.float32, n, f"E[{k}]")
        ea = _ptr_array(E)
    rc = lib().oracle_dp_step_compressed(n, R, M, ctypes.addressof(ga), _ptr(W), _ptr(m), _ptr(v),
                                         ctypes.addressof(pa), ctypes.byref(hp), step, kind,
                                         ctypes.addressof(ea) if ea is not None else None)
    if rc != 0:
        raise RuntimeError(f"oracle_dp_step_compressed failed: {rc}")


def onebit_step(G, W, m, v, P, hp: HParams, step: int, freeze_step: int, R: int, M: int,
                S: int, E, Es) -> None:
    """1-bit Adam step (reading R15) on numpy arrays of n elements each;
    E (R arrays) and Es are updated in place after the warm-up."""
    n = W.size
    for k, g in enumerate(G):
        _check(g, np.uint16, n, f"G[{k}]")
    for k, p in enumerate(P):
        _check(p, np.uint16, n, f"P[{k}]")
    for nm, a in (("W", W), ("m", m), ("v", v), ("Es", Es)):
        _check(a, np.float32, n, nm)
    for k, e in enumerate(E):
        _check(e, np.float32, n, f"E[{k}]")
    ga, pa, ea = _ptr_array(G), _ptr_array(P), _ptr_array(E)
    rc = lib().oracle_onebit_step(n, S, R, M, ctypes.addressof(ga), _ptr(W), _ptr(m), _ptr(v),
                                  ctypes.addressof(pa), ctypes.byref(hp), step, freeze_step,
                                  ctypes.addressof(ea), _ptr(Es))
    if rc != 0:
        raise RuntimeError(f"oracle_onebit_step failed: {rc}")


def zero3_rs_unit(Gu, n: int, R: int, M: int, S: int, lo: int, hi: int, gshard: np.ndarray):
    """Reduce-scatter of the unit [lo, hi) (reading R16) into gshard (n or
    more floats, element i at index i); returns the per-card receive counts."""
    for k, g in enumerate(Gu):
        _check(g, np.uint16, hi - lo, f"Gu[{k}]")
    _check(gshard, np.float32, None, "gshard")
    if gshard.size < n:
        raise ValueError("gshard too small")
    ga = _ptr_array(Gu) if Gu else None
    recv = np.zeros(R, np.int64)
    rc = lib().oracle_zero3_rs_unit(n, R, M, S, ctypes.addressof(ga) if ga is not None else None,
                                    lo, hi, _ptr(gshard), _ptr(recv))
    if rc != 0:
        raise RuntimeError(f"oracle_zero3_rs_unit failed: {rc}")
    return recv


def zero3_update(gshard, W, m, v, Pshard, hp: HParams, step: int, n: int, R: int, M: int,
                 S: int) -> None:
    """Shard update from reduce-scattered gradients (reading R16)."""
    for nm, a in (("gshard", gshard), ("W", W), ("m", m), ("v", v)):
        _check(a, np.float32, None, nm)
    _check(Pshard, np.uint16, None, "Pshard")
    rc = lib().oracle_zero3_update(n, R, M, S, _ptr(gshard), _ptr(W), _ptr(m), _ptr(v),
                                   _ptr(Pshard), ctypes.byref(hp), step)
    if rc != 0:
        raise RuntimeError(f"oracle_zero3_update failed: {rc}")
