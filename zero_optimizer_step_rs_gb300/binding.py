"""Thin ctypes binding of libzero_step.so (include/zero_step.h).

Argument marshalling only: tensors become device pointers, the current
torch stream becomes the cudaStream_t, and status codes become exceptions.
Every step of the optimizer runs in the library's CUDA kernels; there is no
fallback.  If the library has not been built the import of the functions
fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libzero_step.so")

ZERO_OK = 0
ZERO_ERR_INVALID_ARG = -1
ZERO_ERR_NULL = -2
ZERO_ERR_ALIGN = -3
ZERO_ERR_SIZE = -4
ZERO_ERR_OVERLAP = -5
ZERO_ERR_CUDA = -6
ZERO_ERR_DEVICE_TIMEOUT = -7
ZERO_ERR_NONFINITE = -8
ZERO_ERR_IO = -9
ZERO_ERR_CORRUPT = -10
ZERO_DEV_NONFINITE = 1
ZERO_DEV_SKIPPED = 4
ZERO_FLAG_CHECK_FINITE = 1
ZERO_FLAG_SKIP_NONFINITE = 2
ZERO_VARIANT_FUSED = 0
ZERO_VARIANT_STAGED = 1
ZERO_VARIANT_FUSED_TMA = 2
ZERO_DEV_TIMEOUT = 2
ZERO_DEV_DRAIN_FAILED = 8
ZERO_FLAG_DEBUG_EXPIRE_WAITS = 1 << 30
ZERO_COMP_FP16 = 1
ZERO_COMP_INT8 = 2
ZERO_COMP_SIGN = 3
ZERO_MAX_R = 64
ZERO_MAX_RM = 256
ZERO_NOALLOC_MAX_ELEMS = 4 * 1024 * 1024
ZERO_MAX_GATHER_UNITS = 1024

EXPORTED = ("zero_abi_version", "zero_status_string", "zero_plan_create", "zero_plan_destroy",
            "zero_plan_owner", "zero_step", "zero_rs_avg", "zero_adamw_shard", "zero_ag_cast",
            "zero_step_host", "zero_step_staged_noalloc", "zero_step_clipped",
            "zero_clip_scratch_bytes", "zero3_step", "zero3_gather", "zero_ckpt_write_host",
            "zero_ckpt_read_host", "zero_ckpt_save_async", "zero_ckpt_job_wait",
            "zero_ckpt_load", "zero_step_compressed", "zero_check_replicas", "zero_step_onebit",
            "zero3_rs_unit", "zero3_update", "zero_get_device_status",
            "zero3_gather_units")


class ZeroError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {zero_status_string(code)} ({code})")


class zero_plan_t(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("S", ctypes.c_int64), ("padded", ctypes.c_int64),
                ("R", ctypes.c_int32), ("M", ctypes.c_int32), ("stage", ctypes.c_int32),
                ("align_elems", ctypes.c_int32), ("n_tensors", ctypes.c_int32),
                ("tensor_offsets", ctypes.POINTER(ctypes.c_int64)),
                ("bytes_per_rank_dp", ctypes.c_int64), ("bytes_per_rank_z1", ctypes.c_int64),
                ("bytes_per_rank_z2", ctypes.c_int64), ("bytes_per_rank_z3", ctypes.c_int64),
                ("bytes_per_rank", ctypes.c_int64), ("scratch_bytes_staged", ctypes.c_int64)]


class zero_gather_unit(ctypes.Structure):
    _fields_ = [("lo", ctypes.c_int64), ("hi", ctypes.c_int64), ("out", ctypes.c_void_p)]


class zero_adamw_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "zero_optimizer_step_rs_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        P = ctypes.POINTER
        L.zero_abi_version.argtypes = []
        L.zero_abi_version.restype = i32
        L.zero_status_string.argtypes = [ctypes.c_int]
        L.zero_status_string.restype = ctypes.c_char_p
        L.zero_plan_create.argtypes = [vp, i32, i32, i32, i32, i32, P(P(zero_plan_t))]
        L.zero_plan_create.restype = ctypes.c_int
        L.zero_plan_destroy.argtypes = [P(zero_plan_t)]
        L.zero_plan_destroy.restype = None
        L.zero_plan_owner.argtypes = [P(zero_plan_t), i64]
        L.zero_plan_owner.restype = i32
        L.zero_step.argtypes = [P(zero_plan_t), vp, vp, vp, vp, vp, P(zero_adamw_hparams), i64,
                                i32, vp, i64, i32, vp, vp]
        L.zero_step.restype = ctypes.c_int
        L.zero_rs_avg.argtypes = [P(zero_plan_t), vp, vp, i32, vp, vp]
        L.zero_rs_avg.restype = ctypes.c_int
        L.zero_adamw_shard.argtypes = [P(zero_plan_t), vp, vp, vp, vp, P(zero_adamw_hparams),
                                       i64, vp]
        L.zero_adamw_shard.restype = ctypes.c_int
        L.zero_ag_cast.argtypes = [P(zero_plan_t), vp, vp, vp]
        L.zero_ag_cast.restype = ctypes.c_int
        L.zero_step_host.argtypes = [P(zero_plan_t), vp, vp, vp, vp, vp, vp, vp,
                                     P(zero_adamw_hparams), i64, i32, vp, vp]
        L.zero_step_host.restype = ctypes.c_int
        L.zero_step_staged_noalloc.argtypes = [P(zero_plan_t), vp, vp, vp, vp, vp,
                                               P(zero_adamw_hparams), i64, i32, vp, vp]
        L.zero_step_staged_noalloc.restype = ctypes.c_int
        L.zero_step_clipped.argtypes = [P(zero_plan_t), vp, vp, vp, vp, vp, P(zero_adamw_hparams),
                                        i64, ctypes.c_float, vp, i64, i32, vp, vp, vp]
        L.zero_step_clipped.restype = ctypes.c_int
        L.zero_clip_scratch_bytes.argtypes = [P(zero_plan_t)]
        L.zero_clip_scratch_bytes.restype = i64
        L.zero3_step.argtypes = [P(zero_plan_t), vp, vp, vp, vp, vp, P(zero_adamw_hparams), i64,
                                 i32, vp, vp]
        L.zero3_step.restype = ctypes.c_int
        L.zero3_gather.argtypes = [P(zero_plan_t), vp, i64, i64, vp, i32, vp]
        L.zero3_gather.restype = ctypes.c_int
        L.zero_ckpt_write_host.argtypes = [P(zero_plan_t), vp, vp, vp, vp, i64,
                                           P(zero_adamw_hparams), ctypes.c_char_p, i32]
        L.zero_ckpt_write_host.restype = ctypes.c_int
        L.zero_ckpt_read_host.argtypes = [P(zero_plan_t), ctypes.c_char_p, i32, vp, vp, vp, vp,
                                          P(i64), P(zero_adamw_hparams)]
        L.zero_ckpt_read_host.restype = ctypes.c_int
        L.zero_ckpt_save_async.argtypes = [P(zero_plan_t), vp, vp, vp, vp, i64,
                                           P(zero_adamw_hparams), ctypes.c_char_p, i32, vp,
                                           P(vp)]
        L.zero_ckpt_save_async.restype = ctypes.c_int
        L.zero_ckpt_job_wait.argtypes = [vp]
        L.zero_ckpt_job_wait.restype = ctypes.c_int
        L.zero_ckpt_load.argtypes = [P(zero_plan_t), ctypes.c_char_p, vp, i32, vp, vp, vp, P(i64),
                                     P(zero_adamw_hparams), vp]
        L.zero_ckpt_load.restype = ctypes.c_int
        L.zero_step_compressed.argtypes = [P(zero_plan_t), vp, vp, vp, vp, vp,
                                           P(zero_adamw_hparams), i64, i32, vp, vp]
        L.zero_step_compressed.restype = ctypes.c_int
        L.zero_check_replicas.argtypes = [P(zero_plan_t), vp, vp, vp, vp]
        L.zero_check_replicas.restype = ctypes.c_int
        L.zero_step_onebit.argtypes = [P(zero_plan_t), vp, vp, vp, vp, vp,
                                       P(zero_adamw_hparams), i64, i64, vp, vp, vp]
        L.zero_step_onebit.restype = ctypes.c_int
        L.zero3_rs_unit.argtypes = [P(zero_plan_t), vp, i64, i64, vp, i32, vp, vp]
        L.zero3_rs_unit.restype = ctypes.c_int
        L.zero3_update.argtypes = [P(zero_plan_t), vp, vp, vp, vp, vp, P(zero_adamw_hparams), i64,
                                   vp]
        L.zero3_update.restype = ctypes.c_int
        L.zero_get_device_status.argtypes = [vp, vp, P(i32)]
        L.zero_get_device_status.restype = ctypes.c_int
        L.zero3_gather_units.argtypes = [P(zero_plan_t), vp, P(zero_gather_unit), i32, vp]
        L.zero3_gather_units.restype = ctypes.c_int
        _lib = L
    return _lib


def zero_abi_version() -> int:
    return int(lib().zero_abi_version())


def zero_status_string(code: int) -> str:
    return lib().zero_status_string(code).decode()


def _check(code: int, where: str) -> None:
    if code != ZERO_OK:
        raise ZeroError(code, where)


# ------------------------------------------------------------------ plan --

class Plan:
    """Owning handle of a zero_plan_t (the shard layout)."""

    def __init__(self, tensor_numels: Sequence[int], R: int, M: int = 1, stage: int = 1,
                 align_elems: int = 0):
        arr = (ctypes.c_int64 * max(1, len(tensor_numels)))(*[int(n) for n in tensor_numels])
        out = ctypes.POINTER(zero_plan_t)()
        _check(lib().zero_plan_create(ctypes.addressof(arr), len(tensor_numels), R, M, stage,
                                      align_elems, ctypes.byref(out)), "zero_plan_create")
        self._p = out

    @property
    def ptr(self):
        return self._p

    @property
    def c(self) -> zero_plan_t:
        return self._p.contents

    def __getattr__(self, name):
        if name.startswith("_"):
            raise AttributeError(name)
        return getattr(self._p.contents, name)

    def tensor_offsets(self):
        c = self.c
        return [c.tensor_offsets[k] for k in range(c.n_tensors + 1)]

    def owner(self, i: int) -> int:
        return int(lib().zero_plan_owner(self._p, i))

    def close(self):
        if getattr(self, "_p", None):
            lib().zero_plan_destroy(self._p)
            self._p = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zero_plan_create(tensor_numels, R, M=1, stage=1, align_elems=0) -> Plan:
    return Plan(tensor_numels, R, M, stage, align_elems)


def zero_plan_destroy(plan: Plan) -> None:
    plan.close()


def zero_plan_owner(plan: Plan, i: int) -> int:
    return plan.owner(i)


def hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1) -> zero_adamw_hparams:
    return zero_adamw_hparams(lr, beta1, beta2, eps, weight_decay)


# ------------------------------------------------------------ marshalling --

def _ptrs(values) -> ctypes.Array:
    return (ctypes.c_void_p * max(1, len(values)))(*[int(v) if v else None for v in values])


def _addr(x) -> Optional[int]:
    """A device/host address from a torch tensor, an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_tensor(t, dtype_name, numel, where, device="cuda"):
    if isinstance(t, int) or t is None:
        return
    import torch
    want = {"bf16": torch.bfloat16, "f32": torch.float32, "i32": torch.int32}[dtype_name]
    if t.dtype != want:
        raise TypeError(f"{where}: expected {want}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{where}: tensor must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{where}: need {numel} elements, got {t.numel()}")
    if device == "cuda" and not t.is_cuda:
        raise ValueError(f"{where}: must be a CUDA tensor")
    if device == "cpu" and t.is_cuda:
        raise ValueError(f"{where}: must be a host tensor")


# -------------------------------------------------------------- the steps --

def zero_step(plan: Plan, rank_grads, master, m, v, rank_params, hp: zero_adamw_hparams,
              step: int, variant: int = ZERO_VARIANT_FUSED, scratch=None, flags: int = 0,
              dev_status=None, stream=None) -> None:
    c = plan.c
    for k, g in enumerate(rank_grads):
        _check_tensor(g, "bf16", c.N, f"rank_grads[{k}]")
    for k, p in enumerate(rank_params):
        _check_tensor(p, "bf16", c.N, f"rank_params[{k}]")
    for nm, t in (("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.padded, nm)
    _check_tensor(dev_status, "i32", 1, "dev_status")
    if len(rank_grads) != c.R * c.M or len(rank_params) != c.R:
        raise ValueError(f"need {c.R * c.M} gradient buffers and {c.R} replicas")
    sbytes = 0
    if scratch is not None and not isinstance(scratch, int):
        sbytes = scratch.numel() * scratch.element_size()
    elif isinstance(scratch, int):
        sbytes = c.scratch_bytes_staged
    ga, pa = _ptrs([_addr(g) for g in rank_grads]), _ptrs([_addr(p) for p in rank_params])
    _check(lib().zero_step(plan.ptr, ctypes.addressof(ga), _addr(master), _addr(m), _addr(v),
                           ctypes.addressof(pa), ctypes.byref(hp), step, variant,
                           _addr(scratch), sbytes, flags, _addr(dev_status), _stream(stream)),
           "zero_step")


def zero_get_device_status(dev_status, stream=None, raise_on_error: bool = False):
    """Wait for `stream`, read the caller's device status word (an int32
    device tensor, or an address) and return (code, word): code is ZERO_OK,
    ZERO_ERR_DEVICE_TIMEOUT or ZERO_ERR_NONFINITE as the word's bits say.
    Argument and CUDA errors always raise; with raise_on_error the two
    device conditions raise ZeroError as well."""
    _check_tensor(dev_status, "i32", 1, "dev_status")
    word = ctypes.c_int32(0)
    code = int(lib().zero_get_device_status(_addr(dev_status), _stream(stream),
                                            ctypes.byref(word)))
    if code not in (ZERO_OK, ZERO_ERR_DEVICE_TIMEOUT, ZERO_ERR_NONFINITE) or (
            raise_on_error and code != ZERO_OK):
        raise ZeroError(code, "zero_get_device_status")
    return code, int(word.value)


def zero_rs_avg(plan: Plan, rank_grads, g_shards, flags: int = 0, dev_status=None,
                stream=None) -> None:
    c = plan.c
    for k, g in enumerate(rank_grads):
        _check_tensor(g, "bf16", c.N, f"rank_grads[{k}]")
    _check_tensor(g_shards, "f32", c.padded, "g_shards")
    if len(rank_grads) != c.R * c.M:
        raise ValueError(f"need {c.R * c.M} gradient buffers")
    ga = _ptrs([_addr(g) for g in rank_grads])
    _check(lib().zero_rs_avg(plan.ptr, ctypes.addressof(ga), _addr(g_shards), flags,
                             _addr(dev_status), _stream(stream)), "zero_rs_avg")


def zero_adamw_shard(plan: Plan, g_shards, master, m, v, hp: zero_adamw_hparams, step: int,
                     stream=None) -> None:
    c = plan.c
    for nm, t in (("g_shards", g_shards), ("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.padded, nm)
    _check(lib().zero_adamw_shard(plan.ptr, _addr(g_shards), _addr(master), _addr(m), _addr(v),
                                  ctypes.byref(hp), step, _stream(stream)), "zero_adamw_shard")


def zero_ag_cast(plan: Plan, master, rank_params, stream=None) -> None:
    c = plan.c
    _check_tensor(master, "f32", c.padded, "master")
    for k, p in enumerate(rank_params):
        _check_tensor(p, "bf16", c.N, f"rank_params[{k}]")
    if len(rank_params) != c.R:
        raise ValueError(f"need {c.R} replicas")
    pa = _ptrs([_addr(p) for p in rank_params])
    _check(lib().zero_ag_cast(plan.ptr, _addr(master), ctypes.addressof(pa), _stream(stream)),
           "zero_ag_cast")


def zero_step_host(plan: Plan, host_grads, dev_grads, master, m, v, rank_params,
                   host_params_out, hp: zero_adamw_hparams, step: int, flags: int = 0,
                   dev_status=None, stream=None) -> None:
    """End-to-end step from host buffers.  dev_grads=None selects the
    zero-copy mode (the kernel reads pinned host gradients directly); a list
    of device buffers selects the copy-engine mode."""
    c = plan.c
    for k, g in enumerate(host_grads):
        _check_tensor(g, "bf16", c.N, f"host_grads[{k}]", device="cpu")
    if dev_grads is not None:
        for k, g in enumerate(dev_grads):
            _check_tensor(g, "bf16", c.N, f"dev_grads[{k}]")
        if len(dev_grads) != c.R * c.M:
            raise ValueError("wrong number of device gradient buffers")
    for k, p in enumerate(rank_params):
        _check_tensor(p, "bf16", c.N, f"rank_params[{k}]")
    for nm, t in (("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.padded, nm)
    _check_tensor(host_params_out, "bf16", c.N, "host_params_out", device="cpu")
    if len(host_grads) != c.R * c.M or len(rank_params) != c.R:
        raise ValueError("wrong number of buffers")
    ha = _ptrs([_addr(g) for g in host_grads])
    pa = _ptrs([_addr(p) for p in rank_params])
    da = _ptrs([_addr(g) for g in dev_grads]) if dev_grads is not None else None
    _check(lib().zero_step_host(plan.ptr, ctypes.addressof(ha),
                                ctypes.addressof(da) if da is not None else None,
                                _addr(master), _addr(m), _addr(v), ctypes.addressof(pa),
                                _addr(host_params_out), ctypes.byref(hp), step, flags,
                                _addr(dev_status), _stream(stream)), "zero_step_host")


def zero_step_staged_noalloc(plan: Plan, rank_grads, master, m, v, rank_params,
                             hp: zero_adamw_hparams, step: int, flags: int = 0, dev_status=None,
                             stream=None) -> None:
    """The staged step without a scratch argument, for callers that cannot
    allocate device memory: the library keeps the reduced gradient in a fixed
    16 MiB device array (plans with more than ZERO_NOALLOC_MAX_ELEMS padded
    elements are refused).  The first call on a device looks up that array's
    address; calls that overlap on the GPU share the array and race."""
    c = plan.c
    for k, g in enumerate(rank_grads):
        _check_tensor(g, "bf16", c.N, f"rank_grads[{k}]")
    for k, p in enumerate(rank_params):
        _check_tensor(p, "bf16", c.N, f"rank_params[{k}]")
    for nm, t in (("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.padded, nm)
    _check_tensor(dev_status, "i32", 1, "dev_status")
    if len(rank_grads) != c.R * c.M or len(rank_params) != c.R:
        raise ValueError(f"need {c.R * c.M} gradient buffers and {c.R} replicas")
    ga, pa = _ptrs([_addr(g) for g in rank_grads]), _ptrs([_addr(p) for p in rank_params])
    _check(lib().zero_step_staged_noalloc(plan.ptr, ctypes.addressof(ga), _addr(master),
                                          _addr(m), _addr(v), ctypes.addressof(pa),
                                          ctypes.byref(hp), step, flags, _addr(dev_status),
                                          _stream(stream)), "zero_step_staged_noalloc")


def zero_clip_scratch_bytes(plan: Plan) -> int:
    return int(lib().zero_clip_scratch_bytes(plan.ptr))


def zero_step_clipped(plan: Plan, rank_grads, master, m, v, rank_params, hp: zero_adamw_hparams,
                      step: int, max_norm: float, scratch, flags: int = 0, dev_status=None,
                      dev_sumsq=None, stream=None) -> None:
    """Step with global gradient-norm clipping; scratch holds at least
    zero_clip_scratch_bytes(plan) bytes; dev_sumsq (optional, float64
    device tensor of 1) receives the squared norm."""
    c = plan.c
    for k, g in enumerate(rank_grads):
        _check_tensor(g, "bf16", c.N, f"rank_grads[{k}]")
    for k, p in enumerate(rank_params):
        _check_tensor(p, "bf16", c.N, f"rank_params[{k}]")
    for nm, t in (("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.padded, nm)
    _check_tensor(dev_status, "i32", 1, "dev_status")
    if len(rank_grads) != c.R * c.M or len(rank_params) != c.R:
        raise ValueError(f"need {c.R * c.M} gradient buffers and {c.R} replicas")
    sbytes = scratch.numel() * scratch.element_size() if not isinstance(scratch, int) else \
        zero_clip_scratch_bytes(plan)
    ga, pa = _ptrs([_addr(g) for g in rank_grads]), _ptrs([_addr(p) for p in rank_params])
    _check(lib().zero_step_clipped(plan.ptr, ctypes.addressof(ga), _addr(master), _addr(m),
                                   _addr(v), ctypes.addressof(pa), ctypes.byref(hp), step,
                                   max_norm, _addr(scratch), sbytes, flags, _addr(dev_status),
                                   _addr(dev_sumsq), _stream(stream)), "zero_step_clipped")


def zero3_step(plan: Plan, rank_grads, master, m, v, param_shards, hp: zero_adamw_hparams,
               step: int, flags: int = 0, dev_status=None, stream=None) -> None:
    """ZeRO-3 step: reduce-scatter, AdamW, cast into each rank's own shard of
    param_shards (plan.padded bf16, padded layout); no all-gather."""
    c = plan.c
    for k, g in enumerate(rank_grads):
        _check_tensor(g, "bf16", c.N, f"rank_grads[{k}]")
    for nm, t in (("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.padded, nm)
    _check_tensor(param_shards, "bf16", c.padded, "param_shards")
    _check_tensor(dev_status, "i32", 1, "dev_status")
    if len(rank_grads) != c.R * c.M:
        raise ValueError(f"need {c.R * c.M} gradient buffers")
    ga = _ptrs([_addr(g) for g in rank_grads])
    _check(lib().zero3_step(plan.ptr, ctypes.addressof(ga), _addr(master), _addr(m), _addr(v),
                            _addr(param_shards), ctypes.byref(hp), step, flags,
                            _addr(dev_status), _stream(stream)), "zero3_step")


def zero3_gather(plan: Plan, param_shards, lo: int, hi: int, outs, stream=None) -> None:
    """All-gather of unit [lo, hi) into each of the transient buffers in outs."""
    c = plan.c
    _check_tensor(param_shards, "bf16", c.padded, "param_shards")
    for k, o in enumerate(outs):
        _check_tensor(o, "bf16", hi - lo, f"outs[{k}]")
    oa = _ptrs([_addr(o) for o in outs])
    _check(lib().zero3_gather(plan.ptr, _addr(param_shards), lo, hi, ctypes.addressof(oa),
                              len(outs), _stream(stream)), "zero3_gather")


def gather_unit_table(units) -> ctypes.Array:
    """A C array of zero_gather_unit from (lo, hi, out) triples (out a bf16
    device tensor of hi - lo elements, an address, or None for an empty
    unit); build it once and pass it to zero3_gather_units on every call."""
    units = list(units)
    arr = (zero_gather_unit * max(1, len(units)))()
    for k, (lo, hi, out) in enumerate(units):
        _check_tensor(out, "bf16", hi - lo, f"units[{k}].out")
        arr[k] = zero_gather_unit(int(lo), int(hi), _addr(out))
    return arr


def zero3_gather_units(plan: Plan, param_shards, units, n_units: Optional[int] = None,
                       stream=None) -> None:
    """All-gather of a table of units in one launch.  units: a table from
    gather_unit_table, or (lo, hi, out) triples (converted on every call)."""
    c = plan.c
    _check_tensor(param_shards, "bf16", c.padded, "param_shards")
    if not isinstance(units, ctypes.Array):
        units = list(units)
        n_units = len(units)
        units = gather_unit_table(units)
    elif n_units is None:
        n_units = len(units)
    _check(lib().zero3_gather_units(plan.ptr, _addr(param_shards), units, n_units,
                                    _stream(stream)), "zero3_gather_units")


# -------------------------------------------------------------- checkpoints --

def _np_ptr(a):
    return a.ctypes.data


def zero_ckpt_write_host(plan: Plan, params, master, m, v, step: int, hp: zero_adamw_hparams,
                         directory: str, n_threads: int = 8) -> None:
    """Write the checkpoint of host numpy arrays (params uint16 bf16 bits of N,
    master/m/v float32 with element i at [i])."""
    _check(lib().zero_ckpt_write_host(plan.ptr, _np_ptr(params), _np_ptr(master), _np_ptr(m),
                                      _np_ptr(v), step, ctypes.byref(hp),
                                      os.fsencode(directory), n_threads), "zero_ckpt_write_host")


def zero_ckpt_read_host(plan: Plan, directory: str, params, master, m, v, rank: int = -1):
    """Read a checkpoint (any R) into host numpy arrays in plan's layout;
    returns (step, hparams)."""
    step = ctypes.c_int64(0)
    hp = zero_adamw_hparams()
    _check(lib().zero_ckpt_read_host(plan.ptr, os.fsencode(directory), rank, _np_ptr(params),
                                     _np_ptr(master), _np_ptr(m), _np_ptr(v), ctypes.byref(step),
                                     ctypes.byref(hp)), "zero_ckpt_read_host")
    return step.value, hp


class CkptJob:
    def __init__(self, handle):
        self._h = handle

    def wait(self) -> None:
        if self._h:
            code = lib().zero_ckpt_job_wait(self._h)
            self._h = None
            _check(code, "zero_ckpt_job_wait")


def zero_ckpt_save_async(plan: Plan, params, master, m, v, step: int, hp: zero_adamw_hparams,
                         directory: str, n_threads: int = 8, stream=None) -> CkptJob:
    c = plan.c
    _check_tensor(params, "bf16", c.N, "params")
    for nm, t in (("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.N, nm)
    job = ctypes.c_void_p()
    _check(lib().zero_ckpt_save_async(plan.ptr, _addr(params), _addr(master), _addr(m), _addr(v),
                                      step, ctypes.byref(hp), os.fsencode(directory), n_threads,
                                      _stream(stream), ctypes.byref(job)), "zero_ckpt_save_async")
    return CkptJob(job.value)


def zero_ckpt_job_wait(job: CkptJob) -> None:
    job.wait()


def zero_ckpt_load(plan: Plan, directory: str, params_list, master, m, v, stream=None):
    """Load a checkpoint (any R) onto the device in plan's layout; returns
    (step, hparams)."""
    c = plan.c
    for k, p in enumerate(params_list):
        _check_tensor(p, "bf16", c.N, f"params[{k}]")
    for nm, t in (("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.N, nm)
    pa = _ptrs([_addr(p) for p in params_list])
    step = ctypes.c_int64(0)
    hp = zero_adamw_hparams()
    _check(lib().zero_ckpt_load(plan.ptr, os.fsencode(directory), ctypes.addressof(pa),
                                len(params_list), _addr(master), _addr(m), _addr(v),
                                ctypes.byref(step), ctypes.byref(hp), _stream(stream)),
           "zero_ckpt_load")
    return step.value, hp


def zero_step_compressed(plan: Plan, rank_grads, master, m, v, rank_params,
                         hp: zero_adamw_hparams, step: int, kind: int, residuals=None,
                         stream=None) -> None:
    """Step with a compressed reduce-scatter (kind: ZERO_COMP_FP16 / INT8 /
    SIGN); residuals: None, or R float32 device tensors of N (error feedback)."""
    c = plan.c
    for k, g in enumerate(rank_grads):
        _check_tensor(g, "bf16", c.N, f"rank_grads[{k}]")
    for k, p in enumerate(rank_params):
        _check_tensor(p, "bf16", c.N, f"rank_params[{k}]")
    for nm, t in (("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.padded, nm)
    if len(rank_grads) != c.R * c.M or len(rank_params) != c.R:
        raise ValueError(f"need {c.R * c.M} gradient buffers and {c.R} replicas")
    ea = None
    if residuals is not None:
        if len(residuals) != c.R:
            raise ValueError(f"need {c.R} residual buffers")
        for k, e in enumerate(residuals):
            _check_tensor(e, "f32", c.N, f"residuals[{k}]")
        ea = _ptrs([_addr(e) for e in residuals])
    ga, pa = _ptrs([_addr(g) for g in rank_grads]), _ptrs([_addr(p) for p in rank_params])
    _check(lib().zero_step_compressed(plan.ptr, ctypes.addressof(ga), _addr(master), _addr(m),
                                      _addr(v), ctypes.addressof(pa), ctypes.byref(hp), step, kind,
                                      ctypes.addressof(ea) if ea is not None else None,
                                      _stream(stream)), "zero_step_compressed")


def zero_check_replicas(plan: Plan, rank_params, dev_count, dev_first=None, stream=None) -> None:
    """Count (into dev_count, an int64 device tensor of 1) the elements where
    any replica differs from replica 0; dev_first receives the first index."""
    c = plan.c
    for k, p in enumerate(rank_params):
        _check_tensor(p, "bf16", c.N, f"rank_params[{k}]")
    pa = _ptrs([_addr(p) for p in rank_params])
    _check(lib().zero_check_replicas(plan.ptr, ctypes.addressof(pa), _addr(dev_count),
                                     _addr(dev_first), _stream(stream)), "zero_check_replicas")


def zero_step_onebit(plan: Plan, rank_grads, master, m, v, rank_params,
                     hp: zero_adamw_hparams, step: int, freeze_step: int, worker_residuals,
                     server_residual, stream=None) -> None:
    """1-bit Adam: the plain step while step <= freeze_step, then the
    sign-compressed momentum exchange with worker and owner error feedback
    and a frozen variance.  worker_residuals: R float32 device tensors of N;
    server_residual: a float32 device tensor of plan.padded.  The plan's
    shard length must be a multiple of 128 (align_elems a multiple of 128)."""
    c = plan.c
    for k, g in enumerate(rank_grads):
        _check_tensor(g, "bf16", c.N, f"rank_grads[{k}]")
    for k, p in enumerate(rank_params):
        _check_tensor(p, "bf16", c.N, f"rank_params[{k}]")
    for nm, t in (("master", master), ("m", m), ("v", v), ("server_residual", server_residual)):
        _check_tensor(t, "f32", c.padded, nm)
    if len(rank_grads) != c.R * c.M or len(rank_params) != c.R:
        raise ValueError(f"need {c.R * c.M} gradient buffers and {c.R} replicas")
    if len(worker_residuals) != c.R:
        raise ValueError(f"need {c.R} worker residual buffers")
    for k, e in enumerate(worker_residuals):
        _check_tensor(e, "f32", c.N, f"worker_residuals[{k}]")
    ga, pa = _ptrs([_addr(g) for g in rank_grads]), _ptrs([_addr(p) for p in rank_params])
    ea = _ptrs([_addr(e) for e in worker_residuals])
    _check(lib().zero_step_onebit(plan.ptr, ctypes.addressof(ga), _addr(master), _addr(m),
                                  _addr(v), ctypes.addressof(pa), ctypes.byref(hp), step,
                                  freeze_step, ctypes.addressof(ea), _addr(server_residual),
                                  _stream(stream)), "zero_step_onebit")


def zero3_rs_unit(plan: Plan, unit_grads, lo: int, hi: int, grad_shards, flags: int = 0,
                  dev_status=None, stream=None) -> None:
    """Reduce-scatter one unit's gradients (R*M bf16 device tensors of
    hi - lo each) into the owners' fp32 gradient shards (plan.padded floats)."""
    c = plan.c
    if len(unit_grads) != c.R * c.M:
        raise ValueError(f"need {c.R * c.M} unit gradient buffers")
    for k, g in enumerate(unit_grads):
        _check_tensor(g, "bf16", hi - lo, f"unit_grads[{k}]")
    _check_tensor(grad_shards, "f32", c.padded, "grad_shards")
    ga = _ptrs([_addr(g) for g in unit_grads])
    _check(lib().zero3_rs_unit(plan.ptr, ctypes.addressof(ga), lo, hi, _addr(grad_shards), flags,
                               _addr(dev_status), _stream(stream)), "zero3_rs_unit")


def zero3_update(plan: Plan, grad_shards, master, m, v, param_shards, hp: zero_adamw_hparams,
                 step: int, stream=None) -> None:
    """AdamW of every owned element from the reduce-scattered fp32 gradient
    shards, then the bf16 cast into each rank's own parameter shard."""
    c = plan.c
    for nm, t in (("grad_shards", grad_shards), ("master", master), ("m", m), ("v", v)):
        _check_tensor(t, "f32", c.padded, nm)
    _check_tensor(param_shards, "bf16", c.padded, "param_shards")
    _check(lib().zero3_update(plan.ptr, _addr(grad_shards), _addr(master), _addr(m), _addr(v),
                              _addr(param_shards), ctypes.byref(hp), step, _stream(stream)),
           "zero3_update")
