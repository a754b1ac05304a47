"""Benchmark of the ZeRO-1/2 mixed-precision AdamW step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama-3.2-1b] [--variant fused|staged]

One "step" is one pass of the whole hot path (ordered reduce-scatter +
average, AdamW on every shard, bf16 all-gather into all R replicas) over the
workload's synthetic inputs, which are resident in HBM before the timed
region starts.  The default workload is the Llama-3.2-1B-shaped parameter
set (1,235,814,400 params, R=8 emulated ranks, M=1, ZeRO-2, step 100):
69.2 GB of algorithmic traffic per step, far larger than the 129 MB L2, so
no L2 flush is needed between steps.

Timing: W warm-up steps, then K steps bracketed by a barrier and
cuda.synchronize on both sides, CUDA events on the launching stream, max over
ranks.  Each rank (one per GPU) runs its own emulated ZeRO group: the
emulated ranks live in one GPU's memory and nothing crosses GPUs, so N>1
runs N independent replicas ("weak" scaling).  The JSON line also carries the roofline of the dominant
kernel, the end-to-end number through the host-buffer entry point, the
oracle timed on the host cores, and the SM clocks sampled during the timed
region.

--impl reference times the CPU oracle (the plain C definition the kernels
are checked against) on a bounded sample of the same workload, on the host
cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ZeRO AdamW step: params/s and HBM GB/s (% of ~8 TB/s roofline), 1 GB300"
UNIT = "params/s"


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


# ------------------------------------------------------------ clocks --

class _NvmlClocks:
    """Read-only NVML queries of one GPU (SM clock, its maximum, board power
    and the clock-event reasons), through the driver's libnvidia-ml."""

    LIB = "libnvidia-ml.so.1"
    SM = 1                                            # NVML_CLOCK_SM
    BITS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
            "sw_power_cap": 0x4}

    def __init__(self, uuid: str):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL(self.LIB)
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError(f"no NVML handle for {uuid}")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_mhz = self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.SM)

    def _uint(self, fn, *args):
        x = self.c.c_uint(0)
        rc = fn(self.h, *args, self.c.byref(x))
        return x.value if rc == 0 else None

    def line(self) -> str:
        """One sample in nvidia-smi's CSV form (timestamp, then the fields of
        ClockSampler.FIELDS)."""
        import datetime
        sm = self._uint(self.lib.nvmlDeviceGetClockInfo, self.SM)
        mw = self._uint(self.lib.nvmlDeviceGetPowerUsage)
        r = self.c.c_ulonglong(0)
        ok = self.reasons_fn(self.h, self.c.byref(r)) == 0
        stamp = datetime.datetime.now().strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        flags = [("Active" if r.value & b else "Not Active") if ok else "[N/A]"
                 for b in self.BITS.values()]
        return ", ".join([stamp, "0", str(sm if sm is not None else "[N/A]"),
                          str(self.max_mhz if self.max_mhz is not None else "[N/A]"),
                          "%.2f" % (mw / 1e3) if mw is not None else "[N/A]",
                          "0x%016x" % r.value, *flags]) + "\n"


class ClockSampler:
    """SM clocks and throttle reasons sampled in the background while the
    timed region runs; read-only queries.  NVML is polled every 5 ms from a
    thread when the driver's library loads (a 0.2 s timed region still gets
    dozens of samples); otherwise `nvidia-smi -lms 20` runs beside the
    process."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NVML_PERIOD_S = 0.005
    SMI_PERIOD_MS = 20

    def __init__(self, gpu_id: str, use_nvml=None):
        self.gpu_id = gpu_id
        self.use_nvml = use_nvml
        self.proc = None
        self.path = None
        self.thread = None
        self.lines = []
        self.source = None
        self.t_start = self.t_stop = None

    def _start_nvml(self):
        import threading
        try:
            nv = _NvmlClocks(self.gpu_id)
        except (OSError, AttributeError):
            return False
        self._halt = threading.Event()

        def poll():
            while not self._halt.is_set():
                try:
                    self.lines.append(nv.line())
                except Exception:
                    pass
                self._halt.wait(self.NVML_PERIOD_S)

        self.thread = threading.Thread(target=poll, daemon=True)
        self.thread.start()
        self.source = f"nvml every {self.NVML_PERIOD_S * 1e3:.0f} ms"
        return True

    def start(self):
        if self.use_nvml is not False and self._start_nvml():
            time.sleep(0.1)
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.SMI_PERIOD_MS)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            self.source = f"nvidia-smi -lms {self.SMI_PERIOD_MS}"
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def stop(self):
        if self.thread is not None:
            time.sleep(0.05)
            self._halt.set()
            self.thread.join(timeout=5)
            lines = list(self.lines)
        elif self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            with open(self.path) as f:
                lines = f.readlines()
            os.unlink(self.path)
        else:
            return None
        slack = 2 * (self.NVML_PERIOD_S if self.thread is not None
                     else self.SMI_PERIOD_MS / 1e3)
        out = summarise_clocks(lines, self.t_start, self.t_stop, slack)
        if out is not None:
            out["source"] = self.source
        return out


CLOCK_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def summarise_clocks(lines, t_start, t_stop, slack=0.1):
    """Summary of nvidia-smi CSV lines (timestamp, then ClockSampler.FIELDS,
    no header, no units): the median SM clock, the maximum SM clock and the
    throttle reasons that were active, over the samples taken between
    t_start and t_stop (`slack` seconds either side, about one sampling
    period), or over every sample when none fell inside; None without a
    usable sample."""
    import datetime

    rows = [[p.strip() for p in line.split(",")] for line in lines]
    rows = [p for p in rows if len(p) >= 10]

    def ts(p):
        try:
            return datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    inside = [p for p in rows if t_start and t_stop and ts(p) is not None
              and t_start - slack <= ts(p) <= t_stop + slack]
    use = inside or rows
    sm, reasons, sm_max = [], set(), None
    for p in use:
        try:
            mhz, mx = float(p[2]), float(p[3])
        except ValueError:
            continue
        sm_max = mx
        sm.append(mhz)
        for name, flag in zip(CLOCK_REASONS, p[6:10]):
            if flag.lower().startswith("active"):
                reasons.add(name)
    if not sm:
        return None
    sm.sort()
    return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": sm_max, "reasons": sorted(reasons),
            "samples": len(sm), "in_timed_region": bool(inside)}


def gpu_uuid(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device_index)


# --------------------------------------------------------- oracle (CPU) --

def oracle_prepare(wl, n, threads=None):
    """Host inputs of the first n params of the workload (seeded generator,
    built in parallel chunks) for timing the oracle."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor

    from zgen import workloads as W

    threads = threads or os.cpu_count() or 1
    chunks = [(lo, min(n, lo + (1 << 20))) for lo in range(0, n, 1 << 20)]
    G = [np.empty(n, np.uint16) for _ in range(wl.R * wl.M)]
    W0 = np.empty(n, np.float32)
    m0 = np.empty(n, np.float32)
    v0 = np.empty(n, np.float32)

    def work(c):
        lo, hi = c
        idx = np.arange(lo, hi, dtype=np.int64)
        for g, src in zip(G, W.host_grads_at(wl, wl.step, idx)):
            g[lo:hi] = src
        W0[lo:hi] = W.host_w0_at(wl, idx)
        a, b = W.host_mv0_at(wl, idx)
        m0[lo:hi], v0[lo:hi] = a, b

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, chunks))
    P = [np.empty(n, np.uint16) for _ in range(wl.R)]
    return {"G": G, "W0": W0, "m0": m0, "v0": v0, "P": P, "threads": threads, "n": n}


# the oracle function that defines each measured step (only the plain step
# has a multithreaded form; the others run on one core)
ORACLE_FN = {"fused": "oracle_dp_step_mt", "staged": "oracle_dp_step_mt",
             "staged_grads": "oracle_dp_step_mt",
             "tma": "oracle_dp_step_mt", "clipped": "oracle_dp_step_clipped",
             "compressed": "oracle_dp_step_compressed", "onebit": "oracle_onebit_step",
             "zero3": "oracle_zero3_step", "zero3_gather_units": "oracle_zero3_gather"}


def oracle_step_opts(args=None) -> dict:
    """The step a bench line measures, as the oracle leg needs it."""
    if args is None:
        return {"variant": "fused"}
    return {"variant": args.variant, "codec": args.codec, "ef": args.ef,
            "max_norm": args.max_norm}


def oracle_threads(ctx, variant: str) -> int:
    return ctx["threads"] if ORACLE_FN[variant] == "oracle_dp_step_mt" else 1


def oracle_pass(wl, ctx, variant="fused", codec="int8", ef=False, max_norm=1.0):
    """One timed pass of the oracle (unchanged) of the step `variant`
    measures, over the prepared sample; returns seconds.  Buffers the step
    needs besides the sample (zero residuals, padded ZeRO-3 state, the
    parameter shard) are made before the clock starts."""
    import numpy as np

    import oracle
    n, R, M, t = ctx["n"], wl.R, wl.M, wl.step
    hp = oracle.hparams(**wl.hparams())
    G, P = ctx["G"], ctx["P"]
    if variant == "zero3_gather_units":
        # every tensor of the sample (the workload's first n params) gathered
        # from the padded shard buffer, one unit at a time
        S = oracle.shard_len(n, R)
        Ps = np.zeros(R * S, np.uint16)
        cuts = [int(c) for c in wl.offsets if c < n] + [n]
        t0 = time.perf_counter()
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            oracle.zero3_gather(Ps, n, R, S, lo, hi, 0)
        return time.perf_counter() - t0
    if variant == "zero3":
        S = oracle.shard_len(n, R)
        Wc, mc, vc = (np.zeros(R * S, np.float32) for _ in range(3))
        Wc[:n], mc[:n], vc[:n] = ctx["W0"], ctx["m0"], ctx["v0"]
        Ps = np.zeros(R * S, np.uint16)
        t0 = time.perf_counter()
        oracle.zero3_step(G, Wc, mc, vc, Ps, hp, t, R, M, n, S)
        return time.perf_counter() - t0
    Wc, mc, vc = ctx["W0"].copy(), ctx["m0"].copy(), ctx["v0"].copy()
    if variant == "clipped":
        t0 = time.perf_counter()
        oracle.dp_step_clipped(G, Wc, mc, vc, P, hp, t, R, M, max_norm)
    elif variant == "compressed":
        kind = {"fp16": oracle.COMP_FP16, "int8": oracle.COMP_INT8,
                "sign": oracle.COMP_SIGN}[codec]
        E = [np.zeros(n, np.float32) for _ in range(R)] if ef else None
        t0 = time.perf_counter()
        oracle.dp_step_compressed(G, Wc, mc, vc, P, hp, t, R, M, kind, E)
    elif variant == "onebit":
        S = oracle.shard_len(n, R, 128)
        E = [np.zeros(n, np.float32) for _ in range(R)]
        Es = np.zeros(n, np.float32)
        t0 = time.perf_counter()
        oracle.onebit_step(G, Wc, mc, vc, P, hp, t, max(1, t - 1), R, M, S, E, Es)
    else:
        t0 = time.perf_counter()
        oracle.dp_step(G, Wc, mc, vc, P, hp, t, R, M, nthreads=ctx["threads"])
    return time.perf_counter() - t0


def oracle_sample_rate(wl, target_s=12.0, sample_elems=1 << 24, threads=None, opts=None,
                       ctx=None):
    """Time the oracle of the measured step (opts, from oracle_step_opts) on
    the first sample_elems params of the workload, repeated until target_s of
    CPU time; returns params/s, cores, text.  ctx: inputs already prepared
    (oracle_prepare), timed with `threads` threads when given."""
    opts = opts or {"variant": "fused"}
    n = min(sample_elems, wl.N)
    if ctx is None:
        ctx = oracle_prepare(wl, n, threads)
    elif threads:
        ctx = dict(ctx, threads=threads)
    n = ctx["n"]
    reps, elapsed = 0, 0.0
    while elapsed < target_s or reps == 0:
        elapsed += oracle_pass(wl, ctx, **opts)
        reps += 1
    cores = oracle_threads(ctx, opts["variant"])
    desc = (f"{ORACLE_FN[opts['variant']]} over the first {n:,} params of the workload "
            f"(same R, M, distributions), {cores} thread(s), {reps} passes, {elapsed:.1f} s")
    return n * reps / elapsed, cores, desc


def oracle_baseline(wl, opts, target_s=8.0, sample_elems=1 << 24):
    """The cpu_baseline object: the oracle of the measured step on all host
    cores and on one core, over the same prepared sample."""
    n = min(sample_elems, wl.N)
    ctx = oracle_prepare(wl, n)
    rate, cores, desc = oracle_sample_rate(wl, target_s, opts=opts, ctx=ctx)
    cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
    if cores > 1:
        r1, c1, d1 = oracle_sample_rate(wl, target_s, threads=1, opts=opts, ctx=ctx)
    else:
        r1, c1, d1 = rate, cores, desc
    cpu.update({"value_1core": r1, "cores_1core": c1, "sample_1core": d1,
                "host_cores": os.cpu_count()})
    return cpu


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of a per-rank float over all ranks of the default process
    group (the identity without one).  Timing only: no step data crosses
    ranks."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ our arm --

KERNEL_SRC = os.path.join(ROOT, "zero_optimizer_step_rs_gb300", "csrc", "zero_step.cu")
FUSED_PATH_END = "// ================================================== end of the fused path =="


def kernel_source_hash() -> str:
    """Hash of the source the fused path is compiled from: zero_step.cu up to
    its end-of-fused-path marker (helpers, k_fused and its launch)."""
    with open(KERNEL_SRC) as f:
        body = f.read().split(FUSED_PATH_END)[0].rstrip()
    return hashlib.sha256(body.encode()).hexdigest()[:16]


def _mem_available_bytes():
    """MemAvailable of this node from /proc/meminfo, or None."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return None


def e2e_fits_host(host_need: int, device=None):
    """Whether this node's ranks can pin host_need bytes between them (at
    most 60 % of the available memory), decided with a max over ranks so
    that every rank takes the same branch; returns (fits, available bytes
    seen by this rank)."""
    avail = _mem_available_bytes()
    too_big = bool(avail) and host_need > 0.6 * avail
    return max_over_ranks(1.0 if too_big else 0.0, device) == 0.0, avail


def traffic_per_param():
    """Measured DRAM bytes per parameter of the fused kernel from the
    committed ncu summary, if it was taken on the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, None
    if rec.get("source_sha256_16") != kernel_source_hash():
        return None, rec
    return rec, rec


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import zero_optimizer_step_rs_gb300 as z
    from tests import harness as H
    from zgen import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = W.by_name(args.workload)
    if getattr(args, "scale", 0):
        wl = wl.scaled(args.scale)
    variant = {"staged": z.ZERO_VARIANT_STAGED, "staged_grads": z.ZERO_VARIANT_STAGED,
               "tma": z.ZERO_VARIANT_FUSED_TMA}.get(args.variant, z.ZERO_VARIANT_FUSED)
    staged_grads = args.variant == "staged_grads"
    clipped = args.variant == "clipped"
    zero3 = args.variant == "zero3"
    gather_units = args.variant == "zero3_gather_units"
    compressed = args.variant == "compressed"
    onebit = args.variant == "onebit"
    if onebit:                             # 1-bit Adam wants shards on the 128-element block grid
        import dataclasses
        wl = dataclasses.replace(wl, align=128)
    stream = torch.cuda.current_stream()

    ds = H.DeviceState(wl, str(dev), staged_scratch=(args.variant == "staged"))
    restore = None
    if staged_grads:
        # ZeRO-2 without scratch: the reduced gradient in gradient buffers 0 and 1.
        # The step leaves those two buffers unspecified; in training the next
        # backward writes them again.  Here a copy of their inputs is put back
        # before every step, outside the step's own event pair (the timed steps
        # are then summed from those pairs): steps fed the previous step's
        # leftovers would compute on arbitrary bits, NaN and Inf among them.
        if not (wl.stage == 2 and wl.R * wl.M >= 2):
            raise SystemExit("--variant staged_grads needs a ZeRO-2 workload with R*M >= 2")
        ds.step = lambda t, variant=0, flags=0: z.zero_step(
            ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t,
            variant=z.ZERO_VARIANT_STAGED, scratch=None, flags=flags, dev_status=ds.status)
        kept = None

        def restore():
            for g, c in zip(ds.grads[:2], kept):
                g.copy_(c)
    if clipped:
        ds.step = lambda t, variant=0, flags=0: ds.step_clipped(t, args.max_norm, flags=flags)
    elif gather_units:
        # the whole parameter set gathered per tensor, one zero3_gather_units
        # launch over the table of its units; the shards hold the result of a
        # ZeRO-3 step taken before the timed region
        shards = torch.empty(ds.padded, dtype=torch.bfloat16, device=dev)
        offs = [int(x) for x in wl.offsets]
        pairs = list(zip(offs[:-1], offs[1:]))
        unit_outs = [torch.empty(hi - lo, dtype=torch.bfloat16, device=dev) for lo, hi in pairs]
        table = z.gather_unit_table([(lo, hi, o) for (lo, hi), o in zip(pairs, unit_outs)])
        ds.step = lambda t, variant=0, flags=0: z.zero3_gather_units(ds.plan, shards, table,
                                                                     len(pairs))
    elif zero3:
        shards = torch.empty(ds.padded, dtype=torch.bfloat16, device=dev)
        ds.step = lambda t, variant=0, flags=0: z.zero3_step(
            ds.plan, ds.grads, ds.W, ds.m, ds.v, shards, ds.hp, t, flags=flags,
            dev_status=ds.status)
    elif compressed:
        codec = {"fp16": z.ZERO_COMP_FP16, "int8": z.ZERO_COMP_INT8, "sign": z.ZERO_COMP_SIGN}[
            args.codec]
        resid = ([torch.zeros(wl.N, dtype=torch.float32, device=dev) for _ in range(wl.R)]
                 if args.ef else None)
        ds.step = lambda t, variant=0, flags=0: z.zero_step_compressed(
            ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t, codec, resid)
    elif onebit:
        # freeze before the measured step, so every warm-up and timed step is
        # a compressed one
        freeze = max(1, wl.step - 1)
        w_res = [torch.zeros(wl.N, dtype=torch.float32, device=dev) for _ in range(wl.R)]
        s_res = torch.zeros(ds.padded, dtype=torch.float32, device=dev)
        ds.step = lambda t, variant=0, flags=0: z.zero_step_onebit(
            ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t, freeze, w_res, s_res)
    ds.fill_state_device()
    t = wl.first_step()
    while t < wl.step:                     # prior steps build the moments
        ds.fill_grads_device(t)
        ds.step(t, variant=variant)
        t += 1
    ds.fill_grads_device(wl.step)
    if restore is not None:
        kept = [g.clone() for g in ds.grads[:2]]
    if gather_units:
        z.zero3_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, shards, ds.hp, wl.step)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    step_t = wl.step
    for _ in range(args.warmup):
        if restore is not None:
            restore()
        ds.step(step_t, variant=variant)
        step_t += 1
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_uuid(local_rank))
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    e_all0, e_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    sampler.mark_start()
    e_all0.record(stream)
    for k in range(args.steps):
        if restore is not None:
            restore()
        ev[k][0].record(stream)
        ds.step(step_t, variant=variant)
        ev[k][1].record(stream)
        step_t += 1
    e_all1.record(stream)
    torch.cuda.synchronize()
    barrier()
    sampler.mark_stop()
    clocks = sampler.stop()
    total_ms = e_all0.elapsed_time(e_all1)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if restore is not None:
        total_ms = float(sum(launch_ms))          # the steps alone, without the restores

    total_ms = max_over_ranks(total_ms, dev)

    N = wl.N
    ms_per_step = total_ms / args.steps
    value = N * args.steps * world / (total_ms / 1e3)
    if clipped:
        bpp = 2 * wl.R * wl.M + 4 + 4 + 24 + 2 * wl.R      # stash written and read back
    elif gather_units:
        bpp = 4                                             # 2 read from the shards, 2 written
    elif zero3:
        bpp = 2 * wl.R * wl.M + 24 + 2
    elif compressed:
        bpp = wl.bytes_per_param() + (8 * wl.R if args.ef else 0)
    elif onebit:
        bpp = 2 * wl.R * wl.M + 10 * wl.R + 28
    elif variant in (z.ZERO_VARIANT_FUSED, z.ZERO_VARIANT_FUSED_TMA):
        bpp = wl.bytes_per_param()
    else:
        bpp = 2 * wl.R * wl.M + 4 + 4 + 24 + 4 + 2 * wl.R
    alg_bytes = bpp * N
    avg_launch_s = float(np.mean(launch_ms)) / 1e3
    achieved_gbs = alg_bytes / avg_launch_s / 1e9
    peaks = measured_peaks()
    if peaks and "hbm_gbs" in peaks:
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    else:
        peak, peak_src = 6800.0, "fallback"
    rec, _ = traffic_per_param()
    traffic = None
    if (rec and args.variant == "fused" and rec.get("R") == wl.R and rec.get("M") == wl.M):
        traffic = round(rec["dram_bytes_per_param"] * N)
    roofline = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved_gbs / peak, 4), "traffic": traffic,
                "peak_source": peak_src,
                "kernel": ("clipped step (k_rs_norm, k_adamw_ag)" if clipped
                           else f"k_gather_units ({len(pairs)} per-tensor units, one launch)"
                           if gather_units
                           else "k_fused (ZeRO-3 output)" if zero3
                           else f"k_comp ({args.codec}{', error feedback' if args.ef else ''})"
                           if compressed
                           else "k_onebit (1-bit Adam, frozen variance)" if onebit
                           else "staged trio, reduced gradient in gradient buffers 0 and 1"
                           if staged_grads
                           else {0: "k_fused", 1: "staged trio", 2: "k_fused_tma"}[variant]),
                "algorithmic_bytes_per_launch": alg_bytes, "bytes_per_param": bpp}

    # -------- end to end through the host-buffer entry point
    e2e = None
    want_e2e = not args.no_e2e and args.variant == "fused"
    # every rank of this node pins its own copy of the gradients and the
    # replica; decided together before any rank pins, so all ranks take the
    # same branch (the collectives below need every rank)
    host_need = world * (2 * wl.R * wl.M + 2) * N
    fits, host_avail = e2e_fits_host(host_need, dev) if want_e2e else (False, None)
    if want_e2e and not fits:
        e2e = {"unavailable": f"{world} rank(s) would pin {host_need / 1e9:.1f} GB of host memory "
                              f"for the gradients; {(host_avail or 0) / 1e9:.1f} GB is available"}
    elif want_e2e:
        host_g = [torch.empty(N, dtype=torch.bfloat16, pin_memory=True) for _ in ds.grads]
        for h, d in zip(host_g, ds.grads):
            h.copy_(d[:N])
        out = torch.empty(N, dtype=torch.bfloat16, pin_memory=True)
        torch.cuda.synchronize()
        k_e2e = max(2, min(args.steps, 5))

        def e2e_run(dev_grads):
            nonlocal step_t
            z.zero_step_host(ds.plan, host_g, dev_grads, ds.W, ds.m, ds.v, ds.params, out,
                             ds.hp, step_t)
            step_t += 1
            torch.cuda.synchronize()
            barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(k_e2e):
                z.zero_step_host(ds.plan, host_g, dev_grads, ds.W, ds.m, ds.v, ds.params, out,
                                 ds.hp, step_t)
                step_t += 1
            e1.record(stream)
            torch.cuda.synchronize()
            return max_over_ranks(e0.elapsed_time(e1), dev)

        zc_ms = e2e_run(None)                    # zero-copy: kernel reads host memory
        ce_ms = e2e_run(ds.grads)                # copy engine: copies in, step, copy out
        e2e = {"value": N * k_e2e * world / (zc_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": 2 * wl.R * wl.M * N, "d2h_bytes_per_step": 2 * N,
               "ms_per_step": zc_ms / k_e2e, "steps": k_e2e,
               "path": "zero_step_host, zero-copy mode: the fused kernel reads the R*M "
                       "gradient buffers from pinned host memory over the host link and writes "
                       "replica 0 back to pinned host memory",
               "copy_engine_value": N * k_e2e * world / (ce_ms / 1e3),
               "copy_engine_ms_per_step": ce_ms / k_e2e}
        del host_g, out

    if clipped:
        launches_per_step = 2          # rs_norm with the tree up to the groups, update
    else:
        launches_per_step = 3 if variant == z.ZERO_VARIANT_STAGED else 1
    del ds
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(wl, oracle_step_opts(args))

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator; shapes of the named parameter set)",
        "config": {"workload": wl.name, "N": N, "R": wl.R, "M": wl.M, "stage": wl.stage,
                   "step": wl.step, "variant": args.variant,
                   **({"max_norm": args.max_norm} if clipped else {}),
                   **({"codec": args.codec, "error_feedback": args.ef} if compressed else {}),
                   **({"freeze_step": max(1, wl.step - 1), "align": 128} if onebit else {}),
                   **({"units": len(pairs)} if gather_units else {}),
                   "l2": "inputs (%.1f GB/step) far larger than the 129 MB L2; no flush"
                         % (alg_bytes / 1e9),
                   "parallelism": f"{world} independent replica(s) of an R={wl.R} "
                                  "emulated ZeRO group"},
        "hbm_gbs": round(alg_bytes / (ms_per_step / 1e3) / 1e9, 1),
        # the pages' normalised collective bandwidth (CS336 Lecture 7 book,
        # sections 5.2 and 5.3): a reduce-scatter or all-gather of a B-byte
        # message over R ranks counts B (R-1)/R, an all-reduce twice that;
        # the emulated step does one reduce-scatter and one all-gather of
        # 2N-byte bf16 messages (micro-batches summed locally; ZeRO-3 has no
        # all-gather in the step), timed by the whole step
        "emulated_busbw_gbs": round((1 if zero3 or gather_units else 2) * 2 * N * (wl.R - 1) / wl.R
                                    / (ms_per_step / 1e3) / 1e9, 1),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    return line


# -------------------------------------------------------------- table --

def run_table(args):
    """Every workload (fused and staged) and the flat sweep: median kernel
    time over reps with an L2 flush before each rep, params/s, GB/s of
    algorithmic bytes and the fraction of the measured copy peak; the oracle
    on 1 core and on all host cores for each workload."""
    import numpy as np
    import torch

    import zero_optimizer_step_rs_gb300 as z
    from tests import harness as H
    from zgen import workloads as W

    torch.cuda.set_device(0)
    peaks = measured_peaks() or {}
    peak = float(peaks.get("hbm_gbs", 6800.0))
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    # read after the write flush, it leaves L2 holding clean lines of an
    # unrelated buffer: the timed launch then writes back none of the
    # flush's dirty lines (up to the 129 MB of L2 at 6.7 TB/s: ~19 us)
    clean_src = torch.zeros(64 * 1024 * 1024, dtype=torch.float32, device="cuda")
    rows = []
    sampler = ClockSampler(gpu_uuid(0))          # SM clocks over the GPU part
    sampler.start()
    sampler.mark_start()

    def run_step(ds, t, variant):
        if variant == "in_grads":                    # staged, reduced gradient in buffers 0 and 1
            z.zero_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t,
                        variant=z.ZERO_VARIANT_STAGED, scratch=None)
        else:
            ds.step(t, variant=variant)

    def before_step(ds, variant):
        # the in-buffer mode leaves gradient buffers 0 and 1 unspecified: put
        # their inputs back before each step, outside its event pair
        if variant == "in_grads":
            for g, c in zip(ds.grads[:2], ds.kept_grads):
                g.copy_(c)

    def timed(ds, variant, reps, cold=True, clean=False):
        ts = []
        t = ds.wl.step
        for k in range(3 + reps):
            before_step(ds, variant)
            if cold:
                flush.fill_(k & 0xFF)                  # evict L2 (256 MB > 129 MB)
                if clean:
                    clean_src.sum()                    # dirty lines written back here
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run_step(ds, t, variant)
            e1.record()
            torch.cuda.synchronize()
            t += 1
            if k >= 3:
                ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    def timed_small(ds, variant, reps, cold, clean=False):
        """A step of microseconds: every launch is enqueued behind a sleep
        kernel, so the events time the GPU, not the host's launch calls.
        Warm: reps steps back to back between one event pair, the mean per
        step.  Cold: a flush, then an event pair around one step, reps
        times; the mean of the spans (the event timer ticks about every
        2 us, so a median would only pick a tick)."""
        t = ds.wl.step
        for _ in range(3):
            run_step(ds, t, variant)
            t += 1
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000_000)                 # ~0.1 s: the host enqueues meanwhile
        if not cold:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for k in range(reps):
                run_step(ds, t + k, variant)
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps
        ev = []
        for k in range(reps):
            flush.fill_(k & 0xFF)
            if clean:
                clean_src.sum()                        # dirty lines written back here
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run_step(ds, t + k, variant)
            e1.record()
            ev.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in ev]))

    def bpp(wl, variant):
        return wl.bytes_per_param() if variant == 0 else 2 * wl.R * wl.M + 36 + 2 * wl.R

    def measure(wl, label, reps, variants=(0, 1, "in_grads")):
        ds = H.DeviceState(wl, staged_scratch=True)
        ds.fill_state_device()
        ds.fill_grads_device(wl.step)
        ds.kept_grads = [g.clone() for g in ds.grads[:2]] if "in_grads" in variants else []
        torch.cuda.synchronize()
        resident = bpp(wl, 1) * wl.N < 129e6
        for variant in variants:
            if variant == "in_grads" and not (wl.stage == 2 and wl.R * wl.M >= 2):
                continue
            # a workload that fits in L2 is timed twice: after a flush (cold
            # L2, the flush's dirty lines written back during the launch) and
            # back to back with its inputs resident (warm L2)
            for cold in ((True, False) if resident else (True,)):
                ms = timed_small(ds, variant, 200, cold) if resident else timed(ds, variant, reps)
                gbs = bpp(wl, variant) * wl.N / (ms / 1e3) / 1e9
                row = {"workload": label, "R": wl.R, "M": wl.M, "N": wl.N,
                       "variant": {0: "fused", 1: "staged"}.get(
                           variant, "staged, reduced gradient in gradient buffers 0 and 1"),
                       "ms": round(ms, 4),
                       "params_per_s": wl.N / (ms / 1e3), "bytes_per_param": bpp(wl, variant),
                       "GB_s": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
                       "l2": ("cold: 256 MB flush before each launch; mean of 200 event "
                              "spans around one launch (an empty pair spans ~2.1 us)" if cold
                              else "warm: inputs resident, 200 launches back to back, mean")
                       if resident else "inputs far larger than L2; flushed before each launch"}
                if cold:
                    ms_c = (timed(ds, variant, reps, clean=True) if not resident
                            else timed_small(ds, variant, 200, True, clean=True))
                    row["ms_clean_l2"] = round(ms_c, 4)
                    row["frac_clean_l2"] = round(
                        bpp(wl, variant) * wl.N / (ms_c / 1e3) / 1e9 / peak, 4)
                rows.append(row)
                print(json.dumps(row), flush=True)
        del ds
        torch.cuda.empty_cache()

    for name in ("tiny", "gpt2-small", "llama-3.2-1b", "uneven", "large"):
        measure(W.ALL[name](), name, reps=20 if name != "large" else 10)
    # ZeRO-3: the step (cast into each rank's own shard) and the per-unit
    # all-gather of the whole 1B-shaped model at three unit sizes
    for name in ("gpt2-small", "llama-3.2-1b", "large"):
        wl = W.ALL[name]()
        ds = H.DeviceState(wl, staged_scratch=False)
        ds.fill_state_device()
        ds.fill_grads_device(wl.step)
        shards = torch.empty(ds.padded, dtype=torch.bfloat16, device="cuda")
        ts, t = [], wl.step
        for k in range(3 + 10):
            flush.fill_(k & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            z.zero3_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, shards, ds.hp, t)
            e1.record()
            torch.cuda.synchronize()
            t += 1
            if k >= 3:
                ts.append(e0.elapsed_time(e1))
        ms = float(np.median(ts))
        b = 2 * wl.R * wl.M + 26
        row = {"workload": name, "R": wl.R, "M": wl.M, "N": wl.N, "variant": "zero3_step",
               "ms": round(ms, 4), "params_per_s": wl.N / (ms / 1e3), "bytes_per_param": b,
               "GB_s": round(b * wl.N / (ms / 1e3) / 1e9, 1),
               "frac_of_measured_peak": round(b * wl.N / (ms / 1e3) / 1e9 / peak, 4),
               "l2_resident": False}
        rows.append(row)
        print(json.dumps(row), flush=True)
        if name == "llama-3.2-1b":
            offs = [int(x) for x in wl.offsets]
            layers = [0, offs[1]] + [offs[1 + 9 * (l + 1)] for l in range(16)] + [offs[-1]]
            layers = sorted(set(layers))
            full = torch.empty(wl.N, dtype=torch.bfloat16, device="cuda")
            for label, cuts, graph in (("unit = tensor (146 units)", offs, False),
                                       ("unit = tensor (146 units), one CUDA graph", offs, True),
                                       ("unit = tensor (146 units), one zero3_gather_units "
                                        "launch", offs, "table"),
                                       ("unit = layer (18 units)", layers, False),
                                       ("unit = layer (18 units), one CUDA graph", layers, True),
                                       ("unit = layer (18 units), one zero3_gather_units "
                                        "launch", layers, "table"),
                                       ("unit = whole model (1 unit)", [0, wl.N], False)):
                def gather_all():
                    for lo, hi in zip(cuts[:-1], cuts[1:]):
                        z.zero3_gather(ds.plan, shards, lo, hi, [full[:hi - lo]])
                run = gather_all
                if graph == "table":
                    # every unit into its own slice of the model buffer (the
                    # table's destinations may not overlap); the table is
                    # built once and passed as is on every call
                    pairs = list(zip(cuts[:-1], cuts[1:]))
                    table = z.gather_unit_table([(lo, hi, full[lo:hi]) for lo, hi in pairs])

                    def run():
                        z.zero3_gather_units(ds.plan, shards, table, len(pairs))
                elif graph:
                    # the same launches captured once and replayed: no host
                    # work between them (the eager rows above have already
                    # run every kernel once)
                    cg = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(cg):
                        gather_all()
                    run = cg.replay
                ts = []
                for k in range(3 + 10):
                    flush.fill_(k & 0xFF)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                    run()
                    e1.record()
                    torch.cuda.synchronize()
                    if k >= 3:
                        ts.append(e0.elapsed_time(e1))
                ms = float(np.median(ts))
                row = {"workload": name, "variant": "zero3_gather", "unit": label,
                       "launches": 1 if graph == "table" else len(cuts) - 1, "ms": round(ms, 4),
                       "GB_s": round(4 * wl.N / (ms / 1e3) / 1e9, 1),
                       "frac_of_measured_peak": round(4 * wl.N / (ms / 1e3) / 1e9 / peak, 4)}
                rows.append(row)
                print(json.dumps(row), flush=True)
            del full
            # FSDP's backward: each layer's gradient reduce-scattered by its
            # own launch (last layer first), then one update of the shards
            gs = torch.empty(ds.padded, dtype=torch.float32, device="cuda")
            units = list(zip(layers[:-1], layers[1:]))[::-1]
            t_rs, t_up = [], []
            for k in range(3 + 10):
                flush.fill_(k & 0xFF)
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                ev[0].record()
                for lo, hi in units:
                    z.zero3_rs_unit(ds.plan, [g[lo:hi] for g in ds.grads], lo, hi, gs)
                ev[1].record()
                z.zero3_update(ds.plan, gs, ds.W, ds.m, ds.v, shards, ds.hp, t)
                ev[2].record()
                torch.cuda.synchronize()
                t += 1
                if k >= 3:
                    t_rs.append(ev[0].elapsed_time(ev[1]))
                    t_up.append(ev[1].elapsed_time(ev[2]))
            for label, ms, b, n_l in (
                    ("zero3_rs_unit, unit = layer (18 units)", float(np.median(t_rs)),
                     2 * wl.R * wl.M + 4, len(units)),
                    ("zero3_update", float(np.median(t_up)), 30, 1),
                    ("unit reduce-scatter + update", float(np.median(t_rs)) + float(np.median(t_up)),
                     2 * wl.R * wl.M + 34, len(units) + 1)):
                row = {"workload": name, "R": wl.R, "M": wl.M, "N": wl.N,
                       "variant": "zero3_units", "part": label, "launches": n_l,
                       "ms": round(ms, 4), "params_per_s": wl.N / (ms / 1e3), "bytes_per_param": b,
                       "GB_s": round(b * wl.N / (ms / 1e3) / 1e9, 1),
                       "frac_of_measured_peak": round(b * wl.N / (ms / 1e3) / 1e9 / peak, 4)}
                rows.append(row)
                print(json.dumps(row), flush=True)
            # the same backward with each layer's parameters all-gathered
            # again before its reduce-scatter (FSDP materialises a unit for
            # its backward) into one of two transient buffers: all on one
            # stream, then with the next layer's gather prefetched on a second
            # stream (it waits only for its buffer to be released)
            umax = max(hi - lo for lo, hi in units)
            bufs = [torch.empty(umax, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
            main, side = torch.cuda.current_stream(), torch.cuda.Stream()
            unit_grads = [[g[lo:hi] for g in ds.grads] for lo, hi in units]

            def serial():
                for k, (lo, hi) in enumerate(units):
                    z.zero3_gather(ds.plan, shards, lo, hi, [bufs[k % 2][:hi - lo]])
                    z.zero3_rs_unit(ds.plan, unit_grads[k], lo, hi, gs)

            def prefetched():
                gathered = [torch.cuda.Event() for _ in units]
                released = [torch.cuda.Event() for _ in units]
                side.wait_stream(main)

                def issue(k):
                    lo, hi = units[k]
                    if k >= 2:
                        side.wait_event(released[k - 2])
                    z.zero3_gather(ds.plan, shards, lo, hi, [bufs[k % 2][:hi - lo]], stream=side)
                    gathered[k].record(side)

                issue(0)
                for k, (lo, hi) in enumerate(units):
                    if k + 1 < len(units):
                        issue(k + 1)
                    main.wait_event(gathered[k])
                    z.zero3_rs_unit(ds.plan, unit_grads[k], lo, hi, gs)
                    released[k].record(main)

            b = 4 + 2 * wl.R * wl.M + 4
            for label, fn in (("gather + reduce-scatter per layer, one stream", serial),
                              ("gather + reduce-scatter per layer, next gather prefetched "
                               "on a second stream", prefetched)):
                ts = []
                for k in range(3 + 10):
                    flush.fill_(k & 0xFF)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    fn()
                    e1.record()
                    torch.cuda.synchronize()
                    if k >= 3:
                        ts.append(e0.elapsed_time(e1))
                ms = float(np.median(ts))
                row = {"workload": name, "R": wl.R, "M": wl.M, "N": wl.N,
                       "variant": "zero3_backward", "part": label, "launches": 2 * len(units),
                       "ms": round(ms, 4), "params_per_s": wl.N / (ms / 1e3), "bytes_per_param": b,
                       "GB_s": round(b * wl.N / (ms / 1e3) / 1e9, 1),
                       "frac_of_measured_peak": round(b * wl.N / (ms / 1e3) / 1e9 / peak, 4)}
                rows.append(row)
                print(json.dumps(row), flush=True)
            del gs, bufs, unit_grads
        del ds, shards
        torch.cuda.empty_cache()

    # compressed reduce-scatter on the 1B-shaped workload: each codec with and
    # without error feedback
    wl = W.llama32_1b()
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.fill_state_device()
    ds.fill_grads_device(wl.step)
    res = [torch.zeros(wl.N, dtype=torch.float32, device="cuda") for _ in range(wl.R)]
    wire = {z.ZERO_COMP_FP16: 2.0, z.ZERO_COMP_INT8: 1 + 4 / 128, z.ZERO_COMP_SIGN: 1 / 8 + 4 / 128}
    names = {z.ZERO_COMP_FP16: "fp16", z.ZERO_COMP_INT8: "int8/128", z.ZERO_COMP_SIGN: "sign/128"}
    for kind in (z.ZERO_COMP_FP16, z.ZERO_COMP_INT8, z.ZERO_COMP_SIGN):
        for ef in (False, True):
            ts, t = [], wl.step
            for k in range(3 + 10):
                flush.fill_(k & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                z.zero_step_compressed(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t,
                                       kind, res if ef else None)
                e1.record()
                torch.cuda.synchronize()
                t += 1
                if k >= 3:
                    ts.append(e0.elapsed_time(e1))
            ms = float(np.median(ts))
            b = 2 * wl.R * wl.M + 24 + 2 * wl.R + (8 * wl.R if ef else 0)
            row = {"workload": "llama-3.2-1b", "R": wl.R, "M": wl.M, "N": wl.N,
                   "variant": "compressed", "codec": names[kind], "error_feedback": ef,
                   "wire_bytes_per_param_per_rank": round(wire[kind], 4),
                   "ms": round(ms, 4), "params_per_s": wl.N / (ms / 1e3), "bytes_per_param": b,
                   "GB_s": round(b * wl.N / (ms / 1e3) / 1e9, 1),
                   "frac_of_measured_peak": round(b * wl.N / (ms / 1e3) / 1e9 / peak, 4)}
            rows.append(row)
            print(json.dumps(row), flush=True)
    del ds, res
    torch.cuda.empty_cache()

    # 1-bit Adam after its warm-up on the 1B-shaped workload (shards on the
    # 128-element block grid)
    import dataclasses
    wl = dataclasses.replace(W.llama32_1b(), align=128)
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.fill_state_device()
    ds.fill_grads_device(wl.step)
    w_res = [torch.zeros(wl.N, dtype=torch.float32, device="cuda") for _ in range(wl.R)]
    s_res = torch.zeros(ds.padded, dtype=torch.float32, device="cuda")
    ts, t = [], wl.step
    for k in range(3 + 10):
        flush.fill_(k & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        z.zero_step_onebit(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t, wl.step - 1,
                           w_res, s_res)
        e1.record()
        torch.cuda.synchronize()
        t += 1
        if k >= 3:
            ts.append(e0.elapsed_time(e1))
    ms = float(np.median(ts))
    b = 2 * wl.R * wl.M + 10 * wl.R + 28
    row = {"workload": "llama-3.2-1b", "R": wl.R, "M": wl.M, "N": wl.N, "variant": "onebit",
           "wire_bytes_per_param_per_rank": round(2 * (1 / 8 + 4 / 128), 4),
           "ms": round(ms, 4), "params_per_s": wl.N / (ms / 1e3), "bytes_per_param": b,
           "GB_s": round(b * wl.N / (ms / 1e3) / 1e9, 1),
           "frac_of_measured_peak": round(b * wl.N / (ms / 1e3) / 1e9 / peak, 4)}
    rows.append(row)
    print(json.dumps(row), flush=True)
    del ds, w_res, s_res
    torch.cuda.empty_cache()

    # the step with global-norm clipping on the 1B-shaped workload (clipping
    # active: max_norm far below the gradient norm)
    wl = W.llama32_1b()
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.fill_state_device()
    ds.fill_grads_device(wl.step)
    ts, t = [], wl.step
    for k in range(3 + 10):
        flush.fill_(k & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        ds.step_clipped(t, 1e-3)
        e1.record()
        torch.cuda.synchronize()
        t += 1
        if k >= 3:
            ts.append(e0.elapsed_time(e1))
    ms = float(np.median(ts))
    b = 2 * wl.R * wl.M + 4 + 4 + 24 + 2 * wl.R
    row = {"workload": "llama-3.2-1b", "R": wl.R, "M": wl.M, "N": wl.N, "variant": "clipped",
           "launches": 2, "ms": round(ms, 4),
           "params_per_s": wl.N / (ms / 1e3), "bytes_per_param": b,
           "GB_s": round(b * wl.N / (ms / 1e3) / 1e9, 1),
           "frac_of_measured_peak": round(b * wl.N / (ms / 1e3) / 1e9 / peak, 4)}
    rows.append(row)
    print(json.dumps(row), flush=True)
    del ds
    torch.cuda.empty_cache()

    for R in (2, 4, 8):
        S = 1024
        while S <= 256 * 1024 * 1024:
            measure(W.sweep_point(R, S), f"sweep R={R} S={S}", reps=20, variants=(0,))
            S *= 4

    sampler.mark_stop()
    row = {"clocks": sampler.stop(), "scope": "every GPU row of the table"}
    rows.append(row)
    print(json.dumps(row), flush=True)

    # oracle on 1 core and on all cores, per workload, first 2^22 params
    for name in ("tiny", "gpt2-small", "llama-3.2-1b", "uneven", "large"):
        wl = W.ALL[name]()
        n = min(wl.N, 1 << 22)
        for th in (1, os.cpu_count() or 1):
            ctx = oracle_prepare(wl, n, threads=th)
            tpass = min(oracle_pass(wl, ctx) for _ in range(3))
            row = {"workload": name, "oracle_threads": th, "sample_params": n,
                   "params_per_s": n / tpass,
                   "GB_s": round(wl.bytes_per_param() * n / tpass / 1e9, 2)}
            rows.append(row)
            print(json.dumps(row), flush=True)
    for row in oracle_variant_rows():
        rows.append(row)
        print(json.dumps(row), flush=True)
    return rows


TABLE_VARIANT_STEPS = (
    {"variant": "clipped", "max_norm": 1.0},
    *({"variant": "compressed", "codec": c, "ef": ef}
      for c in ("fp16", "int8", "sign") for ef in (False, True)),
    {"variant": "onebit"},
    {"variant": "zero3"},
)


def oracle_variant_rows(name="llama-3.2-1b", n=1 << 22, reps=3):
    """The oracles of the clipped, compressed, 1-bit Adam and ZeRO-3 steps
    (one core each, as they stand) on the first n params of the workload
    their GPU rows measure; best of reps passes each."""
    from zgen import workloads as W
    wl = W.ALL[name]()
    n = min(wl.N, n)
    ctx = oracle_prepare(wl, n, threads=1)
    out = []
    for opts in TABLE_VARIANT_STEPS:
        tpass = min(oracle_pass(wl, ctx, **opts) for _ in range(reps))
        out.append({"workload": name, "oracle": ORACLE_FN[opts["variant"]], **opts,
                    "oracle_threads": 1, "sample_params": n, "params_per_s": n / tpass})
    return out


# --------------------------------------------------------- checkpoints --

def run_ckpt(args):
    """Sharded checkpoint of the GPT-2- and 1B-shaped workloads' state (14 B
    per param: bf16 param, fp32 master, m, v; one file per rank shard): the
    pause on the step's stream (from the call, which pins the staging buffer,
    to the end of the device-to-host copies) and the time until every shard
    file is fsync'ed and renamed; then a load under the same R and one
    resharded to R' = R/2.  The files go to a temporary directory that is
    removed afterwards."""
    import shutil

    import torch

    import zero_optimizer_step_rs_gb300 as z
    from tests import harness as H
    from zgen import workloads as W

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    base = os.environ.get("TMPDIR") or tempfile.gettempdir()
    for name in ("gpt2-small", "llama-3.2-1b"):
        wl = W.ALL[name]()
        nbytes = 14 * wl.N
        free = shutil.disk_usage(base).free
        if free < 2.5 * nbytes:
            print(json.dumps({"workload": name, "variant": "checkpoint",
                              "skipped": f"{free / 1e9:.1f} GB free under {base}, "
                                         f"need {2.5 * nbytes / 1e9:.1f} GB"}), flush=True)
            continue
        ds = H.DeviceState(wl, staged_scratch=False)
        ds.fill_state_device()
        ds.fill_grads_device(wl.step)
        ds.step(wl.step)
        torch.cuda.synchronize()
        d = tempfile.mkdtemp(prefix="zckpt_", dir=base)
        try:
            rows = {}

            def save(sub):
                """One save: GPU-stream pause from the call to the end of the
                copies (events), host time of the call, seconds until every
                file is durable."""
                os.makedirs(sub)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                e0.record(stream)
                job = z.zero_ckpt_save_async(ds.plan, ds.params[0], ds.W, ds.m, ds.v, wl.step,
                                             ds.hp, sub, n_threads=8)
                t_call = time.perf_counter() - t0
                e1.record(stream)
                e1.synchronize()
                job.wait()
                return e0.elapsed_time(e1), t_call, time.perf_counter() - t0

            def settle():
                # background writeback of earlier files can slow the copies
                # into host memory: let it finish between measurements
                os.sync()
                time.sleep(3)

            settle()
            # the library pins its own staging buffer for the save
            rows["pause_ms"], rows["call_s"], rows["save_s"] = save(os.path.join(d, "save1"))
            rows["copy_ms"] = rows["pause_ms"] - 1e3 * rows["call_s"]
            settle()
            sub = os.path.join(d, "save1")
            t0 = time.perf_counter()
            z.zero_ckpt_load(ds.plan, sub, ds.params, ds.W, ds.m, ds.v)
            rows["load_s"] = time.perf_counter() - t0
            R2 = max(1, wl.R // 2)
            plan2 = z.Plan([int(x) for x in (wl.offsets[1:] - wl.offsets[:-1])], R2, wl.M, wl.stage,
                           wl.align)
            W2, m2, v2 = (torch.empty(plan2.c.padded, dtype=torch.float32, device="cuda")
                          for _ in range(3))
            P2 = [torch.empty(plan2.c.N, dtype=torch.bfloat16, device="cuda") for _ in range(R2)]
            t0 = time.perf_counter()
            z.zero_ckpt_load(plan2, sub, P2, W2, m2, v2)
            rows["reshard_load_s"] = time.perf_counter() - t0
            same = torch.equal(W2[:wl.N].view(torch.int32), ds.W[:wl.N].view(torch.int32))
            del W2, m2, v2, P2
        finally:
            shutil.rmtree(d, ignore_errors=True)
        row = {"workload": name, "variant": "checkpoint", "R": wl.R, "N": wl.N,
               "bytes": nbytes, "stream_pause_ms": round(rows["pause_ms"], 2),
               "staging_alloc_and_enqueue_s": round(rows["call_s"], 3),
               "copy_ms": round(rows["copy_ms"], 2),
               "copy_GB_s": round(nbytes / (rows["copy_ms"] / 1e3) / 1e9, 1),
               "save_s": round(rows["save_s"], 3), "save_GB_s": round(nbytes / rows["save_s"] / 1e9, 2),
               "load_s": round(rows["load_s"], 3), "load_GB_s": round(nbytes / rows["load_s"] / 1e9, 2),
               "reshard_R": R2, "reshard_load_s": round(rows["reshard_load_s"], 3),
               "reshard_load_GB_s": round(nbytes / rows["reshard_load_s"] / 1e9, 2),
               "reshard_master_bit_identical": bool(same), "dir": base}
        print(json.dumps(row), flush=True)
        del ds
        torch.cuda.empty_cache()


# ------------------------------------------------------- reference arm --

def run_reference(args):
    """The oracle as it stands, on the host cores: each step is one pass of
    the oracle of the measured step (oracle_dp_step_mt for the default
    fused step) over a bounded sample (the first 2^22 params) of the
    workload."""
    from zgen import workloads as W
    wl = W.by_name(args.workload)
    if getattr(args, "scale", 0):
        wl = wl.scaled(args.scale)
    t0 = time.time()
    sample = min(wl.N, 1 << 22)
    ctx = oracle_prepare(wl, sample)
    opts = oracle_step_opts(args)
    for _ in range(args.warmup):
        oracle_pass(wl, ctx, **opts)
    per_step = [oracle_pass(wl, ctx, **opts) for _ in range(args.steps)]
    cores = oracle_threads(ctx, args.variant)
    mean_s = sum(per_step) / len(per_step)
    value = sample / mean_s
    desc = (f"{ORACLE_FN[args.variant]} over the first {sample:,} params of the workload "
            f"(same R, M, distributions), {cores} thread(s), one pass per step")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * mean_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator; shapes of the named parameter set)",
        "config": {"workload": wl.name, "N": wl.N, "R": wl.R, "M": wl.M, "stage": wl.stage,
                   "step": wl.step, "variant": args.variant,
                   **({"max_norm": args.max_norm} if args.variant == "clipped" else {}),
                   **({"codec": args.codec, "error_feedback": args.ef}
                      if args.variant == "compressed" else {}),
                   **({"freeze_step": max(1, wl.step - 1), "align": 128}
                      if args.variant == "onebit" else {}),
                   "sample_params_per_step": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(time.time() - t0, 1),
    }


def render_table(rows, peak_gbs):
    """The rows of `bench.py --table` (parsed JSON lines) as the markdown
    tables of the all-workload profile; the commentary under them is
    written by hand."""
    out = []
    P = out.append

    def gp(x):                                    # params/s as G params/s
        return f"{x / 1e9:.2f}"

    def t_str(ms):
        return f"{ms * 1e3:.2f} µs" if ms < 0.1 else f"{ms:.4f} ms"

    def clean(r):                                 # the clean-L2 columns
        if "ms_clean_l2" not in r:
            return "– | –"
        return f"{t_str(r['ms_clean_l2'])} | {r['frac_clean_l2']:.3f}"

    def l2_label(r, resident="warm"):
        l2 = r.get("l2", "")
        return "cold" if l2.startswith("cold") else resident if l2.startswith("warm") else "> L2"

    P("# All workloads; the clipped, compressed, 1-bit Adam and ZeRO-3 steps; the flat sweep; "
      "the oracle on 1 and 16 host cores")
    P("")
    P("Commands (one GB300, one call; the tables are rendered from the JSON lines, the reading at "
      "the end is written by hand):")
    P("")
    P("    python bench.py --table > table.jsonl")
    P("    python bench.py --render-table table.jsonl")
    P("")
    P("Timing:")
    P("")
    P("- Workloads larger than L2: a 256 MB write evicts L2 before every timed launch; median of 20 "
      "reps (10 for")
    P("  the ~4B workload, ZeRO-3, the compressed codecs, 1-bit Adam and the clipped step). That "
      "write leaves L2")
    P("  full of dirty lines, and the timed launch writes them back as its own data evicts them: up "
      "to ~19 us at")
    P("  the copy peak, noise at the 1B size but most of the gap at a few million params. The "
      "**clean L2**")
    P("  columns time the same launches after the write and then a 256 MB read of another buffer, "
      "which leaves")
    P("  L2 holding clean, unrelated lines: the kernel's own cost from a cold cache.")
    P("- Workloads that fit in L2 (tiny, small sweep points), every launch enqueued behind a sleep "
      "kernel so the")
    P("  events time the GPU, not the host's launch calls: **cold** = a flush, then an event pair "
      "around one")
    P("  launch, mean of 200 (the event timer ticks about every 2 µs and an empty pair spans "
      "~2.1 µs);")
    P("  **warm** = 200 launches back to back between one event pair, mean per launch.")
    P("")
    P(f"Peak: {peak_gbs:,.1f} GB/s, the pool's measured copy bandwidth (`MEASURED_PEAKS.json`). "
      "Bytes per parameter are algorithmic:")
    P("")
    for line in ("- fused: 2RM + 24 + 2R;",
                 "- staged (scratch, or the reduced gradient in gradient buffers 0 and 1): "
                 "2RM + 36 + 2R;",
                 "- ZeRO-3 step: 2RM + 26;",
                 "- ZeRO-3 gather: 4 per element (2 read, 2 written);",
                 "- ZeRO-3 unit reduce-scatter: 2RM + 4; shard update: 30;",
                 "- compressed: 2RM + 24 + 2R, plus 8R with error feedback;",
                 "- clipped: 2RM + 32 + 2R;",
                 "- 1-bit Adam: 2RM + 10R + 28."):
        P(line)
    P("")
    clk = next((r["clocks"] for r in rows if "clocks" in r), None)
    if clk:
        P(f"SM clock over the GPU rows (NVML every 5 ms): median {clk['sm_mhz']:.0f} MHz of "
          f"{clk['sm_max_mhz']:.0f}, throttle reasons: {', '.join(clk['reasons']) or 'none'} "
          f"({clk['samples']} samples).")
        P("")
    P("## ZeRO-1/2 step, every workload")
    P("")
    P("| workload | R | M | N | variant | L2 | B/param | µs or ms | G params/s | GB/s | "
      "of measured peak | clean L2: µs or ms | of peak |")
    P("|---|---:|---:|---:|---|---|---:|---:|---:|---:|---:|---:|---:|")
    for r in rows:
        v = str(r.get("variant", ""))
        if v not in ("fused", "staged") and not v.startswith("staged, reduced"):
            continue
        if str(r["workload"]).startswith("sweep"):
            continue
        vs = "staged, gradient in buffers 0/1" if v.startswith("staged, reduced") else v
        P(f"| {r['workload']} | {r['R']} | {r['M']} | {r['N']:,} | {vs} | {l2_label(r)} | "
          f"{r['bytes_per_param']} | {t_str(r['ms'])} | {gp(r['params_per_s'])} | {r['GB_s']} | "
          f"{r['frac_of_measured_peak']:.3f} | {clean(r)} |")
    P("")
    P("## ZeRO-3: step (cast into each rank's own shard, no all-gather)")
    P("")
    P("| workload | R | M | N | B/param | ms | G params/s | GB/s | of measured peak |")
    P("|---|---:|---:|---:|---:|---:|---:|---:|---:|")
    for r in rows:
        if r.get("variant") == "zero3_step":
            P(f"| {r['workload']} | {r['R']} | {r['M']} | {r['N']:,} | {r['bytes_per_param']} | "
              f"{r['ms']:.4f} | {gp(r['params_per_s'])} | {r['GB_s']} | "
              f"{r['frac_of_measured_peak']:.3f} |")
    P("")
    P("## ZeRO-3: all-gather of the whole Llama-3.2-1B-shaped model, by unit size "
      "(one destination)")
    P("")
    P("| unit | launches | ms for the whole model | GB/s | of measured peak |")
    P("|---|---:|---:|---:|---:|")
    for r in rows:
        if r.get("variant") == "zero3_gather":
            P(f"| {r['unit']} | {r['launches']} | {r['ms']:.4f} | {r['GB_s']} | "
              f"{r['frac_of_measured_peak']:.3f} |")
    P("")
    P("## ZeRO-3 backward unit by unit (FSDP) on the Llama-3.2-1B-shaped workload: one "
      "reduce-scatter per layer, last layer first, then the shard update")
    P("")
    P("The fp32 gradient shard is written by the reduce-scatters and read by the update: "
      "8 B/param more than the whole-step kernel.")
    P("")
    part_hdr = ("| {} | launches | B/param | ms | G params/s | GB/s | of measured peak |",
                "|---|---:|---:|---:|---:|---:|---:|")
    P(part_hdr[0].format("part"))
    P(part_hdr[1])
    for r in rows:
        if r.get("variant") == "zero3_units":
            P(f"| {r['part']} | {r['launches']} | {r['bytes_per_param']} | {r['ms']:.4f} | "
              f"{gp(r['params_per_s'])} | {r['GB_s']} | {r['frac_of_measured_peak']:.3f} |")
    P("")
    P("With each layer's parameters all-gathered again before its reduce-scatter (FSDP "
      "materialises a unit for its backward) into one of two transient buffers: "
      "4 + 2RM + 4 B/param.")
    P("")
    P(part_hdr[0].format("schedule"))
    P(part_hdr[1])
    for r in rows:
        if r.get("variant") == "zero3_backward":
            P(f"| {r['part']} | {r['launches']} | {r['bytes_per_param']} | {r['ms']:.4f} | "
              f"{gp(r['params_per_s'])} | {r['GB_s']} | {r['frac_of_measured_peak']:.3f} |")
    P("")
    P("## Compressed reduce-scatter on the Llama-3.2-1B-shaped workload (R=8, M=1)")
    P("")
    P("Error feedback reads and writes one fp32 residual per rank: +8R B/param. The compressed "
      "message stays in registers; wire bytes are what a rank would send.")
    P("")
    P("| codec | error feedback | wire B/param per rank | B/param (HBM) | ms | G params/s | GB/s | "
      "of measured peak |")
    P("|---|---|---:|---:|---:|---:|---:|---:|")
    for r in rows:
        if r.get("variant") == "compressed" and "ms" in r:
            P(f"| {r['codec']} | {'yes' if r['error_feedback'] else 'no'} | "
              f"{r['wire_bytes_per_param_per_rank']} | {r['bytes_per_param']} | {r['ms']:.4f} | "
              f"{gp(r['params_per_s'])} | {r['GB_s']} | {r['frac_of_measured_peak']:.3f} |")
    P("")
    P("## Clipped and 1-bit Adam steps on the Llama-3.2-1B-shaped workload (R=8, M=1)")
    P("")
    P("Clipped: 2RM + 8 + 24 + 2R B/param (the fp32 gradient stash written and read back), "
      "clipping active, two launches (the norm pass with the tree up to one partial per group "
      "of tiles; the update, every block finishing the tree first). 1-bit Adam after its "
      "warm-up: 2RM + 10R + 28 B/param, shards on the 128-element grid.")
    P("")
    P("| step | launches | B/param | ms | G params/s | GB/s | of measured peak |")
    P("|---|---:|---:|---:|---:|---:|---:|")
    for r in rows:
        if r.get("variant") in ("onebit", "clipped") and "ms" in r:
            P(f"| {r['variant']} | {r.get('launches', 1)} | {r['bytes_per_param']} | "
              f"{r['ms']:.4f} | {gp(r['params_per_s'])} | {r['GB_s']} | "
              f"{r['frac_of_measured_peak']:.3f} |")
    P("")
    P("## Flat sweep (fused): fp32 master shard of 4 KB ... 1 GB (S = 1 Ki ... 256 Mi elements), "
      "N = R*S")
    P("")
    P("| R | S | N | L2 | µs or ms | G params/s | GB/s | of measured peak | clean L2: µs or ms | "
      "of peak |")
    P("|---:|---:|---:|---|---:|---:|---:|---:|---:|---:|")
    for r in rows:
        if str(r.get("workload", "")).startswith("sweep"):
            S = int(r["workload"].split("S=")[1])
            P(f"| {r['R']} | {S:,} | {r['N']:,} | {l2_label(r, 'warm (L2-resident)')} | "
              f"{t_str(r['ms'])} | {gp(r['params_per_s'])} | {r['GB_s']} | "
              f"{r['frac_of_measured_peak']:.3f} | {clean(r)} |")
    P("")
    P("## Oracle (unchanged) on the box's host cores, first 2^22 params of each workload, "
      "best of 3")
    P("")
    P("`oracle_dp_step_mt` for the plain step, on 1 and 16 threads:")
    P("")
    P("| workload | threads | M params/s | GB/s (same byte model) |")
    P("|---|---:|---:|---:|")
    for r in rows:
        if "oracle_threads" in r and "oracle" not in r:
            P(f"| {r['workload']} | {r['oracle_threads']} | {r['params_per_s'] / 1e6:.1f} | "
              f"{r['GB_s']} |")
    P("")
    P("The oracle of each step variant on the Llama-3.2-1B-shaped workload (one core: these "
      "functions are single-threaded), beside the GPU rows above:")
    P("")
    P("| oracle | variant | M params/s |")
    P("|---|---|---:|")
    for r in rows:
        if "oracle" in r and "oracle_threads" in r:
            v = r["variant"]
            if v == "compressed":
                v = f"compressed {r['codec']}{' + error feedback' if r['ef'] else ''}"
            P(f"| `{r['oracle']}` | {v} | {r['params_per_s'] / 1e6:.1f} |")
    return "\n".join(out) + "\n"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama-3.2-1b")
    ap.add_argument("--variant", choices=["fused", "staged", "staged_grads", "clipped", "tma",
                                          "zero3", "zero3_gather_units", "compressed", "onebit"],
                    default="fused",
                    help="staged_grads: the staged step on a ZeRO-2 plan without scratch; "
                         "zero3_gather_units: the ZeRO-3 all-gather of every tensor, one launch")
    ap.add_argument("--scale", type=int, default=0,
                    help="scale the workload's tensors down to about this many params")
    ap.add_argument("--codec", choices=["fp16", "int8", "sign"], default="int8",
                    help="codec for --variant compressed")
    ap.add_argument("--ef", action="store_true", help="error feedback for --variant compressed")
    ap.add_argument("--max-norm", type=float, default=1.0,
                    help="global-norm clip threshold for --variant clipped")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--table", action="store_true",
                    help="every workload and the flat sweep, one JSON line each")
    ap.add_argument("--ckpt", action="store_true",
                    help="checkpoint save / load / reshard timings of two workloads")
    ap.add_argument("--render-table", metavar="JSONL",
                    help="print the JSON lines of a --table run as markdown tables")
    args = ap.parse_args()
    if args.render_table:
        with open(args.render_table) as f:
            rows = [json.loads(line) for line in f if line.startswith("{")]
        peak = float((measured_peaks() or {}).get("hbm_gbs", 6800.0))
        sys.stdout.write(render_table(rows, peak))
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local_rank = _env_int("LOCAL_RANK", 0)

    if args.table:
        run_table(args)
        return 0
    if args.ckpt:
        run_ckpt(args)
        return 0

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
