"""Host-side checks of the C-ABI library (no GPU needed).

The library loads, exports every entry point include/zero_step.h declares,
its plan reproduces the pages' accounting, and every argument error is
returned synchronously before anything touches a GPU (so these calls are
safe without one: the library returns before any CUDA call).
"""
import os
import re

import pytest
import torch

import zero_optimizer_step_rs_gb300 as z
from zero_optimizer_step_rs_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_rs_gb300 import build
    build.build()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "zero_step.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(zero[0-9]*_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert len(names) >= 10
    L = B.lib()
    for n in names:
        assert hasattr(L, n), n
    assert sorted(B.EXPORTED) == names


def test_version_and_status_strings():
    assert z.zero_abi_version() == 1
    for code in range(-8, 1):
        assert z.zero_status_string(code) != "unknown status"
    assert z.zero_status_string(-99) == "unknown status"


@pytest.mark.parametrize("numels,R,M,align,S,padded", [
    ([65536], 4, 2, 0, 16384, 65536),
    ([100_000_007], 7, 4, 64, 14_285_760, 100_000_320),
    ([5], 4, 1, 64, 64, 256),
    ([3, 4, 5], 3, 1, 4, 4, 12),
    ([], 2, 1, 0, 0, 0),
])
def test_plan_layout(numels, R, M, align, S, padded):
    p = z.Plan(numels, R, M, 2, align)
    assert (p.N, p.S, p.padded, p.R, p.M) == (sum(numels), S, padded, R, M)
    assert p.tensor_offsets()[-1] == sum(numels)
    assert p.scratch_bytes_staged == 4 * padded


def test_plan_owner():
    p = z.Plan([1000], 3, 1, 1, 4)            # S = roundup(334, 4) = 336
    assert p.S == 336
    assert [p.owner(i) for i in (0, 335, 336, 671, 672, 999)] == [0, 0, 1, 1, 2, 2]
    assert p.owner(-1) == -1 and p.owner(1000) == -1


def test_plan_accounting_matches_pages_exercise_1():
    # CS324 Lecture 9 notes, exercise 1: 7B params, 8 cards, 2+2+12 bytes:
    # DP 112, ZeRO-1 38.5, ZeRO-2 26.25, ZeRO-3 14 GB (S divides exactly)
    p = z.Plan([7_000_000_000], 8, 1, 1)
    got = [p.bytes_per_rank_dp, p.bytes_per_rank_z1, p.bytes_per_rank_z2, p.bytes_per_rank_z3]
    assert [g / 1e9 for g in got] == [112.0, 38.5, 26.25, 14.0]
    assert p.bytes_per_rank == p.bytes_per_rank_z1


def test_plan_accounting_matches_pages_summary_item_5():
    # same notes, summary item 5: 7.5B params on 64 cards: 120 / 31.4 / 16.6 / 1.88 GB
    p = z.Plan([7_500_000_000], 64, 1, 2)
    got = [p.bytes_per_rank_dp, p.bytes_per_rank_z1, p.bytes_per_rank_z2, p.bytes_per_rank_z3]
    assert [round(got[0] / 1e9, 1), round(got[1] / 1e9, 1), round(got[2] / 1e9, 1),
            round(got[3] / 1e9, 2)] == [120.0, 31.4, 16.6, 1.88]
    assert p.bytes_per_rank == p.bytes_per_rank_z2


@pytest.mark.parametrize("args,code", [
    (([10], 0, 1, 1, 0), B.ZERO_ERR_INVALID_ARG),
    (([10], 65, 1, 1, 0), B.ZERO_ERR_INVALID_ARG),
    (([10], 4, 0, 1, 0), B.ZERO_ERR_INVALID_ARG),
    (([10], 16, 17, 1, 0), B.ZERO_ERR_INVALID_ARG),    # R*M > 256
    (([10], 4, 1, 3, 0), B.ZERO_ERR_INVALID_ARG),
    (([10], 4, 1, 1, 6), B.ZERO_ERR_INVALID_ARG),      # alignment not a multiple of 4
    (([10], 4, 1, 1, -4), B.ZERO_ERR_INVALID_ARG),
    (([10, -1], 4, 1, 1, 0), B.ZERO_ERR_INVALID_ARG),
    (([2**62, 2**62], 4, 1, 1, 0), B.ZERO_ERR_SIZE),
])
def test_plan_create_errors(args, code):
    with pytest.raises(B.ZeroError) as e:
        z.Plan(*args)
    assert e.value.code == code


# ---------------------------------------------------- step argument errors --
# Fake, 256-byte-aligned, non-overlapping addresses: every case below fails
# validation, which happens on the host before any CUDA call.

BASE = 1 << 40


def fake_bufs(plan, gap=1 << 30):
    # fake addresses are only ever handed to the library where no GPU is
    # visible: a call that got past validation by mistake then fails with
    # ZERO_ERR_CUDA instead of touching memory
    if torch.cuda.is_available():
        pytest.skip("fake device addresses are used only on machines without a GPU")
    c = plan.c
    addr = [BASE + k * gap for k in range(c.R * c.M + c.R + 5)]
    grads = addr[:c.R * c.M]
    params = addr[c.R * c.M:c.R * c.M + c.R]
    Wp, mp, vp, scr, st = addr[c.R * c.M + c.R:]
    return grads, Wp, mp, vp, params, scr, st


def call_step(plan, grads, Wp, mp, vp, params, hp=None, step=1, variant=0, scratch=None,
              sbytes=0, flags=0, status=None):
    import ctypes
    L = B.lib()
    ga = B._ptrs(grads)
    pa = B._ptrs(params)
    hp = hp if hp is not None else z.hparams()
    return L.zero_step(plan.ptr, ctypes.addressof(ga), Wp, mp, vp, ctypes.addressof(pa),
                       ctypes.byref(hp), step, variant, scratch, sbytes, flags, status, None)


@pytest.fixture
def plan():
    return z.Plan([100_000], 4, 2, 2)


def test_step_null_and_align(plan):
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    assert call_step(plan, [0] + g[1:], Wp, mp, vp, P) == B.ZERO_ERR_NULL
    assert call_step(plan, g, 0, mp, vp, P) == B.ZERO_ERR_NULL
    assert call_step(plan, g, Wp, mp, vp, P[:-1] + [0]) == B.ZERO_ERR_NULL
    assert call_step(plan, [g[0] + 2] + g[1:], Wp, mp, vp, P) == B.ZERO_ERR_ALIGN
    assert call_step(plan, g, Wp + 8, mp, vp, P) == B.ZERO_ERR_ALIGN
    assert call_step(plan, g, Wp, mp, vp, [P[0] + 4] + P[1:]) == B.ZERO_ERR_ALIGN


def test_step_invalid_args(plan):
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    assert call_step(plan, g, Wp, mp, vp, P, step=0) == B.ZERO_ERR_INVALID_ARG
    assert call_step(plan, g, Wp, mp, vp, P, variant=3) == B.ZERO_ERR_INVALID_ARG
    assert call_step(plan, g, Wp, mp, vp, P, flags=4) == B.ZERO_ERR_INVALID_ARG
    assert call_step(plan, g, Wp, mp, vp, P, flags=1) == B.ZERO_ERR_NULL     # no status word
    for bad in (dict(beta1=1.0), dict(beta2=1.5), dict(beta1=-0.1), dict(eps=-1.0),
                dict(lr=float("nan")), dict(weight_decay=float("inf"))):
        hp = z.hparams(**bad)
        assert call_step(plan, g, Wp, mp, vp, P, hp=hp) == B.ZERO_ERR_INVALID_ARG, bad


def test_step_overlap(plan):
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    assert call_step(plan, g, Wp, Wp, vp, P) == B.ZERO_ERR_OVERLAP            # master == m
    assert call_step(plan, g, Wp, mp, vp, [g[0]] + P[1:]) == B.ZERO_ERR_OVERLAP
    assert call_step(plan, g, Wp, mp, vp, [P[1]] + P[1:]) == B.ZERO_ERR_OVERLAP
    # W's range is 4*padded bytes: m starting inside it overlaps
    assert call_step(plan, g, Wp, Wp + 4 * plan.padded - 16, vp, P) == B.ZERO_ERR_OVERLAP
    assert call_step(plan, g, Wp, mp, vp, P, status=Wp) == B.ZERO_ERR_OVERLAP


def test_step_staged_scratch(plan):
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    need = plan.scratch_bytes_staged
    assert call_step(plan, g, Wp, mp, vp, P, variant=1, scratch=scr,
                     sbytes=need - 4) == B.ZERO_ERR_SIZE
    assert call_step(plan, g, Wp, mp, vp, P, variant=1, scratch=Wp,
                     sbytes=need) == B.ZERO_ERR_OVERLAP
    # ZeRO-1 keeps its gradients: the staged step needs scratch
    z1 = z.Plan([100_000], 4, 2, 1)
    assert call_step(z1, g, Wp, mp, vp, P, variant=1, scratch=None) == B.ZERO_ERR_NULL
    # one gradient buffer cannot hold the fp32 result: scratch needed
    one = z.Plan([100_000], 1, 1, 2)
    g1, W1, m1, v1, P1, _, _ = fake_bufs(one)
    assert call_step(one, g1, W1, m1, v1, P1, variant=1, scratch=None) == B.ZERO_ERR_NULL


def test_staged_zero2_without_scratch_writes_two_gradient_buffers(plan):
    """ZeRO-2 without scratch: gradient buffers 0 and 1 become outputs (the
    reduced gradient's low and high halves), so they may alias nothing; the
    other gradient buffers stay read-only inputs that may alias each other."""
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    assert call_step(plan, [g[0], g[0]] + g[2:], Wp, mp, vp, P, variant=1) == B.ZERO_ERR_OVERLAP
    assert call_step(plan, g[:2] + [g[1]] + g[3:], Wp, mp, vp, P,
                     variant=1) == B.ZERO_ERR_OVERLAP
    assert call_step(plan, g[:3] + [g[0] + 64] + g[4:], Wp, mp, vp, P,
                     variant=1) == B.ZERO_ERR_OVERLAP
    # inputs 2.. may alias one another; the call then gets past validation and
    # fails at the launch on a machine without a GPU
    assert call_step(plan, g[:2] + [g[2]] * 6, Wp, mp, vp, P, variant=1) == B.ZERO_ERR_CUDA


def test_staged_entry_errors(plan):
    import ctypes
    L = B.lib()
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    ga, pa = B._ptrs(g), B._ptrs(P)
    assert L.zero_rs_avg(plan.ptr, ctypes.addressof(ga), None, 0, None, None) == B.ZERO_ERR_NULL
    assert L.zero_rs_avg(plan.ptr, ctypes.addressof(ga), g[0], 0, None, None) == B.ZERO_ERR_OVERLAP
    hp = z.hparams()
    assert L.zero_adamw_shard(plan.ptr, scr, Wp, mp, vp, ctypes.byref(hp), 0,
                              None) == B.ZERO_ERR_INVALID_ARG
    assert L.zero_adamw_shard(plan.ptr, Wp, Wp, mp, vp, ctypes.byref(hp), 1,
                              None) == B.ZERO_ERR_OVERLAP
    assert L.zero_ag_cast(plan.ptr, Wp + 4, ctypes.addressof(pa), None) == B.ZERO_ERR_ALIGN
    assert L.zero_ag_cast(None, Wp, ctypes.addressof(pa), None) == B.ZERO_ERR_NULL


def test_step_host_errors(plan):
    import ctypes
    L = B.lib()
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    host = [BASE * 2 + k * 4096 for k in range(len(g))]
    ha, da, pa = B._ptrs(host), B._ptrs(g), B._ptrs(P)
    hp = z.hparams()
    assert L.zero_step_host(plan.ptr, ctypes.addressof(ha), ctypes.addressof(da), Wp, mp, vp,
                            ctypes.addressof(pa), None, ctypes.byref(hp), 1, 0, None,
                            None) == B.ZERO_ERR_NULL
    dup = B._ptrs([g[0]] * len(g))                 # copies would overwrite each other
    assert L.zero_step_host(plan.ptr, ctypes.addressof(ha), ctypes.addressof(dup), Wp, mp, vp,
                            ctypes.addressof(pa), BASE * 3, ctypes.byref(hp), 1, 0, None,
                            None) == B.ZERO_ERR_OVERLAP


def test_binding_rejects_host_tensors_for_device_arguments():
    p = z.Plan([1000], 2, 1, 1)
    cpu = [torch.zeros(1000, dtype=torch.bfloat16) for _ in range(2)]
    st = [torch.zeros(p.padded, dtype=torch.float32) for _ in range(3)]
    with pytest.raises(ValueError):
        z.zero_step(p, cpu, *st, cpu, z.hparams(), 1, stream=0)
    with pytest.raises(TypeError):
        z.zero_step(p, [t.float() for t in cpu], *st, cpu, z.hparams(), 1, stream=0)


def test_clip_scratch_bytes_layout():
    # fp32 gradient stash (4 * padded, rounded to 256 bytes) + one fp32 partial
    # per group of tiles (2048 elements a tile; a power-of-two number of tiles
    # a group, the least that leaves at most 8192 groups), rounded to 256
    # bytes; nothing else: no counters, no control record
    def r256(x):
        return -(-x // 256) * 256
    p = z.Plan([65536], 4, 2, 1)                     # 32 tiles, a group each
    assert z.zero_clip_scratch_bytes(p) == 4 * 65536 + 256
    p = z.Plan([1_235_814_400], 8, 1, 2)             # 603,425 tiles: 128 a group
    assert 1_235_814_400 == 603_425 * 2048
    assert -(-603_425 // 64) > 8192 >= -(-603_425 // 128)
    assert z.zero_clip_scratch_bytes(p) == 4 * p.padded + r256(4 * 4_715)
    p = z.Plan([200], 2, 1, 2)                        # one tile
    assert z.zero_clip_scratch_bytes(p) == 4 * p.padded + 256
    p = z.Plan([8192 * 2048 + 1], 1, 1, 2)           # 8193 tiles: 2 a group
    assert z.zero_clip_scratch_bytes(p) == 4 * p.padded + r256(4 * 4097)


def test_clipped_step_argument_errors():
    import ctypes
    plan = z.Plan([100_000], 4, 2, 2)
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    ga, pa = B._ptrs(g), B._ptrs(P)
    hp = z.hparams()
    need = z.zero_clip_scratch_bytes(plan)
    L = B.lib()

    def call(max_norm=1.0, scratch=scr, sbytes=need, flags=0, status=None, sumsq=None):
        return L.zero_step_clipped(plan.ptr, ctypes.addressof(ga), Wp, mp, vp,
                                   ctypes.addressof(pa), ctypes.byref(hp), 1, max_norm, scratch,
                                   sbytes, flags, status, sumsq, None)
    assert call(max_norm=0.0) == B.ZERO_ERR_INVALID_ARG
    assert call(max_norm=float("inf")) == B.ZERO_ERR_INVALID_ARG
    assert call(max_norm=float("nan")) == B.ZERO_ERR_INVALID_ARG
    assert call(sbytes=need - 1) == B.ZERO_ERR_SIZE
    assert call(scratch=None) == B.ZERO_ERR_NULL
    assert call(scratch=Wp) == B.ZERO_ERR_OVERLAP
    assert call(flags=8) == B.ZERO_ERR_INVALID_ARG
    assert call(flags=B.ZERO_FLAG_CHECK_FINITE) == B.ZERO_ERR_NULL
    assert call(sumsq=st + 4) == B.ZERO_ERR_ALIGN


def test_tma_variant_argument_errors(plan):
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    # debug flag needs the TMA variant and a status word
    assert call_step(plan, g, Wp, mp, vp, P, variant=0,
                     flags=B.ZERO_FLAG_DEBUG_EXPIRE_WAITS, status=st) == B.ZERO_ERR_INVALID_ARG
    assert call_step(plan, g, Wp, mp, vp, P, variant=2,
                     flags=B.ZERO_FLAG_DEBUG_EXPIRE_WAITS) == B.ZERO_ERR_NULL
    big = z.Plan([1000], 16, 2, 2)                     # R*M = 32 > 16
    g2, Wp2, mp2, vp2, P2, _, _ = fake_bufs(big)
    assert call_step(big, g2, Wp2, mp2, vp2, P2, variant=2) == B.ZERO_ERR_INVALID_ARG


def test_onebit_argument_errors():
    import ctypes
    plan = z.Plan([100_000], 4, 2, 2, 128)
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    E = [BASE + (1 << 36) + k * (1 << 30) for k in range(plan.R)]
    L = B.lib()

    def call(pl=plan, step=3, freeze=2, worker=E, server=scr, hp=None):
        ga, pa = B._ptrs(g), B._ptrs(P)
        ea = B._ptrs(worker) if worker is not None else None
        hp = hp if hp is not None else z.hparams()
        return L.zero_step_onebit(pl.ptr, ctypes.addressof(ga), Wp, mp, vp,
                                  ctypes.addressof(pa), ctypes.byref(hp), step, freeze,
                                  ctypes.addressof(ea) if ea is not None else None, server, None)
    assert call(freeze=0) == B.ZERO_ERR_INVALID_ARG
    assert call(step=0) == B.ZERO_ERR_INVALID_ARG
    assert call(hp=z.hparams(beta2=1.0)) == B.ZERO_ERR_INVALID_ARG
    # S = 25,024 with the default 64-element alignment: not a multiple of 128
    assert plan.S % 128 == 0
    assert call(pl=z.Plan([100_000], 4, 2, 2)) == B.ZERO_ERR_INVALID_ARG
    assert call(worker=None) == B.ZERO_ERR_NULL
    assert call(server=None) == B.ZERO_ERR_NULL
    assert call(server=scr + 8) == B.ZERO_ERR_ALIGN
    assert call(worker=E[:-1] + [0]) == B.ZERO_ERR_NULL
    assert call(worker=[E[0] + 4] + E[1:]) == B.ZERO_ERR_ALIGN
    # overlaps are checked before the first launch
    assert call(server=Wp) == B.ZERO_ERR_OVERLAP
    assert call(worker=[g[0]] + E[1:]) == B.ZERO_ERR_OVERLAP
    assert call(worker=[E[0], E[0]] + E[2:]) == B.ZERO_ERR_OVERLAP
    assert call(worker=[P[1]] + E[1:]) == B.ZERO_ERR_OVERLAP


def test_committed_fused_traffic_matches_the_fused_source():
    """profiles/traffic.json holds the ncu DRAM bytes of k_fused; it is only
    valid for the source it was captured on (zero_step.cu up to the end of
    the fused path).  Any edit there needs a new capture."""
    import json
    import os
    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    rec = json.load(open(os.path.join(root, "profiles", "traffic.json")))
    assert rec["source_sha256_16"] == bench.kernel_source_hash()


def test_zero3_unit_entry_argument_errors():
    import ctypes
    plan = z.Plan([100_000], 4, 2, 2)
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    L = B.lib()
    hp = z.hparams()

    def rs(lo=10, hi=5000, grads=g, gs=scr, flags=0, status=None):
        ga = B._ptrs(grads) if grads is not None else None
        return L.zero3_rs_unit(plan.ptr, ctypes.addressof(ga) if ga is not None else None, lo, hi,
                               gs, flags, status, None)
    assert rs(lo=-1) == B.ZERO_ERR_INVALID_ARG
    assert rs(lo=6000, hi=5000) == B.ZERO_ERR_INVALID_ARG
    assert rs(hi=100_001) == B.ZERO_ERR_INVALID_ARG
    assert rs(flags=2) == B.ZERO_ERR_INVALID_ARG
    assert rs(flags=B.ZERO_FLAG_CHECK_FINITE) == B.ZERO_ERR_NULL
    assert rs(lo=7, hi=7, grads=None, gs=None) == B.ZERO_OK          # empty unit: nothing to do
    assert rs(grads=None) == B.ZERO_ERR_NULL
    assert rs(grads=g[:-1] + [0]) == B.ZERO_ERR_NULL
    assert rs(grads=[g[0] + 2] + g[1:]) == B.ZERO_ERR_ALIGN
    assert rs(gs=scr + 4) == B.ZERO_ERR_ALIGN
    assert rs(gs=g[3]) == B.ZERO_ERR_OVERLAP
    assert rs(status=scr + 64) == B.ZERO_ERR_OVERLAP

    def upd(gs=scr, W=Wp, m=mp, v=vp, ps=P[0], step=1):
        return L.zero3_update(plan.ptr, gs, W, m, v, ps, ctypes.byref(hp), step, None)
    assert upd(step=0) == B.ZERO_ERR_INVALID_ARG
    assert upd(gs=None) == B.ZERO_ERR_NULL
    assert upd(gs=Wp) == B.ZERO_ERR_OVERLAP
    assert upd(ps=mp) == B.ZERO_ERR_OVERLAP
    assert upd(ps=P[0] + 2) == B.ZERO_ERR_ALIGN


def test_compressed_step_argument_errors(plan):
    import ctypes
    g, Wp, mp, vp, P, scr, st = fake_bufs(plan)
    E = [BASE + (1 << 36) + k * (1 << 30) for k in range(plan.R)]
    L = B.lib()

    def call(kind=B.ZERO_COMP_INT8, residuals=E, step=1, hp=None, grads=g, W=Wp):
        ga, pa = B._ptrs(grads), B._ptrs(P)
        ea = B._ptrs(residuals) if residuals is not None else None
        hp = hp if hp is not None else z.hparams()
        return L.zero_step_compressed(plan.ptr, ctypes.addressof(ga), W, mp, vp,
                                      ctypes.addressof(pa), ctypes.byref(hp), step, kind,
                                      ctypes.addressof(ea) if ea is not None else None, None)
    assert call(kind=7) == B.ZERO_ERR_INVALID_ARG
    assert call(kind=-1) == B.ZERO_ERR_INVALID_ARG
    assert call(step=0) == B.ZERO_ERR_INVALID_ARG
    assert call(hp=z.hparams(eps=-1.0)) == B.ZERO_ERR_INVALID_ARG
    assert call(grads=[0] + g[1:]) == B.ZERO_ERR_NULL
    assert call(W=0) == B.ZERO_ERR_NULL
    assert call(W=Wp + 8) == B.ZERO_ERR_ALIGN
    assert call(residuals=E[:-1] + [0]) == B.ZERO_ERR_NULL
    assert call(residuals=[E[0] + 4] + E[1:]) == B.ZERO_ERR_ALIGN
    # every residual is an output of N floats: it may overlap no other buffer
    assert call(residuals=[Wp] + E[1:]) == B.ZERO_ERR_OVERLAP
    assert call(residuals=[E[0], E[0]] + E[2:]) == B.ZERO_ERR_OVERLAP
    assert call(residuals=[g[3]] + E[1:]) == B.ZERO_ERR_OVERLAP
    assert call(residuals=[P[0]] + E[1:]) == B.ZERO_ERR_OVERLAP
    # residual 1 starting 16 bytes before residual 0 ends overlaps it; right
    # after its end it does not (the call then fails later, at the first CUDA
    # call, on a machine without a GPU)
    assert call(residuals=[E[0], E[0] + 4 * plan.N - 16] + E[2:]) == B.ZERO_ERR_OVERLAP
    assert call(residuals=[E[0], E[0] + 4 * plan.N] + E[2:]) == B.ZERO_ERR_CUDA


def test_no_alloc_step_refuses_plans_beyond_its_array():
    """The allocation-free staged step holds its scratch in a fixed array of
    ZERO_NOALLOC_MAX_ELEMS floats: a plan one element past it is refused
    with ZERO_ERR_SIZE before anything else is looked at."""
    import ctypes
    L = B.lib()
    cap = B.ZERO_NOALLOC_MAX_ELEMS
    fits = z.Plan([cap], 4, 1, 2)
    over = z.Plan([cap + 1], 4, 1, 2)
    assert fits.padded == cap and over.padded > cap
    hp = z.hparams()
    for pl, want in ((over, B.ZERO_ERR_SIZE), (fits, B.ZERO_ERR_NULL)):
        ga = B._ptrs([0] * (pl.R * pl.M))
        pa = B._ptrs([0] * pl.R)
        got = L.zero_step_staged_noalloc(pl.ptr, ctypes.addressof(ga), None, None, None,
                                         ctypes.addressof(pa), ctypes.byref(hp), 1, 0, None,
                                         None)
        assert got == want, (pl.padded, got)


def test_gather_units_argument_errors():
    """zero3_gather_units validates the whole table before any launch: unit
    bounds, NULL and misaligned destinations, overlapping destinations (and a
    destination over the shards), the table size; a table of empty units is
    a no-op that needs no shard pointer."""
    import ctypes
    L = B.lib()
    pl = z.Plan([10_000], 4, 1, 2)
    U = B.zero_gather_unit
    SH = 0x100000                                   # fake, 16-byte aligned; never dereferenced

    def call(units, n=None, shards=SH):
        arr = (U * max(1, len(units)))(*[U(*u) for u in units])
        return L.zero3_gather_units(pl.ptr, shards, arr, len(units) if n is None else n, None)

    far = 0x10000000
    assert call([], 0) == B.ZERO_OK
    assert call([(0, 10, far)], -1) == B.ZERO_ERR_INVALID_ARG
    assert call([(0, 10, far)], B.ZERO_MAX_GATHER_UNITS + 1) == B.ZERO_ERR_INVALID_ARG
    assert L.zero3_gather_units(pl.ptr, SH, None, 1, None) == B.ZERO_ERR_NULL
    assert call([(5, 4, far)]) == B.ZERO_ERR_INVALID_ARG             # hi < lo
    assert call([(-1, 4, far)]) == B.ZERO_ERR_INVALID_ARG
    assert call([(0, 10_001, far)]) == B.ZERO_ERR_INVALID_ARG        # past N
    assert call([(0, 10, None)]) == B.ZERO_ERR_NULL
    assert call([(0, 10, far + 2)]) == B.ZERO_ERR_ALIGN
    assert call([(0, 10, far), (3, 13, far + 16)]) == B.ZERO_ERR_OVERLAP
    assert call([(0, 10, SH + 64)]) == B.ZERO_ERR_OVERLAP            # writes over the shards
    assert call([(0, 10, far)], shards=None) == B.ZERO_ERR_NULL
    assert call([(0, 10, far)], shards=SH + 8) == B.ZERO_ERR_ALIGN
    assert call([(7, 7, None), (10_000, 10_000, None)], shards=None) == B.ZERO_OK
    with pytest.raises(ValueError):
        z.gather_unit_table([(0, 10, torch.zeros(10, dtype=torch.bfloat16))])  # host tensor


def test_device_status_argument_errors():
    """zero_get_device_status checks its word's pointer before any CUDA call:
    NULL -> ZERO_ERR_NULL, not 4-byte aligned -> ZERO_ERR_ALIGN, and the host
    output is left untouched."""
    import ctypes
    L = B.lib()
    out = ctypes.c_int32(-12345)
    assert L.zero_get_device_status(None, None, ctypes.byref(out)) == B.ZERO_ERR_NULL
    for bad in (0x1001, 0x1002, 0x1003):
        assert L.zero_get_device_status(bad, None, ctypes.byref(out)) == B.ZERO_ERR_ALIGN
    assert out.value == -12345
    with pytest.raises(B.ZeroError) as e:
        z.zero_get_device_status(0x1002, stream=0)
    assert e.value.code == B.ZERO_ERR_ALIGN
    # the status codes the call maps the device bits to have names
    for code in (B.ZERO_ERR_DEVICE_TIMEOUT, B.ZERO_ERR_NONFINITE):
        assert z.zero_status_string(code) != "unknown status"


def test_empty_plan_is_a_no_op_for_every_step_entry_point():
    """A plan with N = 0 has nothing to update: after the plan, hyper-parameter
    and flag checks every step entry point returns ZERO_OK without looking at
    a buffer pointer (NULLs here) and without a CUDA call."""
    import ctypes
    L = B.lib()
    pl = z.Plan([0], 4, 2, 2)
    assert (pl.N, pl.S, pl.padded) == (0, 0, 0)
    hp = ctypes.byref(z.hparams())
    g = B._ptrs([0] * (pl.R * pl.M))
    P = B._ptrs([0] * pl.R)
    ga, pa = ctypes.addressof(g), ctypes.addressof(P)
    host_out = (ctypes.c_uint16 * 8)()
    for variant in (B.ZERO_VARIANT_FUSED, B.ZERO_VARIANT_STAGED):
        assert L.zero_step(pl.ptr, ga, None, None, None, pa, hp, 1, variant, None, 0, 0,
                           None, None) == B.ZERO_OK
    assert L.zero_rs_avg(pl.ptr, ga, None, 0, None, None) == B.ZERO_OK
    assert L.zero_adamw_shard(pl.ptr, None, None, None, None, hp, 1, None) == B.ZERO_OK
    assert L.zero_ag_cast(pl.ptr, None, pa, None) == B.ZERO_OK
    assert L.zero_step_host(pl.ptr, ga, None, None, None, None, pa, host_out, hp, 1, 0, None,
                            None) == B.ZERO_OK
    assert L.zero_step_staged_noalloc(pl.ptr, ga, None, None, None, pa, hp, 1, 0, None,
                                      None) == B.ZERO_OK
    assert L.zero3_step(pl.ptr, ga, None, None, None, None, hp, 1, 0, None, None) == B.ZERO_OK
    assert L.zero3_update(pl.ptr, None, None, None, None, None, hp, 1, None) == B.ZERO_OK
    assert L.zero_step_clipped(pl.ptr, ga, None, None, None, pa, hp, 1, 1.0, None, 0, 0, None,
                               None, None) == B.ZERO_OK
    for kind in (B.ZERO_COMP_FP16, B.ZERO_COMP_INT8, B.ZERO_COMP_SIGN):
        assert L.zero_step_compressed(pl.ptr, ga, None, None, None, pa, hp, 1, kind, None,
                                      None) == B.ZERO_OK
    # the checks before the empty return still hold
    assert L.zero_step(pl.ptr, ga, None, None, None, pa, hp, 0, 0, None, 0, 0, None,
                       None) == B.ZERO_ERR_INVALID_ARG
    assert L.zero_step_clipped(pl.ptr, ga, None, None, None, pa, hp, 1, 0.0, None, 0, 0, None,
                               None, None) == B.ZERO_ERR_INVALID_ARG
    assert L.zero_step_compressed(pl.ptr, ga, None, None, None, pa, hp, 1, 9, None,
                                  None) == B.ZERO_ERR_INVALID_ARG
    assert L.zero_step_host(pl.ptr, None, None, None, None, None, pa, host_out, hp, 1, 0, None,
                            None) == B.ZERO_ERR_NULL


def test_binding_fails_loudly_without_the_library(tmp_path):
    """No fallback: with the shared library absent, the first call through
    the binding raises instead of computing anything another way (checked in
    a child process, so this process keeps its loaded library)."""
    import subprocess
    import sys
    code = ("import zero_optimizer_step_rs_gb300.binding as B\n"
            f"B.LIB_PATH = {str(tmp_path / 'libzero_step.so')!r}\n"
            "try:\n"
            "    B.Plan([1000], 2, 1, 1)\n"
            "except RuntimeError as e:\n"
            "    assert 'is missing' in str(e), e\n"
            "    print('raised')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "raised", r.stdout + r.stderr


def test_product_and_oracle_share_no_code():
    """The CUDA path and the oracle are independent: neither library defines
    or references the other's symbols, and neither source tree includes or
    imports the other (the input generator zgen is the one shared module)."""
    import shutil
    import subprocess
    import oracle
    oracle.build()
    pkg = os.path.join(ROOT, "zero_optimizer_step_rs_gb300")
    if shutil.which("nm"):
        prod = subprocess.run(["nm", "-D", B.LIB_PATH], capture_output=True, text=True,
                              check=True).stdout
        orc = subprocess.run(["nm", "-D", oracle.LIB_PATH], capture_output=True, text=True,
                             check=True).stdout
        assert "oracle_" not in prod
        assert not re.search(r"\bzero_[a-z]", orc) and "zgen_" not in orc
    for d in (pkg, os.path.join(pkg, "csrc"), os.path.join(ROOT, "include")):
        for f in os.listdir(d):
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                src = open(os.path.join(d, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert not re.search(r"^\s*#\s*include\s+.*oracle", src, re.M), f
                assert "liboracle" not in src, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            src = open(os.path.join(ROOT, "oracle", f)).read()
            assert not re.search(r"^\s*#\s*include\s+.*(zero_step|csrc)", src, re.M), f
            assert not re.search(r"^\s*(import|from)\s+zero_optimizer_step_rs_gb300\b",
                                 src, re.M), f
            assert "libzero_step" not in src, f


def test_header_is_plain_c_and_a_c_program_links_the_library(tmp_path):
    """include/zero_step.h compiles as strict C99, and a C program linked
    against libzero_step.so calls its host-only entry points: a plan with the
    pages' exercise-1 accounting, status strings, and the argument errors of
    the device-status call (returned before any CUDA call)."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("gcc needed")
    src = tmp_path / "abi.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "zero_step.h"
int main(void)
{
    const int64_t n[1] = {7000000000LL};
    zero_plan_t* p = NULL;
    if (zero_plan_create(n, 1, 8, 1, 1, 0, &p) != ZERO_OK) return 1;
    /* 7B parameters on 8 cards, ZeRO-1: 2+2 bytes replicated, 12 sharded */
    if (p->bytes_per_rank_z1 != 4 * p->N + 12 * p->S) return 2;
    zero_plan_destroy(p);
    if (strcmp(zero_status_string(ZERO_ERR_DEVICE_TIMEOUT), "unknown status") == 0) return 3;
    int32_t word = -1;
    if (zero_get_device_status(NULL, NULL, &word) != ZERO_ERR_NULL) return 4;
    if (zero_get_device_status((const int32_t*)(uintptr_t)0x1002, NULL, &word) != ZERO_ERR_ALIGN) return 5;
    if (word != -1) return 6;
    if (zero3_gather_units(NULL, NULL, NULL, 0, NULL) != ZERO_ERR_NULL) return 7;
    printf("abi ok %d\n", zero_abi_version());
    return 0;
}
''')
    exe = tmp_path / "abi"
    libdir = os.path.join(ROOT, "zero_optimizer_step_rs_gb300")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lzero_step", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip() == "abi ok 1"
