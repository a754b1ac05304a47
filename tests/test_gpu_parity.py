"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Element by element on seeded inputs small enough for the oracle: every
workload recipe scaled down (same R, M, stage, distributions, tensor count),
the tiny workload at full size, ragged sizes around every vector/tile/shard
boundary, run-time (R, M) pairs, special values, guard bands and padding.
Bar: replicas bit-exact, fp32 state within 1e-6 relative (the design makes
both sides run the same operation sequence, so the state is also checked
bit for bit).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu

VARIANTS = [z.ZERO_VARIANT_FUSED, z.ZERO_VARIANT_STAGED]


def _run_both(wl, variant, steps=None, flags=0):
    steps = steps or list(range(wl.first_step(), wl.step + 1))
    _, W0, m0, v0 = H.host_inputs(wl, steps[0])
    idx = np.arange(wl.N, dtype=np.int64)
    Gs = {t: W.host_grads_at(wl, t, idx) for t in steps}
    want = H.oracle_run(wl, Gs, W0, m0, v0, steps)
    ds = H.DeviceState(wl)
    ds.upload_state(W0, m0, v0)
    for t in steps:
        ds.upload_grads(Gs[t])
        ds.step(t, variant=variant, flags=flags)
    torch.cuda.synchronize()
    return ds, ds.result(), want


def _assert_parity(res, bitwise=True):
    bad = {k: v for k, v in res.items() if v and (bitwise or not k.endswith("_bits"))}
    assert not bad, bad


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_full_size(variant):
    _, got, want = _run_both(W.tiny(), variant)
    _assert_parity(H.compare(got, want))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name,target", [("gpt2-small", 300_000), ("llama-3.2-1b", 400_000),
                                         ("uneven", 250_000), ("large", 300_000)])
def test_workload_recipes_scaled(name, target, variant):
    wl = W.ALL[name]().scaled(target)
    if wl.state == "prior":
        wl = dataclasses.replace(wl, step=4, prior_steps=3)
    _, got, want = _run_both(wl, variant)
    _assert_parity(H.compare(got, want))


RAGGED = [1, 2, 3, 4, 5, 7, 8, 9, 63, 64, 65, 1023, 1024, 1025, 2047, 2048, 2049, 4095, 4097,
          8191, 8192 + 5, 100_003]


@pytest.mark.parametrize("n", RAGGED)
@pytest.mark.parametrize("R,M", [(8, 1), (4, 2), (3, 1), (5, 3)])
def test_ragged_sizes(n, R, M):
    wl = W.flat(R, M, n, seed=n, step=3)
    for variant in VARIANTS:
        _, got, want = _run_both(wl, variant)
        _assert_parity(H.compare(got, want))


@pytest.mark.parametrize("R,M", [(1, 1), (2, 1), (4, 1), (16, 1), (7, 4), (8, 2), (4, 4),
                                 (2, 2), (3, 3), (6, 1), (9, 2), (64, 1), (1, 256), (64, 4)])
def test_rank_microbatch_pairs(R, M):
    # compile-time specialisations and the run-time path, up to the limits
    wl = W.flat(R, M, 20_000 + 37, seed=R * 1000 + M, step=2)
    for variant in VARIANTS:
        _, got, want = _run_both(wl, variant)
        _assert_parity(H.compare(got, want))


@pytest.mark.parametrize("R,M", [(3, 1), (5, 3), (6, 1)])
def test_generic_rank_counts_at_full_size_tiling(R, M):
    """(R, M) pairs without a compile-time case, at a size where the fused
    kernel takes its full-size tiling (2-unit tiles, several per persistent
    block) and every staged grid row loops over many tiles."""
    wl = W.flat(R, M, 3_000_017, seed=R * 100 + M, step=3)
    for variant in VARIANTS:
        _, got, want = _run_both(wl, variant)
        _assert_parity(H.compare(got, want))


@pytest.mark.parametrize("align", [4, 8, 64, 128, 4096])
def test_shard_alignment_and_empty_shards(align):
    for n, R in ((5, 4), (130, 7), (10_000, 8), (4096 * 3 + 1, 4)):
        wl = W.Workload(f"align{align}", R=R, M=1, stage=2, tensors=(("flat", n, "normal"),),
                        seed=9, step=1, state="synthetic", align=align)
        for variant in VARIANTS:
            _, got, want = _run_both(wl, variant)
            _assert_parity(H.compare(got, want))


def test_many_odd_tensors_layout():
    # tensor boundaries are irrelevant to the flat step but must not be
    # treated as shard boundaries: 37 odd tensors, R = 7, M = 4
    wl = W.uneven().scaled(60_001)
    for variant in VARIANTS:
        _, got, want = _run_both(wl, variant)
        _assert_parity(H.compare(got, want))


def _special_case(variant):
    wl = W.flat(4, 2, 4099, seed=17, step=5)
    G, W0, m0, v0 = H.host_inputs(wl, 5)
    rng = np.random.default_rng(0)
    specials16 = np.array([0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001, 0x8000, 0x0000, 0x7F7F,
                           0xFF7F, 0x0080], np.uint16)
    for g in G:
        pos = rng.choice(wl.N, 64, replace=False)
        g[pos] = rng.choice(specials16, 64)
    W0 = W0.copy()
    W0[:8] = np.array([1e-40, -1e-42, 3.39e38, -3.39e38, 0.0, -0.0, np.inf, np.nan], np.float32)
    W0[8:12] = np.array([1.00390625, 1.01171875, -1.00390625, 2.0 ** -130], np.float32)
    v0 = v0.copy()
    v0[20:24] = np.array([0.0, 1e-45, 3e38, np.inf], np.float32)
    want = H.oracle_run(wl, {5: G}, W0, m0, v0, [5])
    ds = H.DeviceState(wl)
    ds.upload_state(W0, m0, v0)
    ds.upload_grads(G)
    ds.step(5, variant=variant, flags=z.ZERO_FLAG_CHECK_FINITE)
    torch.cuda.synchronize()
    return ds, ds.result(), want


@pytest.mark.parametrize("variant", VARIANTS)
def test_special_values(variant):
    # Inf/NaN/subnormal/signed-zero gradients, bf16 overflow, subnormal and
    # halfway master values: NaN positions match, everything else bit for bit
    ds, got, want = _special_case(variant)
    res = H.compare(got, want)
    _assert_parity({k: v for k, v in res.items() if not k.endswith("_bits")})
    for name, a, b in zip(("W", "m", "v"), got[:3], want[:3]):
        fin = ~(np.isnan(a) | np.isnan(b))
        assert np.array_equal(a[fin].view(np.uint32), b[fin].view(np.uint32)), name
    assert int(ds.status.item()) & z.ZERO_DEV_NONFINITE


@pytest.mark.parametrize("variant", VARIANTS)
def test_finite_check_stays_clear(variant):
    wl = W.flat(8, 1, 50_000, seed=3, step=1)
    ds, _, _ = _run_both(wl, variant, flags=z.ZERO_FLAG_CHECK_FINITE)
    assert int(ds.status.item()) == 0


def test_fused_and_staged_identical_and_deterministic():
    wl = W.llama32_1b().scaled(200_000)
    outs = []
    for variant in VARIANTS + [z.ZERO_VARIANT_FUSED]:
        _, got, _ = _run_both(wl, variant)
        outs.append(got)
    for o in outs[1:]:
        for a, b in zip(o[:3], outs[0][:3]):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        for p, q in zip(o[3], outs[0][3]):
            assert np.array_equal(p, q)


def test_guard_bands_and_padding_untouched():
    # every buffer is carved out of a larger allocation with canaries around
    # it; after fused and staged steps the canaries and the state pad hold
    # their fill pattern
    wl = W.uneven().scaled(30_011)
    plan = z.Plan(wl.numels, wl.R, wl.M, wl.stage, wl.align)
    N, padded, RM = plan.N, plan.padded, wl.R * wl.M
    GB = 64                                       # guard elements (x4 bytes = 256 B)
    dev = torch.device("cuda")
    canary = 0x7FA5A5A5

    def carve_f32(n):
        buf = torch.full((n + 2 * GB,), canary, dtype=torch.int32, device=dev)
        return buf, buf[GB:GB + n].view(torch.float32)

    def carve_bf16(n):
        buf = torch.full((n + 2 * 2 * GB,), -1, dtype=torch.int16, device=dev)
        return buf, buf[2 * GB:2 * GB + n].view(torch.bfloat16)

    G, W0, m0, v0 = H.host_inputs(wl, 1)
    gbufs, grads = zip(*[carve_bf16(N) for _ in range(RM)])
    pbufs, params = zip(*[carve_bf16(N) for _ in range(wl.R)])
    sbufs, (Wt, mt, vt, scr) = zip(*[carve_f32(padded) for _ in range(4)])
    for t, g in zip(grads, G):
        t.copy_(H.bf16_from_u16(g, dev))
    for t, a in ((Wt, W0), (mt, m0), (vt, v0)):
        t[:N].copy_(torch.from_numpy(a))
    before_g = [b.clone() for b in gbufs]
    hp = z.hparams(**wl.hparams())
    z.zero_step(plan, list(grads), Wt, mt, vt, list(params), hp, 1, z.ZERO_VARIANT_FUSED)
    z.zero_step(plan, list(grads), Wt, mt, vt, list(params), hp, 2, z.ZERO_VARIANT_STAGED,
                scratch=scr)
    torch.cuda.synchronize()
    for b, b0 in zip(gbufs, before_g):            # gradients are read only
        assert torch.equal(b, b0)
    for b in pbufs:
        assert torch.all(b[:2 * GB] == -1) and torch.all(b[-2 * GB:] == -1)
    for b in sbufs:
        assert torch.all(b[:GB] == canary) and torch.all(b[-GB:] == canary)
    for t in (Wt, mt, vt):
        assert torch.all(t.view(torch.int32)[N:] == canary), "state pad touched"


@pytest.mark.parametrize("name,target", [("uneven", 250_003), ("llama-3.2-1b", 400_000),
                                         ("tiny", 65_536),
                                         # many tiles per block in every staged grid row
                                         ("uneven", 3_000_017), ("llama-3.2-1b", 6_000_000)])
def test_staged_zero2_without_scratch_matches_oracle(name, target):
    """ZeRO-2 gives up the gradients once reduced: the staged step without
    scratch keeps the fp32 reduced gradient in gradient buffers 0 and 1 and
    must give the oracle's bits, over two steps with fresh gradients."""
    wl = dataclasses.replace(W.ALL[name]().scaled(target), stage=2)
    steps = [wl.first_step(), wl.first_step() + 1]
    _, W0, m0, v0 = H.host_inputs(wl, steps[0])
    idx = np.arange(wl.N, dtype=np.int64)
    Gs = {t: W.host_grads_at(wl, t, idx) for t in steps}
    want = H.oracle_run(wl, Gs, W0, m0, v0, steps)
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.upload_state(W0, m0, v0)
    for t in steps:
        ds.upload_grads(Gs[t])
        z.zero_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t,
                    variant=z.ZERO_VARIANT_STAGED, scratch=None, flags=z.ZERO_FLAG_CHECK_FINITE,
                    dev_status=ds.status)
    torch.cuda.synchronize()
    _assert_parity(H.compare(ds.result(), want))
    assert int(ds.status.item()) == 0


def test_staged_scratch_contents_on_entry_do_not_matter():
    """The staged step's caller scratch carries nothing between calls: filled
    with 0xFF bytes (NaN in every fp32 slot) before each step, two steps with
    fresh gradients still give the oracle's bits."""
    wl = W.uneven().scaled(250_003)
    steps = [wl.first_step(), wl.first_step() + 1]
    _, W0, m0, v0 = H.host_inputs(wl, steps[0])
    idx = np.arange(wl.N, dtype=np.int64)
    Gs = {t: W.host_grads_at(wl, t, idx) for t in steps}
    want = H.oracle_run(wl, Gs, W0, m0, v0, steps)
    ds = H.DeviceState(wl)
    ds.upload_state(W0, m0, v0)
    for t in steps:
        ds.upload_grads(Gs[t])
        ds.scratch.view(torch.uint8).fill_(0xFF)
        ds.step(t, variant=z.ZERO_VARIANT_STAGED, flags=z.ZERO_FLAG_CHECK_FINITE)
    torch.cuda.synchronize()
    _assert_parity(H.compare(ds.result(), want))
    assert int(ds.status.item()) == 0


def test_staged_zero2_without_scratch_touches_only_two_gradient_buffers():
    """Guard bands around every buffer: the mode writes gradient buffers 0
    and 1 and nothing else beside the state and the replicas; the other
    gradient buffers, the guards and the state pad keep their bits."""
    wl = dataclasses.replace(W.uneven().scaled(30_011), stage=2)
    plan = z.Plan(wl.numels, wl.R, wl.M, wl.stage, wl.align)
    N, padded, RM = plan.N, plan.padded, wl.R * wl.M
    GB = 64
    dev = torch.device("cuda")
    canary = 0x7FA5A5A5
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    gbufs = [torch.full((N + 4 * GB,), -1, dtype=torch.int16, device=dev) for _ in range(RM)]
    grads = [b[2 * GB:2 * GB + N].view(torch.bfloat16) for b in gbufs]
    pbufs = [torch.full((N + 4 * GB,), -1, dtype=torch.int16, device=dev) for _ in range(wl.R)]
    params = [b[2 * GB:2 * GB + N].view(torch.bfloat16) for b in pbufs]
    sbufs = [torch.full((padded + 2 * GB,), canary, dtype=torch.int32, device=dev)
             for _ in range(3)]
    Wt, mt, vt = [b[GB:GB + padded].view(torch.float32) for b in sbufs]
    for t, g in zip(grads, G):
        t.copy_(H.bf16_from_u16(g, dev))
    for t, a in ((Wt, W0), (mt, m0), (vt, v0)):
        t[:N].copy_(torch.from_numpy(a))
    before = [b.clone() for b in gbufs]
    hp = z.hparams(**wl.hparams())
    z.zero_step(plan, grads, Wt, mt, vt, params, hp, 1, z.ZERO_VARIANT_STAGED, scratch=None)
    torch.cuda.synchronize()
    for q, (b, b0) in enumerate(zip(gbufs, before)):
        assert torch.equal(b[:2 * GB], b0[:2 * GB]) and torch.equal(b[-2 * GB:], b0[-2 * GB:])
        if q >= 2:
            assert torch.equal(b, b0), f"gradient buffer {q} written"
    for b in pbufs:
        assert torch.all(b[:2 * GB] == -1) and torch.all(b[-2 * GB:] == -1)
    for b in sbufs:
        assert torch.all(b[:GB] == canary) and torch.all(b[-GB:] == canary)
    for t in (Wt, mt, vt):
        assert torch.all(t.view(torch.int32)[N:] == canary), "state pad touched"
    # buffers 0 and 1 hold the reduced gradient's halves: reassembled, the oracle's average
    import ctypes
    ga = (ctypes.c_void_p * RM)(*[g.ctypes.data for g in G])
    L = oracle.lib()
    want_g = np.array([L.oracle_avg_grad(ctypes.addressof(ga), wl.R, wl.M, i,
                                         float(RM)) for i in range(N)], np.float32)
    lo = H.u16_from_bf16(grads[0]).astype(np.uint32)
    hi = H.u16_from_bf16(grads[1]).astype(np.uint32)
    assert np.array_equal(lo | (hi << 16), want_g.view(np.uint32))
    want = H.oracle_run(wl, {1: G}, W0, m0, v0, [1])
    got = (Wt[:N].cpu().numpy(), mt[:N].cpu().numpy(), vt[:N].cpu().numpy(),
           [H.u16_from_bf16(p) for p in params])
    _assert_parity(H.compare(got, want))


def test_staged_entry_points_one_by_one():
    wl = W.uneven().scaled(40_000)
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    ds = H.DeviceState(wl)
    ds.upload_state(W0, m0, v0)
    ds.upload_grads(G)
    z.zero_rs_avg(ds.plan, ds.grads, ds.scratch)
    torch.cuda.synchronize()
    import ctypes
    ga = (ctypes.c_void_p * len(G))(*[g.ctypes.data for g in G])
    L = oracle.lib()
    want_g = np.array([L.oracle_avg_grad(ctypes.addressof(ga), wl.R, wl.M, i,
                                         float(wl.R * wl.M)) for i in range(wl.N)], np.float32)
    got_g = ds.scratch[:wl.N].cpu().numpy()
    assert np.array_equal(got_g.view(np.uint32), want_g.view(np.uint32))
    z.zero_adamw_shard(ds.plan, ds.scratch, ds.W, ds.m, ds.v, ds.hp, 1)
    z.zero_ag_cast(ds.plan, ds.W, ds.params)
    torch.cuda.synchronize()
    want = H.oracle_run(wl, {1: G}, W0, m0, v0, [1])
    _assert_parity(H.compare(ds.result(), want))


def test_zero_emulation_oracle_agrees_with_gpu():
    # the oracle's card-by-card ZeRO emulation (explicit RS copies, per-card
    # shard update, AG copies) against the GPU replicas
    wl = W.uneven().scaled(20_000)
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    S = oracle.shard_len(wl.N, wl.R, wl.align)
    Wz = np.zeros(wl.R * S, np.float32)
    mz, vz = Wz.copy(), Wz.copy()
    Wz[:wl.N], mz[:wl.N], vz[:wl.N] = W0, m0, v0
    Pz = [np.zeros(wl.N, np.uint16) for _ in range(wl.R)]
    oracle.zero_step(G, Wz, mz, vz, Pz, oracle.hparams(**wl.hparams()), 1, wl.R, wl.M, wl.N, S)
    ds = H.DeviceState(wl)
    ds.upload_state(W0, m0, v0)
    ds.upload_grads(G)
    ds.step(1)
    torch.cuda.synchronize()
    gW, gm, gv, gP = ds.result()
    assert np.array_equal(gW.view(np.uint32), Wz[:wl.N].view(np.uint32))
    for p, q in zip(gP, Pz):
        assert np.array_equal(p, q)


@pytest.mark.parametrize("mode", ["zero_copy", "copy_engine"])
@pytest.mark.parametrize("target", [100_000, 3_000_000])   # small-vector path, full-size tiling
def test_step_from_host_buffers(mode, target):
    wl = W.llama32_1b().scaled(target)
    G, W0, m0, v0 = H.host_inputs(wl, wl.step)
    want = H.oracle_run(wl, {wl.step: G}, W0, m0, v0, [wl.step])
    ds = H.DeviceState(wl)
    ds.upload_state(W0, m0, v0)
    host_g = [torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
              for g in G]
    out = torch.empty(wl.N, dtype=torch.bfloat16).pin_memory()
    z.zero_step_host(ds.plan, host_g, ds.grads if mode == "copy_engine" else None, ds.W, ds.m,
                     ds.v, ds.params, out, ds.hp, wl.step, flags=z.ZERO_FLAG_CHECK_FINITE,
                     dev_status=ds.status)
    torch.cuda.synchronize()
    assert np.array_equal(out.view(torch.int16).numpy().view(np.uint16), want[3][0])
    _assert_parity(H.compare(ds.result(), want))
    assert int(ds.status.item()) == 0


def test_step_from_host_pageable_memory():
    # pageable host memory: refused (ZERO_ERR_INVALID_ARG) unless the GPU can
    # reach it through the host page tables, in which case the step runs and
    # must give the same bits as the device replica
    wl = W.flat(2, 1, 4096)
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    ds = H.DeviceState(wl)
    ds.upload_state(W0, m0, v0)
    host_g = [torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16) for g in G]
    out = torch.empty(wl.N, dtype=torch.bfloat16)
    try:
        z.zero_step_host(ds.plan, host_g, None, ds.W, ds.m, ds.v, ds.params, out, ds.hp, 1)
        torch.cuda.synchronize()
    except z.ZeroError as e:
        assert e.code == -1
        return
    want = H.oracle_run(wl, {1: G}, W0, m0, v0, [1])
    assert np.array_equal(out.view(torch.int16).numpy().view(np.uint16), want[3][0])


def test_generator_device_matches_host():
    wl = W.uneven().scaled(50_000)
    ds = H.DeviceState(wl)
    ds.fill_state_device()
    ds.fill_grads_device(1)
    torch.cuda.synchronize()
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    assert np.array_equal(ds.W[:wl.N].cpu().numpy().view(np.uint32), W0.view(np.uint32))
    for g, t in zip(G, ds.grads):
        assert np.array_equal(H.u16_from_bf16(t[:wl.N]), g)
    wl2 = W.llama32_1b().scaled(50_000)
    ds2 = H.DeviceState(wl2)
    ds2.fill_state_device()
    torch.cuda.synchronize()
    _, W0, m0, v0 = H.host_inputs(wl2, wl2.step)
    for t, a in ((ds2.W, W0), (ds2.m, m0), (ds2.v, v0)):
        assert np.array_equal(t[:wl2.N].cpu().numpy().view(np.uint32), a.view(np.uint32))


@pytest.mark.parametrize("variant", ["fused", "staged", "staged_grads_refill", "clipped", "zero3"])
def test_back_to_back_steps_on_one_stream_match_oracle(variant):
    """Six steps enqueued back to back on one stream with no host sync and no
    copy in between (the same gradients every step), so each step's kernels
    follow the previous step's kernels directly and overlap their launch with
    them: every step must still read the state the previous one wrote.  The
    result equals the oracle run of the same six steps."""
    wl = W.flat(8, 1, 1_000_003, seed=31, step=1)
    steps = list(range(1, 7))
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    ds = H.DeviceState(wl)
    ds.upload_state(W0, m0, v0)
    ds.upload_grads(G)
    torch.cuda.synchronize()
    hp = oracle.hparams(**wl.hparams())
    Wc, mc, vc = W0.copy(), m0.copy(), v0.copy()
    P = [np.zeros(wl.N, np.uint16) for _ in range(wl.R)]
    if variant == "clipped":
        for t in steps:
            ds.step_clipped(t, 1e-3)
            oracle.dp_step_clipped(G, Wc, mc, vc, P, hp, t, wl.R, wl.M, max_norm=1e-3)
    elif variant == "zero3":
        plan = ds.plan
        Pz = np.zeros(plan.padded, np.uint16)
        shards = torch.zeros(plan.padded, dtype=torch.bfloat16, device="cuda")
        Wz = np.zeros(plan.padded, np.float32)
        mz, vz = Wz.copy(), Wz.copy()
        Wz[:wl.N], mz[:wl.N], vz[:wl.N] = W0, m0, v0
        for t in steps:
            z.zero3_step(plan, ds.grads, ds.W, ds.m, ds.v, shards, ds.hp, t)
            oracle.zero3_step(G, Wz, mz, vz, Pz, hp, t, wl.R, wl.M, wl.N, plan.S)
        torch.cuda.synchronize()
        assert np.array_equal(H.u16_from_bf16(shards), Pz)
        assert np.array_equal(ds.W[:wl.N].cpu().numpy().view(np.uint32), Wz[:wl.N].view(np.uint32))
        return
    else:
        for t in steps:
            if variant == "fused":
                ds.step(t, variant=z.ZERO_VARIANT_FUSED)
            elif variant == "staged":
                ds.step(t, variant=z.ZERO_VARIANT_STAGED)
            else:
                # in-buffer mode: its two gradient buffers are written again from
                # the third one (a device copy, as a backward would) before each step
                if t > 1:
                    for q in (0, 1):
                        ds.grads[q].copy_(ds.kept[q])
                else:
                    ds.kept = [g.clone() for g in ds.grads[:2]]
                z.zero_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t,
                            variant=z.ZERO_VARIANT_STAGED, scratch=None)
            oracle.dp_step(G, Wc, mc, vc, P, hp, t, wl.R, wl.M)
    torch.cuda.synchronize()
    _assert_parity(H.compare(ds.result(), (Wc, mc, vc, P)))
