"""GPU parity of the ZeRO-3 step and the per-unit all-gather.

zero3_step and zero3_gather through the C ABI against oracle.zero3_step and
oracle.zero3_gather: shard buffer and fp32 state bit for bit, pad and guard
bands untouched, every unit misalignment (lo mod 8), units at the very end
of an unpadded buffer, 1..R destinations; at full size (Llama-3.2-1B-shaped)
on sampled elements, and the gathered model equals the shards everywhere.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu
CANARY = 0x5A5A


def _zero3_run(wl, steps):
    _, W0, m0, v0 = H.host_inputs(wl, steps[0])
    idx = np.arange(wl.N, dtype=np.int64)
    plan = z.Plan(wl.numels, wl.R, wl.M, wl.stage, wl.align)
    S, N, padded = plan.S, plan.N, plan.padded
    # oracle, card by card
    Wz = np.zeros(padded, np.float32)
    mz, vz = Wz.copy(), Wz.copy()
    Wz[:N], mz[:N], vz[:N] = W0, m0, v0
    Ps = np.full(padded, CANARY, np.uint16)
    hp = oracle.hparams(**wl.hparams())
    # GPU
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.upload_state(W0, m0, v0)
    shards = torch.full((padded,), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    for t in steps:
        G = W.host_grads_at(wl, t, idx)
        oracle.zero3_step(G, Wz, mz, vz, Ps, hp, t, wl.R, wl.M, N, S)
        ds.upload_grads(G)
        z.zero3_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, shards, ds.hp, t,
                     flags=z.ZERO_FLAG_CHECK_FINITE, dev_status=ds.status)
    torch.cuda.synchronize()
    return plan, ds, shards, (Wz, mz, vz, Ps)


@pytest.mark.parametrize("name,target", [("uneven", 200_000), ("llama-3.2-1b", 300_000),
                                         ("gpt2-small", 150_000)])
def test_zero3_step_matches_oracle(name, target):
    import dataclasses
    wl = W.ALL[name]().scaled(target)
    if wl.state == "prior":
        wl = dataclasses.replace(wl, step=3, prior_steps=2)
    plan, ds, shards, (Wz, mz, vz, Ps) = _zero3_run(wl, list(range(wl.first_step(), wl.step + 1)))
    got_s = H.u16_from_bf16(shards)
    assert np.array_equal(got_s, Ps)                       # includes the untouched pad
    for t, a in ((ds.W, Wz), (ds.m, mz), (ds.v, vz)):
        assert np.array_equal(t.cpu().numpy().view(np.uint32)[:plan.N],
                              a.view(np.uint32)[:plan.N])
    assert int(ds.status.item()) == 0


@pytest.mark.parametrize("n,R,M", [(1, 2, 1), (7, 4, 1), (2049, 3, 1), (4096 * 8, 8, 1),
                                   (100_003, 7, 1), (100_003, 64, 4), (2049, 1, 256),
                                   (3_000_017, 3, 2)])   # run-time path, full-size tiling
def test_zero3_step_ragged(n, R, M):
    wl = W.flat(R, M, n, seed=n, step=2)
    plan, ds, shards, (Wz, mz, vz, Ps) = _zero3_run(wl, [2])
    assert np.array_equal(H.u16_from_bf16(shards), Ps)


def _gather_case(plan, shards_np, shards, lo, hi, n_out):
    L = hi - lo
    G = 64                                                 # guard elements (128 B)
    bufs = [torch.full((L + 2 * G + 8,), -7, dtype=torch.int16, device="cuda")
            for _ in range(n_out)]
    outs = [b[G:G + L].view(torch.bfloat16) for b in bufs]
    z.zero3_gather(plan, shards, lo, hi, outs)
    torch.cuda.synchronize()
    for card, (b, o) in enumerate(zip(bufs, outs)):
        want, _ = oracle.zero3_gather(shards_np, plan.N, plan.R, plan.S, lo, hi, card % plan.R)
        assert np.array_equal(H.u16_from_bf16(o), want), (lo, hi)
        assert torch.all(b[:G] == -7) and torch.all(b[G + L:] == -7), (lo, hi)


def test_gather_every_alignment_and_length():
    N, R = 8 * 4096, 8                                     # no padding: the last shard ends the buffer
    plan = z.Plan([N], R, 1, 2, 64)
    assert plan.padded == N
    rng = np.random.default_rng(0)
    shards_np = rng.integers(0, 2 ** 16, N, dtype=np.uint16)
    shards = torch.from_numpy(shards_np.view(np.int16).copy()).cuda().view(torch.bfloat16)
    cases = []
    for lo in list(range(0, 24)) + [N - 40 + k for k in range(8)]:
        for L in (0, 1, 3, 7, 8, 9, 15, 16, 17, 31, 33):
            if lo + L <= N:
                cases.append((lo, lo + L))
    for s in range(8):                                     # units that end exactly at N
        cases.append((N - 1000 - s, N))
        cases.append((s, N))
    cases += [(4096 * 3 - 5, 4096 * 5 + 3)]               # crosses two shard boundaries
    for k, (lo, hi) in enumerate(cases):
        _gather_case(plan, shards_np, shards, lo, hi, n_out=1 + k % R)


def test_full_size_zero3_llama():
    wl = W.llama32_1b()
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.fill_state_device()
    ds.fill_grads_device(wl.step)
    shards = torch.empty(ds.padded, dtype=torch.bfloat16, device="cuda")
    z.zero3_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, shards, ds.hp, wl.step,
                 flags=z.ZERO_FLAG_CHECK_FINITE, dev_status=ds.status)
    # gather every tensor as its own unit; each must equal its slice of the shards
    offs = wl.offsets
    for lo, hi in zip(offs[:-1], offs[1:]):
        lo, hi = int(lo), int(hi)
        unit = torch.empty(hi - lo, dtype=torch.bfloat16, device="cuda")
        z.zero3_gather(ds.plan, shards, lo, hi, [unit])
        assert torch.equal(unit.view(torch.int16), shards[lo:hi].view(torch.int16)), (lo, hi)
    full = torch.empty(ds.N, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    pick = np.unique(np.concatenate([rng.integers(0, ds.N, 20_000), np.arange(ds.N - 3000, ds.N)]))
    it = torch.from_numpy(pick).cuda()
    W0 = W.host_w0_at(wl, pick)
    m0, v0 = W.host_mv0_at(wl, pick)
    want = H.oracle_run(wl, {wl.step: W.host_grads_at(wl, wl.step, pick)}, W0, m0, v0, [wl.step])
    got_s = H.u16_from_bf16(shards[it])
    assert np.array_equal(got_s, want[3][0])
    assert np.array_equal(ds.W[it].cpu().numpy().view(np.uint32), want[0].view(np.uint32))
    assert int(ds.status.item()) == 0
    # the whole model gathered in one unit equals the shards, element for element
    z.zero3_gather(ds.plan, shards, 0, ds.N, [full])
    torch.cuda.synchronize()
    assert torch.equal(full.view(torch.int16), shards[:ds.N].view(torch.int16))


@pytest.mark.parametrize("R", [4, 8])
def test_zero3_step_sampled_at_a_persistent_grid_size(R):
    """200 M elements: the ZeRO-3 step runs its persistent grid below the
    resident maximum (R = 4 and R = 8); sampled elements against the oracle,
    and the shards' bf16 equal to the updated master everywhere."""
    wl = W.flat(R, 1, 200_000_003, seed=R + 50, step=3, state="synthetic")
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.fill_state_device()
    ds.fill_grads_device(wl.step)
    shards = torch.zeros(ds.padded, dtype=torch.bfloat16, device="cuda")
    z.zero3_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, shards, ds.hp, wl.step)
    torch.cuda.synchronize()
    rng = np.random.default_rng(R)
    pick = np.unique(np.concatenate([rng.integers(0, ds.N, 20_000), np.arange(ds.N - 3000, ds.N),
                                     np.arange(0, 3000)]))
    it = torch.from_numpy(pick).cuda()
    W0 = W.host_w0_at(wl, pick)
    m0, v0 = W.host_mv0_at(wl, pick)
    want = H.oracle_run(wl, {wl.step: W.host_grads_at(wl, wl.step, pick)}, W0, m0, v0, [wl.step])
    assert np.array_equal(H.u16_from_bf16(shards[it]), want[3][0])
    for got, exp in ((ds.W, want[0]), (ds.m, want[1]), (ds.v, want[2])):
        assert np.array_equal(got[it].cpu().numpy().view(np.uint32), exp.view(np.uint32))
    assert torch.equal(shards[:ds.N].view(torch.int16), ds.W[:ds.N].to(torch.bfloat16).view(torch.int16))


# ----------------------------------------- per-unit reduce-scatter (FSDP) --

def _random_units(n, rng, pieces):
    if n == 1:
        return [(0, 1)]
    cuts = np.sort(rng.choice(np.arange(1, n), size=min(pieces, n - 1), replace=False))
    b = [0] + cuts.tolist() + [n]
    units = [(b[k], b[k + 1]) for k in range(len(b) - 1)]
    rng.shuffle(units)
    return units


@pytest.mark.parametrize("n,R,M,pieces", [(1, 2, 1, 1), (1000, 4, 2, 7), (4099, 7, 4, 30),
                                          (8192, 8, 1, 3), (20_011, 3, 2, 64), (100_003, 8, 1, 9),
                                          (5003, 64, 4, 5), (2049, 1, 256, 4),
                                          (3_000_017, 3, 2, 5)])   # run-time path, many waves
def test_unit_reduce_scatter_then_update_matches_oracle(n, R, M, pieces):
    """Random units (any start, so the fp32 shard stores take both the
    vector and the scalar path) in shuffled order, each unit's gradient in
    buffers of its own; then the update.  Gradient shards, state and
    parameter shards bit for bit against the oracle, and against zero3_step."""
    wl = W.flat(R, M, n, seed=n + R, step=3)
    G, W0, m0, v0 = H.host_inputs(wl, 3)
    plan = z.Plan(wl.numels, R, M, wl.stage, wl.align)
    S, padded = plan.S, plan.padded
    hp = oracle.hparams(**wl.hparams())
    rng = np.random.default_rng(n)
    units = _random_units(n, rng, pieces)
    # oracle
    g_or = np.full(padded, np.nan, np.float32)
    for lo, hi in units:
        oracle.zero3_rs_unit([np.ascontiguousarray(g[lo:hi]) for g in G], n, R, M, S, lo, hi, g_or)
    Wz = np.zeros(padded, np.float32)
    mz, vz = Wz.copy(), Wz.copy()
    Wz[:n], mz[:n], vz[:n] = W0, m0, v0
    Ps = np.full(padded, CANARY, np.uint16)
    oracle.zero3_update(g_or, Wz, mz, vz, Ps, hp, 3, n, R, M, S)
    # GPU, unit by unit
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.upload_state(W0, m0, v0)
    gs = torch.full((padded,), float("nan"), dtype=torch.float32, device="cuda")
    for lo, hi in units:
        ug = [H.bf16_from_u16(np.ascontiguousarray(g[lo:hi]), "cuda") for g in G]
        z.zero3_rs_unit(ds.plan, ug, lo, hi, gs, flags=z.ZERO_FLAG_CHECK_FINITE,
                        dev_status=ds.status)
    shards = torch.full((padded,), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    z.zero3_update(ds.plan, gs, ds.W, ds.m, ds.v, shards, ds.hp, 3)
    torch.cuda.synchronize()
    g_gpu = gs.cpu().numpy()
    assert np.array_equal(np.isnan(g_gpu), np.isnan(g_or))          # pad untouched
    fin = ~np.isnan(g_or)
    assert np.array_equal(g_gpu[fin].view(np.uint32), g_or[fin].view(np.uint32))
    for t, a in ((ds.W, Wz), (ds.m, mz), (ds.v, vz)):
        assert np.array_equal(t.cpu().numpy().view(np.uint32)[:n], a.view(np.uint32)[:n])
    assert np.array_equal(H.u16_from_bf16(shards), Ps)              # pad included
    assert int(ds.status.item()) == 0
    # the whole-step kernel gives the same bits
    ds2 = H.DeviceState(wl, staged_scratch=False)
    ds2.upload_state(W0, m0, v0)
    ds2.upload_grads(G)
    shards2 = torch.full((padded,), CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    z.zero3_step(ds2.plan, ds2.grads, ds2.W, ds2.m, ds2.v, shards2, ds2.hp, 3)
    torch.cuda.synchronize()
    assert torch.equal(shards2.view(torch.int16), shards.view(torch.int16))
    assert torch.equal(ds2.W.view(torch.int32), ds.W.view(torch.int32))


def test_unit_reduce_scatter_reports_non_finite():
    wl = W.flat(4, 1, 3000, seed=5, step=1)
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    G[2][1234] = 0x7F80                                      # +Inf in rank 2's gradient
    ds = H.DeviceState(wl, staged_scratch=False)
    gs = torch.zeros(ds.padded, dtype=torch.float32, device="cuda")
    lo, hi = 1001, 2999
    ug = [H.bf16_from_u16(np.ascontiguousarray(g[lo:hi]), "cuda") for g in G]
    z.zero3_rs_unit(ds.plan, ug, lo, hi, gs, flags=z.ZERO_FLAG_CHECK_FINITE, dev_status=ds.status)
    torch.cuda.synchronize()
    assert int(ds.status.item()) & z.ZERO_DEV_NONFINITE
    assert torch.isinf(gs[1234]).item()


def test_full_size_unit_reduce_scatter_llama_layers():
    """The 1B-shaped workload with one unit per transformer layer (plus the
    embedding and the final norm), the backward's order (last unit first),
    each unit's gradient read in place from the full gradient buffers; the
    result equals zero3_step everywhere."""
    wl = W.llama32_1b()
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.fill_state_device()
    ds.fill_grads_device(wl.step)
    offs = [int(o) for o in wl.offsets]
    # embedding, 16 layers of 9 tensors, final norm
    bounds = [offs[0], offs[1]] + [offs[1 + 9 * k] for k in range(1, 17)] + [offs[-1]]
    bounds = sorted(set(bounds))
    units = list(zip(bounds[:-1], bounds[1:]))[::-1]
    assert units[-1][0] == 0 and max(h for _, h in units) == ds.N
    gs = torch.empty(ds.padded, dtype=torch.float32, device="cuda")
    for lo, hi in units:
        assert lo % 8 == 0                                   # slices stay 16-byte aligned
        z.zero3_rs_unit(ds.plan, [g[lo:hi] for g in ds.grads], lo, hi, gs,
                        flags=z.ZERO_FLAG_CHECK_FINITE, dev_status=ds.status)
    shards = torch.empty(ds.padded, dtype=torch.bfloat16, device="cuda")
    W1 = ds.W.clone()
    m1, v1 = ds.m.clone(), ds.v.clone()
    z.zero3_update(ds.plan, gs, W1, m1, v1, shards, ds.hp, wl.step)
    shards_ref = torch.empty(ds.padded, dtype=torch.bfloat16, device="cuda")
    z.zero3_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, shards_ref, ds.hp, wl.step)
    torch.cuda.synchronize()
    N = ds.N
    assert torch.equal(shards[:N].view(torch.int16), shards_ref[:N].view(torch.int16))
    for a, b in ((W1, ds.W), (m1, ds.m), (v1, ds.v)):
        assert torch.equal(a[:N].view(torch.int32), b[:N].view(torch.int32))
    assert int(ds.status.item()) == 0


# ------------------------------------------- the table of units, one launch --

def _table_case(plan, shards_np, shards, units):
    """Gather `units` ((lo, hi) pairs) in one zero3_gather_units call into
    guarded buffers; every unit must equal oracle.zero3_gather bit for bit
    and the guards must be untouched."""
    G = 64
    bufs, outs = [], []
    for lo, hi in units:
        b = torch.full((hi - lo + 2 * G + 8,), -7, dtype=torch.int16, device="cuda")
        bufs.append(b)
        outs.append(b[G:G + hi - lo].view(torch.bfloat16) if hi > lo else None)
    z.zero3_gather_units(plan, shards, [(lo, hi, o) for (lo, hi), o in zip(units, outs)])
    torch.cuda.synchronize()
    for k, ((lo, hi), b, o) in enumerate(zip(units, bufs, outs)):
        if hi > lo:
            want, _ = oracle.zero3_gather(shards_np, plan.N, plan.R, plan.S, lo, hi, k % plan.R)
            assert np.array_equal(H.u16_from_bf16(o), want), (k, lo, hi)
        L = hi - lo
        assert torch.all(b[:G] == -7) and torch.all(b[G + L:] == -7), (k, lo, hi)


def _random_shards(plan, seed):
    rng = np.random.default_rng(seed)
    shards_np = rng.integers(0, 2 ** 16, plan.padded, dtype=np.uint16)
    shards = torch.from_numpy(shards_np.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return shards_np, shards


def test_gather_units_every_alignment_length_and_empty_units():
    N, R = 8 * 4096, 8                                     # no padding: the last shard ends the buffer
    plan = z.Plan([N], R, 1, 2, 64)
    shards_np, shards = _random_shards(plan, 3)
    units = []
    for lo in list(range(0, 24)) + [N - 40 + k for k in range(8)]:
        for L in (0, 1, 7, 8, 9, 17, 33, 2047, 2048, 2049, 4103):
            if lo + L <= N:
                units.append((lo, lo + L))
    units += [(N - 1000 - s, N) for s in range(8)] + [(s, N) for s in range(3)]
    units += [(4096 * 3 - 5, 4096 * 5 + 3), (100, 100), (N, N)]
    rng = np.random.default_rng(4)
    rng.shuffle(units)
    for k in range(0, len(units), 300):                   # several tables, any order
        _table_case(plan, shards_np, shards, units[k:k + 300])


def test_gather_units_full_table_and_overlapping_sources():
    """A table of ZERO_MAX_GATHER_UNITS units over a padded, uneven layout,
    many of them reading the same source ranges."""
    plan = z.Plan([500_003], 7, 1, 2, 64)
    assert plan.padded > plan.N
    shards_np, shards = _random_shards(plan, 5)
    rng = np.random.default_rng(6)
    lo = rng.integers(0, plan.N, z.ZERO_MAX_GATHER_UNITS)
    ln = rng.integers(0, 3000, z.ZERO_MAX_GATHER_UNITS)
    units = [(int(a), int(min(plan.N, a + b))) for a, b in zip(lo, ln)]
    units[:8] = [(0, 8), (0, 8), (plan.N - 3, plan.N), (plan.N - 3, plan.N), (5, 5),
                 (plan.S - 1, plan.S + 1), (2 * plan.S - 9, 2 * plan.S + 9), (1, plan.N)]
    _table_case(plan, shards_np, shards, units)


def test_gather_units_equal_one_unit_gathers_on_the_1b_tables():
    """The 146 per-tensor units and the 18 per-layer units of the
    Llama-3.2-1B-shaped set, over shards filled by the seeded generator: one
    table launch equals the oracle's gather of each unit, every element."""
    import zgen
    wl = W.llama32_1b()
    plan = z.Plan(wl.numels, wl.R, wl.M, wl.stage, wl.align)
    shards = torch.empty(plan.padded, dtype=torch.bfloat16, device="cuda")
    stream_id = (1 << 50) + 17
    zgen.dev_grad(shards.data_ptr(), wl.seed, stream_id, 0, plan.padded, 1e-2,
                  cuda_stream=torch.cuda.current_stream().cuda_stream)
    shards_np = zgen.host_grad(wl.seed, stream_id, 0, plan.padded, 1e-2)
    offs = [int(x) for x in wl.offsets]
    per_tensor = list(zip(offs[:-1], offs[1:]))
    # per layer: the embedding, 16 decoder layers of 9 tensors, the final norm
    layer_bounds = [offs[0], offs[1]] + [offs[1 + 9 * (k + 1)] for k in range(16)] + [offs[-1]]
    per_layer = list(zip(layer_bounds[:-1], layer_bounds[1:]))
    assert len(per_tensor) == 146 and len(per_layer) == 18
    for table in (per_tensor, per_layer):
        outs = [torch.empty(hi - lo, dtype=torch.bfloat16, device="cuda") for lo, hi in table]
        z.zero3_gather_units(plan, shards, [(lo, hi, o) for (lo, hi), o in zip(table, outs)])
        torch.cuda.synchronize()
        for (lo, hi), o in zip(table, outs):
            want, _ = oracle.zero3_gather(shards_np, plan.N, plan.R, plan.S, lo, hi, 0)
            assert np.array_equal(H.u16_from_bf16(o), want), (lo, hi)
        del outs
