"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.

Inputs are generated on the device by the seeded generator; the oracle
regenerates the same inputs on the host at sampled indices (random ones plus
every shard boundary, tensor boundary, the first and last elements and the
last partial tile) and runs the same steps on them, since the step is
elementwise.  Properties that hold at any size are checked on every element:
all R replicas are bitwise identical and the state pad is untouched.
"""
import numpy as np
import pytest
import torch

import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu

N_RANDOM = 20_000


def _sample_indices(wl, plan, seed=123):
    N, S = plan.N, plan.S
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, N, N_RANDOM)]
    special = [0, 1, 2, 3, 4, 5, N - 1, N - 2, N - 3, N - 4, N - 5]
    for r in range(1, wl.R + 1):
        special += [r * S - 2, r * S - 1, r * S, r * S + 1]
    for off in wl.offsets:
        special += [int(off) - 1, int(off), int(off) + 1]
    tail = max(0, N - 4096)
    idx.append(np.arange(tail, N, 7))
    idx.append(np.array([i for i in special if 0 <= i < N]))
    return np.unique(np.concatenate(idx).astype(np.int64))


def _oracle_at(wl, idx, steps):
    W0 = W.host_w0_at(wl, idx)
    m0, v0 = W.host_mv0_at(wl, idx)
    Gs = {t: W.host_grads_at(wl, t, idx) for t in steps}
    return H.oracle_run(wl, Gs, W0, m0, v0, steps)


def _run_full(wl, variant):
    steps = list(range(wl.first_step(), wl.step + 1))
    ds = H.DeviceState(wl, staged_scratch=(variant == z.ZERO_VARIANT_STAGED))
    ds.fill_state_device()
    for t in steps:
        ds.fill_grads_device(t)
        ds.step(t, variant=variant, flags=z.ZERO_FLAG_CHECK_FINITE)
    torch.cuda.synchronize()
    idx = _sample_indices(wl, ds.plan)
    it = torch.from_numpy(idx).to(ds.W.device)
    got = (ds.W[it].cpu().numpy(), ds.m[it].cpu().numpy(), ds.v[it].cpu().numpy(),
           [H.u16_from_bf16(p[it]) for p in ds.params])
    want = _oracle_at(wl, idx, steps)
    res = H.compare(got, want)
    # properties on every element
    replicas_equal = all(torch.equal(p, ds.params[0]) for p in ds.params[1:])
    pad_clean = all(int(torch.count_nonzero(t[ds.N:])) == 0 for t in (ds.W, ds.m, ds.v))
    status = int(ds.status.item())
    del ds
    torch.cuda.empty_cache()
    return res, replicas_equal, pad_clean, status, idx.size


@pytest.mark.parametrize("variant", [z.ZERO_VARIANT_FUSED, z.ZERO_VARIANT_STAGED])
@pytest.mark.parametrize("name", ["gpt2-small", "llama-3.2-1b", "uneven", "large"])
def test_full_size_sampled(name, variant):
    wl = W.ALL[name]()
    res, replicas_equal, pad_clean, status, k = _run_full(wl, variant)
    bad = {key: v for key, v in res.items() if v}
    assert not bad, (name, bad, k)
    assert replicas_equal, "replicas differ somewhere"
    assert pad_clean, "state pad written"
    assert status == 0, f"device status {status}"


@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("S", [1 << 10, 1 << 16, 1 << 22, 1 << 28])
def test_flat_sweep_points_sampled(R, S):
    """The flat-vector sweep (fp32 master shard of 4 KB to 1 GB, N = R*S) at
    its smallest, two middle and largest shard sizes: sampled parity of the
    fused step against the oracle, replicas and pad checked everywhere.  The
    largest point at R = 8 holds about 88 GB on the device."""
    wl = W.sweep_point(R, S)
    res, replicas_equal, pad_clean, status, k = _run_full(wl, z.ZERO_VARIANT_FUSED)
    bad = {key: v for key, v in res.items() if v}
    assert not bad, (wl.name, bad, k)
    assert replicas_equal and pad_clean and status == 0


@pytest.mark.parametrize("name", ["gpt2-small", "llama-3.2-1b"])
def test_full_size_sampled_tma_variant(name):
    """The TMA-bulk-staged variant (R*M <= 16) at full size, sampled against
    the oracle like the other variants."""
    wl = W.ALL[name]()
    res, replicas_equal, pad_clean, status, k = _run_full(wl, z.ZERO_VARIANT_FUSED_TMA)
    bad = {key: v for key, v in res.items() if v}
    assert not bad, (name, bad, k)
    assert replicas_equal and pad_clean and status == 0
