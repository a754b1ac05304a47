"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times.

Inputs are generated on the device by the seeded generator.  For the
GPT-2-small, Llama-3.2-1B, uneven and ~4B workloads every element is
compared: the host regenerates the inputs of one chunk of the flat vector at
a time (the generator is a pure function of seed, stream and index), the
oracle runs the same steps on that chunk on all host cores (the step is
elementwise, so a chunk's result is the whole run's at those indices), and
the device's W, m, v and replica 0 over the same chunk must match bit for
bit.  Every replica must equal replica 0 and the state pad must be
untouched, checked on the device over the whole vector.  The TMA-staged
variant is compared on every element of the GPT-2 and 1B workloads too.  The
flat sweep points keep a sampled comparison (random indices plus every shard and tensor
boundary and the last partial tile).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu

N_RANDOM = 20_000
CHUNK = 1 << 25                      # elements compared per round trip to the host
THREADS = max(1, os.cpu_count() or 1)


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


def _device_run(wl, variant):
    steps = list(range(wl.first_step(), wl.step + 1))
    ds = H.DeviceState(wl, staged_scratch=(variant == z.ZERO_VARIANT_STAGED))
    ds.fill_state_device()
    for t in steps:
        ds.fill_grads_device(t)
        ds.step(t, variant=variant, flags=z.ZERO_FLAG_CHECK_FINITE)
    torch.cuda.synchronize()
    return ds, steps


def _everywhere(ds):
    """Properties checked on the device over every element."""
    replicas_equal = all(torch.equal(p, ds.params[0]) for p in ds.params[1:])
    pad_clean = all(int(torch.count_nonzero(t[ds.N:])) == 0 for t in (ds.W, ds.m, ds.v))
    return replicas_equal, pad_clean, int(ds.status.item())


def _host_chunk(wl, steps, lo, n, pool):
    """The inputs of elements [lo, lo + n), regenerated on the host cores."""
    W0 = np.empty(n, np.float32)
    m0, v0 = np.empty_like(W0), np.empty_like(W0)
    G = {t: [np.empty(n, np.uint16) for _ in range(wl.R * wl.M)] for t in steps}
    part = -(-n // THREADS)

    def fill(k):
        a, b = k * part, min(n, (k + 1) * part)
        if a >= b:
            return
        idx = np.arange(lo + a, lo + b, dtype=np.int64)
        W0[a:b] = W.host_w0_at(wl, idx)
        mm, vv = W.host_mv0_at(wl, idx)
        m0[a:b], v0[a:b] = mm, vv
        for t in steps:
            for q, g in enumerate(W.host_grads_range(wl, t, lo + a, b - a)):
                G[t][q][a:b] = g

    list(pool.map(fill, range(THREADS)))
    return W0, m0, v0, G


def _whole_vector_mismatches(wl, ds, steps):
    """Chunk by chunk: the oracle over every element against the device."""
    hp = oracle.hparams(**wl.hparams())
    total = {}
    with ThreadPoolExecutor(THREADS) as pool:
        for lo in range(0, ds.N, CHUNK):
            n = min(CHUNK, ds.N - lo)
            Wc, mc, vc, G = _host_chunk(wl, steps, lo, n, pool)
            P = [np.zeros(n, np.uint16) for _ in range(wl.R)]
            for t in steps:
                oracle.dp_step(G[t], Wc, mc, vc, P, hp, t, wl.R, wl.M, nthreads=THREADS)
            del G
            sl = slice(lo, lo + n)
            got = (ds.W[sl].cpu().numpy(), ds.m[sl].cpu().numpy(), ds.v[sl].cpu().numpy(),
                   [H.u16_from_bf16(ds.params[0][sl])])
            want = (Wc, mc, vc, P[:1])
            if all(np.array_equal(a.view(np.uint32), b.view(np.uint32))
                   for a, b in zip(got[:3], want[:3])) and np.array_equal(got[3][0], P[0]):
                continue                           # every bit equal: nothing to count
            res = H.compare(got, want)
            for k, v in res.items():
                total[k] = total.get(k, 0) + v
    return total


@pytest.mark.parametrize("variant", [z.ZERO_VARIANT_FUSED, z.ZERO_VARIANT_STAGED])
@pytest.mark.parametrize("name", ["gpt2-small", "llama-3.2-1b", "uneven", "large"])
def test_full_size_every_element(name, variant):
    wl = W.ALL[name]()
    ds, steps = _device_run(wl, variant)
    replicas_equal, pad_clean, status = _everywhere(ds)
    assert replicas_equal, "replicas differ somewhere"
    assert pad_clean, "state pad written"
    assert status == 0, f"device status {status}"
    res = _whole_vector_mismatches(wl, ds, steps)
    del ds
    torch.cuda.empty_cache()
    bad = {key: v for key, v in res.items() if v}
    assert not bad, (name, bad)


def _run_sampled(wl, variant):
    ds, steps = _device_run(wl, variant)
    idx = _sample_indices(wl, ds.plan)
    it = torch.from_numpy(idx).to(ds.W.device)
    got = (ds.W[it].cpu().numpy(), ds.m[it].cpu().numpy(), ds.v[it].cpu().numpy(),
           [H.u16_from_bf16(p[it]) for p in ds.params])
    res = H.compare(got, _oracle_at(wl, idx, steps))
    replicas_equal, pad_clean, status = _everywhere(ds)
    del ds
    torch.cuda.empty_cache()
    return res, replicas_equal, pad_clean, status, idx.size


@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("S", [1 << 10, 1 << 16, 1 << 22, 1 << 28])
def test_flat_sweep_points_sampled(R, S):
    """The flat-vector sweep (fp32 master shard of 4 KB to 1 GB, N = R*S) at
    its smallest, two middle and largest shard sizes: sampled parity of the
    fused step against the oracle, replicas and pad checked everywhere.  The
    largest point at R = 8 holds about 88 GB on the device."""
    wl = W.sweep_point(R, S)
    res, replicas_equal, pad_clean, status, k = _run_sampled(wl, z.ZERO_VARIANT_FUSED)
    bad = {key: v for key, v in res.items() if v}
    assert not bad, (wl.name, bad, k)
    assert replicas_equal and pad_clean and status == 0


@pytest.mark.parametrize("name", ["gpt2-small", "llama-3.2-1b"])
def test_full_size_every_element_tma_variant(name):
    """The TMA-bulk-staged variant (R*M <= 16) at full size, every element
    against the oracle like the fused and staged steps."""
    wl = W.ALL[name]()
    ds, steps = _device_run(wl, z.ZERO_VARIANT_FUSED_TMA)
    replicas_equal, pad_clean, status = _everywhere(ds)
    assert replicas_equal and pad_clean and status == 0, (replicas_equal, pad_clean, status)
    res = _whole_vector_mismatches(wl, ds, steps)
    del ds
    torch.cuda.empty_cache()
    bad = {key: v for key, v in res.items() if v}
    assert not bad, (name, bad)
