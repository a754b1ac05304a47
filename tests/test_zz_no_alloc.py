"""The allocation-free staged step (zero_step_staged_noalloc).

Some callers cannot allocate device memory (a runtime that has reserved the
GPU's memory for its own pool, or a latency-critical caller that may not call
cudaMalloc); this entry point gives them the staged step with its scratch in
a fixed device array owned by the library.  The test calls it through the C
ABI twice in a row and checks each result both against the CPU oracle on the
same inputs and against the existing staged entry point (zero_step with
caller scratch), with the bar the other parity tests use: replicas bit for
bit, fp32 state within 1e-6 (and, by design, bit for bit).  One case fills
the array to its last element.
This file sorts last so that a run stopping at its first failure has run
every other test; it passes alone in a fresh process and after the others.
"""
import numpy as np
import pytest
import torch

import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zero_optimizer_step_rs_gb300 import binding as B
from zgen import workloads as W

pytestmark = pytest.mark.gpu


def _pair(wl, G, W0, m0, v0):
    ref = H.DeviceState(wl, staged_scratch=True)
    new = H.DeviceState(wl, staged_scratch=False)
    for ds in (ref, new):
        ds.upload_state(W0, m0, v0)
        ds.upload_grads(G)
    return ref, new


def _no_alloc_step(ds, t, flags=0):
    z.zero_step_staged_noalloc(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t,
                               flags=flags, dev_status=ds.status)


def _assert_same(got, want, what):
    res = H.compare(got, want)
    bad = {k: v for k, v in res.items() if v}
    assert not bad, (what, bad)


def _two_calls_against_oracle_and_staged(wl):
    t0 = wl.first_step()
    steps = [t0, t0 + 1]
    idx = np.arange(wl.N, dtype=np.int64)
    Gs = {t: W.host_grads_at(wl, t, idx) for t in steps}
    W0 = W.host_w0_at(wl, idx)
    m0, v0 = W.host_mv0_at(wl, idx)
    ref, new = _pair(wl, Gs[t0], W0, m0, v0)
    for k, t in enumerate(steps):
        if k:
            ref.upload_grads(Gs[t])
            new.upload_grads(Gs[t])
        ref.step(t, variant=z.ZERO_VARIANT_STAGED, flags=z.ZERO_FLAG_CHECK_FINITE)
        _no_alloc_step(new, t, flags=z.ZERO_FLAG_CHECK_FINITE)
        torch.cuda.synchronize()
        got = new.result()
        want = H.oracle_run(wl, Gs, W0, m0, v0, steps[:k + 1])
        _assert_same(got, want, f"oracle, call {k + 1}")
        _assert_same(got, ref.result(), f"staged zero_step, call {k + 1}")
        assert int(new.status.item()) == 0


@pytest.mark.parametrize("name,target", [("uneven", 300_000), ("llama-3.2-1b", 1_000_000)])
def test_no_alloc_step_matches_oracle_and_staged_step_on_two_calls(name, target):
    wl = W.ALL[name]().scaled(target)
    assert H.DeviceState(wl, staged_scratch=False).padded <= B.ZERO_NOALLOC_MAX_ELEMS
    _two_calls_against_oracle_and_staged(wl)


def test_no_alloc_step_fills_the_array_to_its_last_element():
    # R = 8 ranks over exactly ZERO_NOALLOC_MAX_ELEMS elements: padded equals
    # the array's size, so the last shard's last element is the array's last
    wl = W.flat(8, 1, B.ZERO_NOALLOC_MAX_ELEMS, seed=77, step=3)
    plan = z.Plan(wl.numels, wl.R, wl.M, wl.stage, wl.align)
    assert plan.padded == plan.N == B.ZERO_NOALLOC_MAX_ELEMS
    _two_calls_against_oracle_and_staged(wl)


def test_no_alloc_array_reused_by_a_smaller_plan():
    # the array keeps the previous call's contents; a smaller plan after a
    # larger one must still match (nothing in it needs clearing)
    for target in (900_000, 70_001):
        wl = W.uneven().scaled(target)
        G, W0, m0, v0 = H.host_inputs(wl, 1)
        ref, new = _pair(wl, G, W0, m0, v0)
        ref.step(1, variant=z.ZERO_VARIANT_STAGED)
        _no_alloc_step(new, 1)
        torch.cuda.synchronize()
        got = new.result()
        _assert_same(got, H.oracle_run(wl, {1: G}, W0, m0, v0, [1]), ("oracle", target))
        _assert_same(got, ref.result(), ("staged zero_step", target))


def test_no_alloc_refuses_plans_beyond_the_array():
    wl = W.flat(8, 1, B.ZERO_NOALLOC_MAX_ELEMS + 1)
    plan = z.Plan(wl.numels, wl.R, wl.M, wl.stage, wl.align)
    assert plan.padded > B.ZERO_NOALLOC_MAX_ELEMS
    dev = torch.device("cuda")
    one = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    st = torch.zeros(16, dtype=torch.float32, device=dev)
    # size is checked before any pointer or launch: nothing runs
    with pytest.raises(B.ZeroError) as e:
        B.lib()
        import ctypes
        ga = B._ptrs([one.data_ptr()] * (wl.R * wl.M))
        pa = B._ptrs([one.data_ptr()] * wl.R)
        hp = z.hparams()
        code = B.lib().zero_step_staged_noalloc(plan.ptr, ctypes.addressof(ga), st.data_ptr(),
                                                st.data_ptr(), st.data_ptr(),
                                                ctypes.addressof(pa), ctypes.byref(hp), 1, 0,
                                                None, None)
        B._check(code, "zero_step_staged_noalloc")
    assert e.value.code == B.ZERO_ERR_SIZE
