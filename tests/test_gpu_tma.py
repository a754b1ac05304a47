"""The TMA-bulk-staged fused variant (ZERO_VARIANT_FUSED_TMA): parity with the
oracle over tile boundaries and (R, M), and its bounded-wait timeout path.

The timeout is made without a fault: the test-only flag makes every bounded
wait give up at once; the kernel must then let its in-flight bulk copies
land, report ZERO_DEV_TIMEOUT in the status word and return, leaving the
context usable - the next, normal step must still match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu


def _tma_vs_oracle(wl, steps):
    _, W0, m0, v0 = H.host_inputs(wl, steps[0])
    idx = np.arange(wl.N, dtype=np.int64)
    Gs = {t: W.host_grads_at(wl, t, idx) for t in steps}
    want = H.oracle_run(wl, Gs, W0, m0, v0, steps)
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.upload_state(W0, m0, v0)
    for t in steps:
        ds.upload_grads(Gs[t])
        ds.step(t, variant=z.ZERO_VARIANT_FUSED_TMA, flags=z.ZERO_FLAG_CHECK_FINITE)
    torch.cuda.synchronize()
    res = H.compare(ds.result(), want)
    assert not {k: v for k, v in res.items() if v}, res
    assert int(ds.status.item()) == 0
    return ds


@pytest.mark.parametrize("n", [1, 1023, 1024, 1025, 3 * 4096 + 5, 100_003, 1_000_003])
@pytest.mark.parametrize("R,M", [(8, 1), (4, 2), (7, 2), (16, 1), (1, 1)])
def test_tma_variant_matches_oracle(n, R, M):
    _tma_vs_oracle(W.flat(R, M, n, seed=n + R, step=2), [2, 3])


def test_tma_variant_workload_recipes():
    _tma_vs_oracle(W.llama32_1b().scaled(2_000_000), [100])
    _tma_vs_oracle(W.gpt2_small().scaled(500_000), [1, 2])


def test_bounded_wait_timeout_reports_and_leaves_the_context_usable():
    wl = W.flat(8, 1, 300_000, seed=9, step=1)
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.upload_state(W0, m0, v0)
    ds.upload_grads(G)
    before = ds.result()
    ds.step(1, variant=z.ZERO_VARIANT_FUSED_TMA, flags=z.ZERO_FLAG_DEBUG_EXPIRE_WAITS)
    torch.cuda.synchronize()
    assert int(ds.status.item()) & z.ZERO_DEV_TIMEOUT
    after = ds.result()
    # no tile was computed: the state and the replicas are as they were
    for a, b in zip(after[:3], before[:3]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    for a, b in zip(after[3], before[3]):
        assert np.array_equal(a, b)
    # the same buffers, a normal step: matches the oracle
    ds.status.zero_()
    ds.step(1, variant=z.ZERO_VARIANT_FUSED_TMA)
    torch.cuda.synchronize()
    want = H.oracle_run(wl, {1: G}, W0, m0, v0, [1])
    res = H.compare(ds.result(), want)
    assert not {k: v for k, v in res.items() if v}, res
    assert int(ds.status.item()) == 0
