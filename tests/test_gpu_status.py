"""zero_get_device_status: the device status word as a status code.

The steps OR ZERO_DEV_* bits into a caller-owned device word; this call waits
for the stream, reads the word and maps it to ZERO_OK, ZERO_ERR_NONFINITE or
ZERO_ERR_DEVICE_TIMEOUT (failure detection: find and report, do not hang;
LLM infra 06, section 15.4).  Every condition is made without a GPU fault: a
clean step, an Inf gradient planted on the host, the clipped step's skip on a
non-finite norm, and the TMA variant's test-only flag that makes every
bounded wait give up at once (the kernel drains its copies and returns).
"""
import numpy as np
import pytest
import torch

import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zero_optimizer_step_rs_gb300 import binding as B
from zgen import workloads as W

pytestmark = pytest.mark.gpu


def _state(n=300_000, R=8, M=1, seed=21):
    wl = W.flat(R, M, n, seed=seed, step=1)
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    ds = H.DeviceState(wl, staged_scratch=True)
    ds.upload_state(W0, m0, v0)
    return wl, G, ds


@pytest.mark.parametrize("variant", [z.ZERO_VARIANT_FUSED, z.ZERO_VARIANT_STAGED,
                                     z.ZERO_VARIANT_FUSED_TMA])
def test_clean_step_reads_ok(variant):
    wl, G, ds = _state()
    ds.upload_grads(G)
    ds.step(1, variant=variant, flags=z.ZERO_FLAG_CHECK_FINITE)
    code, word = z.zero_get_device_status(ds.status)
    assert (code, word) == (B.ZERO_OK, 0)


@pytest.mark.parametrize("variant", [z.ZERO_VARIANT_FUSED, z.ZERO_VARIANT_STAGED,
                                     z.ZERO_VARIANT_FUSED_TMA])
def test_inf_gradient_reads_nonfinite(variant):
    wl, G, ds = _state()
    G = [g.copy() for g in G]
    G[5][123_457] = 0x7F80                          # +Inf, rank 5
    ds.upload_grads(G)
    ds.step(1, variant=variant, flags=z.ZERO_FLAG_CHECK_FINITE)
    code, word = z.zero_get_device_status(ds.status)
    assert code == B.ZERO_ERR_NONFINITE
    assert word == B.ZERO_DEV_NONFINITE
    with pytest.raises(B.ZeroError) as e:
        z.zero_get_device_status(ds.status, raise_on_error=True)
    assert e.value.code == B.ZERO_ERR_NONFINITE
    # the word is read, not cleared: zeroing it makes the next clean step read OK
    ds.status.zero_()
    ds.upload_grads(H.host_inputs(wl, 1)[0])
    ds.step(2, variant=variant, flags=z.ZERO_FLAG_CHECK_FINITE)
    assert z.zero_get_device_status(ds.status) == (B.ZERO_OK, 0)


def test_clipped_skip_reads_nonfinite_with_the_skip_bit():
    wl, G, ds = _state(n=200_003, R=4, M=2)
    G = [g.copy() for g in G]
    G[3][1234] = 0xFF80                             # -Inf
    ds.upload_grads(G)
    ds.step_clipped(1, 1.0, flags=z.ZERO_FLAG_SKIP_NONFINITE)
    code, word = z.zero_get_device_status(ds.status)
    assert code == B.ZERO_ERR_NONFINITE
    assert word == B.ZERO_DEV_NONFINITE | B.ZERO_DEV_SKIPPED


def test_expired_waits_read_timeout_and_the_context_stays_usable():
    wl, G, ds = _state()
    ds.upload_grads(G)
    ds.step(1, variant=z.ZERO_VARIANT_FUSED_TMA,
            flags=z.ZERO_FLAG_DEBUG_EXPIRE_WAITS | z.ZERO_FLAG_CHECK_FINITE)
    code, word = z.zero_get_device_status(ds.status)
    assert code == B.ZERO_ERR_DEVICE_TIMEOUT
    assert word & B.ZERO_DEV_TIMEOUT
    # every block's copies landed before it left: the drain never ran out
    assert not word & B.ZERO_DEV_DRAIN_FAILED
    # timeout outranks a non-finite bit in the same word
    ds.status.fill_(B.ZERO_DEV_TIMEOUT | B.ZERO_DEV_NONFINITE)
    assert z.zero_get_device_status(ds.status)[0] == B.ZERO_ERR_DEVICE_TIMEOUT
    # a normal step on the same context afterwards matches the oracle
    ds.status.zero_()
    ds.step(1, variant=z.ZERO_VARIANT_FUSED_TMA, flags=z.ZERO_FLAG_CHECK_FINITE)
    assert z.zero_get_device_status(ds.status) == (B.ZERO_OK, 0)
    _, W0, m0, v0 = H.host_inputs(wl, 1)
    want = H.oracle_run(wl, {1: G}, W0, m0, v0, [1])
    res = H.compare(ds.result(), want)
    assert not {k: v for k, v in res.items() if v}, res


def test_status_read_is_ordered_after_the_step_on_its_stream():
    """The read is enqueued on the step's stream: a side stream whose step
    reports a non-finite gradient is seen without a device-wide sync."""
    wl, G, ds = _state()
    G = [g.copy() for g in G]
    G[0][7] = 0x7FC1                                # NaN
    ds.upload_grads(G)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ds.step(1, flags=z.ZERO_FLAG_CHECK_FINITE)
    code, word = z.zero_get_device_status(ds.status, stream=side)
    assert code == B.ZERO_ERR_NONFINITE and word == B.ZERO_DEV_NONFINITE
    assert np.isnan(ds.W[7].item())
