"""Silent-data-corruption detection without a GPU fault: the failure is made on
the host (one element of one rank's replica is overwritten through torch),
and zero_check_replicas must find it (LLM infra 06, section 15.4)."""
import numpy as np
import pytest
import torch

import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu


def _check(ds):
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    first = torch.zeros(1, dtype=torch.int64, device="cuda")
    z.zero_check_replicas(ds.plan, ds.params, cnt, first)
    torch.cuda.synchronize()
    return int(cnt.item()), int(first.item())


@pytest.mark.parametrize("n", [1, 9, 4096 + 3, 1_000_003])
def test_clean_step_has_equal_replicas(n):
    wl = W.flat(8, 1, n, seed=n, step=1)
    ds = H.DeviceState(wl)
    ds.fill_state_device()
    ds.fill_grads_device(1)
    ds.step(1)
    assert _check(ds) == (0, 2 ** 63 - 1)


@pytest.mark.parametrize("n", [9, 4096 + 3, 1_000_003])
def test_corrupted_replica_is_found(n):
    wl = W.flat(8, 1, n, seed=n + 1, step=1)
    ds = H.DeviceState(wl)
    ds.fill_state_device()
    ds.fill_grads_device(1)
    ds.step(1)
    torch.cuda.synchronize()
    rng = np.random.default_rng(n)
    hits = sorted(set(int(i) for i in rng.integers(0, n, 3)))
    for i in hits:                        # one bit flipped in rank 5's copy (host-side write)
        r = ds.params[5].view(torch.int16)
        r[i] = r[i] ^ 0x0001
    assert _check(ds) == (len(hits), hits[0])
    # an untouched rank pair stays consistent once the corruption is repaired
    ds.params[5].copy_(ds.params[0])
    assert _check(ds) == (0, 2 ** 63 - 1)
