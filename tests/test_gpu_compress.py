"""GPU parity of the step with a compressed reduce-scatter (reading R14):
zero_step_compressed through the C ABI against oracle.dp_step_compressed,
for fp16, block-int8 and sign codecs, with and without error feedback, over
several steps (the residuals carried between them), ragged sizes around the
128-element blocks, and run-time (R, M).  Everything bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu

KINDS = [(z.ZERO_COMP_FP16, oracle.COMP_FP16), (z.ZERO_COMP_INT8, oracle.COMP_INT8),
         (z.ZERO_COMP_SIGN, oracle.COMP_SIGN)]


def _run(wl, kind, ef, steps):
    gk, ok = kind
    _, W0, m0, v0 = H.host_inputs(wl, steps[0])
    idx = np.arange(wl.N, dtype=np.int64)
    Wc, mc, vc = W0.copy(), m0.copy(), v0.copy()
    Pc = [np.zeros(wl.N, np.uint16) for _ in range(wl.R)]
    Ec = [np.zeros(wl.N, np.float32) for _ in range(wl.R)] if ef else None
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.upload_state(W0, m0, v0)
    Ed = [torch.zeros(wl.N, dtype=torch.float32, device="cuda") for _ in range(wl.R)] if ef else None
    hp = oracle.hparams(**wl.hparams())
    for t in steps:
        G = W.host_grads_at(wl, t, idx)
        oracle.dp_step_compressed(G, Wc, mc, vc, Pc, hp, t, wl.R, wl.M, ok, Ec)
        ds.upload_grads(G)
        z.zero_step_compressed(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t, gk, Ed)
    torch.cuda.synchronize()
    res = H.compare(ds.result(), (Wc, mc, vc, Pc))
    assert not {k: v for k, v in res.items() if v}, res
    if ef:
        for e_d, e_c in zip(Ed, Ec):
            assert np.array_equal(e_d.cpu().numpy().view(np.uint32), e_c.view(np.uint32))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("n", [1, 127, 128, 129, 1000, 4099, 100_003])
def test_compressed_step_matches_oracle(kind, ef, n):
    _run(W.flat(4, 1, n, seed=n, step=1, state="synthetic"), kind, ef, [1, 2, 3])


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("R,M", [(8, 1), (7, 4), (3, 2), (64, 4), (1, 256)])
def test_compressed_rank_microbatch_pairs(kind, R, M):
    _run(W.flat(R, M, 20_011, seed=R + M, step=1, state="synthetic"), kind, True, [1, 2])


def test_compressed_uneven_workload_scaled():
    _run(W.uneven().scaled(200_000), KINDS[1], True, [1, 2])
