"""CUDA graph capture of the step entry points.

A training loop can capture its optimizer step once and replay it: the
entry points only enqueue kernels on the caller's stream (no allocation, no
host synchronisation, launch attributes allowed in capture). Three steps
(t = 1, 2, 3) of one entry point are captured into one graph, and the graph
is replayed twice. The step scalars are kernel arguments, so the replays run
t = 1, 2, 3, 1, 2, 3. The result must equal the oracle over that same
sequence, bit for bit. A first call on buffers of the same plan before the
capture fills the library's per-device caches (occupancy, kernel attributes).
"""
import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu

STEPS = [1, 2, 3]
MAX_NORM = 1e-3


def _enqueue(variant, ds, t, extra):
    if variant == "fused":
        ds.step(t, variant=z.ZERO_VARIANT_FUSED)
    elif variant == "staged":
        ds.step(t, variant=z.ZERO_VARIANT_STAGED)
    elif variant == "clipped":
        z.zero_step_clipped(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t, MAX_NORM,
                            extra)
    else:                                                   # zero3
        z.zero3_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, extra, ds.hp, t)


def _extra(variant, ds):
    if variant == "clipped":
        return torch.empty(z.zero_clip_scratch_bytes(ds.plan), dtype=torch.uint8, device="cuda")
    if variant == "zero3":
        return torch.zeros(ds.padded, dtype=torch.bfloat16, device="cuda")
    return None


@pytest.mark.parametrize("variant", ["fused", "staged", "clipped", "zero3"])
def test_steps_captured_in_a_cuda_graph_match_the_oracle(variant):
    wl = W.flat(8, 1, 1_000_003, seed=61, step=1)
    G, W0, m0, v0 = H.host_inputs(wl, 1)
    seq = STEPS * 2

    # warm-up on buffers of the same plan, then the capture on fresh ones
    warm = H.DeviceState(wl)
    warm.upload_state(W0, m0, v0)
    warm.upload_grads(G)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _enqueue(variant, warm, 1, _extra(variant, warm))
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    ds = H.DeviceState(wl)
    ds.upload_state(W0, m0, v0)
    ds.upload_grads(G)
    extra = _extra(variant, ds)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for t in STEPS:
            _enqueue(variant, ds, t, extra)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()

    hp = oracle.hparams(**wl.hparams())
    Wc, mc, vc = W0.copy(), m0.copy(), v0.copy()
    if variant in ("fused", "staged", "clipped"):
        P = [np.zeros(wl.N, np.uint16) for _ in range(wl.R)]
        for t in seq:
            if variant == "clipped":
                oracle.dp_step_clipped(G, Wc, mc, vc, P, hp, t, wl.R, wl.M, max_norm=MAX_NORM)
            else:
                oracle.dp_step(G, Wc, mc, vc, P, hp, t, wl.R, wl.M)
        res = H.compare(ds.result(), (Wc, mc, vc, P))
        assert not {k: v for k, v in res.items() if v}, res
    else:
        plan = ds.plan
        Wz = np.zeros(plan.padded, np.float32)
        mz, vz = Wz.copy(), Wz.copy()
        Wz[:wl.N], mz[:wl.N], vz[:wl.N] = Wc, mc, vc
        Ps = np.zeros(plan.padded, np.uint16)
        for t in seq:
            oracle.zero3_step(G, Wz, mz, vz, Ps, hp, t, wl.R, wl.M, plan.N, plan.S)
        assert np.array_equal(H.u16_from_bf16(extra), Ps)
        for dev, want in ((ds.W, Wz), (ds.m, mz), (ds.v, vz)):
            assert np.array_equal(dev.cpu().numpy().view(np.uint32)[:wl.N],
                                  want.view(np.uint32)[:wl.N])
