"""Device checkpoints: asynchronous save ordered before the next step, load
under another rank count, and a bit-identical resume (CS324 Lecture 9 notes,
section 3.1: PaLM reruns bitwise from any checkpoint)."""
import numpy as np
import pytest
import torch

import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu


def _device_state(wl):
    ds = H.DeviceState(wl)
    ds.fill_state_device()
    return ds


def test_resume_is_bit_identical(tmp_path):
    wl = W.uneven().scaled(300_000)
    a = _device_state(wl)
    for t in (1, 2, 3):
        a.fill_grads_device(t)
        a.step(t)
    job = z.zero_ckpt_save_async(a.plan, a.params[0][:a.N], a.W[:a.N], a.m[:a.N], a.v[:a.N], 3,
                                 a.hp, str(tmp_path))
    job.wait()
    # uninterrupted: step 4
    a.fill_grads_device(4)
    a.step(4)
    torch.cuda.synchronize()
    # resumed: fresh buffers, load, step 4
    b = H.DeviceState(wl)
    step, hp = z.zero_ckpt_load(b.plan, str(tmp_path), [p[:b.N] for p in b.params], b.W[:b.N],
                                b.m[:b.N], b.v[:b.N])
    assert step == 3 and hp.lr == np.float32(wl.lr)
    b.fill_grads_device(4)
    b.step(4)
    torch.cuda.synchronize()
    ra, rb = a.result(), b.result()
    for x, y in zip(ra[:3], rb[:3]):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    for x, y in zip(ra[3], rb[3]):
        assert np.array_equal(x, y)


def test_async_save_snapshots_the_state_before_the_next_step(tmp_path):
    wl = W.llama32_1b().scaled(2_000_000)
    ds = _device_state(wl)
    ds.fill_grads_device(wl.step)
    ds.step(wl.step)
    torch.cuda.synchronize()
    before = ds.result()
    job = z.zero_ckpt_save_async(ds.plan, ds.params[0][:ds.N], ds.W[:ds.N], ds.m[:ds.N],
                                 ds.v[:ds.N], wl.step, ds.hp, str(tmp_path))
    ds.step(wl.step + 1)                 # enqueued right away; the copies come first
    job.wait()
    N = ds.N
    params = np.zeros(N, np.uint16)
    Wh = np.zeros(ds.padded, np.float32)
    mh, vh = Wh.copy(), Wh.copy()
    step, _ = z.zero_ckpt_read_host(ds.plan, str(tmp_path), params, Wh, mh, vh)
    assert step == wl.step
    assert np.array_equal(params, before[3][0])
    assert np.array_equal(Wh[:N].view(np.uint32), before[0].view(np.uint32))
    assert np.array_equal(mh[:N].view(np.uint32), before[1].view(np.uint32))
    assert np.array_equal(vh[:N].view(np.uint32), before[2].view(np.uint32))
    # the step after the save did change all three, so the snapshot is not the later state
    after = ds.result()
    for k in range(3):
        assert not np.array_equal(after[k].view(np.uint32), before[k].view(np.uint32))


@pytest.mark.parametrize("R_new", [7, 1, 16])
def test_load_under_another_rank_count(tmp_path, R_new):
    import dataclasses
    wl = W.uneven().scaled(400_000)
    ds = _device_state(wl)
    ds.fill_grads_device(1)
    ds.step(1)
    job = z.zero_ckpt_save_async(ds.plan, ds.params[0][:ds.N], ds.W[:ds.N], ds.m[:ds.N],
                                 ds.v[:ds.N], 1, ds.hp, str(tmp_path))
    job.wait()
    torch.cuda.synchronize()
    want = ds.result()
    wl2 = dataclasses.replace(wl, R=R_new, M=1)
    ds2 = H.DeviceState(wl2)
    z.zero_ckpt_load(ds2.plan, str(tmp_path), [p[:ds2.N] for p in ds2.params], ds2.W[:ds2.N],
                     ds2.m[:ds2.N], ds2.v[:ds2.N])
    got = ds2.result()
    for x, y in zip(got[:3], want[:3]):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    for p in got[3]:
        assert np.array_equal(p, want[3][0])


def test_zero3_shard_buffer_checkpoint(tmp_path):
    wl = W.llama32_1b().scaled(500_000)
    ds = _device_state(wl)
    ds.fill_grads_device(wl.step)
    shards = torch.zeros(ds.padded, dtype=torch.bfloat16, device="cuda")
    z.zero3_step(ds.plan, ds.grads, ds.W, ds.m, ds.v, shards, ds.hp, wl.step)
    job = z.zero_ckpt_save_async(ds.plan, shards[:ds.N], ds.W[:ds.N], ds.m[:ds.N], ds.v[:ds.N],
                                 wl.step, ds.hp, str(tmp_path))
    job.wait()
    shards2 = torch.zeros(ds.padded, dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros_like(ds.W)
    m2, v2 = torch.zeros_like(ds.W), torch.zeros_like(ds.W)
    z.zero_ckpt_load(ds.plan, str(tmp_path), [shards2[:ds.N]], W2[:ds.N], m2[:ds.N], v2[:ds.N])
    assert torch.equal(shards2.view(torch.int16), shards.view(torch.int16))
    assert torch.equal(W2.view(torch.int32), ds.W.view(torch.int32))
