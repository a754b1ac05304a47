"""GPU parity of the 1-bit Adam step (reading R15 of oracle/zero_oracle.h):
zero_step_onebit through the C ABI against oracle.onebit_step, bit for bit.

- Small cases: ragged sizes around the 128-element blocks, and several
  (R, M) pairs, compile-time and run-time.  The warm-up steps and several
  compressed steps run in sequence, so the residuals carry from one step to
  the next.
- Full-size cases: the GPT-2, Llama-3.2-1B and uneven workloads, in the
  launch configuration the benchmark times.  The oracle runs on sampled
  whole 128-element blocks (random ones, the first, the last ragged one,
  and those at shard and tensor boundaries), because a block is the
  codec's unit.  Properties that hold at any size are checked everywhere:
  the replicas agree bitwise, and the pad of the state and of the owner
  residual stays untouched.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import zero_optimizer_step_rs_gb300 as z
from tests import harness as H
from zgen import workloads as W

pytestmark = pytest.mark.gpu

BLOCK = 128


def _with_align(wl, align=BLOCK):
    return dataclasses.replace(wl, align=align)


def _bits(t):
    return t.detach().cpu().numpy().view(np.uint32)


def _run(wl, steps, freeze):
    """Host inputs, every element compared."""
    _, W0, m0, v0 = H.host_inputs(wl, steps[0])
    idx = np.arange(wl.N, dtype=np.int64)
    Wc, mc, vc = W0.copy(), m0.copy(), v0.copy()
    Pc = [np.zeros(wl.N, np.uint16) for _ in range(wl.R)]
    Ec = [np.zeros(wl.N, np.float32) for _ in range(wl.R)]
    Esc = np.zeros(wl.N, np.float32)
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.upload_state(W0, m0, v0)
    Ed = [torch.zeros(max(1, wl.N), dtype=torch.float32, device="cuda") for _ in range(wl.R)]
    Esd = torch.zeros(max(1, ds.padded), dtype=torch.float32, device="cuda")
    hp = oracle.hparams(**wl.hparams())
    for t in steps:
        G = W.host_grads_at(wl, t, idx)
        oracle.onebit_step(G, Wc, mc, vc, Pc, hp, t, freeze, wl.R, wl.M, ds.S, Ec, Esc)
        ds.upload_grads(G)
        z.zero_step_onebit(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t, freeze,
                           Ed, Esd)
    torch.cuda.synchronize()
    res = H.compare(ds.result(), (Wc, mc, vc, Pc))
    assert not {k: v for k, v in res.items() if v}, res
    N = wl.N
    for e_d, e_c in zip(Ed, Ec):
        assert np.array_equal(_bits(e_d[:N]), e_c.view(np.uint32))
    assert np.array_equal(_bits(Esd[:N]), Esc.view(np.uint32))
    assert int(torch.count_nonzero(Esd[N:])) == 0


@pytest.mark.parametrize("n", [1, 127, 128, 129, 1000, 4099, 100_003])
def test_onebit_matches_oracle(n):
    wl = _with_align(W.flat(4, 1, n, seed=n, step=1, state="synthetic"))
    _run(wl, [1, 2, 3, 4, 5], freeze=2)


@pytest.mark.parametrize("R,M", [(8, 1), (4, 1), (7, 4), (3, 2), (2, 2), (1, 1), (64, 4),
                                 (64, 1), (1, 256)])
def test_onebit_rank_microbatch_pairs(R, M):
    wl = _with_align(W.flat(R, M, 20_011, seed=R + M, step=1, state="synthetic"))
    _run(wl, [1, 2, 3, 4], freeze=1)


def test_onebit_generic_rank_count_at_a_persistent_grid_size():
    """(R, M) = (3, 2), the run-time path, over enough 128-element blocks
    that every warp of the persistent grid loops; warm-up, then the frozen
    phase."""
    _run(_with_align(W.flat(3, 2, 2_000_003, seed=44, step=1, state="synthetic")), [1, 2, 3],
         freeze=1)


def test_onebit_uneven_workload_scaled():
    _run(_with_align(W.uneven().scaled(200_000)), [1, 2, 3], freeze=1)


def test_onebit_wider_alignment():
    # S a multiple of 256: each owner's shard holds whole blocks either way
    _run(_with_align(W.flat(4, 2, 50_000, seed=3, step=1, state="synthetic"), 256), [1, 2, 3],
         freeze=1)


def test_onebit_rejects_shards_off_the_block_grid():
    wl = W.flat(4, 1, 100_000, seed=1, step=1, state="synthetic")       # align 64: S % 128 = 64
    ds = H.DeviceState(wl, staged_scratch=False)
    assert ds.S % BLOCK != 0
    Ed = [torch.zeros(wl.N, dtype=torch.float32, device="cuda") for _ in range(wl.R)]
    Esd = torch.zeros(ds.padded, dtype=torch.float32, device="cuda")
    with pytest.raises(z.ZeroError) as e:
        z.zero_step_onebit(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, 3, 2, Ed, Esd)
    assert e.value.code == -1


# ------------------------------------------------------------- full size --

def _sample_blocks(wl, plan, seed=321, n_random=160):
    N, S = plan.N, plan.S
    nblk = (N + BLOCK - 1) // BLOCK
    rng = np.random.default_rng(seed)
    blocks = set(rng.integers(0, nblk, n_random).tolist())
    blocks |= {0, 1, nblk - 2, nblk - 1}
    for r in range(1, wl.R):
        b = r * S // BLOCK
        blocks |= {b - 1, b}
    for off in wl.offsets[1:-1]:
        blocks.add(int(off) // BLOCK)
    blocks = sorted(b for b in blocks if 0 <= b < nblk)
    # the ragged last block goes last so that every block of the sample
    # starts at a multiple of 128 of the concatenation
    idx = np.concatenate([np.arange(b * BLOCK, min((b + 1) * BLOCK, N)) for b in blocks])
    return idx.astype(np.int64)


def _oracle_blocks(wl, idx, warm_steps, comp_steps, freeze):
    n = idx.size
    per = -(-n // wl.R)
    S = -(-per // BLOCK) * BLOCK          # shards on the block grid: server blocks = 128-blocks
    Wc = W.host_w0_at(wl, idx)
    mc, vc = W.host_mv0_at(wl, idx)
    Pc = [np.zeros(n, np.uint16) for _ in range(wl.R)]
    Ec = [np.zeros(n, np.float32) for _ in range(wl.R)]
    Esc = np.zeros(n, np.float32)
    hp = oracle.hparams(**wl.hparams())
    for t in warm_steps + comp_steps:
        G = W.host_grads_at(wl, t, idx)
        oracle.onebit_step(G, Wc, mc, vc, Pc, hp, t, freeze, wl.R, wl.M, S, Ec, Esc)
    return (Wc, mc, vc, Pc), Ec, Esc


@pytest.mark.parametrize("name", ["gpt2-small", "llama-3.2-1b", "uneven"])
def test_onebit_full_size_sampled_blocks(name):
    wl = _with_align(W.ALL[name]())
    freeze = wl.step
    warm = list(range(wl.first_step(), wl.step + 1))
    comp = [wl.step + 1, wl.step + 2]
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.fill_state_device()
    Ed = [torch.zeros(ds.N, dtype=torch.float32, device="cuda") for _ in range(wl.R)]
    Esd = torch.zeros(ds.padded, dtype=torch.float32, device="cuda")
    for t in warm + comp:
        ds.fill_grads_device(t)
        z.zero_step_onebit(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t, freeze,
                           Ed, Esd)
    torch.cuda.synchronize()
    idx = _sample_blocks(wl, ds.plan)
    it = torch.from_numpy(idx).to(ds.W.device)
    got = (ds.W[it].cpu().numpy(), ds.m[it].cpu().numpy(), ds.v[it].cpu().numpy(),
           [H.u16_from_bf16(p[it]) for p in ds.params])
    got_E = [_bits(e[it]) for e in Ed]
    got_Es = _bits(Esd[it])
    replicas_equal = all(torch.equal(p, ds.params[0]) for p in ds.params[1:])
    pad_clean = all(int(torch.count_nonzero(t[ds.N:])) == 0 for t in (ds.W, ds.m, ds.v, Esd))
    del ds, Ed, Esd, it
    torch.cuda.empty_cache()
    want, Ec, Esc = _oracle_blocks(wl, idx, warm, comp, freeze)
    res = H.compare(got, want)
    assert not {k: v for k, v in res.items() if v}, (name, res, idx.size)
    for g, e in zip(got_E, Ec):
        assert np.array_equal(g, e.view(np.uint32))
    assert np.array_equal(got_Es, Esc.view(np.uint32))
    assert replicas_equal, "replicas differ somewhere"
    assert pad_clean, "pad written"
