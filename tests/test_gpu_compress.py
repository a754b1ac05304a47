"""GPU parity of the step with a compressed reduce-scatter (reading R14 of
oracle/zero_oracle.h): zero_step_compressed through the C ABI against
oracle.dp_step_compressed,
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
@pytest.mark.parametrize("R,M", [(8, 1), (4, 1), (7, 4), (3, 2), (64, 4), (1, 256)])
@pytest.mark.parametrize("ef", [False, True])
def test_compressed_rank_microbatch_pairs(kind, R, M, ef):
    _run(W.flat(R, M, 20_011, seed=R + M, step=1, state="synthetic"), kind, ef, [1, 2])


def test_compressed_uneven_workload_scaled():
    _run(W.uneven().scaled(200_000), KINDS[1], True, [1, 2])


def _split3(x):
    """bf16 bit patterns (hi, mid, lo) whose fp32 sum ((hi + mid) + lo) is x
    exactly, or None when three pieces do not carry x's bits."""
    x = np.float32(x)
    pieces, rest = [], x
    for _ in range(3):
        b = oracle.bf16_rne(float(rest))
        f = np.float32(oracle.bf16_to_float(b))
        pieces.append(b)
        rest = np.float32(rest - f)
    f = [np.float32(oracle.bf16_to_float(b)) for b in pieces]
    return pieces if np.float32(np.float32(f[0] + f[1]) + f[2]) == x else None


def test_int8_codes_at_half_integer_quotients():
    """Without error feedback a rank's x is the fp32 sum of its M bf16
    micro-batch values, so with M = 3 any fp32 x can be built exactly.  Each
    block holds its max A and values within a few ulps of (j +- 1/2) * s,
    s = A / 127: the quotients x / s land on and around the half-integers
    where the rounded code changes.  Some blocks have scales outside the
    reciprocal path's range (2^-100 .. 2^100), one block is all zero."""
    R, M = 2, 3
    rng = np.random.default_rng(2024)
    scales = [float(2.0 ** e * rng.uniform(1, 2)) for e in rng.integers(-60, 40, 90)]
    scales += [2.0 ** -118 * 1.3, 2.0 ** -105, 2.0 ** 108 * 1.7, 2.0 ** 110]   # fallback path
    scales += [2.0 ** -93 * 1.01, 2.0 ** 106 * 1.9]           # s just inside the range
    xs = [[] for _ in range(R)]
    for A in scales + [0.0]:
        A = np.float32(oracle.bf16_to_float(oracle.bf16_rne(A)))     # one bf16 piece
        s = np.float32(A / np.float32(127.0))
        for r in range(R):
            blk = [A if r == 0 else -A]
            while len(blk) < 128:
                if A == 0:
                    blk.append(np.float32(0.0))
                    continue
                j = int(rng.integers(-127, 127))
                t = np.float32((j + 0.5) * np.float64(s))
                t = (np.array([t], np.float32).view(np.int32) + int(rng.integers(-3, 4))).view(np.float32)[0]
                if abs(t) <= A and _split3(t) is not None:
                    blk.append(t)
            xs[r].extend(blk)
    n = len(xs[0])
    G = [np.zeros(n, np.uint16) for _ in range(R * M)]
    for r in range(R):
        for i, x in enumerate(xs[r]):
            p = _split3(x)
            assert p is not None
            for j in range(M):
                G[r * M + j][i] = p[j]
    wl = W.flat(R, M, n, seed=1, step=1, state="zero")
    W0 = np.zeros(n, np.float32)
    m0, v0 = np.zeros(n, np.float32), np.zeros(n, np.float32)
    Wc, mc, vc = W0.copy(), m0.copy(), v0.copy()
    Pc = [np.zeros(n, np.uint16) for _ in range(R)]
    hp = oracle.hparams(**wl.hparams())
    oracle.dp_step_compressed(G, Wc, mc, vc, Pc, hp, 1, R, M, oracle.COMP_INT8, None)
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.upload_state(W0, m0, v0)
    ds.upload_grads(G)
    z.zero_step_compressed(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, 1,
                           z.ZERO_COMP_INT8, None)
    torch.cuda.synchronize()
    res = H.compare(ds.result(), (Wc, mc, vc, Pc))
    assert not {k: v for k, v in res.items() if v}, res


def _regime_block(rng, regime):
    """128 bf16 bit patterns of one block in one magnitude regime."""
    sign = rng.integers(0, 2, 128).astype(np.uint32) << 31
    if regime == "zero":
        f = np.zeros(128, np.float32)
    elif regime == "single":
        f = np.zeros(128, np.float32)
        f[rng.integers(0, 128)] = np.float32(2.0 ** int(rng.integers(-20, 20)))
    elif regime == "subnormal":                    # bf16 subnormals, 2^-133 .. 2^-127
        f = (rng.uniform(1, 2, 128) * 2.0 ** rng.integers(-133, -127, 128)).astype(np.float32)
    elif regime == "tiny":                         # block scale below 2^-100
        f = (rng.uniform(1, 2, 128) * 2.0 ** int(rng.integers(-126, -108))).astype(np.float32)
    elif regime == "huge":                         # block scale around and above 2^100
        f = (rng.uniform(1, 2, 128) * 2.0 ** int(rng.integers(100, 114))).astype(np.float32)
    elif regime == "halfint":                      # quotients near j + 1/2 (as bf16 allows)
        A = np.float32(rng.uniform(1, 2) * 2.0 ** int(rng.integers(-40, 40)))
        s = np.float64(A) / 127.0
        j = rng.integers(-127, 127, 128)
        f = np.minimum(np.abs(((j + 0.5) * s).astype(np.float32)), A)
        f[0] = A
    else:                                          # "normal": mixed magnitudes
        f = (rng.standard_normal(128) * 10.0 ** int(rng.integers(-6, 1))).astype(np.float32)
    bits = (np.abs(f).view(np.uint32) | sign) >> 16
    return bits.astype(np.uint16)


@pytest.mark.parametrize("kind", KINDS[1:])
@pytest.mark.parametrize("R,M", [(8, 1), (4, 1), (7, 4), (2, 3)])
@pytest.mark.parametrize("ef", [False, True])
def test_codecs_on_extreme_blocks(kind, R, M, ef):
    """int8 and sign codecs on blocks of zeros, a single value, bf16
    subnormals, scales far below and above the reciprocal path's range,
    quotients near half-integers and mixed magnitudes, for the compile-time
    (R, M) cases (8, 1), (4, 1), (7, 4) and a run-time one, with a ragged last
    block; two steps, so the error-feedback residuals are used."""
    gk, ok = kind
    rng = np.random.default_rng(R * 100 + M + (7 if ef else 0) + gk)
    regimes = ["zero", "single", "subnormal", "tiny", "huge", "halfint", "normal"]
    nblk = 3 * len(regimes)
    n = nblk * 128 + 37
    idx = np.arange(n, dtype=np.int64)
    wl = W.flat(R, M, n, seed=R + M, step=1, state="synthetic")
    _, W0, m0, v0 = H.host_inputs(wl, 1)
    Wc, mc, vc = W0.copy(), m0.copy(), v0.copy()
    Pc = [np.zeros(n, np.uint16) for _ in range(R)]
    Ec = [np.zeros(n, np.float32) for _ in range(R)] if ef else None
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.upload_state(W0, m0, v0)
    Ed = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(R)] if ef else None
    hp = oracle.hparams(**wl.hparams())
    for t in (1, 2):
        G = []
        for q in range(R * M):
            g = np.empty(n, np.uint16)
            for b in range(nblk + 1):
                blk = _regime_block(rng, regimes[int(rng.integers(0, len(regimes)))])
                g[b * 128:min(n, b * 128 + 128)] = blk[:min(128, n - b * 128)]
            G.append(g)
        oracle.dp_step_compressed(G, Wc, mc, vc, Pc, hp, t, R, M, ok, Ec)
        ds.upload_grads(G)
        z.zero_step_compressed(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t, gk, Ed)
    torch.cuda.synchronize()
    res = H.compare(ds.result(), (Wc, mc, vc, Pc))
    assert not {k: v for k, v in res.items() if v}, res
    if ef:
        for e_d, e_c in zip(Ed, Ec):
            got, want = e_d.cpu().numpy(), e_c
            nan = np.isnan(want)
            assert np.array_equal(np.isnan(got), nan)
            assert np.array_equal(got.view(np.uint32)[~nan], want.view(np.uint32)[~nan])


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("ef", [False, True])
def test_compressed_step_at_a_persistent_grid_size(kind, ef):
    """4 M elements at R = 8: enough 128-element blocks that every launch
    runs its persistent grid (for the sign codec without error feedback the
    grid below the resident maximum), whole vector against the oracle."""
    _run(W.flat(8, 1, 4_000_037, seed=41, step=1, state="synthetic"), kind, ef, [1, 2])


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("ef", [False, True])
def test_generic_rank_count_at_a_persistent_grid_size(kind, ef):
    """(R, M) = (3, 2) has no compile-time case: the run-time path, over
    enough blocks that every warp of the persistent grid loops, whole vector
    against the oracle."""
    _run(W.flat(3, 2, 2_000_003, seed=43, step=1, state="synthetic"), kind, ef, [1, 2])


# ------------------------------------------------------------- full size --

def _sample_blocks(wl, plan, seed=777, n_random=160):
    """Whole 128-element compression blocks: random ones, the first and
    last, those at shard and tensor boundaries; the ragged last block last,
    so every block of the concatenation starts at a multiple of 128."""
    N, S = plan.N, plan.S
    nblk = (N + 127) // 128
    rng = np.random.default_rng(seed)
    blocks = set(rng.integers(0, nblk, n_random).tolist()) | {0, 1, nblk - 2, nblk - 1}
    for r in range(1, wl.R):
        blocks |= {r * S // 128 - 1, r * S // 128}
    for off in wl.offsets[1:-1]:
        blocks.add(int(off) // 128)
    blocks = sorted(b for b in blocks if 0 <= b < nblk)
    return np.concatenate([np.arange(b * 128, min((b + 1) * 128, N)) for b in blocks]).astype(np.int64)


@pytest.mark.parametrize("name,kind,ef", [
    ("llama-3.2-1b", KINDS[2], False), ("llama-3.2-1b", KINDS[1], False),
    ("llama-3.2-1b", KINDS[1], True), ("gpt2-small", KINDS[2], True),
    ("gpt2-small", KINDS[0], False), ("uneven", KINDS[2], False), ("uneven", KINDS[1], True)])
def test_compressed_full_size_sampled_blocks(name, kind, ef):
    """The workloads at full size, in the launch configuration the benchmark
    times: every step from the workload's first to its measured step on the
    device, the oracle on sampled whole blocks (the codec acts per block,
    the rest per element); replicas equal and the pad untouched everywhere."""
    gk, ok = kind
    wl = W.ALL[name]()
    steps = list(range(wl.first_step(), wl.step + 1))
    ds = H.DeviceState(wl, staged_scratch=False)
    ds.fill_state_device()
    Ed = [torch.zeros(ds.N, dtype=torch.float32, device="cuda") for _ in range(wl.R)] if ef else None
    for t in steps:
        ds.fill_grads_device(t)
        z.zero_step_compressed(ds.plan, ds.grads, ds.W, ds.m, ds.v, ds.params, ds.hp, t, gk, Ed)
    torch.cuda.synchronize()
    idx = _sample_blocks(wl, ds.plan)
    it = torch.from_numpy(idx).to(ds.W.device)
    got = (ds.W[it].cpu().numpy(), ds.m[it].cpu().numpy(), ds.v[it].cpu().numpy(),
           [H.u16_from_bf16(p[it]) for p in ds.params])
    got_E = [e[it].cpu().numpy() for e in Ed] if ef else None
    replicas_equal = all(torch.equal(p, ds.params[0]) for p in ds.params[1:])
    pad_clean = all(int(torch.count_nonzero(t[ds.N:])) == 0 for t in (ds.W, ds.m, ds.v))
    del ds, Ed, it
    torch.cuda.empty_cache()
    Wc = W.host_w0_at(wl, idx)
    mc, vc = W.host_mv0_at(wl, idx)
    Pc = [np.zeros(idx.size, np.uint16) for _ in range(wl.R)]
    Ec = [np.zeros(idx.size, np.float32) for _ in range(wl.R)] if ef else None
    hp = oracle.hparams(**wl.hparams())
    for t in steps:
        oracle.dp_step_compressed(W.host_grads_at(wl, t, idx), Wc, mc, vc, Pc, hp, t, wl.R, wl.M,
                                  ok, Ec)
    res = H.compare(got, (Wc, mc, vc, Pc))
    assert not {k: v for k, v in res.items() if v}, (name, res, idx.size)
    if ef:
        for g, e in zip(got_E, Ec):
            assert np.array_equal(g.view(np.uint32), e.view(np.uint32))
    assert replicas_equal and pad_clean
