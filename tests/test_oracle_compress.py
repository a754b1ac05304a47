"""Pins of the oracle's gradient compression (reading R14 of
oracle/zero_oracle.h): binary16 rounding against numpy's float16 (an
independent implementation of the same rule) and hand-worked int8 / sign
blocks; the compressed step reduces to the plain step whenever compression is
exact; error feedback keeps exactly what was dropped."""
import numpy as np
import pytest

import oracle
from tests.conftest import load_golden


def test_fp16_rne_matches_numpy():
    rng = np.random.default_rng(0)
    u = rng.integers(0, 2 ** 32, 300_000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    # bias towards the half range: subnormals, normals, overflow
    x = np.concatenate([x, rng.uniform(-70000, 70000, 50_000).astype(np.float32),
                        (rng.uniform(-1, 1, 50_000) * 2.0 ** -14).astype(np.float32),
                        (rng.uniform(-1, 1, 50_000) * 2.0 ** -24).astype(np.float32)])
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.fp16_rne(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


def test_fp16_to_float_every_pattern():
    h = np.arange(2 ** 16, dtype=np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = np.array([oracle.fp16_to_float(int(b)) for b in h], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_fp16_hand_cases():
    gd = load_golden("compress_examples.txt")
    for x, b in zip(gd["fp16_x"], gd["fp16_bits"]):
        assert oracle.fp16_rne(x) == int(b), x
    assert oracle.fp16_rne(float("nan")) == 0x7E00


@pytest.mark.parametrize("key,kind", [("int8", oracle.COMP_INT8), ("int8b", oracle.COMP_INT8),
                                      ("int8c", oracle.COMP_INT8),
                                      ("sign", oracle.COMP_SIGN), ("signz", oracle.COMP_SIGN)])
def test_hand_worked_blocks(key, kind):
    gd = load_golden("compress_examples.txt")
    x = np.array(gd[key + "_x"], np.float32)
    d = oracle.compress(kind, x)
    assert d.tolist() == gd[key + "_d"]


def test_int8_scale_is_per_block():
    # the pages: with one scale for the whole vector, many small gradients
    # round to 0; real systems quantise per block.  Block 0 holds large
    # values, block 1 small ones: per block, none of block 1 is lost.
    x = np.concatenate([np.linspace(-127, 127, 128), np.full(128, 0.01)]).astype(np.float32)
    d = oracle.compress(oracle.COMP_INT8, x)
    assert np.all(d[128:] != 0)
    assert np.all(np.abs(d[128:] - x[128:]) <= 0.01 / 127 / 2 * 1.0001)
    whole = np.clip(np.rint(x / (np.abs(x).max() / 127)), -127, 127) * (np.abs(x).max() / 127)
    assert np.all(whole[128:] == 0)                       # the whole-vector scale loses them


def test_block_boundaries_and_tail():
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1, 300).astype(np.float32)         # blocks of 128, 128, 44
    for kind in (oracle.COMP_INT8, oracle.COMP_SIGN):
        d = oracle.compress(kind, x)
        for lo in (0, 128, 256):
            blk = x[lo:lo + 128]
            assert np.array_equal(d[lo:lo + 128], oracle.compress(kind, blk.copy()))
    s_tail = oracle.compress(oracle.COMP_SIGN, x)[256:]
    assert np.allclose(np.abs(s_tail), np.abs(x[256:]).mean(), rtol=1e-6)


def _grads(n, R, M, seed, values=None):
    rng = np.random.default_rng(seed)
    if values is None:
        return [np.array([oracle.bf16_rne(v) for v in rng.normal(0, 1e-3, n)], np.uint16)
                for _ in range(R * M)]
    return [np.array([oracle.bf16_rne(float(v)) for v in values(rng)], np.uint16)
            for _ in range(R * M)]


def _run_both(G, n, R, M, kind, E=None):
    rng = np.random.default_rng(1)
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    hp = oracle.hparams()
    a = [W0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    b = [W0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    Pa = [np.zeros(n, np.uint16) for _ in range(R)]
    Pb = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.dp_step(G, *a, Pa, hp, 1, R, M)
    oracle.dp_step_compressed(G, *b, Pb, hp, 1, R, M, kind, E)
    return a, b, Pa, Pb


@pytest.mark.parametrize("ef", [False, True])
def test_fp16_exact_inputs_give_the_plain_step(ef):
    # bf16 values in the fp16 normal range have <= 8 significant bits: exact in fp16
    n, R = 1000, 4
    G = _grads(n, R, 1, 3, values=lambda rng: rng.choice([-1.0, 1.0], n)
               * rng.uniform(1e-4, 3e-3, n))
    E = [np.zeros(n, np.float32) for _ in range(R)] if ef else None
    a, b, Pa, Pb = _run_both(G, n, R, 1, oracle.COMP_FP16, E)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    assert all(np.array_equal(p, q) for p, q in zip(Pa, Pb))
    if ef:
        assert all(not e.any() for e in E)


def test_int8_exact_inputs_give_the_plain_step():
    # integer values in [-127, 127] with +-127 in every block: scale 1, exact
    n, R = 512, 3
    def vals(rng):
        v = rng.integers(-127, 128, n).astype(np.float64)
        v[::128] = 127
        return v
    G = _grads(n, R, 1, 4, values=vals)
    a, b, Pa, Pb = _run_both(G, n, R, 1, oracle.COMP_INT8)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


@pytest.mark.parametrize("kind", [oracle.COMP_FP16, oracle.COMP_INT8, oracle.COMP_SIGN])
def test_error_feedback_keeps_what_was_dropped(kind):
    n, R, M = 700, 3, 2
    G = _grads(n, R, M, 5)
    E0 = [np.random.default_rng(k).normal(0, 1e-4, n).astype(np.float32) for k in range(R)]
    E = [e.copy() for e in E0]
    W = np.zeros(n, np.float32)
    oracle.dp_step_compressed(G, W, np.zeros(n, np.float32), np.zeros(n, np.float32),
                              [np.zeros(n, np.uint16) for _ in range(R)], oracle.hparams(), 1,
                              R, M, kind, E)
    for r in range(R):
        loc = (G[r * M].astype(np.uint32) << 16).view(np.float32)
        for j in range(1, M):
            loc = (loc + (G[r * M + j].astype(np.uint32) << 16).view(np.float32)).astype(np.float32)
        x = (loc + E0[r]).astype(np.float32)
        d = oracle.compress(kind, x)
        assert np.array_equal(E[r], (x - d).astype(np.float32))


def test_none_is_the_plain_step():
    n, R, M = 333, 2, 2
    G = _grads(n, R, M, 6)
    a, b, Pa, Pb = _run_both(G, n, R, M, oracle.COMP_NONE)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
