"""Pins of the oracle's 1-bit Adam step (reading R15 of oracle/zero_oracle.h).

- The warm-up steps are the plain step, bit for bit.
- A hand-worked two-rank example (tests/golden/onebit_example.txt) fixes the
  worker and server error feedback, the sign codec's zero rule and the
  server blocks counted from each shard's start.
- When the sign codec happens to be lossless and beta2 = 0 (so the frozen
  and the live second moment coincide), the step is the plain AdamW step.
- A closed form (W = 0, wd = 0, eps = 0, v = g^2) fixes the frozen bias
  correction of v.
- On random inputs, the codec's defining properties and the error-feedback
  bookkeeping hold at every element: every block decodes to one magnitude,
  the mean |input| of that block, with the input's sign; decoded value plus
  new residual gives back the input.
"""
import numpy as np
import pytest

import oracle
from tests.conftest import load_golden


def _bf16_exact(vals):
    """bf16 bits of values that bf16 represents exactly."""
    x = np.asarray(vals, np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, x), "value not exact in bf16"
    return bits


def _bf16_round(x):
    return np.array([oracle.bf16_rne(float(v)) for v in np.asarray(x, np.float32)], np.uint16)


def _bf16_float(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _state(n, R, seed, scale=1e-2):
    rng = np.random.default_rng(seed)
    W = rng.normal(0, 0.02, n).astype(np.float32)
    m = rng.normal(0, scale, n).astype(np.float32)
    v = (rng.normal(0, scale, n) ** 2).astype(np.float32)
    E = [rng.normal(0, scale / 4, n).astype(np.float32) for _ in range(R)]
    Es = rng.normal(0, scale / 4, n).astype(np.float32)
    return W, m, v, E, Es


def _grads(n, R, M, seed, scale=1e-2):
    rng = np.random.default_rng(seed)
    return [_bf16_round(rng.normal(0, scale, n)) for _ in range(R * M)]


# -------------------------------------------------------------- warm-up --

@pytest.mark.parametrize("step,freeze", [(1, 1), (3, 5), (5, 5)])
def test_warmup_is_the_plain_step(step, freeze):
    n, R, M, S = 700, 3, 2, 256
    G = _grads(n, R, M, 1)
    W, m, v, E, Es = _state(n, R, 2)
    E0 = [e.copy() for e in E]
    Es0 = Es.copy()
    hp = oracle.hparams()
    ref = [W.copy(), m.copy(), v.copy()]
    Pref = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.dp_step(G, *ref, Pref, hp, step, R, M)
    P = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.onebit_step(G, W, m, v, P, hp, step, freeze, R, M, S, E, Es)
    for a, b in zip((W, m, v), ref):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    for p, q in zip(P, Pref):
        assert np.array_equal(p, q)
    for e, e0 in zip(E, E0):
        assert np.array_equal(e, e0)
    assert np.array_equal(Es, Es0)


# ---------------------------------------------------- hand-worked example --

def test_hand_worked_example():
    gd = load_golden("onebit_example.txt")
    R, M, n, S = 2, 1, 4, 2
    hp = oracle.hparams(lr=2.0 ** -10, beta1=0.5, beta2=0.75, eps=0.0, weight_decay=0.5)
    G = [_bf16_exact(gd["g_rank0"]), _bf16_exact(gd["g_rank1"])]
    W = np.array(gd["W0"], np.float32)
    m = np.array(gd["m0"], np.float32)
    v = np.array(gd["v"], np.float32)
    v0 = v.copy()
    E = [np.array(gd["E_rank0"], np.float32), np.array(gd["E_rank1"], np.float32)]
    Es = np.array(gd["Es0"], np.float32)
    P = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.onebit_step(G, W, m, v, P, hp, 2, 1, R, M, S, E, Es)
    assert m.tolist() == gd["m1"]
    assert E[0].tolist() == gd["E1_rank0"]
    assert E[1].tolist() == gd["E1_rank1"]
    assert Es.tolist() == gd["Es1"]
    assert np.array_equal(v, v0)
    step_size = np.float32(2.0 ** -10 / 0.75)
    wdec = np.array(gd["W0"], np.float32) * np.float32(1 - 2.0 ** -11)
    want = wdec - step_size * np.array(gd["ratio"], np.float32)
    assert np.array_equal(W, want)
    for p in P:
        assert np.array_equal(p, _bf16_round(want))


# ---------------------------------------- lossless codec: the plain step --

@pytest.mark.parametrize("R,M,n,S,step", [(1, 1, 300, 320, 2), (1, 1, 1000, 1024, 9),
                                          (2, 2, 600, 320, 4), (4, 1, 1000, 256, 3)])
def test_lossless_codec_with_beta2_zero_is_the_plain_step(R, M, n, S, step):
    """With beta2 = 0 the live v is g^2 and both bias corrections of v are
    1, so with v = g^2 the frozen preconditioner equals the live one.  With
    m = 0, beta1 = 1/2 and |g| constant over every block, every sign block
    is lossless: the residuals stay 0 and the step is plain AdamW."""
    rng = np.random.default_rng(7 + n)
    if R == 1:
        # one magnitude per 128-element block (worker and server blocks
        # coincide for one rank)
        mags = 2.0 ** rng.integers(-12, -4, (n + 127) // 128)
        mag = np.repeat(mags, 128)[:n]
    else:
        mag = np.full(n, 2.0 ** -7)
    g = (mag * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    G = [_bf16_exact(g) for _ in range(R * M)]
    W = rng.normal(0, 0.02, n).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = (g * g).astype(np.float32)
    hp = oracle.hparams(lr=1e-3, beta1=0.5, beta2=0.0, eps=1e-8, weight_decay=0.1)
    ref = [W.copy(), m.copy(), v.copy()]
    Pref = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.dp_step(G, *ref, Pref, hp, step, R, M)
    E = [np.zeros(n, np.float32) for _ in range(R)]
    Es = np.zeros(n, np.float32)
    P = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.onebit_step(G, W, m, v, P, hp, step, 1, R, M, S, E, Es)
    for a, b in zip((W, m, v), ref):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    for p, q in zip(P, Pref):
        assert np.array_equal(p, q)
    for e in E:
        assert not e.any()
    assert not Es.any()


# ------------------------------------------- frozen preconditioner closed form --

@pytest.mark.parametrize("beta2,quarter", [(0.75, 0.25), (0.9375, 0.125)])
@pytest.mark.parametrize("step", [2, 3, 7])
def test_frozen_bias_correction_closed_form(beta2, quarter, step):
    """W = 0, wd = 0, eps = 0, m = 0, beta1 = 1/2, v = g^2, freeze at T_w = 1:
    the momentum is g/2 (lossless for one magnitude), the preconditioner is
    |g| / sqrt(1 - beta2), so W' = -sign(g) * step_size * sqrt(1 - beta2) / 2,
    i.e. step_size/4 for beta2 = 3/4 and step_size/8 for beta2 = 15/16,
    whatever t is."""
    n, R, M = 256, 1, 1
    rng = np.random.default_rng(step)
    g = (2.0 ** -6 * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    G = [_bf16_exact(g)]
    W = np.zeros(n, np.float32)
    m = np.zeros(n, np.float32)
    v = (g * g).astype(np.float32)
    v0 = v.copy()
    lr, b1 = 2.0 ** -10, 0.5
    hp = oracle.hparams(lr=lr, beta1=b1, beta2=beta2, eps=0.0, weight_decay=0.0)
    E = [np.zeros(n, np.float32)]
    Es = np.zeros(n, np.float32)
    P = [np.zeros(n, np.uint16)]
    oracle.onebit_step(G, W, m, v, P, hp, step, 1, R, M, 256, E, Es)
    step_size = np.float32(lr / (1.0 - b1 ** step))
    assert np.array_equal(W, (-np.sign(g) * step_size * np.float32(quarter)).astype(np.float32))
    assert np.array_equal(v, v0)


# -------------------------------------------- codec and bookkeeping invariants --

def _blocks(lo, hi, size=128):
    b = lo
    while b < hi:
        yield b, min(b + size, hi)
        b += size


def _check_sign_blocks(x, d, blocks, what):
    """Every block decodes to one magnitude, mean |x| over the block, with
    x's sign (a zero is sent as +)."""
    for lo, hi in blocks:
        xb, db = x[lo:hi].astype(np.float64), d[lo:hi].astype(np.float64)
        s = np.abs(xb).mean()
        assert np.allclose(np.abs(db), s, rtol=2e-6, atol=0), (what, lo, hi)
        assert np.all((db < 0) == (xb < 0)), (what, lo, hi)


@pytest.mark.parametrize("R,M,n,S", [(2, 2, 552, 320), (3, 1, 900, 320), (4, 3, 1030, 320)])
def test_codec_and_error_feedback_invariants(R, M, n, S):
    """S = 320 is a multiple of 64 but not of 128, so the shards' server
    blocks differ from the flat vector's 128-element worker blocks; n leaves
    ragged last blocks.  Two compression steps, so the second one starts from
    the residuals the first one left."""
    b1 = 0.875
    hp = oracle.hparams(lr=1e-3, beta1=b1, beta2=0.95, eps=1e-8, weight_decay=0.1)
    W, m, v, E, Es = _state(n, R, 11 + n)
    for step in (6, 7):
        G = _grads(n, R, M, 100 + step + n)
        m0, E0, Es0, v0 = m.copy(), [e.copy() for e in E], Es.copy(), v.copy()
        P = [np.zeros(n, np.uint16) for _ in range(R)]
        oracle.onebit_step(G, W, m, v, P, hp, step, 5, R, M, S, E, Es)
        assert np.array_equal(v, v0)
        dsum = np.zeros(n)
        for r in range(R):
            gl = sum(_bf16_float(G[r * M + j]).astype(np.float64) for j in range(M)) / M
            x = b1 * m0.astype(np.float64) + (1 - b1) * gl + E0[r]
            d = x - E[r].astype(np.float64)            # decoded value = input - new residual
            _check_sign_blocks(x, d, list(_blocks(0, n)), f"worker {r}")
            dsum += d
        y = dsum / R + Es0
        # the owner's decoded momentum plus its new residual is its input
        assert np.allclose(m.astype(np.float64) + Es, y, rtol=0, atol=1e-6 * np.abs(y).max())
        server_blocks = [b for r in range(R) for b in _blocks(r * S, min((r + 1) * S, n))]
        _check_sign_blocks(y, m, server_blocks, "server")
        # every replica holds bf16 of the new master weights
        for p in P:
            assert np.array_equal(p, _bf16_round(W))


def test_argument_errors():
    n, R, M = 8, 2, 1
    G = [np.zeros(n, np.uint16) for _ in range(R)]
    W, m, v = (np.zeros(n, np.float32) for _ in range(3))
    E = [np.zeros(n, np.float32) for _ in range(R)]
    Es = np.zeros(n, np.float32)
    P = [np.zeros(n, np.uint16) for _ in range(R)]
    hp = oracle.hparams()
    with pytest.raises(RuntimeError):
        oracle.onebit_step(G, W, m, v, P, hp, 2, 0, R, M, 4, E, Es)     # no warm-up
    with pytest.raises(RuntimeError):
        oracle.onebit_step(G, W, m, v, P, hp, 2, 1, R, M, 3, E, Es)     # R*S < n
