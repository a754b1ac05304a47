"""The oracle's cross-function invariants over random shapes and values.

Each property ties two separately written oracle functions together, so a
slip in either shows (CS324 Lecture 9 notes, section 3.4: the ZeRO stages and
plain DP differ by 0.0 because AdamW is elementwise):
- the card-by-card ZeRO-1/2 emulation equals the unsharded DP step bit for bit;
- ZeRO-3 (step, or unit reduce-scatters over a random partition then the
  update) equals DP, and gathering every unit rebuilds the DP replica;
- the compressed step with the identity codec, the clipped step with a
  threshold never reached, and the 1-bit step in its warm-up each equal DP.
"""
import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


@st.composite
def cases(draw, max_n=3000):
    n = draw(st.integers(0, max_n))
    R = draw(st.integers(1, 16))
    M = draw(st.integers(1, 4))
    align = draw(st.sampled_from([1, 4, 64]))
    t = draw(st.integers(1, 50))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    G = [np.array([oracle.bf16_rne(x) for x in rng.normal(0, 1e-3, n)], np.uint16)
         for _ in range(R * M)]
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    m0 = rng.normal(0, 1e-5, n).astype(np.float32)
    v0 = (rng.normal(0, 1e-4, n) ** 2).astype(np.float32)
    return n, R, M, align, t, G, W0, m0, v0


def _dp(case):
    n, R, M, _, t, G, W0, m0, v0 = case
    W, m, v = W0.copy(), m0.copy(), v0.copy()
    P = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.dp_step(G, W, m, v, P, oracle.hparams(), t, R, M)
    return W, m, v, P


def _bits_equal(a, b):
    return np.array_equal(np.asarray(a).view(np.uint32), np.asarray(b).view(np.uint32))


def _padded(x, size):
    out = np.zeros(size, np.float32)
    out[:x.size] = x
    return out


SETTINGS = dict(max_examples=40, deadline=None)


@hypothesis.settings(**SETTINGS)
@hypothesis.given(cases())
def test_zero_emulation_equals_dp(case):
    n, R, M, align, t, G, W0, m0, v0 = case
    Wd, md, vd, Pd = _dp(case)
    S = oracle.shard_len(n, R, align)
    W, m, v = (_padded(x, R * S) for x in (W0, m0, v0))
    P = [np.full(n, 0xDEAD, np.uint16) for _ in range(R)]
    oracle.zero_step(G, W, m, v, P, oracle.hparams(), t, R, M, n, S)
    assert _bits_equal(W[:n], Wd) and _bits_equal(m[:n], md) and _bits_equal(v[:n], vd)
    assert all(np.array_equal(p, Pd[0]) for p in P)
    assert not W[n:].any() and not m[n:].any() and not v[n:].any()


@hypothesis.settings(**SETTINGS)
@hypothesis.given(cases(), st.data())
def test_zero3_step_units_and_gathers_equal_dp(case, data):
    n, R, M, align, t, G, W0, m0, v0 = case
    Wd, md, vd, Pd = _dp(case)
    S = oracle.shard_len(n, R, align)
    hp = oracle.hparams()
    # whole step
    W, m, v = (_padded(x, R * S) for x in (W0, m0, v0))
    Ps = np.zeros(R * S, np.uint16)
    oracle.zero3_step(G, W, m, v, Ps, hp, t, R, M, n, S)
    assert _bits_equal(W[:n], Wd) and _bits_equal(m[:n], md) and _bits_equal(v[:n], vd)
    # units of a random partition, reduce-scattered in a random order, then the update
    cuts = sorted(set(data.draw(st.lists(st.integers(0, n), max_size=6)) + [0, n]))
    units = list(zip(cuts[:-1], cuts[1:]))
    order = data.draw(st.permutations(units)) if units else []
    gshard = np.full(max(1, R * S), np.nan, np.float32)
    for lo, hi in order:
        oracle.zero3_rs_unit([g[lo:hi].copy() for g in G], n, R, M, S, lo, hi, gshard)
    W2, m2, v2 = (_padded(x, R * S) for x in (W0, m0, v0))
    Ps2 = np.zeros(R * S, np.uint16)
    oracle.zero3_update(gshard, W2, m2, v2, Ps2, hp, t, n, R, M, S)
    assert _bits_equal(W2[:n], Wd) and np.array_equal(Ps2[:n], Ps[:n])
    # gathering every unit for any card rebuilds the DP replica
    card = data.draw(st.integers(0, R - 1))
    got = np.concatenate([oracle.zero3_gather(Ps, n, R, S, lo, hi, card)[0]
                          for lo, hi in units] or [np.zeros(0, np.uint16)])
    assert np.array_equal(got, Pd[0])


@hypothesis.settings(**SETTINGS)
@hypothesis.given(cases())
def test_identity_codec_unreached_clip_and_onebit_warmup_equal_dp(case):
    n, R, M, align, t, G, W0, m0, v0 = case
    Wd, md, vd, Pd = _dp(case)
    hp = oracle.hparams()

    def fresh():
        return W0.copy(), m0.copy(), v0.copy(), [np.zeros(n, np.uint16) for _ in range(R)]

    W, m, v, P = fresh()
    oracle.dp_step_compressed(G, W, m, v, P, hp, t, R, M, oracle.COMP_NONE, None)
    assert _bits_equal(W, Wd) and _bits_equal(m, md) and _bits_equal(v, vd)
    assert all(np.array_equal(a, b) for a, b in zip(P, Pd))
    W, m, v, P = fresh()
    ss, skipped = oracle.dp_step_clipped(G, W, m, v, P, hp, t, R, M, max_norm=1e30)
    assert not skipped and np.isfinite(ss)
    assert _bits_equal(W, Wd) and _bits_equal(m, md) and _bits_equal(v, vd)
    W, m, v, P = fresh()
    S = max(128, oracle.shard_len(n, R, 128))                 # the 1-bit oracle wants S >= 1
    E = [np.full(n, 7.0, np.float32) for _ in range(R)]
    Es = np.full(n, 7.0, np.float32)
    oracle.onebit_step(G, W, m, v, P, hp, t, t, R, M, S, E, Es)      # t <= freeze: warm-up
    assert _bits_equal(W, Wd) and _bits_equal(m, md) and _bits_equal(v, vd)
    assert all(np.all(e == 7.0) for e in E) and np.all(Es == 7.0)    # residuals untouched
