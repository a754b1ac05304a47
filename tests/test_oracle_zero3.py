"""Pins of the oracle's ZeRO-3 emulation (reading R13): bit-identical to plain
DP (CS324 Lecture 9 notes, section 3.4), per-unit all-gathers that rebuild
the DP replica, and the pages' per-card traffic (exercise 7)."""
import numpy as np
import pytest

import oracle
from tests.conftest import load_golden


def _inputs(n, R, M, seed):
    rng = np.random.default_rng(seed)
    G = [np.array([oracle.bf16_rne(x) for x in rng.normal(0, 1e-3, n)], np.uint16)
         for _ in range(R * M)]
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    m0 = rng.normal(0, 1e-5, n).astype(np.float32)
    v0 = (rng.normal(0, 1e-4, n) ** 2).astype(np.float32)
    return G, W0, m0, v0


@pytest.mark.parametrize("n,R,M,align", [(1000, 4, 2, 64), (4099, 7, 4, 64), (5, 4, 1, 64),
                                         (8192, 8, 1, 64), (130, 3, 3, 4)])
def test_zero3_step_bit_identical_to_dp(n, R, M, align):
    G, W0, m0, v0 = _inputs(n, R, M, n + R)
    S = oracle.shard_len(n, R, align)
    hp = oracle.hparams()
    Wd, md, vd = W0.copy(), m0.copy(), v0.copy()
    Pd = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.dp_step(G, Wd, md, vd, Pd, hp, 3, R, M)
    Wz = np.zeros(R * S, np.float32)
    mz, vz = Wz.copy(), Wz.copy()
    Wz[:n], mz[:n], vz[:n] = W0, m0, v0
    Ps = np.full(R * S, 0xBEEF, np.uint16)
    oracle.zero3_step(G, Wz, mz, vz, Ps, hp, 3, R, M, n, S)
    for a, b in ((Wz[:n], Wd), (mz[:n], md), (vz[:n], vd)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.array_equal(Ps[:n], Pd[0])                  # each card's shard = the DP bits
    assert np.all(Ps[n:] == 0xBEEF)                       # pad never written


def test_unit_gathers_rebuild_the_dp_replica():
    n, R, M = 10_007, 7, 2
    G, W0, m0, v0 = _inputs(n, R, M, 3)
    S = oracle.shard_len(n, R, 64)
    hp = oracle.hparams()
    Wd, md, vd = W0.copy(), m0.copy(), v0.copy()
    Pd = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.dp_step(G, Wd, md, vd, Pd, hp, 1, R, M)
    Wz = np.zeros(R * S, np.float32)
    mz, vz = Wz.copy(), Wz.copy()
    Wz[:n], mz[:n], vz[:n] = W0, m0, v0
    Ps = np.zeros(R * S, np.uint16)
    oracle.zero3_step(G, Wz, mz, vz, Ps, hp, 1, R, M, n, S)
    rng = np.random.default_rng(0)
    cuts = np.unique(np.concatenate([[0, n], rng.integers(0, n, 40)]))
    for card in range(R):
        parts = []
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            vals, _ = oracle.zero3_gather(Ps, n, R, S, int(lo), int(hi), card)
            parts.append(vals)
        assert np.array_equal(np.concatenate(parts), Pd[card])


def test_per_card_traffic_matches_the_pages():
    gd = load_golden("zero_comm_volumes.txt")
    p = int(gd["p"])
    n = p * 1024                                          # shards divide exactly
    G, W0, m0, v0 = _inputs(n, p, 1, 11)
    S = oracle.shard_len(n, p, 64)
    assert S * p == n
    W, m, v = W0.copy(), m0.copy(), v0.copy()
    Ps = np.zeros(n, np.uint16)
    rs_recv = oracle.zero3_step(G, W, m, v, Ps, oracle.hparams(), 1, p, 1, n, S)
    ag_recv = [oracle.zero3_gather(Ps, n, p, S, 0, n, c)[1] for c in range(p)]
    for c in range(p):
        zero12 = (rs_recv[c] + ag_recv[c]) / n            # RS + one AG after the update
        zero3 = (rs_recv[c] + 2 * ag_recv[c]) / n         # RS + AG before forward and backward
        assert zero12 == gd["zero12_per_card"]
        assert zero3 == gd["zero3_per_card"]
        assert zero3 / zero12 == gd["zero3_over_zero12"]


@pytest.mark.parametrize("M", [1, 2, 4])
def test_reduce_scatter_traffic_independent_of_microbatches(M):
    # each rank accumulates its M micro-batches locally, then sends one number
    # per element of every other card's chunk: (p-1)/p of Psi per card
    p, n = 4, 4 * 256
    G, W0, m0, v0 = _inputs(n, p, M, 5 + M)
    S = oracle.shard_len(n, p, 64)
    recv = oracle.zero3_step(G, W0.copy(), m0.copy(), v0.copy(), np.zeros(n, np.uint16),
                             oracle.hparams(), 1, p, M, n, S)
    assert list(recv) == [(p - 1) * S] * p
