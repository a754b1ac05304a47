"""Pins of the oracle's ZeRO-3 emulation (reading R13 of oracle/zero_oracle.h):
bit-identical to plain DP (CS324 Lecture 9 notes, section 3.4), per-unit all-gathers that rebuild
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


# ------------------------------------------------- per-unit reduce-scatter --
# Reading R16: each unit's gradient is reduce-scattered right after its
# backward into the owners' fp32 gradient shards; the step then updates the
# shards from them.


def _unit_grads(G, lo, hi):
    return [np.ascontiguousarray(g[lo:hi]) for g in G]


def _partition(n, rng, pieces):
    cuts = np.sort(rng.choice(np.arange(1, n), size=min(pieces, n - 1), replace=False))
    b = [0] + cuts.tolist() + [n]
    units = [(b[k], b[k + 1]) for k in range(len(b) - 1)]
    rng.shuffle(units)                       # any order: the backward runs last unit first
    return units


@pytest.mark.parametrize("n,R,M,align,pieces", [(1000, 4, 2, 64, 7), (4099, 7, 4, 64, 30),
                                                (5, 4, 1, 64, 3), (8192, 8, 1, 64, 1),
                                                (130, 3, 3, 4, 129), (10_007, 2, 2, 8, 11)])
def test_unit_reduce_scatter_then_update_is_the_zero3_step(n, R, M, align, pieces):
    G, W0, m0, v0 = _inputs(n, R, M, n + 5 * R)
    S = oracle.shard_len(n, R, align)
    hp = oracle.hparams()
    # the whole-step oracle (itself pinned to plain DP above)
    Wz = np.zeros(R * S, np.float32)
    mz, vz = Wz.copy(), Wz.copy()
    Wz[:n], mz[:n], vz[:n] = W0, m0, v0
    Ps = np.full(R * S, 0xBEEF, np.uint16)
    recv_step = oracle.zero3_step(G, Wz, mz, vz, Ps, hp, 4, R, M, n, S)
    # unit by unit, in a shuffled order
    rng = np.random.default_rng(n)
    gshard = np.full(R * S, np.nan, np.float32)
    recv = np.zeros(R, np.int64)
    for lo, hi in _partition(n, rng, pieces):
        recv += oracle.zero3_rs_unit(_unit_grads(G, lo, hi), n, R, M, S, lo, hi, gshard)
    assert not np.isnan(gshard[:n]).any()              # every element reduced once
    assert np.isnan(gshard[n:]).all()                  # the pad never written
    Wu = np.zeros(R * S, np.float32)
    mu, vu = Wu.copy(), Wu.copy()
    Wu[:n], mu[:n], vu[:n] = W0, m0, v0
    Pu = np.full(R * S, 0xBEEF, np.uint16)
    oracle.zero3_update(gshard, Wu, mu, vu, Pu, hp, 4, n, R, M, S)
    for a, b in ((Wu, Wz), (mu, mz), (vu, vz)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.array_equal(Pu, Ps)
    assert np.array_equal(recv, recv_step)


def test_unit_reduce_scatter_worked_example():
    # the pages' 4-rank example as one unit of 4 elements, one per rank
    gd = load_golden("rs_worked_example.txt")
    G = [np.array([oracle.bf16_rne(x) for x in gd[f"rank{r}"]], np.uint16) for r in range(4)]
    g = np.zeros(4, np.float32)
    recv = oracle.zero3_rs_unit(G, 4, 4, 1, 1, 0, 4, g)
    assert g.tolist() == gd["rs_avg"]
    assert recv.tolist() == [3, 3, 3, 3]                # one number from each other rank


def test_unit_receive_counts_and_untouched_elements():
    n, R, M, S = 300, 3, 2, 128                         # shards [0,128) [128,256) [256,300)
    G, _, _, _ = _inputs(n, R, M, 9)
    g = np.full(n, -1.0, np.float32)
    lo, hi = 100, 270
    recv = oracle.zero3_rs_unit(_unit_grads(G, lo, hi), n, R, M, S, lo, hi, g)
    # card 0 owns 100..127 (28), card 1 128..255 (128), card 2 256..269 (14);
    # each receives one number per element from each of the other 2 ranks
    assert recv.tolist() == [2 * 28, 2 * 128, 2 * 14]
    assert np.all(g[:lo] == -1.0) and np.all(g[hi:] == -1.0)
    assert np.all(g[lo:hi] != -1.0)
    with pytest.raises(RuntimeError):                   # hi beyond n
        oracle.zero3_rs_unit([np.zeros(296, np.uint16)] * (R * M), n, R, M, S, 5, 301, g)
