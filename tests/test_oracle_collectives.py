"""Pins of the oracle's collective emulation and accounting against the
pages' worked examples (fixtures under tests/golden/, each with its source)."""
import numpy as np
import pytest

import oracle
from tests.conftest import load_golden


def test_reduce_scatter_worked_example():
    gd = load_golden("rs_worked_example.txt")
    ranks = [np.array(gd[f"rank{r}"], np.float32) for r in range(4)]
    shards = oracle.reduce_scatter_sum(ranks, S=1)
    assert [float(s[0]) for s in shards] == gd["rs_sum"]


def test_reduce_scatter_average_of_worked_example():
    # The same four ranks as bf16 gradients (all values exact in bf16), one
    # micro-batch each: the averaged gradient of element r is rs_sum[r] / 4.
    import ctypes
    gd = load_golden("rs_worked_example.txt")
    G = [np.array([oracle.bf16_rne(x) for x in gd[f"rank{r}"]], np.uint16) for r in range(4)]
    ga = (ctypes.c_void_p * 4)(*[g.ctypes.data for g in G])
    L = oracle.lib()
    got = [L.oracle_avg_grad(ctypes.addressof(ga), 4, 1, i, 4.0) for i in range(4)]
    assert got == gd["rs_avg"]


def test_ring_allreduce_demo():
    gd = load_golden("ring_demo.txt")
    p, n = int(gd["p"]), int(gd["n"])
    cards = [np.arange(n, dtype=np.float32) * (k + 1) for k in range(p)]
    sent = oracle.ring_allreduce(cards)
    for c in cards:
        assert c.tolist() == gd["result"]
    chunk = n // p
    assert all(s == gd["numbers_per_card"] for s in sent)
    assert all(s // chunk == gd["sends_per_card"] for s in sent)
    assert gd["steps"] == 2 * (p - 1)


@pytest.mark.parametrize("p", [2, 4, 8, 16])
def test_ring_volume_ratio(p, golden):
    gd = golden("ring_demo.txt")
    n = 16 * 64
    cards = [np.full(n, float(k), np.float32) for k in range(p)]
    sent = oracle.ring_allreduce(cards)
    assert np.all(sent / n == gd[f"volume_ratio_p{p}"])


@pytest.mark.parametrize("p,n", [(3, 10), (4, 8), (5, 23), (8, 64), (2, 1)])
def test_allreduce_equals_reduce_scatter_plus_all_gather(p, n):
    # AllReduce = ReduceScatter + AllGather.  Small integers keep every sum
    # exact, so the ring's rotated summation order cannot matter.
    rng = np.random.default_rng(p * 100 + n)
    data = [rng.integers(-50, 50, n).astype(np.float32) for _ in range(p)]
    ring = [d.copy() for d in data]
    oracle.ring_allreduce(ring)
    S = oracle.shard_len(n, p, 1)
    shards = oracle.reduce_scatter_sum(data, S)
    gathered = np.concatenate(shards)             # all-gather of the shards
    for c in ring:
        assert np.array_equal(c, gathered)
    assert np.array_equal(gathered, np.sum(data, axis=0))


def test_zero_bytes_exercise_1():
    gd = load_golden("zero_memory_exercises.txt")
    out = oracle.zero_bytes(gd["ex1_N"], int(gd["ex1_P"]), *gd["ex1_bytes"]) / 1e9
    assert np.allclose(out, gd["ex1_GB"], rtol=0, atol=1e-9)


def test_zero_bytes_summary_item_5():
    gd = load_golden("zero_memory_exercises.txt")
    out = oracle.zero_bytes(gd["sum5_N"], int(gd["sum5_P"]), *gd["sum5_bytes"]) / 1e9
    for o, want, d in zip(out, gd["sum5_GB"], gd["sum5_decimals"]):
        assert round(float(o), int(d)) == want


def test_zero_bytes_exercise_7_units():
    gd = load_golden("zero_memory_exercises.txt")
    out = oracle.zero_bytes(1.0, int(gd["ex7_P"]), *gd["ex7_units"])
    assert out.tolist() == gd["ex7_psi"]


@pytest.mark.parametrize("n,R,align,S", [
    (65536, 4, 64, 16384),                 # tiny: 65,536 / 4
    (124439808, 8, 64, 15555008),          # 15,554,976 -> next multiple of 64
    (1235814400, 8, 64, 154476800),        # divides exactly
    (100000007, 7, 64, 14285760),          # ceil = 14,285,716 -> 14,285,760
    (3959073792, 4, 64, 989768448),
    (5, 4, 64, 64), (0, 3, 64, 0), (7, 7, 1, 1),
])
def test_shard_len_hand_computed(n, R, align, S):
    assert oracle.shard_len(n, R, align) == S


def test_uneven_layout_padding_count():
    S = oracle.shard_len(100000007, 7, 64)
    assert 7 * S - 100000007 == 313


def _replica_mismatches(P):
    """Indices where any replica differs from replica 0, in order (the check
    zero_check_replicas makes on the device)."""
    bad = np.zeros(P[0].size, bool)
    for p in P[1:]:
        bad |= p != P[0]
    return np.flatnonzero(bad)


@pytest.mark.parametrize("n,R,c,d", [(1000, 4, 2, 0), (4099, 8, 7, 3), (130, 7, 0, 6)])
def test_dropped_allgather_message_is_found_by_replica_equality(n, R, c, d):
    """A rank failure made in the card-by-card emulation (LLM infra 06,
    section 15.4, silent data corruption): card d never receives card c's
    all-gather message, so its replica keeps last step's values on c's shard.
    Replica equality finds exactly the elements of that shard whose bf16
    value changed this step, and no others; a clean step has none."""
    M, align = 1, 64
    rng = np.random.default_rng(n + R)
    S = oracle.shard_len(n, R, align)
    G = [np.array([oracle.bf16_rne(x) for x in rng.normal(0, 1e-3, n)], np.uint16)
         for _ in range(R * M)]
    W = np.zeros(R * S, np.float32)
    W[:n] = rng.normal(0, 0.02, n)
    m = np.zeros(R * S, np.float32)
    v = np.zeros(R * S, np.float32)
    before = np.array([oracle.bf16_rne(x) for x in W[:n]], np.uint16)
    P = [before.copy() for _ in range(R)]
    oracle.zero_step(G, W, m, v, P, oracle.hparams(), 1, R, M, n, S)
    assert _replica_mismatches(P).size == 0
    lo, hi = c * S, min((c + 1) * S, n)
    assert hi > lo
    P[d][lo:hi] = before[lo:hi]                   # the dropped message
    got = _replica_mismatches(P)
    good = P[(d + 1) % R]                         # a card that did receive it
    changed = lo + np.flatnonzero(good[lo:hi] != before[lo:hi])
    assert changed.size > 0
    assert np.array_equal(got, changed)


def test_corrupted_replica_element_is_found_by_replica_equality():
    """One bit flipped in one card's list element after a clean step."""
    n, R, M = 777, 4, 2
    rng = np.random.default_rng(5)
    S = oracle.shard_len(n, R)
    G = [np.array([oracle.bf16_rne(x) for x in rng.normal(0, 1e-3, n)], np.uint16)
         for _ in range(R * M)]
    W = np.zeros(R * S, np.float32)
    W[:n] = rng.normal(0, 0.02, n)
    m = np.zeros(R * S, np.float32)
    v = np.zeros(R * S, np.float32)
    P = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.zero_step(G, W, m, v, P, oracle.hparams(), 1, R, M, n, S)
    P[3][500] ^= np.uint16(1)
    assert _replica_mismatches(P).tolist() == [500]
