"""Resharding properties of the host checkpoint over random layouts: a
checkpoint written by R ranks (one shard file each, 14 bytes per parameter,
CS324 Lecture 9 notes, section 2.1) and read back under any R' (exercise 11:
a different card count needs the optimizer state merged) gives the same
bits, and the R' rank-local reads together cover [0, N) exactly once."""
import os
import tempfile

import numpy as np
import pytest

import zero_optimizer_step_rs_gb300 as z

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


@hypothesis.settings(max_examples=60, deadline=None)
@hypothesis.given(N=st.integers(0, 5000), R=st.integers(1, 64), R2=st.integers(1, 64),
                  align=st.sampled_from([0, 4, 16, 128]), align2=st.sampled_from([0, 4, 16]),
                  seed=st.integers(0, 2 ** 31 - 1))
def test_reshard_round_trip_and_rank_local_cover(N, R, R2, align, align2, seed):
    rng = np.random.default_rng(seed)
    plan = z.Plan([N], R, 1, 2, align)
    params = rng.integers(0, 2 ** 16, max(1, N), dtype=np.uint16)
    W = np.zeros(max(1, plan.padded), np.float32)
    m, v = W.copy(), W.copy()
    W[:N] = rng.normal(0, 0.02, N)
    m[:N] = rng.normal(0, 1e-5, N)
    v[:N] = rng.normal(0, 1e-4, N) ** 2
    with tempfile.TemporaryDirectory() as d:
        z.zero_ckpt_write_host(plan, params, W, m, v, 5, z.hparams(), d)
        assert sorted(os.listdir(d)) == [f"shard-{r:05d}-of-{R:05d}.zck" for r in range(R)]
        plan2 = z.Plan([N], R2, 1, 2, align2)
        P2 = max(1, plan2.padded)
        # whole read under R'
        p2 = np.zeros(max(1, N), np.uint16)
        W2 = np.full(P2, np.nan, np.float32)
        m2, v2 = W2.copy(), W2.copy()
        step, _ = z.zero_ckpt_read_host(plan2, d, p2, W2, m2, v2)
        assert step == 5
        assert np.array_equal(p2[:N], params[:N])
        for a, b in ((W2, W), (m2, m), (v2, v)):
            assert np.array_equal(a[:N].view(np.uint32), b[:N].view(np.uint32))
        # rank-local reads: each fills its own new shard only
        seen = np.zeros(max(1, N), np.int32)
        for r in range(R2):
            pr = np.full(max(1, N), 0xABCD, np.uint16)
            Wr = np.full(P2, np.nan, np.float32)
            z.zero_ckpt_read_host(plan2, d, pr, Wr, Wr.copy(), Wr.copy(), rank=r)
            lo, hi = min(N, r * plan2.S), min(N, (r + 1) * plan2.S)
            assert np.array_equal(Wr[lo:hi].view(np.uint32), W[lo:hi].view(np.uint32))
            outside = np.ones(N, bool)
            outside[lo:hi] = False
            assert np.all(np.isnan(Wr[:N][outside])) and np.all(pr[:N][outside] == 0xABCD)
            seen[lo:hi] += 1
        assert np.all(seen[:N] == 1)
