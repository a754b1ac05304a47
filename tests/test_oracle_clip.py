"""Pins of the oracle's global-norm clipping (readings R10-R12 of oracle/zero_oracle.h).

The squared norm is pinned by closed forms, by math.fsum, and by a hand-worked
case whose pairwise, left-to-right and exact sums all differ
(tests/golden/clip_tree_order.txt).  The clipped step is pinned by
invariants (no clipping == the plain step; a coefficient of exactly 1/2 ==
the plain step on halved gradients) and by torch.nn.utils.clip_grad_norm_
followed by torch.optim.AdamW.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import load_golden


def bf16(x):
    return np.array([oracle.bf16_rne(float(v)) for v in np.ravel(x)], np.uint16)


def f32_of(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("n", [1, 3, 8, 1000, 4097])
def test_sumsq_of_ones(n):
    assert oracle.grad_sumsq(np.ones(n, np.float32)) == float(n)


@pytest.mark.parametrize("n", [1, 2, 17, 64, 300])
def test_sumsq_of_integers_closed_form(n):
    # every partial sum stays below 2^24, so the fp32 tree is exact
    g = np.arange(n, dtype=np.float32)
    assert oracle.grad_sumsq(g) == (n - 1) * n * (2 * n - 1) // 6


def test_sumsq_tree_order_hand_worked():
    gd = load_golden("clip_tree_order.txt")
    for k in ("8", "16"):
        g = np.array(gd["g" + k], np.float32)
        got = oracle.grad_sumsq(g)
        assert got == 2.0 ** 24 + gd[f"sumsq{k}_minus_2p24"]
        assert got != math.fsum(float(x) ** 2 for x in g)          # not the exact sum
        seq = np.float32(0.0)
        for x in g:
            seq = np.float32(seq + np.float32(x) * np.float32(x))
        assert got != float(seq)                                   # not left to right


def test_sumsq_close_to_exact_sum():
    # fp32 pairwise error bound: about log2(n) half-ulps, 17 * 2^-24 here
    rng = np.random.default_rng(4)
    g = rng.normal(0, 1e-3, 100_003).astype(np.float32)
    exact = math.fsum(float(x) ** 2 for x in g)
    assert abs(oracle.grad_sumsq(g) - exact) <= 18 * 2.0 ** -24 * exact


def test_clip_coef_cases():
    c, clip = oracle.clip_coef(4.0, 1.0)                 # norm 2 > 1
    assert clip and c == np.float32(1.0 / (2.0 + 1e-6))
    c, clip = oracle.clip_coef(0.25, 1.0)                # norm 0.5 < 1: untouched
    assert not clip and c == 1.0
    c, clip = oracle.clip_coef(float("inf"), 1.0)        # coef 1/inf = 0
    assert clip and c == 0.0
    c, clip = oracle.clip_coef(float("nan"), 1.0)        # NaN coef: no clipping
    assert not clip and c == 1.0
    c, clip = oracle.clip_coef((1.0 - 2e-6) ** 2, 1.0)   # norm + 1e-6 < max_norm
    assert not clip
    c, clip = oracle.clip_coef((1.0 - 0.5e-6) ** 2, 1.0)  # norm + 1e-6 > max_norm
    assert clip and c < 1.0


def _inputs(n, R, M, seed, sigma=1e-3):
    rng = np.random.default_rng(seed)
    G = [bf16(rng.normal(0, sigma, n)) for _ in range(R * M)]
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    m0 = rng.normal(0, 1e-5, n).astype(np.float32)
    v0 = (rng.normal(0, 1e-4, n) ** 2).astype(np.float32)
    return G, W0, m0, v0


@pytest.mark.parametrize("R,M", [(1, 1), (4, 2), (7, 4)])
def test_no_clipping_equals_plain_step(R, M):
    n = 3001
    G, W0, m0, v0 = _inputs(n, R, M, R * 7 + M)
    hp = oracle.hparams()
    a = [W0.copy(), m0.copy(), v0.copy()]
    b = [W0.copy(), m0.copy(), v0.copy()]
    Pa = [np.zeros(n, np.uint16) for _ in range(R)]
    Pb = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.dp_step(G, *a, Pa, hp, 3, R, M)
    ss, sk = oracle.dp_step_clipped(G, *b, Pb, hp, 3, R, M, max_norm=1e6)
    assert not sk and ss > 0
    for x, y in zip(a + Pa, b + Pb):
        assert np.array_equal(x.view(np.uint16 if x.dtype == np.uint16 else np.uint32),
                              y.view(np.uint16 if y.dtype == np.uint16 else np.uint32))


@pytest.mark.parametrize("R,M", [(1, 1), (4, 2), (3, 1)])
def test_clipping_scales_the_averaged_gradient(R, M):
    # At step 1 with m = v = 0 the moments are m' = (1-b1) g' and
    # v' = ((1-b2) g') g', so they expose g' = g * coef directly.  The norm is
    # checked against math.fsum; the coefficient is then formed from the
    # oracle's own squared norm (pinned above) to test where it is applied.
    n = 2049
    G, W0, _, _ = _inputs(n, R, M, 11 * R + M)
    g = None
    for r in range(R):
        loc = f32_of(G[r * M])
        for j in range(1, M):
            loc = (loc + f32_of(G[r * M + j])).astype(np.float32)
        g = loc if r == 0 else (g + loc).astype(np.float32)
    g = (g / np.float32(R * M)).astype(np.float32)
    norm = math.sqrt(math.fsum(float(x) ** 2 for x in g))
    max_norm = float(np.float32(0.3 * norm))
    hp = oracle.hparams()
    W, m, v = W0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    ss, sk = oracle.dp_step_clipped(G, W, m, v, [np.zeros(n, np.uint16)] * R, hp, 1, R, M,
                                    max_norm=max_norm)
    assert not sk and abs(math.sqrt(ss) - norm) <= 1e-6 * norm
    coef = np.float32(max_norm / (math.sqrt(ss) + 1e-6))
    gp = (g * coef).astype(np.float32)
    omb1, omb2 = np.float32(1.0 - np.float64(np.float32(0.9))), \
        np.float32(1.0 - np.float64(np.float32(0.95)))
    assert np.array_equal(m, (omb1 * gp).astype(np.float32))
    assert np.array_equal(v, ((omb2 * gp).astype(np.float32) * gp).astype(np.float32))


def test_clipped_step_matches_torch_clip_grad_norm_and_adamw():
    # torch.nn.utils.clip_grad_norm_ (fp32 norm) then torch.optim.AdamW, with
    # clipping active every step.  The hyper-parameters are exact in binary;
    # torch's fp32 norm and lerp differ from the oracle by ulps, so the bound
    # is 1e-6 of the term scale for m and 2 ulp + t * 1e-5 * lr for w.
    rng = np.random.default_rng(9)
    n, steps = 4096, 10
    hp_d = dict(lr=2.0 ** -10, beta1=0.875, beta2=0.9375, eps=2.0 ** -27, weight_decay=0.125)
    hp = oracle.hparams(**hp_d)
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    W, m, v = W0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    p = torch.nn.Parameter(torch.from_numpy(W0.copy()))
    opt = torch.optim.AdamW([p], lr=hp_d["lr"], betas=(hp_d["beta1"], hp_d["beta2"]),
                            eps=hp_d["eps"], weight_decay=hp_d["weight_decay"],
                            foreach=False, fused=False)
    max_norm = 0.01                                   # the norm is about 0.064
    scale_m = np.zeros(n)
    for t in range(1, steps + 1):
        g16 = bf16(rng.normal(0, 1e-3, n))
        gf = f32_of(g16)
        ss, sk = oracle.dp_step_clipped([g16], W, m, v, [np.zeros(n, np.uint16)], hp, t, 1, 1,
                                        max_norm=max_norm)
        assert not sk and math.sqrt(ss) > max_norm
        p.grad = torch.from_numpy(gf.copy())
        tn = torch.nn.utils.clip_grad_norm_([p], max_norm)
        assert abs(float(tn) - math.sqrt(ss)) <= 1e-6 * math.sqrt(ss)
        opt.step()
        st = opt.state[p]
        tw, tm, tv = p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        gc = np.abs(gf) * (max_norm / math.sqrt(ss))
        scale_m = hp_d["beta1"] * scale_m + (1 - hp_d["beta1"]) * gc
        assert np.all(np.abs(m - tm) <= 2e-6 * scale_m + 1e-30), t
        assert np.all(np.abs(v - tv) <= 2e-6 * np.abs(tv) + 1e-30), t
        tol_w = 2 * np.spacing(np.abs(tw)) + t * 1e-5 * hp_d["lr"]
        assert np.all(np.abs(W.astype(np.float64) - tw) <= tol_w), t


def test_nonfinite_skip_and_propagate():
    n = 100
    G, W0, m0, v0 = _inputs(n, 2, 1, 5)
    G[1][7] = 0x7F80                                  # +Inf gradient on rank 1
    hp = oracle.hparams()
    # skip: nothing changes
    W, m, v = W0.copy(), m0.copy(), v0.copy()
    P = [np.full(n, 0x1234, np.uint16) for _ in range(2)]
    ss, sk = oracle.dp_step_clipped(G, W, m, v, P, hp, 4, 2, 1, max_norm=1.0,
                                    skip_nonfinite=True)
    assert sk and math.isinf(ss)
    assert np.array_equal(W, W0) and np.array_equal(m, m0) and np.array_equal(v, v0)
    assert all(np.all(p == 0x1234) for p in P)
    # no skip: coef = 1/inf = 0 scales every gradient to 0 (the Inf one to NaN)
    W, m, v = W0.copy(), m0.copy(), v0.copy()
    Z = [np.zeros(n, np.uint16), np.zeros(n, np.uint16)]
    ss, sk = oracle.dp_step_clipped(G, W, m, v, [np.zeros(n, np.uint16)] * 2, hp, 4, 2, 1,
                                    max_norm=1.0)
    Wz, mz, vz = W0.copy(), m0.copy(), v0.copy()
    oracle.dp_step(Z, Wz, mz, vz, [np.zeros(n, np.uint16)] * 2, hp, 4, 2, 1)
    assert not sk and np.isnan(W[7])
    keep = np.arange(n) != 7
    assert np.array_equal(W[keep], Wz[keep]) and np.array_equal(m[keep], mz[keep])
