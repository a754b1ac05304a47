"""Pins of the CPU oracle against values the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the bf16
format, a hand-worked example, a closed form, torch.optim.AdamW (an
independent implementation of the same documented algorithm), exact sums on
small-integer inputs, and the pages' own ZeRO == DP result.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import load_golden


def f32(x):
    return np.float32(x)


def bits(x):
    return int(np.float32(x).view(np.uint32))


def from_bits(u):
    return float(np.uint32(u).view(np.float32))


# --------------------------------------------------------------- bf16 cast --

@pytest.mark.parametrize("u32,expect", [
    (0x3F800000, 0x3F80),      # 1.0 exact
    (0x3F808000, 0x3F80),      # halfway, kept part even -> down
    (0x3F818000, 0x3F82),      # halfway, kept part odd  -> up (to even)
    (0x3F808001, 0x3F81),      # just above halfway      -> up
    (0x3F807FFF, 0x3F80),      # just below halfway      -> down
    (0xBF818000, 0xBF82),      # negative halfway, odd   -> away from zero
    (0x7F800000, 0x7F80),      # +Inf kept
    (0xFF800000, 0xFF80),      # -Inf kept
    (0x7F7FFFFF, 0x7F80),      # largest float rounds up to +Inf
    (0x7F7F7FFF, 0x7F7F),      # largest bf16 stays finite
    (0x80000000, 0x8000),      # -0 keeps its sign
    (0x00008000, 0x0000),      # subnormal halfway, even -> down
    (0x00018000, 0x0002),      # subnormal halfway, odd  -> up
    (0x7FC00000, 0x7FC0),      # quiet NaN -> 0x7FC0
    (0xFFC00001, 0x7FC0),      # negative NaN with payload -> 0x7FC0
    (0x7F800001, 0x7FC0),      # signalling NaN -> 0x7FC0
])
def test_bf16_rne_format_cases(u32, expect):
    assert oracle.bf16_rne(from_bits(u32)) == expect


def test_bf16_rne_matches_torch_cast():
    # torch's float32 -> bfloat16 conversion rounds to nearest even: an
    # independent implementation of the same format rule.
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_to_float_is_high_half():
    for h in (0x0000, 0x3F80, 0xC2F7, 0x7F80, 0x0001):
        assert bits(oracle.bf16_to_float(h)) == h << 16


# ------------------------------------------------------------ step scalars --

def test_scalars_closed_form_step1_and_step2():
    hp = oracle.hparams(lr=0.25, beta1=0.5, beta2=0.75, eps=0.0, weight_decay=0.5)
    s1 = oracle.make_scalars(hp, 1, R=3, M=5)
    assert (s1.step_size, s1.bc2_sqrt, s1.decay) == (0.5, 0.5, 0.875)
    assert (s1.one_minus_beta1, s1.one_minus_beta2) == (0.5, 0.25)
    assert s1.denom_rm == 15.0
    s2 = oracle.make_scalars(hp, 2)
    assert bits(s2.step_size) == 0x3EAAAAAB            # float(1/3)
    assert s2.bc2_sqrt == f32(math.sqrt(7) / 4)        # sqrt(1 - 0.75^2)


def test_scalars_bias_correction_vanishes_for_large_t():
    hp = oracle.hparams(lr=1e-3, beta1=0.9, beta2=0.95)
    s = oracle.make_scalars(hp, 10**6)
    assert s.step_size == f32(1e-3) and s.bc2_sqrt == 1.0


# ---------------------------------------------------------- AdamW element --

def _run_hand_example():
    gd = load_golden("adamw_hand_example.txt")
    hp = oracle.hparams(gd["lr"], gd["beta1"], gd["beta2"], gd["eps"], gd["weight_decay"])
    W = np.array(gd["w0"], np.float32)
    m = np.zeros(3, np.float32)
    v = np.zeros(3, np.float32)
    hist = []
    for t, gk in ((1, "g1"), (2, "g2")):
        G = [np.array([oracle.bf16_rne(x) for x in gd[gk]], np.uint16)]
        P = [np.zeros(3, np.uint16)]
        oracle.dp_step(G, W, m, v, P, hp, t, R=1, M=1)
        hist.append((W.copy(), m.copy(), v.copy(), P[0].copy()))
    return gd, hist


def test_adamw_hand_worked_step1_exact():
    gd, hist = _run_hand_example()
    W, m, v, P = hist[0]
    assert np.array_equal(W, np.array(gd["w1"], np.float32))
    assert np.array_equal(m, np.array(gd["m1"], np.float32))
    assert np.array_equal(v, np.array(gd["v1"], np.float32))
    assert np.array_equal(P, np.array([oracle.bf16_rne(x) for x in gd["w1"]], np.uint16))


def test_adamw_hand_worked_step2():
    gd, hist = _run_hand_example()
    W, m, v, _ = hist[1]
    assert np.array_equal(m, np.array(gd["m2"], np.float32))
    assert np.array_equal(v, np.array(gd["v2"], np.float32))
    exact = np.array(gd["w2_num"], np.float64) / np.array(gd["w2_den"], np.float64)
    rel = np.abs(W.astype(np.float64) - exact) / np.abs(exact)
    assert rel.max() <= 1e-6, (W, exact)


def test_adamw_step1_closed_form():
    # With m = v = 0 at t = 1: (1-b1) g * lr/(1-b1) = lr g and
    # sqrt((1-b2) g^2)/sqrt(1-b2) = |g|, so w' = w(1 - lr wd) - lr g/(|g| + eps).
    rng = np.random.default_rng(3)
    n = 4096
    lr, wd, eps = 1e-3, 0.1, 1e-8
    hp = oracle.hparams(lr=lr, beta1=0.9, beta2=0.95, eps=eps, weight_decay=wd)
    g16 = np.array([oracle.bf16_rne(x) for x in rng.normal(0, 1e-3, n)], np.uint16)
    g = g16.astype(np.uint32) << 16
    g = g.view(np.float32).astype(np.float64)
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    W, m, v = W0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    P = [np.zeros(n, np.uint16)]
    oracle.dp_step([g16], W, m, v, P, hp, 1, R=1, M=1)
    lr32, wd32, eps32 = float(f32(lr)), float(f32(wd)), float(f32(eps))
    closed = W0.astype(np.float64) * (1 - lr32 * wd32) - lr32 * g / (np.abs(g) + eps32)
    err = np.abs(W.astype(np.float64) - closed)
    ulp = np.spacing(np.abs(W)).astype(np.float64)
    assert np.all(err <= 4 * ulp + lr32 * 1e-6)
    # |g| >> eps: every parameter moves by lr (up to rounding) past the decay
    big = np.abs(g) > 1e-3                        # eps/|g| <= 1e-5
    decayed = (W0 * np.float32(1 - lr32 * wd32)).astype(np.float64)
    step = np.abs(W.astype(np.float64) - decayed)
    assert np.allclose(step[big], lr32, rtol=1e-4)


def test_adamw_matches_torch_optim_adamw_20_steps():
    # torch.optim.AdamW (single-tensor path) is an independent implementation
    # of the same documented algorithm.  The hyper-parameters are exact in
    # binary32, so both sides start from the same scalars.  torch forms the
    # first moment with lerp, m + (1-b1)(g - m), which rounds differently from
    # b1*m + (1-b1)*g; everything else agrees.  Bounds: step 1 and the second
    # moment bit for bit; m within 1e-6 of the magnitude of the terms it
    # averages; w within 2 ulp plus t * 1e-6 * lr (a 1e-6-relative difference
    # in m/den moves each update by at most that much).
    rng = np.random.default_rng(5)
    n = 4096
    hp_d = dict(lr=2.0**-10, beta1=0.875, beta2=0.9375, eps=2.0**-27, weight_decay=0.125)
    hp = oracle.hparams(**hp_d)
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    W, m, v = W0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    p = torch.nn.Parameter(torch.from_numpy(W0.copy()))
    opt = torch.optim.AdamW([p], lr=hp_d["lr"], betas=(hp_d["beta1"], hp_d["beta2"]),
                            eps=hp_d["eps"], weight_decay=hp_d["weight_decay"],
                            foreach=False, fused=False)
    scale_m = np.zeros(n)
    for t in range(1, 21):
        g16 = np.array([oracle.bf16_rne(x) for x in rng.normal(0, 1e-3, n)], np.uint16)
        gf = (g16.astype(np.uint32) << 16).view(np.float32)
        oracle.dp_step([g16], W, m, v, [np.zeros(n, np.uint16)], hp, t, R=1, M=1)
        p.grad = torch.from_numpy(gf.copy())
        opt.step()
        st = opt.state[p]
        tw = p.detach().numpy()
        tm = st["exp_avg"].numpy()
        tv = st["exp_avg_sq"].numpy()
        scale_m = hp_d["beta1"] * scale_m + (1 - hp_d["beta1"]) * np.abs(gf)
        assert np.array_equal(v, tv), t
        if t == 1:
            assert np.array_equal(W, tw) and np.array_equal(m, tm)
        assert np.all(np.abs(m - tm) <= 1e-6 * scale_m), t
        tol_w = 2 * np.spacing(np.abs(tw)) + t * 1e-6 * hp_d["lr"]
        assert np.all(np.abs(W.astype(np.float64) - tw) <= tol_w), t


def test_zero_gradient_invariants():
    rng = np.random.default_rng(8)
    n = 1000
    hp = oracle.hparams(lr=1e-3, weight_decay=0.0)
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    # m = v = 0, g = 0, wd = 0: nothing moves
    W, m, v = W0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    Z = np.zeros(n, np.uint16)
    oracle.dp_step([Z, Z], W, m, v, [np.zeros(n, np.uint16)] * 2, hp, 7, R=2, M=1)
    assert np.array_equal(W, W0) and not m.any() and not v.any()
    # g = 0 with live moments: the moments just decay by beta
    m0 = rng.normal(0, 1e-4, n).astype(np.float32)
    v0 = np.abs(rng.normal(0, 1e-6, n)).astype(np.float32)
    W, m, v = W0.copy(), m0.copy(), v0.copy()
    oracle.dp_step([Z], W, m, v, [np.zeros(n, np.uint16)], hp, 3, R=1, M=1)
    assert np.array_equal(m, np.float32(0.9) * m0)
    assert np.array_equal(v, np.float32(0.95) * v0)


# ------------------------------------------------------- gradient average --

@pytest.mark.parametrize("R,M", [(1, 1), (3, 1), (4, 2), (7, 4), (8, 1), (5, 3)])
def test_identical_microbatches_average_to_the_gradient(R, M):
    # k copies of a bf16 value sum exactly in fp32 (k * g needs at most
    # 8 + log2(k) significant bits) and the exact quotient (k g)/k = g is
    # representable, so the averaged gradient is g itself for any R, M.
    rng = np.random.default_rng(R * 10 + M)
    n = 2048
    g16 = np.array([oracle.bf16_rne(x) for x in rng.normal(0, 1e-2, n)], np.uint16)
    hp = oracle.hparams()
    W1, m1, v1 = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    W2, m2, v2 = W1.copy(), m1.copy(), v1.copy()
    oracle.dp_step([g16] * (R * M), W1, m1, v1, [np.zeros(n, np.uint16)] * R, hp, 1, R, M)
    oracle.dp_step([g16], W2, m2, v2, [np.zeros(n, np.uint16)], hp, 1, 1, 1)
    assert np.array_equal(W1, W2) and np.array_equal(m1, m2) and np.array_equal(v1, v2)


@pytest.mark.parametrize("R,M", [(4, 2), (7, 4), (2, 3), (8, 1)])
def test_average_against_bruteforce_exact_sums(R, M):
    # Gradients that are small integers times 2^-10 make every partial sum
    # exact, so any summation order gives the same fp32 sum; a numpy sum in
    # reverse order, divided by R*M, must then agree with the oracle.  This
    # catches a dropped or repeated buffer, a wrong r*M+j index or a wrong
    # divisor (R or M instead of R*M).
    rng = np.random.default_rng(R + 100 * M)
    n = 512
    vals = rng.integers(-100, 101, size=(R * M, n)).astype(np.float32) * np.float32(2.0**-10)
    vals[:, :R * M] = 0
    for k in range(R * M):
        vals[k, k] = 1.0 + k                 # buffer k leaves a unique mark
    G = [np.array([oracle.bf16_rne(x) for x in row], np.uint16) for row in vals]
    gp = [g.ctypes.data for g in G]
    import ctypes
    ga = (ctypes.c_void_p * len(gp))(*gp)
    L = oracle.lib()
    ref = vals[::-1].astype(np.float64).sum(axis=0) / (R * M)
    got = np.array([L.oracle_avg_grad(ctypes.addressof(ga), R, M, i, float(R * M))
                    for i in range(n)], np.float32)
    assert np.array_equal(got, ref.astype(np.float32))


# --------------------------------------------------- ZeRO == DP (the pages) --

@pytest.mark.parametrize("n,R,M,align", [
    (65536, 4, 2, 64), (1000, 7, 4, 64), (5, 4, 1, 64), (1, 3, 2, 1),
    (4099, 8, 1, 64), (777, 2, 3, 16), (4096, 1, 1, 64), (130, 7, 2, 8),
])
def test_zero_emulation_bit_identical_to_dp(n, R, M, align):
    # CS324 Lecture 9 notes, section 3.4: the ZeRO stages and plain DP differ
    # by 0.0 because AdamW is elementwise and RS + AG does what all-reduce does.
    rng = np.random.default_rng(n + R)
    S = oracle.shard_len(n, R, align)
    G = [np.array([oracle.bf16_rne(x) for x in rng.normal(0, 1e-3, n)], np.uint16)
         for _ in range(R * M)]
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    m0 = rng.normal(0, 1e-5, n).astype(np.float32)
    v0 = (rng.normal(0, 1e-4, n) ** 2).astype(np.float32)
    hp = oracle.hparams()
    Wd, md, vd = W0.copy(), m0.copy(), v0.copy()
    Pd = [np.zeros(n, np.uint16) for _ in range(R)]
    oracle.dp_step(G, Wd, md, vd, Pd, hp, 5, R, M)
    sentinel = np.float32(np.nan).view(np.uint32) | np.uint32(0x1234)
    pad = np.full(R * S, sentinel, np.uint32).view(np.float32)
    Wz, mz, vz = pad.copy(), pad.copy(), pad.copy()
    Wz[:n], mz[:n], vz[:n] = W0, m0, v0
    Pz = [np.full(n, 0xDEAD, np.uint16) for _ in range(R)]
    oracle.zero_step(G, Wz, mz, vz, Pz, hp, 5, R, M, n, S)
    for a, b in ((Wz[:n], Wd), (mz[:n], md), (vz[:n], vd)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    for a in (Wz, mz, vz):                       # pad never touched
        assert np.all(a[n:].view(np.uint32) == sentinel)
    for r in range(R):                           # every replica identical
        assert np.array_equal(Pz[r], Pd[r])
        assert np.array_equal(Pz[r], Pz[0])
    assert np.array_equal(Pz[0], np.array([oracle.bf16_rne(x) for x in Wd], np.uint16))


def test_dp_step_thread_count_invariant():
    rng = np.random.default_rng(21)
    n, R, M = 100003, 3, 2
    G = [np.array(rng.integers(0, 2**16, n), np.uint16) & np.uint16(0xBFFF) for _ in range(R * M)]
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    hp = oracle.hparams()
    outs = []
    for th in (1, 2, 5, 8):
        W, m, v = W0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        P = [np.zeros(n, np.uint16) for _ in range(R)]
        oracle.dp_step(G, W, m, v, P, hp, 2, R, M, nthreads=th)
        outs.append((W.view(np.uint32), m.view(np.uint32), v.view(np.uint32), P[0]))
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert np.array_equal(a, b)


def test_nonfinite_gradients_propagate():
    # Reading R8: a non-finite gradient is not skipped; it flows through the
    # arithmetic and the bf16 replica holds Inf or the NaN 0x7FC0.
    hp = oracle.hparams()
    inf16, nan16 = 0x7F80, 0x7FC0
    G = [np.array([inf16, nan16, 0x3F80], np.uint16)]
    W = np.ones(3, np.float32)
    m, v = np.zeros(3, np.float32), np.zeros(3, np.float32)
    P = [np.zeros(3, np.uint16)]
    oracle.dp_step(G, W, m, v, P, hp, 1, 1, 1)
    assert np.isnan(W[0]) and np.isnan(W[1]) and np.isfinite(W[2])
    assert P[0][0] == 0x7FC0 and P[0][1] == 0x7FC0


def test_compiled_oracle_rounds_every_operation_on_its_own():
    """Reading R2 is a property of the compiled oracle, not only of its source:
    a compiler that contracted a*b + c into one fused multiply-add (GNU C's
    default on some targets, Arm among them) would change low bits.  Over
    200,000 random elements the compiled step must equal the same sequence
    evaluated in numpy float32, where every operation is rounded on its own
    and sqrt and division are correctly rounded."""
    rng = np.random.default_rng(2024)
    n, t = 200_000, 7
    hp = oracle.hparams(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    g16 = np.array([oracle.bf16_rne(x) for x in rng.normal(0, 1e-2, n)], np.uint16)
    W0 = rng.normal(0, 0.02, n).astype(np.float32)
    m0 = rng.normal(0, 1e-3, n).astype(np.float32)
    v0 = (rng.normal(0, 1e-2, n) ** 2).astype(np.float32)
    W, m, v = W0.copy(), m0.copy(), v0.copy()
    P = [np.zeros(n, np.uint16)]
    oracle.dp_step([g16], W, m, v, P, hp, t, 1, 1)
    s = oracle.make_scalars(hp, t, 1, 1)
    f = np.float32
    g = (g16.astype(np.uint32) << 16).view(np.float32) / f(s.denom_rm)
    wd = W0 * f(s.decay)
    m1 = f(s.beta1) * m0 + f(s.one_minus_beta1) * g
    v1 = f(s.beta2) * v0 + (f(s.one_minus_beta2) * g) * g
    den = np.sqrt(v1) / f(s.bc2_sqrt) + f(s.eps)
    w1 = wd - f(s.step_size) * (m1 / den)
    for got, want in ((W, w1), (m, m1), (v, v1)):
        assert got.dtype == want.dtype == np.float32
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
