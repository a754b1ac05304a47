"""The clipped step's tree decomposition against the oracle's tree (no GPU).

The GPU norm pass never builds the pairwise tree level by level. It reduces
power-of-two groups of tiles, each an aligned subtree. Inside a group it
reduces per-warp subtrees, combines them in rounds of slots padded with
zeros, and combines the rounds pairwise on a stack. The update pass then
reduces the group partials, padded with zeros to a fixed count. This module
replays that decomposition in numpy float32, with the kernel's constants and
with scaled-down ones that reach every path (several rounds per group, a
ragged last group, the group count at its cap) at small sizes. It checks the
result against oracle.grad_sumsq, the plain tree over the leaves padded to
the next power of two. The claim under test is the one the kernel relies on:
any split into aligned power-of-two subtrees, with zero padding, gives the
same fp32 root. A zero leaf or subtree changes no value, because the leaves
are squares (never -0).
"""
import numpy as np
import pytest

import oracle

f32 = np.float32


def _tree(x):
    """Perfect pairwise tree of float32 values, padded with zeros."""
    y = np.asarray(x, dtype=f32)
    n = 1
    while n < len(y):
        n *= 2
    y = np.concatenate([y, np.zeros(n - len(y), f32)])
    while len(y) > 1:
        y = (y[0::2] + y[1::2]).astype(f32)
    return y[0]


def _decomposed(sq, tile, warp_leaves, round_tiles_max, max_groups):
    n = len(sq)
    tiles = max(1, -(-n // tile))
    gt = 1
    while -(-tiles // gt) > max_groups:
        gt *= 2
    groups = -(-tiles // gt)
    warps = tile // warp_leaves
    rt = min(gt, round_tiles_max)
    padded = np.zeros(groups * gt * tile, f32)
    padded[:n] = sq
    parts = []
    for grp in range(groups):
        stack, rounds = [], 0
        for t0 in range(grp * gt, (grp + 1) * gt, rt):
            slots = [_tree(padded[(t0 + j) * tile + w * warp_leaves:
                                  (t0 + j) * tile + (w + 1) * warp_leaves])
                     for j in range(rt) for w in range(warps)]
            slots += [f32(0)] * (round_tiles_max * warps - len(slots))
            v = _tree(slots)
            c = rounds
            rounds += 1
            while c & 1:                      # merge equal-sized subtrees
                v = f32(stack.pop() + v)
                c >>= 1
            stack.append(v)
        assert len(stack) == 1                # rounds per group: 1 or a power of two
        parts.append(stack[0])
    assert len(parts) <= max_groups
    return _tree(parts + [f32(0)] * (max_groups - len(parts))), gt


# (tile, warp leaves, round tiles, max groups): the kernel's constants and
# scaled-down ones with the same structure
KERNEL = (2048, 256, 32, 8192)
SMALL = [(16, 4, 2, 8), (32, 8, 4, 4), (64, 16, 2, 16)]


def _sizes(tile, rt, gmax):
    return [1, 3, tile - 1, tile, tile + 1, tile * gmax, tile * gmax + 1,
            tile * gmax * 4 + 7, tile * gmax * rt * 2 + 5, tile * gmax * rt * 8 - 1]


@pytest.mark.parametrize("consts", SMALL)
def test_scaled_decomposition_equals_the_oracle_tree(consts):
    tile, wl, rt, gmax = consts
    rng = np.random.default_rng(tile + rt)
    seen_rounds = set()
    for n in _sizes(tile, rt, gmax):
        g = (rng.standard_normal(n) * 1e-3).astype(f32)
        got, gt = _decomposed((g * g).astype(f32), tile, wl, rt, gmax)
        seen_rounds.add(max(1, gt // rt))
        assert float(got) == oracle.grad_sumsq(g), (consts, n)
    assert max(seen_rounds) >= 4                  # several rounds per group were reached


@pytest.mark.parametrize("n", [1, 2047, 2048, 2049, 100_003, 2048 * 8192, 2048 * 8192 + 1])
def test_kernel_constants_decomposition_equals_the_oracle_tree(n):
    rng = np.random.default_rng(n % 1000)
    g = (rng.standard_normal(n) * 1e-2).astype(f32)
    g[rng.integers(0, n, size=max(1, n // 1000))] = 0.0     # zero leaves inside groups
    got, gt = _decomposed((g * g).astype(f32), *KERNEL)
    assert gt == (2 if n > 2048 * 8192 else 1)
    assert float(got) == oracle.grad_sumsq(g)


def test_decomposition_differs_from_a_left_to_right_sum():
    """The comparison can fail: a left-to-right sum of the same leaves gives
    other bits, so agreement above is not an accident of the inputs."""
    rng = np.random.default_rng(5)
    g = (rng.standard_normal(4099) * 1e-3).astype(f32)
    sq = (g * g).astype(f32)
    seq = f32(0)
    for x in sq:
        seq = f32(seq + x)
    got, _ = _decomposed(sq, *SMALL[0])
    assert float(got) == oracle.grad_sumsq(g) != float(seq)
