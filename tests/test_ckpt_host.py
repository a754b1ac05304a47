"""Checkpoint format, checksums, atomic writes and R -> R' resharding, on host
memory (no GPU): BLOOM's 14 bytes/param layout (CS324 Lecture 9 notes,
section 2.1) and the merge a different card count needs (exercise 11)."""
import os

import numpy as np
import pytest

import zero_optimizer_step_rs_gb300 as z
from zero_optimizer_step_rs_gb300 import binding as B
from tests.conftest import load_golden


@pytest.fixture(scope="module", autouse=True)
def built():
    from zero_optimizer_step_rs_gb300 import build
    build.build()


def _state(N, R, seed):
    plan = z.Plan([N], R, 1, 2)
    rng = np.random.default_rng(seed)
    params = rng.integers(0, 2 ** 16, N, dtype=np.uint16)
    W = np.zeros(plan.padded, np.float32)
    m, v = W.copy(), W.copy()
    W[:N] = rng.normal(0, 0.02, N)
    m[:N] = rng.normal(0, 1e-5, N)
    v[:N] = rng.normal(0, 1e-4, N) ** 2
    return plan, params, W, m, v


def _read(plan, d, rank=-1, fill=None):
    N, P = plan.N, plan.padded
    params = np.full(max(1, N), 0xABCD if fill is None else fill, np.uint16)
    W = np.full(max(1, P), np.nan, np.float32)
    m, v = W.copy(), W.copy()
    step, hp = z.zero_ckpt_read_host(plan, str(d), params, W, m, v, rank=rank)
    return step, hp, params, W, m, v


def test_round_trip_and_14_bytes_per_param(tmp_path):
    gd = load_golden("ckpt_bytes.txt")
    N, R = 100_003, 8
    plan, params, W, m, v = _state(N, R, 1)
    hp = z.hparams(lr=3e-4, weight_decay=0.05)
    z.zero_ckpt_write_host(plan, params, W, m, v, 1234, hp, str(tmp_path))
    files = sorted(os.listdir(tmp_path))
    assert files == [f"shard-{r:05d}-of-{R:05d}.zck" for r in range(R)]   # no .tmp left
    sizes = [os.path.getsize(tmp_path / f) for f in files]
    lens = [min(plan.S, N - r * plan.S) for r in range(R)]
    assert sizes == [128 + gd["bytes_per_param"] * n for n in lens]
    assert sum(sizes) - 128 * R == gd["bytes_per_param"] * N
    # BLOOM at the same 14 bytes/param: 176B params -> 2.46 TB
    assert round(gd["bloom_params"] * gd["bytes_per_param"] / 1e12, 2) == gd["bloom_total_TB"]
    step, hp2, p2, W2, m2, v2 = _read(plan, tmp_path)
    assert step == 1234 and (hp2.lr, hp2.weight_decay) == (np.float32(3e-4), np.float32(0.05))
    assert np.array_equal(p2, params)
    for a, b in ((W2, W), (m2, m), (v2, v)):
        assert np.array_equal(a[:N].view(np.uint32), b[:N].view(np.uint32))


@pytest.mark.parametrize("R_new", [1, 3, 7, 8, 9, 64])
def test_reshard_to_another_rank_count(tmp_path, R_new):
    N = 100_003
    plan, params, W, m, v = _state(N, 8, 2)
    z.zero_ckpt_write_host(plan, params, W, m, v, 7, z.hparams(), str(tmp_path))
    plan2 = z.Plan([N], R_new, 1, 2)
    _, _, p2, W2, m2, v2 = _read(plan2, tmp_path)
    assert np.array_equal(p2, params)
    for a, b in ((W2, W), (m2, m), (v2, v)):
        assert np.array_equal(a[:N].view(np.uint32), b[:N].view(np.uint32))
    assert np.all(np.isnan(W2[N:]))                     # the new pad is not written
    # and back: the R_new checkpoint, read under R = 8, is the same state
    d2 = tmp_path / "again"
    z.zero_ckpt_write_host(plan2, p2, W2, m2, v2, 7, z.hparams(), str(d2))
    _, _, p3, W3, _, _ = _read(plan, d2)
    assert np.array_equal(p3, params) and np.array_equal(W3[:N], W[:N])


def test_rank_local_load_fills_only_the_new_shard(tmp_path):
    N = 50_001
    plan, params, W, m, v = _state(N, 4, 3)
    z.zero_ckpt_write_host(plan, params, W, m, v, 1, z.hparams(), str(tmp_path))
    plan2 = z.Plan([N], 7, 1, 2)
    for r in range(7):
        _, _, p2, W2, _, _ = _read(plan2, tmp_path, rank=r, fill=0xABCD)
        lo, hi = r * plan2.S, min((r + 1) * plan2.S, N)
        assert np.array_equal(p2[lo:hi], params[lo:hi])
        assert np.all(p2[:lo] == 0xABCD) and np.all(p2[hi:] == 0xABCD)
        assert np.array_equal(W2[lo:hi], W[lo:hi]) and np.all(np.isnan(W2[hi:N]))


def test_empty_shards(tmp_path):
    plan, params, W, m, v = _state(5, 4, 4)               # S = 64: ranks 1..3 own nothing
    z.zero_ckpt_write_host(plan, params, W, m, v, 2, z.hparams(), str(tmp_path))
    assert [os.path.getsize(tmp_path / f"shard-{r:05d}-of-00004.zck") for r in range(4)] == \
        [128 + 14 * 5, 128, 128, 128]
    _, _, p2, W2, _, _ = _read(plan, tmp_path)
    assert np.array_equal(p2[:5], params) and np.array_equal(W2[:5], W[:5])


def _corrupt(path, offset):
    b = bytearray(open(path, "rb").read())
    b[offset] ^= 0x01
    open(path, "wb").write(bytes(b))


@pytest.mark.parametrize("where", ["payload", "header", "truncate", "missing", "stale_tmp",
                                   "other_N"])
def test_damage_is_detected(tmp_path, where):
    N = 20_000
    plan, params, W, m, v = _state(N, 4, 5)
    z.zero_ckpt_write_host(plan, params, W, m, v, 3, z.hparams(), str(tmp_path))
    f = tmp_path / "shard-00002-of-00004.zck"
    if where == "payload":
        _corrupt(f, 128 + 14 * 100 + 3)
        code = B.ZERO_ERR_CORRUPT
    elif where == "header":
        _corrupt(f, 40)                                   # the S field
        code = B.ZERO_ERR_CORRUPT
    elif where == "truncate":
        os.truncate(f, os.path.getsize(f) - 2)
        code = B.ZERO_ERR_CORRUPT
    elif where == "missing":
        os.unlink(f)
        code = B.ZERO_ERR_IO
    elif where == "stale_tmp":
        # a writer that died before its rename leaves a .tmp file: ignored
        (tmp_path / "shard-00002-of-00004.zck.tmp").write_bytes(b"partial")
        _, _, p2, W2, _, _ = _read(plan, tmp_path)
        assert np.array_equal(p2, params)
        return
    else:
        plan = z.Plan([N + 1], 4, 1, 2)
        code = B.ZERO_ERR_SIZE
    with pytest.raises(B.ZeroError) as e:
        _read(plan, tmp_path)
    assert e.value.code == code


def test_write_errors(tmp_path):
    plan, params, W, m, v = _state(100, 2, 6)
    blocker = tmp_path / "file"
    blocker.write_text("x")
    with pytest.raises(B.ZeroError) as e:                 # the directory path is a file
        z.zero_ckpt_write_host(plan, params, W, m, v, 1, z.hparams(), str(blocker))
    assert e.value.code == B.ZERO_ERR_IO
    with pytest.raises(B.ZeroError) as e:
        _read(plan, tmp_path / "nothing-here")
    assert e.value.code == B.ZERO_ERR_IO
