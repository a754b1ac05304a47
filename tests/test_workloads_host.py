"""The synthetic input recipe on the host: the parameter-set shapes of the
five workloads, the shard layout they give, and the value distributions of
the seeded counter-based generator (no GPU; the device generator is checked
against this one bit for bit by the GPU suite)."""
import numpy as np
import pytest

from zgen import workloads as W


def _f32_of_bf16(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)


# (name, R, M, stage, tensors, N, S, bytes/param, measured step)
RECIPES = [
    ("tiny", 4, 2, 1, 1, 65_536, 16_384, 48, 1),
    ("gpt2-small", 8, 1, 1, 148, 124_439_808, 15_555_008, 56, 11),
    ("llama-3.2-1b", 8, 1, 2, 146, 1_235_814_400, 154_476_800, 56, 100),
    ("uneven", 7, 4, 2, 37, 100_000_007, 14_285_760, 94, 1),
    ("large", 4, 1, 2, 255, 3_959_073_792, 989_768_448, 40, 100),
]


@pytest.mark.parametrize("name,R,M,stage,nt,N,S,bpp,step", RECIPES)
def test_workload_shapes_and_layout(name, R, M, stage, nt, N, S, bpp, step):
    wl = W.ALL[name]()
    assert (wl.R, wl.M, wl.stage, len(wl.tensors), wl.N, wl.S) == (R, M, stage, nt, N, S)
    assert wl.bytes_per_param() == bpp and wl.step == step
    assert wl.offsets[0] == 0 and wl.offsets[-1] == N and np.all(np.diff(wl.offsets) > 0)
    # the layout rule: S is ceil(N/R) rounded up to 64 elements, and the last
    # shard is the short one
    assert S % 64 == 0 and (R - 1) * S < N <= R * S and S - (-(-N // R)) < 64


def test_gpt2_and_llama_tensor_shapes():
    g = {n: k for n, k, _ in W.gpt2_small().tensors}
    assert g["wte"] == 50257 * 768 and g["wpe"] == 1024 * 768
    assert g["h0.attn.c_attn.weight"] == 768 * 2304 and g["h11.mlp.c_proj.weight"] == 3072 * 768
    ll = {n: k for n, k, _ in W.llama32_1b().tensors}
    assert ll["embed_tokens"] == 128256 * 2048 and "lm_head" not in ll     # tied
    assert ll["layers.0.k_proj"] == 2048 * 512 and ll["layers.15.down_proj"] == 8192 * 2048
    big = {n: k for n, k, _ in W.large().tensors}
    assert big["lm_head"] == 128256 * 3072 and big["layers.27.v_proj"] == 3072 * 3072


def test_uneven_sizes_are_odd_and_drawn_from_the_stated_range():
    sizes = W.uneven().numels
    assert len(sizes) == 37 and all(n % 2 == 1 for n in sizes)
    assert all(1 <= n <= 5_000_000 for n in sizes[:36]) and sizes[36] >= 1
    assert W.uneven().S * 7 - W.uneven().N == 313                 # 313 pad elements


def test_master_weights_distribution_and_init_classes():
    wl = W.gpt2_small()
    idx = np.arange(0, 1 << 20, dtype=np.int64)                   # inside wte
    w = W.host_w0_at(wl, idx).astype(np.float64)
    assert abs(w.std() / 0.02 - 1) < 0.01 and abs(w.mean()) < 1e-4
    assert np.abs(w).max() <= 4.9 * 0.02                           # Irwin-Hall bound
    off = dict(zip([t[0] for t in wl.tensors], wl.offsets[:-1]))
    ln = W.host_w0_at(wl, np.arange(off["h3.ln_1.weight"], off["h3.ln_1.weight"] + 768))
    bias = W.host_w0_at(wl, np.arange(off["h3.ln_1.bias"], off["h3.ln_1.bias"] + 768))
    assert np.all(ln == 1.0) and np.all(bias == 0.0)


def test_gradient_distribution_and_outliers():
    idx = np.arange(0, 1 << 20, dtype=np.int64)
    g = _f32_of_bf16(W.host_grads_at(W.llama32_1b(), 100, idx)[3]).astype(np.float64)
    assert abs(g.std() / 1e-4 - 1) < 0.02 and abs(g.mean()) < 1e-6
    gu = _f32_of_bf16(W.host_grads_at(W.uneven(), 1, idx)[5]).astype(np.float64)
    out = np.isclose(np.abs(gu), 1e-2, rtol=1e-2)
    assert abs(out.mean() - 0.01) < 0.001                          # 1 % outliers
    pos = (gu[out] > 0).mean()
    assert 0.45 < pos < 0.55                                       # random sign
    rest = gu[~out]
    assert abs(rest.std() / 1e-3 - 1) < 0.02


def test_synthetic_moments():
    wl = W.llama32_1b()
    idx = np.arange(0, 1 << 20, dtype=np.int64)
    m, v = W.host_mv0_at(wl, idx)
    assert abs(m.astype(np.float64).std() / 1e-5 - 1) < 0.01
    assert np.all(v >= 0) and abs(v.astype(np.float64).mean() / 1e-8 - 1) < 0.02
    m0, v0 = W.host_mv0_at(W.uneven(), idx[:100])
    assert not m0.any() and not v0.any()                           # zero state


def test_generator_is_counter_based():
    """Each value is a function of (seed, stream, index) alone: any subset of
    indices gives the values of the whole range at those indices, and other
    steps, ranks, micro-batches or seeds give other values."""
    wl = W.uneven()
    full = W.host_grads_range(wl, 1, 1000, 5000)
    pick = np.array([1000, 1001, 2500, 5999], np.int64)
    sub = W.host_grads_at(wl, 1, pick)
    for a, b in zip(full, sub):
        assert np.array_equal(a[pick - 1000], b)
    assert not np.array_equal(full[0], full[1])                   # micro-batches differ
    assert not np.array_equal(full[0], full[4])                   # ranks differ
    assert not np.array_equal(full[0], W.host_grads_range(wl, 2, 1000, 5000)[0])
    w = W.host_w0_range(wl, 0, 1000)
    assert np.array_equal(w, W.host_w0_range(wl, 0, 1000))
    assert not np.array_equal(w, W.host_w0_range(W.flat(7, 4, 1000, seed=9), 0, 1000))


def test_scaled_workloads_keep_the_recipe():
    for name in ("gpt2-small", "uneven", "llama-3.2-1b"):
        wl = W.ALL[name]()
        s = wl.scaled(300_000)
        assert (s.R, s.M, s.stage, s.seed, s.step, len(s.tensors)) == \
            (wl.R, wl.M, wl.stage, wl.seed, wl.step, len(wl.tensors))
        assert [t[2] for t in s.tensors] == [t[2] for t in wl.tensors]
        assert all(k % 2 == 1 for (_, n, _), (_, k, _) in zip(wl.tensors, s.tensors) if n % 2)
        assert s.N < 2 * 300_000 + 2 * len(wl.tensors)
