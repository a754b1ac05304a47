"""Workload recipes: parameter-set shapes, value distributions and seeds.

Shapes follow the five configurations the method is measured on: a tiny flat
vector, a GPT-2-small-shaped parameter set, a Llama-3.2-1B-shaped set, an
uneven set of 37 odd-sized tensors, and a Llama-3-shaped ~4B set, plus a flat
sweep.  Values are synthetic (no datasets or trained weights): master weights
~N(0, 0.02) with norm weights 1 and biases 0, bf16 gradients ~N(0, sigma),
and Adam moments either zero, synthetic mid-training values, or the result of
prior steps with fresh gradients.

Every input is a pure function of (seed, buffer stream, element index), so a
sampled element can be produced on the host without producing the rest.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional, Tuple

import numpy as np

import zgen

W_STREAM, M_STREAM, V_STREAM = 1 << 60, (1 << 60) + 1, (1 << 60) + 2
SIZE_STREAM = (1 << 60) + 3
GRAD_TAG = 1 << 40


def grad_stream(step: int, r: int, j: int, M: int) -> int:
    """Stream id of the gradient of rank r, micro-batch j at step `step`."""
    return GRAD_TAG + step * 65536 + r * M + j


@dataclass(frozen=True)
class Workload:
    name: str
    R: int
    M: int
    stage: int
    tensors: Tuple[Tuple[str, int, str], ...]     # (name, numel, init: normal|ones|zeros)
    seed: int
    step: int                                     # the measured step t
    grad_sigma: float = 1e-3
    outlier: float = 0.0
    outlier_pct: int = 0
    w_sigma: float = 0.02
    state: str = "zero"                           # zero | synthetic | prior
    m_sigma: float = 1e-5
    v_sigma: float = 1e-4                         # v = (N(0, v_sigma))^2
    prior_steps: int = 0                          # state == "prior": steps 1..prior_steps
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    align: int = 64

    @property
    def N(self) -> int:
        return sum(t[1] for t in self.tensors)

    @property
    def numels(self) -> List[int]:
        return [t[1] for t in self.tensors]

    @property
    def offsets(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.numels)]).astype(np.int64)

    @property
    def S(self) -> int:
        per = -(-self.N // self.R)
        return -(-per // self.align) * self.align

    def bytes_per_param(self) -> int:
        """Algorithmic bytes per parameter of the fused step: bf16 gradient
        reads, fp32 master/m/v read and write, bf16 replica writes."""
        return 2 * self.R * self.M + 12 + 12 + 2 * self.R

    def hparams(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay)

    def first_step(self) -> int:
        """First step the state is driven through: 1 for prior-step workloads
        (which run steps 1..step), else the measured step itself."""
        return 1 if self.state == "prior" else self.step

    # ------------------------------------------------------------ scaling --
    def scaled(self, target_n: int, name: Optional[str] = None) -> "Workload":
        """Same recipe (R, M, stage, seed, distributions, tensor count and
        init classes, odd sizes staying odd) with every tensor shrunk so the
        total is about target_n."""
        f = max(1, self.N // max(1, target_n))
        ts = []
        for nm, n, kind in self.tensors:
            k = max(1, n // f)
            if n % 2 == 1 and k % 2 == 0:
                k += 1
            ts.append((nm, k, kind))
        return replace(self, name=name or f"{self.name}/scaled{target_n}", tensors=tuple(ts))

    def with_tensors(self, tensors, name=None) -> "Workload":
        return replace(self, tensors=tuple(tensors), name=name or self.name)


# ------------------------------------------------------------- recipes --

def _gpt2_small():
    d, ff, V, ctx, L = 768, 3072, 50257, 1024, 12
    ts = [("wte", V * d, "normal"), ("wpe", ctx * d, "normal")]
    for l in range(L):
        p = f"h{l}."
        ts += [(p + "ln_1.weight", d, "ones"), (p + "ln_1.bias", d, "zeros"),
               (p + "attn.c_attn.weight", d * 3 * d, "normal"), (p + "attn.c_attn.bias", 3 * d, "zeros"),
               (p + "attn.c_proj.weight", d * d, "normal"), (p + "attn.c_proj.bias", d, "zeros"),
               (p + "ln_2.weight", d, "ones"), (p + "ln_2.bias", d, "zeros"),
               (p + "mlp.c_fc.weight", d * ff, "normal"), (p + "mlp.c_fc.bias", ff, "zeros"),
               (p + "mlp.c_proj.weight", ff * d, "normal"), (p + "mlp.c_proj.bias", d, "zeros")]
    ts += [("ln_f.weight", d, "ones"), ("ln_f.bias", d, "zeros")]
    return ts


def _llama(d, L, ff, V, kv, tied):
    ts = [("embed_tokens", V * d, "normal")]
    for l in range(L):
        p = f"layers.{l}."
        ts += [(p + "q_proj", d * d, "normal"), (p + "k_proj", d * kv, "normal"),
               (p + "v_proj", d * kv, "normal"), (p + "o_proj", d * d, "normal"),
               (p + "gate_proj", d * ff, "normal"), (p + "up_proj", d * ff, "normal"),
               (p + "down_proj", ff * d, "normal"),
               (p + "input_layernorm", d, "ones"), (p + "post_attention_layernorm", d, "ones")]
    ts += [("norm", d, "ones")]
    if not tied:
        ts += [("lm_head", V * d, "normal")]
    return ts


def _uneven_sizes(N=100_000_007, count=37, seed=3, hi=5_000_000):
    """36 sizes drawn uniform odd in [1, hi]; the last one is the remainder
    (odd, because N is odd and 36 odd numbers sum to an even number); redraw
    with seed + 1 if the remainder is below 1."""
    s = seed
    while True:
        sizes = [2 * (zgen.draw_u64(s, SIZE_STREAM, k) % (hi // 2)) + 1 for k in range(count - 1)]
        rest = N - sum(sizes)
        if rest >= 1:
            return sizes + [rest]
        s += 1


def tiny():
    return Workload("tiny R=4 M=2 ZeRO-1 flat 65,536", R=4, M=2, stage=1,
                    tensors=(("flat", 65536, "normal"),), seed=0, step=1,
                    grad_sigma=1e-3, state="zero")


def gpt2_small():
    return Workload("gpt2-small-shaped R=8 M=1 ZeRO-1 (124,439,808 params)", R=8, M=1, stage=1,
                    tensors=tuple(_gpt2_small()), seed=1, step=11, grad_sigma=1e-3,
                    state="prior", prior_steps=10)


def llama32_1b():
    return Workload("llama-3.2-1b-shaped R=8 M=1 ZeRO-2 (1,235,814,400 params)", R=8, M=1,
                    stage=2, tensors=tuple(_llama(2048, 16, 8192, 128256, 512, tied=True)),
                    seed=2, step=100, grad_sigma=1e-4, state="synthetic",
                    m_sigma=1e-5, v_sigma=1e-4)


def uneven():
    sizes = _uneven_sizes()
    return Workload("uneven R=7 M=4 ZeRO-2 (100,000,007 params in 37 odd tensors)", R=7, M=4,
                    stage=2, tensors=tuple((f"t{k}", n, "normal") for k, n in enumerate(sizes)),
                    seed=3, step=1, grad_sigma=1e-3, outlier=1e-2, outlier_pct=1, state="zero")


def large():
    return Workload("llama-3-shaped ~4B R=4 M=1 ZeRO-2 (3,959,073,792 params)", R=4, M=1,
                    stage=2, tensors=tuple(_llama(3072, 28, 8192, 128256, 3072, tied=False)),
                    seed=4, step=100, grad_sigma=1e-4, state="synthetic",
                    m_sigma=1e-5, v_sigma=1e-4)


def sweep_point(R: int, S: int):
    return Workload(f"sweep R={R} S={S}", R=R, M=1, stage=2,
                    tensors=(("flat", R * S, "normal"),), seed=5, step=1, state="synthetic")


def flat(R: int, M: int, N: int, seed: int = 7, step: int = 1, state: str = "synthetic"):
    return Workload(f"flat R={R} M={M} N={N}", R=R, M=M, stage=2,
                    tensors=(("flat", N, "normal"),), seed=seed, step=step, state=state)


ALL = {"tiny": tiny, "gpt2-small": gpt2_small, "llama-3.2-1b": llama32_1b,
       "uneven": uneven, "large": large}


def by_name(name: str) -> Workload:
    if name.startswith("flat:"):
        kv = dict(p.split("=") for p in name[5:].split(","))
        return flat(int(kv.get("R", 8)), int(kv.get("M", 1)), int(kv["N"]))
    return ALL[name]()


# ---------------------------------------------------- host-side inputs --

def _init_kind_of(wl: Workload, idx: np.ndarray) -> np.ndarray:
    """Init class index (0 normal, 1 ones, 2 zeros) of each element."""
    kinds = np.array([{"normal": 0, "ones": 1, "zeros": 2}[t[2]] for t in wl.tensors], np.int8)
    t = np.searchsorted(wl.offsets, idx, side="right") - 1
    return kinds[t]


def host_w0_at(wl: Workload, idx: np.ndarray) -> np.ndarray:
    idx = np.asarray(idx, np.int64)
    w = zgen.host_state_at(wl.seed, W_STREAM, idx, wl.w_sigma)
    kind = _init_kind_of(wl, idx)
    w[kind == 1] = 1.0
    w[kind == 2] = 0.0
    return w


def host_w0_range(wl: Workload, lo: int, n: int) -> np.ndarray:
    return host_w0_at(wl, np.arange(lo, lo + n, dtype=np.int64))


def host_mv0_at(wl: Workload, idx: np.ndarray):
    idx = np.asarray(idx, np.int64)
    if wl.state == "synthetic":
        m = zgen.host_state_at(wl.seed, M_STREAM, idx, wl.m_sigma)
        v = zgen.host_state_at(wl.seed, V_STREAM, idx, wl.v_sigma, square=True)
    else:
        m = np.zeros(idx.size, np.float32)
        v = np.zeros(idx.size, np.float32)
    return m, v


def host_grads_at(wl: Workload, step: int, idx: np.ndarray):
    """The R*M bf16 gradient arrays (uint16 bits) of `step` at indices idx,
    ordered r*M + j."""
    idx = np.asarray(idx, np.int64)
    return [zgen.host_grad_at(wl.seed, grad_stream(step, r, j, wl.M), idx, wl.grad_sigma,
                              wl.outlier, wl.outlier_pct)
            for r in range(wl.R) for j in range(wl.M)]


def host_grads_range(wl: Workload, step: int, lo: int, n: int):
    return [zgen.host_grad(wl.seed, grad_stream(step, r, j, wl.M), lo, n, wl.grad_sigma,
                           wl.outlier, wl.outlier_pct)
            for r in range(wl.R) for j in range(wl.M)]


# -------------------------------------------------- device-side inputs --

def dev_fill_state(wl: Workload, W_ptr: int, m_ptr: int, v_ptr: int, cuda_stream: int = 0):
    """Fill the first N elements of master/m/v on the device (the pad of the
    R*S arrays is left to the caller, who zeroes it)."""
    for (nm, n, kind), lo in zip(wl.tensors, wl.offsets[:-1]):
        lo = int(lo)
        if kind == "normal":
            zgen.dev_state(W_ptr + 4 * lo, wl.seed, W_STREAM, lo, n, wl.w_sigma,
                           cuda_stream=cuda_stream)
        else:
            zgen.dev_const(W_ptr + 4 * lo, n, 1.0 if kind == "ones" else 0.0, cuda_stream)
    N = wl.N
    if wl.state == "synthetic":
        zgen.dev_state(m_ptr, wl.seed, M_STREAM, 0, N, wl.m_sigma, cuda_stream=cuda_stream)
        zgen.dev_state(v_ptr, wl.seed, V_STREAM, 0, N, wl.v_sigma, square=True,
                       cuda_stream=cuda_stream)
    else:
        zgen.dev_const(m_ptr, N, 0.0, cuda_stream)
        zgen.dev_const(v_ptr, N, 0.0, cuda_stream)


def dev_fill_grads(wl: Workload, step: int, grad_ptrs, cuda_stream: int = 0):
    """Fill the R*M gradient buffers (device pointers, order r*M + j)."""
    assert len(grad_ptrs) == wl.R * wl.M
    for r in range(wl.R):
        for j in range(wl.M):
            zgen.dev_grad(grad_ptrs[r * wl.M + j], wl.seed, grad_stream(step, r, j, wl.M), 0,
                          wl.N, wl.grad_sigma, wl.outlier, wl.outlier_pct, cuda_stream)
