"""Shared set-up for the GPU parity tests and __graft_entry__.smoke().

Builds device buffers for a workload, fills them with the seeded inputs
(host-generated and uploaded for small cases, device-generated for full-size
ones), runs the CUDA path through the C ABI, and runs the CPU oracle on the
same inputs.  The oracle never sees a value produced by the CUDA path.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import zero_optimizer_step_rs_gb300 as z
from zgen import workloads as W


def bf16_from_u16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(a.view(np.int16).copy()).to(device).view(torch.bfloat16)


def u16_from_bf16(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceState:
    """The device buffers of one emulated ZeRO group."""

    def __init__(self, wl: W.Workload, device="cuda:0", staged_scratch=True):
        self.wl = wl
        self.dev = torch.device(device)
        self.plan = z.Plan(wl.numels, wl.R, wl.M, wl.stage, wl.align)
        c = self.plan.c
        self.N, self.S, self.padded = c.N, c.S, c.padded
        n = max(1, self.N)
        self.grads = [torch.empty(n, dtype=torch.bfloat16, device=self.dev)
                      for _ in range(wl.R * wl.M)]
        self.params = [torch.zeros(n, dtype=torch.bfloat16, device=self.dev) for _ in range(wl.R)]
        self.W = torch.zeros(max(1, self.padded), dtype=torch.float32, device=self.dev)
        self.m = torch.zeros_like(self.W)
        self.v = torch.zeros_like(self.W)
        self.scratch = (torch.zeros(max(1, self.padded), dtype=torch.float32, device=self.dev)
                        if staged_scratch else None)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.hp = z.hparams(**wl.hparams())

    # ------------------------------------------------------------ inputs --
    def upload_state(self, W0, m0, v0):
        N = self.N
        self.W[:N].copy_(torch.from_numpy(W0))
        self.m[:N].copy_(torch.from_numpy(m0))
        self.v[:N].copy_(torch.from_numpy(v0))

    def upload_grads(self, G):
        for t, g in zip(self.grads, G):
            t[:self.N].copy_(bf16_from_u16(g, self.dev))

    def fill_state_device(self):
        W.dev_fill_state(self.wl, self.W.data_ptr(), self.m.data_ptr(), self.v.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)

    def fill_grads_device(self, step):
        W.dev_fill_grads(self.wl, step, [g.data_ptr() for g in self.grads],
                         torch.cuda.current_stream().cuda_stream)

    # -------------------------------------------------------------- step --
    def step(self, t, variant=z.ZERO_VARIANT_FUSED, flags=0):
        z.zero_step(self.plan, self.grads, self.W, self.m, self.v, self.params, self.hp, t,
                    variant=variant, scratch=self.scratch if variant else None, flags=flags,
                    dev_status=self.status)

    def step_clipped(self, t, max_norm, flags=0, sumsq=None):
        if getattr(self, "clip_scratch", None) is None:
            self.clip_scratch = torch.empty(z.zero_clip_scratch_bytes(self.plan),
                                            dtype=torch.uint8, device=self.dev)
        z.zero_step_clipped(self.plan, self.grads, self.W, self.m, self.v, self.params, self.hp,
                            t, max_norm, self.clip_scratch, flags=flags, dev_status=self.status,
                            dev_sumsq=sumsq)

    def result(self):
        N = self.N
        return (self.W[:N].cpu().numpy().copy(), self.m[:N].cpu().numpy().copy(),
                self.v[:N].cpu().numpy().copy(), [u16_from_bf16(p[:N]) for p in self.params])


def host_inputs(wl: W.Workload, step: int):
    N = wl.N
    idx = np.arange(N, dtype=np.int64)
    G = W.host_grads_at(wl, step, idx)
    W0 = W.host_w0_at(wl, idx)
    m0, v0 = W.host_mv0_at(wl, idx)
    return G, W0, m0, v0


def oracle_run(wl: W.Workload, G_by_step, W0, m0, v0, steps):
    """Run the oracle's unsharded DP step for each t in steps (gradients
    G_by_step[t]); returns W, m, v and the R replicas."""
    Wc, mc, vc = W0.copy(), m0.copy(), v0.copy()
    P = [np.zeros(Wc.size, np.uint16) for _ in range(wl.R)]
    hp = oracle.hparams(**wl.hparams())
    for t in steps:
        oracle.dp_step(G_by_step[t], Wc, mc, vc, P, hp, t, wl.R, wl.M)
    return Wc, mc, vc, P


def compare(got, want, rel_tol=1e-6):
    """Replicas bit for bit; fp32 state within rel_tol (NaN where NaN).
    Returns a dict of mismatch counts (all zero on success) and the number
    of state elements whose bits differ."""
    gW, gm, gv, gP = got
    eW, em, ev, eP = want
    out = {}
    for name, a, b in (("W", gW, eW), ("m", gm, em), ("v", gv, ev)):
        na, nb = np.isnan(a), np.isnan(b)
        fin = ~(na | nb)
        a64, b64 = a[fin].astype(np.float64), b[fin].astype(np.float64)
        same = a64 == b64                          # includes equal infinities
        with np.errstate(invalid="ignore", over="ignore"):
            rel = np.abs(a64 - b64) / np.maximum(np.abs(b64), 1e-38)
        bad = ~same & ~(rel <= rel_tol)            # NaN rel (inf vs -inf) is bad
        out[name] = int(np.sum(na != nb) + np.sum(bad))
        out[name + "_bits"] = int(np.sum(a.view(np.uint32)[fin] != b.view(np.uint32)[fin]))
    out["replicas"] = int(sum(np.sum(p != eP[0]) for p in gP))
    out["replica_vs_oracle"] = int(sum(np.sum(p != q) for p, q in zip(gP, eP)))
    return out
