"""Seeded synthetic workloads for the DSpark per-step hot path.

This module only draws random tensors with the shapes and value distributions
of the five workloads; it performs none of the method's arithmetic (no Markov
bias, no softmax, no sampling, no scheduling).  Both the CUDA path and the CPU
oracle consume what it produces, and random numbers the method itself draws
(the draft, acceptance and final uniforms) are produced here and passed in as
inputs.

Readings of the workload descriptions:

* ``N(mu, s)`` is a normal with standard deviation ``s``.
* The target logits themselves are formed by the target-model stand-in
  (``target_model.py``) from the draws made here (``target_draws``): the
  correlation ``alpha``, the noise, the fresh bonus-row logits ``z'`` and,
  for the greedy workload, which token each row plants.
* Uniforms are 24-bit: ``k * 2**-24`` with ``k`` uniform in ``[0, 2**24)``.
* Hidden states are ``N(0, 1)``; confidence weights ``N(0, 0.05)`` for every
  workload (the tiny workload's stated value carried to the others).
* The RNN head's recurrence matrix U (``rnn_recurrence``) is ``N(0,
  0.5 / sqrt(r))`` in the workload's dtype: a spectral radius near 0.5, so
  the state is a decaying sum over the prefix.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    R: int  # requests
    gamma: int  # draft block length
    V: int  # vocabulary
    r: int  # Markov rank
    d: int  # confidence-head hidden size (0 = head skipped, confidences given)
    dtype: str  # 'f32' or 'bf16' for logits, E, W, hidden states
    T: float  # sampling temperature (0 = greedy)
    target: str  # 'mix' or 'greedy'
    alpha: float | tuple = 0.9  # target = alpha * z + N(0, noise); tuple = U(lo, hi) per request
    noise_std: float | None = None  # None: sqrt(1 - alpha^2) * z_std
    sts: str = "ones"  # 'ones' or 'ramp' (1 + 0.6 (k-1)/(gamma-1))
    sps: str = "linear"  # 'quadratic' | 'linear' | 'sawtooth'
    n_sps: int = 0  # 0 = R(1+gamma)+1
    c_beta: tuple | None = None  # confidences supplied directly ~ Beta(a, b)
    z_std: float = 2.0
    ew_std: float = 0.1
    w_std: float = 0.05
    h_std: float = 1.0
    index: int = 0

    @property
    def n_sps_eff(self) -> int:
        return self.n_sps if self.n_sps > 0 else self.R * (1 + self.gamma) + 1

    @property
    def seed(self) -> int:
        return 1234 + self.index

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def scaled(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "tiny": Workload("tiny", R=4, gamma=4, V=1024, r=16, d=64, dtype="f32", T=1.0,
                     target="mix", alpha=0.8, noise_std=0.5, sts="ones",
                     sps="quadratic", index=1),
    "qwen3_4b": Workload("qwen3_4b", R=64, gamma=7, V=151936, r=256, d=2560, dtype="bf16",
                         T=1.0, target="mix", alpha=0.9, sts="ramp", sps="linear",
                         n_sps=4096, index=2),
    "deepseek": Workload("deepseek", R=256, gamma=16, V=129280, r=256, d=7168, dtype="bf16",
                         T=0.7, target="mix", alpha=(0.6, 0.95), sts="ramp", sps="linear",
                         index=3),
    "greedy": Workload("greedy", R=512, gamma=7, V=151936, r=256, d=2560, dtype="bf16",
                       T=0.0, target="greedy", sts="ramp", sps="linear", index=4),
    "stress": Workload("stress", R=2048, gamma=16, V=32000, r=128, d=0, dtype="bf16",
                       T=1.0, target="mix", alpha=0.9, sps="sawtooth", n_sps=65536,
                       c_beta=(8.0, 2.0), index=5),
}

# Tensor ids: one generator stream per tensor.
_TID = dict(z=1, E=2, W=3, anchor=4, u_draft=5, u_acc=6, u_fin=7, h=8, w=9, c=10,
            tnoise=11, zbonus=12, alpha=13, gpick=14, gother=15, U=16)


def _gen(seed: int, tid: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1009 + _TID[tid])
    return g


def _normal(shape, std, dtype, seed, tid, device, chunk_rows=64):
    """N(0, std) drawn in fp32 and rounded to ``dtype``, in chunks along dim 0."""
    g = _gen(seed, tid, device)
    out = torch.empty(shape, dtype=dtype, device=device)
    n0 = shape[0]
    for s in range(0, n0, chunk_rows):
        e = min(n0, s + chunk_rows)
        t = torch.randn((e - s,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32)
        out[s:e] = (t * std).to(dtype)
    return out


def uniforms24(shape, seed, tid, device):
    g = _gen(seed, tid, device)
    k = torch.randint(0, 1 << 24, tuple(shape), generator=g, device=device, dtype=torch.int64)
    return (k.to(torch.float64) * 2.0 ** -24).to(torch.float32)


def sps_table(wl: Workload) -> torch.Tensor:
    """Steps-per-second lookup table SPS[B], B = 0..n-1 (fp32)."""
    n = wl.n_sps_eff
    B = np.arange(n, dtype=np.float64)
    if wl.sps == "quadratic":
        t_ms = 12.0 + 0.1 * B + 0.0008 * B * B
    elif wl.sps == "linear":
        t_ms = 10.0 + 0.05 * B
    elif wl.sps == "sawtooth":
        t_ms = 12.0 + 0.02 * B + 3.0 * np.ceil(B / 128.0)
    else:
        raise ValueError(wl.sps)
    return torch.from_numpy((1000.0 / t_ms).astype(np.float32))


def sts_temperatures(wl: Workload) -> torch.Tensor:
    g = wl.gamma
    if wl.sts == "ramp" and g > 1:
        t = 1.0 + 0.6 * np.arange(g, dtype=np.float64) / (g - 1)
    else:
        t = np.ones(g, dtype=np.float64)
    return torch.from_numpy(t.astype(np.float32))


@dataclass
class Inputs:
    wl: Workload
    z: torch.Tensor  # [R, gamma, V] base draft logits
    E: torch.Tensor  # [V, r] Markov embedding (also the confidence head's E1)
    W: torch.Tensor  # [r, V] Markov output projection (pages' layout)
    anchor: torch.Tensor  # [R] int32, x_0
    u_draft: torch.Tensor  # [R, gamma] f32
    u_acc: torch.Tensor  # [R, gamma] f32
    u_fin: torch.Tensor  # [R] f32
    h: torch.Tensor | None  # [R, gamma, d]
    w_conf: torch.Tensor | None  # [d + r] f32
    sts_t: torch.Tensor  # [gamma] f32
    c_in: torch.Tensor | None  # [R, gamma] f32
    sps: torch.Tensor  # [n_sps] f32
    extra: dict = field(default_factory=dict)

    def Wt(self) -> torch.Tensor:
        """W transposed to [V, r], the layout the CUDA library takes."""
        return self.W.t().contiguous()


def make_inputs(wl: Workload, device="cpu", seed: int | None = None) -> Inputs:
    s = wl.seed if seed is None else seed
    dt = wl.torch_dtype
    R, G, V, r, d = wl.R, wl.gamma, wl.V, wl.r, wl.d
    z = _normal((R, G, V), wl.z_std, dt, s, "z", device)
    E = _normal((V, r), wl.ew_std, dt, s, "E", device, chunk_rows=1 << 16)
    W = _normal((r, V), wl.ew_std, dt, s, "W", device)
    anchor = torch.randint(0, V, (R,), generator=_gen(s, "anchor", device), device=device,
                           dtype=torch.int64).to(torch.int32)
    u_draft = uniforms24((R, G), s, "u_draft", device)
    u_acc = uniforms24((R, G), s, "u_acc", device)
    u_fin = uniforms24((R,), s, "u_fin", device)
    if wl.d > 0:
        h = _normal((R, G, d), wl.h_std, dt, s, "h", device)
        w_conf = _normal((d + r,), wl.w_std, torch.float32, s, "w", device, chunk_rows=1 << 20)
    else:
        h, w_conf = None, None
    c_in = None
    if wl.c_beta is not None:
        rng = np.random.Generator(np.random.Philox(key=s * 1009 + _TID["c"]))
        c = rng.beta(wl.c_beta[0], wl.c_beta[1], size=(R, G)).astype(np.float32)
        c_in = torch.from_numpy(c).to(device)
    return Inputs(wl, z, E, W, anchor, u_draft, u_acc, u_fin, h, w_conf,
                  sts_temperatures(wl).to(device), c_in, sps_table(wl).to(device))


def rnn_recurrence(wl: Workload, device="cpu", seed: int | None = None) -> torch.Tensor:
    """U [r, r] for the RNN head, N(0, 0.5 / sqrt(r)) in the workload's dtype."""
    s = wl.seed if seed is None else seed
    return _normal((wl.r, wl.r), 0.5 / math.sqrt(wl.r), wl.torch_dtype, s, "U", device)


@dataclass
class TargetDraws:
    """Random draws of the target-model stand-in (no arithmetic of the
    method): per-request correlation alpha and noise scale, the fresh bonus
    row z', and for the greedy workload which token each row plants."""
    alpha: torch.Tensor  # [R] f32
    noise_std: torch.Tensor  # [R] f32
    z_bonus: torch.Tensor  # [R, 1, V] in the workload's dtype
    keep: torch.Tensor | None  # [R, gamma] bool: plant the drafted token (greedy)
    other: torch.Tensor | None  # [R, gamma] int64 in [0, V-1): offset of the other token
    seed: int
    chunk: int = 16

    def noise_chunks(self, wl: Workload, device):
        """N(0, 1) fp32 noise [r1 - r0, gamma + 1, V] for consecutive chunks
        of requests, always drawn in the same order from one stream."""
        g = _gen(self.seed, "tnoise", device)
        for r0 in range(0, wl.R, self.chunk):
            r1 = min(wl.R, r0 + self.chunk)
            yield r0, r1, torch.randn((r1 - r0, wl.gamma + 1, wl.V), generator=g, device=device,
                                      dtype=torch.float32)


def target_draws(inp: Inputs, seed: int | None = None) -> TargetDraws:
    wl = inp.wl
    s = wl.seed if seed is None else seed
    dev = inp.z.device
    R, G, V = wl.R, wl.gamma, wl.V
    zb = _normal((R, 1, V), wl.z_std, wl.torch_dtype, s, "zbonus", dev)
    if isinstance(wl.alpha, tuple):
        lo, hi = wl.alpha
        alpha = lo + (hi - lo) * torch.rand((R,), generator=_gen(s, "alpha", dev), device=dev,
                                            dtype=torch.float32)
    else:
        alpha = torch.full((R,), float(wl.alpha), device=dev, dtype=torch.float32)
    if wl.noise_std is None:
        nstd = torch.sqrt(1.0 - alpha * alpha) * wl.z_std
    else:
        nstd = torch.full_like(alpha, float(wl.noise_std))
    keep = other = None
    if wl.target == "greedy":
        keep = torch.rand((R, G), generator=_gen(s, "gpick", dev), device=dev) < 0.8
        other = torch.randint(0, V - 1, (R, G), generator=_gen(s, "gother", dev), device=dev,
                              dtype=torch.int64)
    return TargetDraws(alpha, nstd, zb, keep, other, s)


def to_f64(t: torch.Tensor | None) -> np.ndarray | None:
    """Exact conversion of an input tensor to a float64 numpy array."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()
