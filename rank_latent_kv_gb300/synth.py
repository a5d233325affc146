"""Seeded synthetic workloads for the latent KV cache.

This module only draws input data (prefill keys/values, decode-step q/k/v).
It holds none of the cache's arithmetic: no projection, no quantization, no
attention. It is the one module shared by the CPU oracle's tests and the GPU
path's tests and benchmark, so both sides see identical inputs.

The five workloads describe group-head latent caches of the shapes of
Llama-3.2-3B / Qwen2.5-7B style models (head_dim 128, GQA).  Their data are
low-rank structured like real keys and values: a per-group singular spectrum
sigma_i ~ i^-alpha over 128 directions, a random orthogonal basis and a random
mean per head group.

Draw order (seed = base seed + workload index): layer -> tensor (K, V) ->
group -> (basis, mean, per-head noise).  Small parameters (basis, mean,
outlier channels) are always drawn on the CPU so they are identical whatever
device holds the big arrays; the big Gaussian factors are drawn with a
generator on the target device.
"""
from __future__ import annotations

import dataclasses
import math

import torch

HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    batch: int
    hq: int
    hkv: int
    n_groups: int
    prefill: int
    decode_steps: int
    # data model
    kind: str              # "planted" (z.A_g + mu + 0.05 eps) or "spectrum"
    alpha: float = 1.0     # sigma_i ~ i^-alpha ("spectrum" kind)
    drift: bool = False    # + 0.1 sin(t/4096) on every channel of the mean
    k_outliers: int = 0    # number of key channels scaled by 20 after generation
    # cache configuration
    rank_k: int = 0        # 0 -> energy threshold
    rank_v: int = 0
    energy_threshold: float = 0.90
    quantize_values: bool = True
    layers_timed: int = 0  # 0 -> all layers

    @property
    def gq(self) -> int:
        return self.hq // self.hkv

    @property
    def seed(self) -> int:
        return 20260000 + WORKLOAD_INDEX[self.name]


WORKLOADS = {
    # Tiny parity case: planted rank-24 signal per group, explicit rank 32.
    "tiny": Workload("tiny", layers=1, batch=1, hq=24, hkv=8, n_groups=4, prefill=512,
                     decode_steps=16, kind="planted", rank_k=32, rank_v=32),
    # Llama-3.2-3B-shaped cache.
    "llama3b": Workload("llama3b", layers=28, batch=1, hq=24, hkv=8, n_groups=4, prefill=4096,
                        decode_steps=256, kind="spectrum", alpha=1.0),
    # Serving batch: explicit rank 32, values kept as fp16 latents.
    "serving": Workload("serving", layers=28, batch=32, hq=24, hkv=8, n_groups=4, prefill=8192,
                        decode_steps=128, kind="spectrum", alpha=1.2, rank_k=32, rank_v=32,
                        quantize_values=False),
    # Long context with a slowly drifting mean; one layer of 28 timed.
    "longctx": Workload("longctx", layers=28, batch=4, hq=24, hkv=8, n_groups=4, prefill=131072,
                        decode_steps=64, kind="spectrum", alpha=1.0, drift=True, layers_timed=1),
    # Qwen2.5-7B-shaped cache: GQA 7:1, two fixed 20x outlier key channels.
    "qwen7b": Workload("qwen7b", layers=28, batch=16, hq=28, hkv=4, n_groups=2, prefill=32768,
                       decode_steps=128, kind="spectrum", alpha=1.2, k_outliers=2),
}
WORKLOAD_INDEX = {"tiny": 0, "llama3b": 1, "serving": 2, "longctx": 3, "qwen7b": 4}


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _dev_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def spectrum(alpha: float, d: int = HEAD_DIM) -> torch.Tensor:
    """sigma_i ~ i^-alpha, normalised to sum(sigma^2) = d (unit RMS per element)."""
    i = torch.arange(1, d + 1, dtype=torch.float64)
    s = i ** (-alpha)
    return s * math.sqrt(d / float((s * s).sum()))


def haar_orthogonal(gen: torch.Generator, d: int = HEAD_DIM) -> torch.Tensor:
    """Random orthogonal matrix: QR of a Gaussian with the sign of diag(R) fixed."""
    a = torch.randn(d, d, generator=gen, dtype=torch.float64)
    q, r = torch.linalg.qr(a)
    return q * torch.sign(torch.diagonal(r)).unsqueeze(0)


@dataclasses.dataclass
class GroupParams:
    basis: torch.Tensor      # [D, D] fp64 (spectrum) or A_g [24, D] (planted)
    mean: torch.Tensor       # [D] fp64
    sigma: torch.Tensor      # [D] fp64 (spectrum) / unused (planted)


def group_params(w: Workload, layer: int, tensor: int, group: int) -> GroupParams:
    """Per (layer, tensor, group) parameters, drawn on the CPU."""
    seed = w.seed * 1000003 + (layer * 2 + tensor) * 1009 + group
    gen = _cpu_gen(seed)
    if w.kind == "planted":
        a = torch.randn(24, HEAD_DIM, generator=gen, dtype=torch.float64) * math.sqrt(1.0 / 24.0)
        mu = torch.randn(HEAD_DIM, generator=gen, dtype=torch.float64) * math.sqrt(0.5)
        return GroupParams(a, mu, torch.zeros(HEAD_DIM, dtype=torch.float64))
    q = haar_orthogonal(gen)
    mu = torch.randn(HEAD_DIM, generator=gen, dtype=torch.float64) * math.sqrt(0.5)
    return GroupParams(q, mu, spectrum(w.alpha))


def outlier_channels(w: Workload, layer: int) -> list[int]:
    """The fixed key channels scaled by 20 (drawn once per layer from the seed)."""
    if w.k_outliers == 0:
        return []
    gen = _cpu_gen(w.seed * 7919 + layer)
    return sorted(torch.randperm(HEAD_DIM, generator=gen)[: w.k_outliers].tolist())


def _draw_rows(w: Workload, p: GroupParams, n_rows: int, gen, device, t_index=None):
    """n_rows fp32 rows of one head of a group (before the mean drift)."""
    if w.kind == "planted":
        z = torch.randn(n_rows, 24, generator=gen, device=device, dtype=torch.float32)
        eps = torch.randn(n_rows, HEAD_DIM, generator=gen, device=device, dtype=torch.float32)
        x = z @ p.basis.to(device=device, dtype=torch.float32) + p.mean.to(device, torch.float32) + 0.05 * eps
        return x
    z = torch.randn(n_rows, HEAD_DIM, generator=gen, device=device, dtype=torch.float32)
    m = (p.sigma.unsqueeze(1) * p.basis.T).to(device=device, dtype=torch.float32)  # diag(s) Q^T
    x = z @ m + p.mean.to(device, torch.float32)
    if w.drift:
        t = t_index.to(device=device, dtype=torch.float32).unsqueeze(1)
        x = x + 0.1 * torch.sin(t / 4096.0)
    return x


def prefill(w: Workload, layer: int, tensor: int, device="cpu", tokens: int | None = None) -> torch.Tensor:
    """Keys (tensor=0) or values (tensor=1) of one layer's prefill, fp16 [B, Hkv, T, D]."""
    T = w.prefill if tokens is None else tokens
    hg = w.hkv // w.n_groups
    out = torch.empty(w.batch, w.hkv, T, HEAD_DIM, dtype=torch.float16, device=device)
    t_index = torch.arange(0, T, dtype=torch.float64)
    for g in range(w.n_groups):
        p = group_params(w, layer, tensor, g)
        for b in range(w.batch):
            for hh in range(hg):
                h = g * hg + hh
                seed = (w.seed * 31 + layer * 2 + tensor) * 100003 + (b * w.hkv + h) * 7
                gen = _dev_gen(seed, device)
                out[b, h] = _draw_rows(w, p, T, gen, device, t_index).to(torch.float16)
    if tensor == 0:
        for c in outlier_channels(w, layer):
            out[..., c] = (out[..., c].float() * 20.0).to(torch.float16)
    return out


def decode_inputs(w: Workload, layer: int, step: int, device="cpu", n_steps: int = 1):
    """Decode-step inputs for steps [step, step + n_steps) of one layer, fp16:
    q [n, B, Hq, D], k [n, B, Hkv, 1, D], v [n, B, Hkv, 1, D].

    The tiny workload draws q, k, v ~ N(0, 1).  The others draw q ~ N(0, 1)
    and new keys/values from the same low-rank model as the prefill (same
    group basis, spectrum and mean; the drift continues with the position).
    """
    gen = _dev_gen((w.seed * 131 + layer) * 1000003 + step, device)
    n = n_steps
    q = torch.randn(n, w.batch, w.hq, HEAD_DIM, generator=gen, device=device).to(torch.float16)
    if w.kind == "planted":
        k = torch.randn(n, w.batch, w.hkv, 1, HEAD_DIM, generator=gen, device=device).to(torch.float16)
        v = torch.randn(n, w.batch, w.hkv, 1, HEAD_DIM, generator=gen, device=device).to(torch.float16)
        return q, k, v
    hg = w.hkv // w.n_groups
    kv = []
    for tensor in (0, 1):
        z = torch.randn(n, w.batch, w.hkv, HEAD_DIM, generator=gen, device=device, dtype=torch.float32)
        x = torch.empty_like(z)
        for g in range(w.n_groups):
            p = group_params(w, layer, tensor, g)
            m = (p.sigma.unsqueeze(1) * p.basis.T).to(device=device, dtype=torch.float32)
            x[:, :, g * hg:(g + 1) * hg] = z[:, :, g * hg:(g + 1) * hg] @ m + p.mean.to(device, torch.float32)
        if w.drift:
            t = torch.arange(w.prefill + step, w.prefill + step + n, device=device, dtype=torch.float32)
            x = x + 0.1 * torch.sin(t / 4096.0).view(n, 1, 1, 1)
        x = x.to(torch.float16)
        if tensor == 0:
            for c in outlier_channels(w, layer):
                x[..., c] = (x[..., c].float() * 20.0).to(torch.float16)
        kv.append(x.unsqueeze(3))
    return q, kv[0], kv[1]
