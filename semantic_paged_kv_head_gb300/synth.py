"""Seeded synthetic inputs for the IceCache decode-time path.

This module only draws random numbers. It holds none of the method's
arithmetic (no transform, projection, partition, search or attention), so both
the CUDA path and the CPU oracle may consume what it produces.

Workload shapes follow the IceCache pages: LongBench-length contexts
(1.2k-18k tokens), the 36k-token latency study (Figure 1 and the blog's
latency table), RULER lengths up to 250k, and the GQA models named there
(Llama-3.1-8B, Mistral-7B, Qwen3-4B: 32 query heads over 8 KV heads, head
dim 128). The public benchmarks themselves are not available; clustered
Gaussian keys stand in for them:

* keys of a unit: ``mu_c + spread * N(0, I)`` with ``c`` uniform over
  ``n_centers`` centres ``mu_c ~ N(0, I)``; optionally a fraction of tokens is
  replaced by uniform noise in ``[-noise_range, noise_range]^d``;
* values: ``N(0, I)``;
* queries: the ``G`` query heads of a KV group are ``mu_{c*} + spread * N(0, I)``
  around one centre ``c*`` drawn per unit;
* generated tokens (dynamic insertion): the centres drift linearly,
  ``mu_c(t) = mu_c(0) + (t / n_steps) * delta_c`` with ``delta_c ~ N(0, drift^2 I)``.

A "unit" is one (sequence, layer, KV head). Tensors are laid out
``[batch][layer][kv_head][token][d]`` for keys/values and
``[batch][layer][q_head][d]`` for queries, which is the layout the C ABI
expects. Values are drawn in float32 and rounded to the storage dtype with
torch's round-to-nearest-even conversion.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import math

import torch


@dataclass(frozen=True)
class Workload:
    """Shape and distribution of one synthetic workload."""

    name: str
    batch: int
    n_layers: int
    n_kv_heads: int
    group: int  # query heads per KV head (G)
    d: int
    n_tokens: int
    dtype: torch.dtype
    n_centers: int
    spread: float = 0.3
    noise_frac: float = 0.0
    noise_range: float = 3.0
    page_size: int = 16
    budget: int = 256
    n_proj: int = 8
    n_composite: int = 2
    seed: int = 0
    dir_kind: int = 0  # projection directions of the index: 0 Rademacher, 1 Gaussian
    # dynamic-insert workloads
    n_insert: int = 0
    drift: float = 0.5
    extra: dict = field(default_factory=dict)

    @property
    def n_units(self) -> int:
        return self.batch * self.n_layers * self.n_kv_heads

    @property
    def n_q_heads(self) -> int:
        return self.n_kv_heads * self.group


# The five workloads: a small fp32 case the oracle finishes in seconds, then the
# Llama-3.1-8B 36k decode step, a Mistral-7B long-generation run, batched
# serving, and a 250k-token Qwen3-4B context.
WORKLOADS = {
    "tiny_fp32_4k": Workload("tiny_fp32_4k", 1, 1, 1, 2, 128, 4096, torch.float32, 64,
                             page_size=16, budget=256, n_composite=1),
    "llama8b_36k": Workload("llama8b_36k", 1, 32, 8, 4, 128, 36864, torch.bfloat16, 512,
                            page_size=16, budget=256, n_composite=2),
    "mistral7b_gen8k": Workload("mistral7b_gen8k", 1, 1, 8, 4, 128, 8192, torch.bfloat16, 64,
                                page_size=16, budget=256, n_composite=2, n_insert=8192),
    "llama8b_batch16_32k": Workload("llama8b_batch16_32k", 16, 1, 8, 4, 128, 32768,
                                    torch.bfloat16, 256, page_size=32, budget=1024,
                                    n_composite=2),
    "qwen3_4b_250k": Workload("qwen3_4b_250k", 1, 36, 8, 4, 128, 250000, torch.bfloat16,
                              4096, noise_frac=0.1, page_size=16, budget=256, n_composite=2),
}


def scaled(w: Workload, **over) -> Workload:
    """A copy of ``w`` with some fields replaced (smaller test sizes)."""
    kw = {f: getattr(w, f) for f in w.__dataclass_fields__}
    kw.update(over)
    return Workload(**kw)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & ((1 << 63) - 1))
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def make_kv(w: Workload, device="cpu", seed: int | None = None):
    """Prefill keys, values and the mixture centres.

    Returns ``(keys, values, centers)`` with keys/values shaped
    ``[batch, n_layers, n_kv_heads, n_tokens, d]`` in ``w.dtype`` and centres
    ``[n_units, n_centers, d]`` in float32 (kept for drawing queries and
    generated tokens around them).
    """
    seed = w.seed if seed is None else seed
    g = _gen(seed * 1_000_003 + 17, device)
    U, n, d = w.n_units, w.n_tokens, w.d
    centers = _randn((U, w.n_centers, d), g, device)
    keys = torch.empty((U, n, d), dtype=w.dtype, device=device)
    values = torch.empty((U, n, d), dtype=w.dtype, device=device)
    # one unit at a time keeps the float32 staging buffer small
    for u in range(U):
        asg = torch.randint(0, w.n_centers, (n,), generator=g, device=device)
        k = centers[u][asg] + w.spread * _randn((n, d), g, device)
        if w.noise_frac > 0:
            mask = torch.rand((n,), generator=g, device=device) < w.noise_frac
            noise = (torch.rand((n, d), generator=g, device=device) * 2.0 - 1.0) * w.noise_range
            k = torch.where(mask[:, None], noise, k)
        keys[u] = k.to(w.dtype)
        values[u] = _randn((n, d), g, device).to(w.dtype)
    shape = (w.batch, w.n_layers, w.n_kv_heads, n, d)
    return keys.view(shape), values.view(shape), centers


def make_queries(w: Workload, centers: torch.Tensor, step: int = 0, device=None,
                 drift_deltas: torch.Tensor | None = None):
    """Queries ``[batch, n_layers, n_q_heads, d]`` near one centre per unit.

    With ``drift_deltas`` the centres are moved to their position at ``step``
    of an ``n_insert``-step generation.
    """
    device = centers.device if device is None else device
    g = _gen((w.seed * 1_000_003 + 29) * 65_537 + step, device)
    U, d, G = w.n_units, w.d, w.group
    c_star = torch.randint(0, w.n_centers, (U,), generator=g, device=device)
    mu = centers[torch.arange(U, device=device), c_star]
    if drift_deltas is not None and w.n_insert > 0:
        mu = mu + (step / w.n_insert) * drift_deltas[torch.arange(U, device=device), c_star]
    q = mu[:, None, :] + w.spread * _randn((U, G, d), g, device)
    return q.to(w.dtype).view(w.batch, w.n_layers, w.n_kv_heads * G, d)


def make_query_stream(w: Workload, centers: torch.Tensor, n_steps: int, rho: float, device=None):
    """Queries of ``n_steps`` consecutive decode steps: each unit's queries stay
    around one centre and their noise follows an AR(1) process
    ``z_t = rho z_(t-1) + sqrt(1 - rho^2) e_t`` (consecutive queries of a head
    are correlated; ``rho`` sets how much). Returns a list of tensors shaped
    like ``make_queries``."""
    device = centers.device if device is None else device
    g = _gen(w.seed * 1_000_003 + 61, device)
    U, d, G = w.n_units, w.d, w.group
    c_star = torch.randint(0, w.n_centers, (U,), generator=g, device=device)
    mu = centers[torch.arange(U, device=device), c_star]
    z = _randn((U, G, d), g, device)
    a = math.sqrt(max(0.0, 1.0 - rho * rho))
    out = []
    for t in range(n_steps):
        if t:
            z = rho * z + a * _randn((U, G, d), g, device)
        q = mu[:, None, :] + w.spread * z
        out.append(q.to(w.dtype).view(w.batch, w.n_layers, w.n_kv_heads * G, d))
    return out


def make_drift(w: Workload, centers: torch.Tensor):
    """Per-centre drift directions ``delta_c ~ N(0, drift^2 I)``."""
    g = _gen(w.seed * 1_000_003 + 41, centers.device)
    return w.drift * _randn(tuple(centers.shape), g, centers.device)


def make_insert_token(w: Workload, centers: torch.Tensor, deltas: torch.Tensor, step: int):
    """One generated key/value per unit at generation step ``step``.

    Returns ``(k, v)`` shaped ``[batch, n_layers, n_kv_heads, d]``.
    """
    device = centers.device
    g = _gen((w.seed * 1_000_003 + 53) * 65_537 + step, device)
    U, d = w.n_units, w.d
    c = torch.randint(0, w.n_centers, (U,), generator=g, device=device)
    ar = torch.arange(U, device=device)
    mu = centers[ar, c] + (step / max(w.n_insert, 1)) * deltas[ar, c]
    k = mu + w.spread * _randn((U, d), g, device)
    v = _randn((U, d), g, device)
    shape = (w.batch, w.n_layers, w.n_kv_heads, d)
    return k.to(w.dtype).view(shape), v.to(w.dtype).view(shape)
