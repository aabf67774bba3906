"""Seeded synthetic inputs for the TQ1_0 mat-vec workloads.

This module holds input recipes only: random draws and the plain
construction of fp32 weights ``w = d * t`` from drawn trits ``t`` and drawn
fp16 block scales ``d``.  It holds none of the method's arithmetic (no byte
code, no quantisation, no dot product), so both the CUDA path and the CPU
oracle can be fed from it.

Workloads (shapes and distributions of the mat-vec workloads the pages
discuss; no public dataset is involved):

* ``c1``  N=256,  K=1024, T=1;  trits uniform on {-1,0,1}, d ~ U[0.01, 0.1]
* ``c2``  N=5120, K=6144, T=1;  P(0)=0.4, P(+-1)=0.3, d ~ U[0.005, 0.05]
* ``c3``  N=5120, K=6144, T=1..32; c1's distribution
* ``c4``  128 experts of N=768, K=2048, top-8 Zipf(1.1) routing, T=1 and 32
* ``c5``  N=14336, K=4096, T=512; c1's distribution

Activations are fp32 N(0, 1).  Seeds: c1 uses 0, cN uses N.  Each problem
spawns independent child streams (numpy PCG64 via ``SeedSequence.spawn``) in
the order: weight trits, weight scales, activations, routing.  MoE experts
get one grandchild stream each, so any subset of experts can be rebuilt
without drawing the others.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

QK = 256

CONFIGS = {
    "c1": dict(n=256, k=1024, t=1, p_zero=1.0 / 3.0, d_lo=0.01, d_hi=0.1, seed=0),
    "c2": dict(n=5120, k=6144, t=1, p_zero=0.4, d_lo=0.005, d_hi=0.05, seed=2),
    "c3": dict(n=5120, k=6144, t=32, p_zero=1.0 / 3.0, d_lo=0.01, d_hi=0.1, seed=3),
    "c4": dict(n_experts=128, n=768, k=2048, top_k=8, t=(1, 32), zipf_s=1.1,
               p_zero=1.0 / 3.0, d_lo=0.01, d_hi=0.1, seed=4),
    "c5": dict(n=14336, k=4096, t=512, p_zero=1.0 / 3.0, d_lo=0.01, d_hi=0.1, seed=5),
}


def _children(seed: int, count: int = 4):
    return np.random.SeedSequence(seed).spawn(count)


def draw_trits(rng: np.random.Generator, shape, p_zero: float) -> np.ndarray:
    """i.i.d. trits: P(0) = p_zero, P(-1) = P(+1) = (1 - p_zero) / 2."""
    if abs(p_zero - 1.0 / 3.0) < 1e-12:
        return rng.integers(-1, 2, size=shape, dtype=np.int8)
    u = rng.random(shape, dtype=np.float32)
    half = np.float32((1.0 - p_zero) / 2.0)
    t = np.zeros(shape, dtype=np.int8)
    t[u < half] = -1
    t[(u >= half) & (u < 2 * half)] = 1
    return t


def draw_scales(rng: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    """Block scales drawn uniformly in fp64 and rounded (nearest-even) to fp16."""
    return rng.uniform(lo, hi, size=shape).astype(np.float16)


def weights_from(trits: np.ndarray, scales16: np.ndarray) -> np.ndarray:
    """fp32 weights w[n][k] = d[n][k/256] * t[n][k] (exact: |t| <= 1)."""
    n, k = trits.shape
    w = trits.reshape(n, k // QK, QK).astype(np.float32) * scales16.astype(np.float32)[:, :, None]
    return w.reshape(n, k)


def draw_activations(rng: np.random.Generator, t: int, k: int) -> np.ndarray:
    return rng.standard_normal((t, k), dtype=np.float32)


@dataclass
class Matvec:
    n: int
    k: int
    t: int
    trits: np.ndarray      # int8 [n][k]
    scales: np.ndarray     # fp16 [n][k/256]
    w: np.ndarray          # fp32 [n][k]
    x: np.ndarray          # fp32 [t][k]


def matvec(n: int, k: int, t: int, p_zero: float = 1.0 / 3.0, d_lo: float = 0.01, d_hi: float = 0.1,
           seed: int = 0) -> Matvec:
    s_trits, s_scales, s_act, _ = _children(seed)
    tr = draw_trits(np.random.default_rng(s_trits), (n, k), p_zero)
    sc = draw_scales(np.random.default_rng(s_scales), (n, k // QK), d_lo, d_hi)
    x = draw_activations(np.random.default_rng(s_act), t, k)
    return Matvec(n, k, t, tr, sc, weights_from(tr, sc), x)


def config_matvec(name: str, t: int | None = None) -> Matvec:
    c = CONFIGS[name]
    return matvec(c["n"], c["k"], c["t"] if t is None else t, c["p_zero"], c["d_lo"], c["d_hi"], c["seed"])


def zipf_topk(rng: np.random.Generator, t: int, n_experts: int, top_k: int, s: float) -> np.ndarray:
    """Routing ids int32 [t][top_k]: top_k distinct experts per token.

    Ranks 1..E are drawn with P(rank r) proportional to r^-s; a draw that
    repeats a rank already chosen for the token is rejected and redrawn.
    Ranks map to expert ids through one seeded permutation (drawn first)."""
    perm = rng.permutation(n_experts)
    p = np.arange(1, n_experts + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    ids = np.empty((t, top_k), dtype=np.int32)
    for i in range(t):
        chosen: list[int] = []
        while len(chosen) < top_k:
            r = int(rng.choice(n_experts, p=p))
            if r not in chosen:
                chosen.append(r)
        ids[i] = perm[np.array(chosen)]
    return ids


@dataclass
class Moe:
    n_experts: int
    n: int
    k: int
    t: int
    top_k: int
    ids: np.ndarray        # int32 [t][top_k]
    x: np.ndarray          # fp32 [t][k]
    p_zero: float
    d_lo: float
    d_hi: float
    _trit_seeds: list = field(repr=False, default_factory=list)
    _scale_seeds: list = field(repr=False, default_factory=list)

    def expert(self, e: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
        """(trits int8 [n][k], scales fp16 [n][k/256], w fp32 [n][k]) of expert e."""
        tr = draw_trits(np.random.default_rng(self._trit_seeds[e]), (self.n, self.k), self.p_zero)
        sc = draw_scales(np.random.default_rng(self._scale_seeds[e]), (self.n, self.k // QK), self.d_lo, self.d_hi)
        return tr, sc, weights_from(tr, sc)

    def expert_weights(self, e: int) -> np.ndarray:
        return self.expert(e)[2]


def moe(n_experts: int, n: int, k: int, t: int, top_k: int, zipf_s: float = 1.1, p_zero: float = 1.0 / 3.0,
        d_lo: float = 0.01, d_hi: float = 0.1, seed: int = 4) -> Moe:
    s_trits, s_scales, s_act, s_route = _children(seed)
    x = draw_activations(np.random.default_rng(s_act), t, k)
    ids = zipf_topk(np.random.default_rng(s_route), t, n_experts, top_k, zipf_s)
    return Moe(n_experts, n, k, t, top_k, ids, x, p_zero, d_lo, d_hi,
               s_trits.spawn(n_experts), s_scales.spawn(n_experts))


def config_moe(t: int) -> Moe:
    c = CONFIGS["c4"]
    return moe(c["n_experts"], c["n"], c["k"], t, c["top_k"], c["zipf_s"], c["p_zero"], c["d_lo"], c["d_hi"],
               c["seed"])


def device_weights(n: int, k: int, p_zero: float, d_lo: float, d_hi: float, generator, device="cuda"):
    """The same weight recipe drawn on the device with a seeded torch generator
    (for workloads too large to draw on the host, e.g. many distinct weight
    copies).  Returns fp32 [n][k] = fp16(d) * t."""
    import torch

    u = torch.rand((n, k), generator=generator, device=device)
    half = (1.0 - p_zero) / 2.0
    t = torch.zeros((n, k), dtype=torch.float32, device=device)
    t[u < half] = -1.0
    t[(u >= half) & (u < 2 * half)] = 1.0
    d = torch.empty((n, k // QK, 1), dtype=torch.float32, device=device).uniform_(d_lo, d_hi, generator=generator)
    d = d.half().float()
    return (t.view(n, k // QK, QK) * d).view(n, k)


def device_activations(shape, generator, device="cuda"):
    import torch

    return torch.randn(shape, generator=generator, device=device, dtype=torch.float32)
