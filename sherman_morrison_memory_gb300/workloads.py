"""Seeded synthetic inputs for the VLA forward recurrence.

This module only draws random numbers and arranges them into the input
tensors q, k, v, u of shape [B, H, T, d]. It holds none of the method's
arithmetic (no normalisation of k or u, no feature map, no recurrence), so
both the CUDA path and the fp64 oracle can be fed from it without sharing
any of the computation they are compared on.

Every generator returns float32 numpy arrays. Configurations whose inputs
are bf16 are rounded to bf16 (round-to-nearest-even, via torch) and the
returned float32 arrays hold exactly the bf16 values, so the GPU (fed the
bf16 bits) and the oracle (fed those values widened to fp64) see identical
inputs.

Workloads (Variational Linear Attention, arXiv 2605.11196, §3.3 eq. 9-11;
the head dimension d_h = 96 is the paper's own):

  1  B=1,  H=2,  T=256,   d=32,  fp32, q,k,v,u ~ N(0,1)
  2  B=4,  H=8,  T=4096,  d=64,  bf16, q,k,v,u ~ N(0,1)
  3  B=8,  H=16, T=4096,  d=96,  bf16, q,k,v,u ~ N(0,1), v_t clipped to norm <= 4
  4  B=1,  H=32, T=65536, d=128, bf16, q,k,v,u ~ N(0,1)
  5  B=64, H=8,  T=1024,  d=64,  fp32, associative-recall structure (see recall())

Draw order for the plain N(0,1) workloads: q, k, v, u, each one
``rng.standard_normal((B, H, T, d), dtype=float32)`` from
``numpy.random.default_rng(seed)``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "normal",
    "recall",
    "make",
    "upstream_grad",
    "to_bf16_values",
]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    dtype: str  # "f32" or "bf16": the dtype the inputs are handed to the op in
    structure: str  # "normal", "vclip4" or "recall"
    lambda0: float = 0.1
    eps: float = 1e-4
    seed: int = 0

    @property
    def heads(self) -> int:
        return self.B * self.H

    @property
    def head_tokens(self) -> int:
        return self.B * self.H * self.T

    def describe(self) -> str:
        extra = {
            "normal": "q,k,v,u N(0,1)",
            "vclip4": "q,k,v,u N(0,1), v_t clipped to ||v_t||<=4",
            "recall": "associative-recall keys from a 48-vector pool, u=k+0.1N(0,1)",
        }[self.structure]
        return (f"{self.name}: B={self.B},H={self.H},T={self.T},d_h={self.d}, "
                f"{self.dtype} inputs ({extra}), fp32 state, lambda0={self.lambda0}, "
                f"eps={self.eps}, seed={self.seed}")


WORKLOADS = {
    1: Workload("small", 1, 2, 256, 32, "f32", "normal"),
    2: Workload("d64", 4, 8, 4096, 64, "bf16", "normal"),
    3: Workload("d96", 8, 16, 4096, 96, "bf16", "vclip4"),
    4: Workload("long", 1, 32, 65536, 128, "bf16", "normal"),
    5: Workload("recall", 64, 8, 1024, 64, "f32", "recall"),
}


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and return them as float32."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def normal(B, H, T, d, seed=0, vclip=None):
    """q, k, v, u i.i.d. N(0,1) in that draw order.

    If ``vclip`` is given, each value vector is scaled by min(1, vclip/||v_t||)
    in float32 (before any bf16 rounding), so that ||v_t|| <= vclip.
    """
    rng = np.random.default_rng(seed)
    shape = (B, H, T, d)
    q = rng.standard_normal(shape, dtype=np.float32)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    u = rng.standard_normal(shape, dtype=np.float32)
    if vclip is not None:
        nrm = np.sqrt(np.sum(v.astype(np.float64) ** 2, axis=-1, keepdims=True))
        scale = np.minimum(1.0, vclip / np.maximum(nrm, 1e-30)).astype(np.float32)
        v = (v * scale).astype(np.float32)
    return q, k, v, u


def recall(B, H, T, d, seed=0, pool=48, noise=0.1):
    """Associative-recall structured inputs (shape borrowed from MQAR).

    Per (b, h) stream: a pool of ``pool`` random unit vectors P and one N(0,1)
    value vector per pool entry. The first half of the tokens writes pairs:
    idx ~ U{0..pool-1} with replacement, k_t = q_t = P[idx], v_t = V[idx].
    The second half re-presents keys written in the first half (idx uniform
    over the distinct indices written) as queries with v_t = 0. The penalty
    direction is u_t = k_t + noise * N(0,1).
    """
    rng = np.random.default_rng(seed)
    P = rng.standard_normal((B, H, pool, d), dtype=np.float32)
    P = (P / np.sqrt(np.sum(P.astype(np.float64) ** 2, axis=-1, keepdims=True))).astype(np.float32)
    V = rng.standard_normal((B, H, pool, d), dtype=np.float32)
    half = T // 2
    idx1 = rng.integers(0, pool, size=(B, H, half))
    r2 = rng.random((B, H, T - half))
    idx2 = np.empty((B, H, T - half), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            written = np.unique(idx1[b, h])
            idx2[b, h] = written[np.minimum((r2[b, h] * len(written)).astype(np.int64), len(written) - 1)]
    idx = np.concatenate([idx1, idx2], axis=2)
    bi = np.arange(B)[:, None, None]
    hi = np.arange(H)[None, :, None]
    k = P[bi, hi, idx]
    q = k.copy()
    v = V[bi, hi, idx]
    v[:, :, half:, :] = 0.0
    u = (k + np.float32(noise) * rng.standard_normal((B, H, T, d), dtype=np.float32)).astype(np.float32)
    return (np.ascontiguousarray(q), np.ascontiguousarray(k),
            np.ascontiguousarray(v), np.ascontiguousarray(u))


def make(w: Workload, B=None, H=None, T=None):
    """Draw the inputs of workload ``w`` (optionally with B, H or T overridden).

    Returns float32 arrays (q, k, v, u); for bf16 workloads the values are
    already rounded to bf16.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    if w.structure == "recall":
        arrs = recall(B, H, T, w.d, seed=w.seed)
    elif w.structure == "vclip4":
        arrs = normal(B, H, T, w.d, seed=w.seed, vclip=4.0)
    else:
        arrs = normal(B, H, T, w.d, seed=w.seed)
    if w.dtype == "bf16":
        arrs = tuple(to_bf16_values(a) for a in arrs)
    return arrs


def upstream_grad(w: Workload, B=None, H=None, T=None, seed_offset=1000):
    """A seeded upstream gradient dL/do of workload ``w`` for the backward
    pass: float32 N(0,1) of shape [B, H, T, d], from
    ``default_rng(w.seed + seed_offset)``."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    rng = np.random.default_rng(w.seed + seed_offset)
    return rng.standard_normal((B, H, T, w.d), dtype=np.float32)
