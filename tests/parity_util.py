"""Helpers for comparing the CUDA path with the fp64 oracle.

Error metric (the paper fixes none; the target is 2e-3 relative):
  o     max over (head, t) of ||o_t - o^_t||_inf / ||o^_t||_inf   (per token)
  S, A  max over heads of  ||X - X^||_max / ||X^||_max            (per head)
  zk    max over heads of  ||zk - zk^||_max / ||zk^||_max
A per-token / per-head normwise error is robust to individual entries that
are near zero, which an elementwise relative error is not.
"""
from __future__ import annotations

import numpy as np
import torch

TOL = 2e-3


def rel_rows(x, ref, floor=1e-30):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.max(np.abs(x - ref), axis=-1)
    den = np.maximum(np.max(np.abs(ref), axis=-1), floor)
    return float(np.max(num / den)) if num.size else 0.0


def rel_heads(x, ref, floor=1e-30):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.size == 0:
        return 0.0
    lead = ref.shape[:2]
    xf = x.reshape(lead + (-1,))
    rf = ref.reshape(lead + (-1,))
    num = np.max(np.abs(xf - rf), axis=-1)
    den = np.maximum(np.max(np.abs(rf), axis=-1), floor)
    return float(np.max(num / den))


def to_dev(arrs, dtype: str, device="cuda"):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return [torch.from_numpy(np.ascontiguousarray(a)).to(device).to(tdt) for a in arrs]


def errors(gpu_out, ref):
    o, (S, A, zk) = gpu_out
    e = {}
    if ref.o is not None and o is not None:
        e["o"] = rel_rows(o.cpu().numpy(), ref.o)
    e["S"] = rel_heads(S.cpu().numpy(), ref.S)
    e["A"] = rel_heads(A.cpu().numpy(), ref.A)
    e["zk"] = rel_heads(zk.cpu().numpy(), ref.zk)
    return e


def assert_close(errs, tol=TOL, what=""):
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, f"{what} errors above {tol}: {bad} (all: {errs})"
