"""Helpers for comparing the CUDA path with the fp64 oracle.

Error metric (the paper fixes none; the target is 2e-3 relative):
  o     max over (head, t) of ||o_t - o^_t||_inf / ||o^_t||_inf   (per token)
  S, A  max over heads of  ||X - X^||_max / ||X^||_max            (per head)
  zk    max over heads of  ||zk - zk^||_max / ||zk^||_max
A per-token / per-head normwise error is robust to individual entries that
are near zero, which an elementwise relative error is not. The gate is the
normwise error; the elementwise relative error |x - x^| / (|x^| + f), with an
absolute floor f = 1e-3 of the token's / head's largest |x^|, is recorded
beside it for information (entries below the floor are measured against it).

Every comparison that goes through assert_close is recorded in RECORD, and
the test session prints the worst errors per test at its end (conftest.py).
"""
from __future__ import annotations

import os

import numpy as np
import torch

TOL = 2e-3
ELEM_FLOOR = 1e-3
# test name -> {quantity: worst error}; filled by assert_close / record
RECORD = {}


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


def elem_rows(x, ref, floor_frac=ELEM_FLOOR):
    """max over elements of |x - ref| / (|ref| + floor_frac * max|ref| of the row)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.size == 0:
        return 0.0
    scale = np.max(np.abs(ref), axis=-1, keepdims=True)
    return float(np.max(np.abs(x - ref) / (np.abs(ref) + floor_frac * scale + 1e-30)))


def elem_heads(x, ref, floor_frac=ELEM_FLOOR):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if x.size == 0:
        return 0.0
    lead = ref.shape[:2]
    return elem_rows(x.reshape(lead + (-1,)), ref.reshape(lead + (-1,)), floor_frac)


def errors(gpu_out, ref, elementwise=True):
    """Normwise errors of (o, (S, A, zk)) against the oracle result `ref`, and
    (keys ending in "_el") the elementwise relative errors beside them."""
    o, (S, A, zk) = gpu_out
    e = {}
    if ref.o is not None and o is not None:
        on = o.cpu().numpy()
        e["o"] = rel_rows(on, ref.o)
        if elementwise:
            e["o_el"] = elem_rows(on, ref.o)
    for name, x, r in (("S", S, ref.S), ("A", A, ref.A), ("zk", zk, ref.zk)):
        xn = x.cpu().numpy()
        e[name] = rel_heads(xn, r)
        if elementwise:
            e[name + "_el"] = elem_heads(xn, r)
    return e


def _test_name():
    cur = os.environ.get("PYTEST_CURRENT_TEST", "")
    return cur.split(" ")[0].split("::")[-1].split("[")[0] or "?"


def record(errs, name=None):
    """Keep the worst value of every error in `errs` under the current test's name."""
    slot = RECORD.setdefault(name or _test_name(), {"n": 0})
    slot["n"] += 1
    for k, v in errs.items():
        if isinstance(v, (int, float)) and np.isfinite(v):
            slot[k] = max(slot.get(k, 0.0), float(v))


def assert_close(errs, tol=TOL, what=""):
    """Gate the normwise errors (keys without the "_el" suffix) at `tol`."""
    record(errs)
    gated = {k: v for k, v in errs.items() if not k.endswith("_el")}
    bad = {k: v for k, v in gated.items() if not (v <= tol)}
    assert not bad, f"{what} errors above {tol}: {bad} (all: {errs})"
