"""fp64 CPU oracle for the Variational Linear Attention forward recurrence.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package. The
product (``sherman_morrison_memory_gb300``) never imports it and shares no code
with it; the two meet only at the seeded input generator.

The arithmetic lives in ``vla_oracle.c`` (plain C loops in fp64, one head per
OpenMP thread, following §3.3 eq. 9-11 of "Variational Linear Attention",
arXiv 2605.11196); this module compiles it with gcc and calls it through
ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vla_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libvla_oracle.so")

__all__ = ["build", "Oracle", "load", "vla_forward", "linear_attention_state", "OracleResult"]


def build(src: str = SRC, out: str = LIB, openmp: bool = True) -> str:
    """Compile the oracle with gcc into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", out, "-lm"]
    if openmp:
        cmd.insert(1, "-fopenmp")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        if openmp:
            return build(src, out, openmp=False)
        raise RuntimeError("oracle build failed:\n" + r.stderr)
    return out


_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)


def _ptr(a, typ):
    if a is None:
        return ctypes.cast(None, typ)
    return a.ctypes.data_as(typ)


@dataclass
class OracleResult:
    o: Optional[np.ndarray]
    S: np.ndarray
    A: np.ndarray
    zk: np.ndarray
    delta: Optional[np.ndarray] = None
    alpha: Optional[np.ndarray] = None
    khat: Optional[np.ndarray] = None
    uhat: Optional[np.ndarray] = None
    e: Optional[np.ndarray] = None
    threads: int = 1


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        self.lib = ctypes.CDLL(path)
        f = self.lib.vla_oracle_forward
        f.restype = ctypes.c_int
        f.argtypes = ([ctypes.c_int] * 3 + [_fp] * 4 + [ctypes.c_double] * 2
                      + [_dp] * 3 + [_dp] * 4 + [_dp] * 5 + [ctypes.c_int])
        g = self.lib.vla_oracle_linear_attention_state
        g.restype = ctypes.c_int
        g.argtypes = [ctypes.c_int] * 3 + [_fp] * 2 + [_dp, ctypes.c_int]
        h = self.lib.vla_oracle_forward_f64
        h.restype = ctypes.c_int
        h.argtypes = [ctypes.c_int] * 3 + [_dp] * 4 + [ctypes.c_double] * 2 + [_dp] * 3 + [_dp] * 4
        b = self.lib.vla_oracle_backward
        b.restype = ctypes.c_int
        b.argtypes = ([ctypes.c_int] * 3 + [_dp] * 4 + [ctypes.c_double] * 2 + [_dp] * 3 + [_dp] * 4
                      + [_dp] * 4 + [_dp] * 3 + [ctypes.c_int])

    def forward(self, q, k, v, u, lambda0=0.1, eps=1e-4, S0=None, A0=None, zk0=None,
                want_o=True, trace=False, threads=0) -> OracleResult:
        """Run the recurrence for every head.

        q, k, v, u: arrays [..., T, d] (any leading shape; flattened to heads),
        converted to float32 (exact for fp32 and bf16 values). Optional state
        S0, A0 [..., d, d] and zk0 [..., d]. Returns fp64 outputs shaped like
        the inputs.
        """
        q = np.ascontiguousarray(q, dtype=np.float32)
        k = np.ascontiguousarray(k, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        u = np.ascontiguousarray(u, dtype=np.float32)
        lead = q.shape[:-2]
        T, d = q.shape[-2], q.shape[-1]
        BH = int(np.prod(lead)) if lead else 1
        for x in (k, v, u):
            assert x.shape == q.shape
        S0 = None if S0 is None else np.ascontiguousarray(S0, dtype=np.float64)
        A0 = None if A0 is None else np.ascontiguousarray(A0, dtype=np.float64)
        zk0 = None if zk0 is None else np.ascontiguousarray(zk0, dtype=np.float64)
        o = np.empty(lead + (T, d)) if want_o else None
        S = np.empty(lead + (d, d))
        A = np.empty(lead + (d, d))
        zk = np.empty(lead + (d,))
        tr = {}
        if trace:
            tr = dict(delta=np.empty(lead + (T,)), alpha=np.empty(lead + (T, d)),
                      khat=np.empty(lead + (T, d)), uhat=np.empty(lead + (T, d)),
                      e=np.empty(lead + (T, d)))
        n = self.lib.vla_oracle_forward(
            BH, T, d, _ptr(q, _fp), _ptr(k, _fp), _ptr(v, _fp), _ptr(u, _fp),
            float(lambda0), float(eps), _ptr(S0, _dp), _ptr(A0, _dp), _ptr(zk0, _dp),
            _ptr(o, _dp), _ptr(S, _dp), _ptr(A, _dp), _ptr(zk, _dp),
            _ptr(tr.get("delta"), _dp), _ptr(tr.get("alpha"), _dp), _ptr(tr.get("khat"), _dp),
            _ptr(tr.get("uhat"), _dp), _ptr(tr.get("e"), _dp), int(threads))
        return OracleResult(o=o, S=S, A=A, zk=zk, threads=n, **tr)

    def forward_f64(self, q, k, v, u, lambda0=0.1, eps=1e-4, S0=None, A0=None, zk0=None):
        """The recurrence with fp64 inputs (for finite-difference checks):
        returns (o, S, A, zk) as fp64 arrays shaped like the inputs."""
        q, k, v, u = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, u))
        lead = q.shape[:-2]
        T, d = q.shape[-2], q.shape[-1]
        BH = int(np.prod(lead)) if lead else 1
        f = lambda x: None if x is None else np.ascontiguousarray(x, dtype=np.float64)
        o, S, A, zk = np.empty(lead + (T, d)), np.empty(lead + (d, d)), np.empty(lead + (d, d)), np.empty(lead + (d,))
        self.lib.vla_oracle_forward_f64(BH, T, d, _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(u, _dp),
                                        float(lambda0), float(eps), _ptr(f(S0), _dp), _ptr(f(A0), _dp),
                                        _ptr(f(zk0), _dp), _ptr(o, _dp), _ptr(S, _dp), _ptr(A, _dp), _ptr(zk, _dp))
        return o, S, A, zk

    def backward(self, q, k, v, u, lambda0=0.1, eps=1e-4, S0=None, A0=None, zk0=None,
                 gO=None, gS=None, gA=None, gzk=None, threads=0):
        """Reverse-mode gradient of the recurrence (fp64) for the loss seeds
        gO = dL/do [..., T, d] and gS, gA = dL/dS_T, dL/dA_T [..., d, d], gzk =
        dL/dz^key_T [..., d] (each optional). Returns dict dq, dk, dv, du,
        dS0, dA0, dzk0 and the number of threads used."""
        q, k, v, u = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, u))
        lead = q.shape[:-2]
        T, d = q.shape[-2], q.shape[-1]
        BH = int(np.prod(lead)) if lead else 1
        f = lambda x: None if x is None else np.ascontiguousarray(x, dtype=np.float64)
        out = {n: np.empty(lead + (T, d)) for n in ("dq", "dk", "dv", "du")}
        out.update(dS0=np.empty(lead + (d, d)), dA0=np.empty(lead + (d, d)), dzk0=np.empty(lead + (d,)))
        n = self.lib.vla_oracle_backward(
            BH, T, d, _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(u, _dp), float(lambda0), float(eps),
            _ptr(f(S0), _dp), _ptr(f(A0), _dp), _ptr(f(zk0), _dp),
            _ptr(f(gO), _dp), _ptr(f(gS), _dp), _ptr(f(gA), _dp), _ptr(f(gzk), _dp),
            _ptr(out["dq"], _dp), _ptr(out["dk"], _dp), _ptr(out["dv"], _dp), _ptr(out["du"], _dp),
            _ptr(out["dS0"], _dp), _ptr(out["dA0"], _dp), _ptr(out["dzk0"], _dp), int(threads))
        out["threads"] = n
        return out

    def linear_attention_state(self, k, v, threads=0) -> np.ndarray:
        """S = sum_t v_t phi(k_t)^T per head, fp64, shape [..., d, d]."""
        k = np.ascontiguousarray(k, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        lead = k.shape[:-2]
        T, d = k.shape[-2], k.shape[-1]
        BH = int(np.prod(lead)) if lead else 1
        S = np.empty(lead + (d, d))
        self.lib.vla_oracle_linear_attention_state(BH, T, d, _ptr(k, _fp), _ptr(v, _fp),
                                                   _ptr(S, _dp), int(threads))
        return S


_default: Optional[Oracle] = None


def load(rebuild: bool = False) -> Oracle:
    """The oracle compiled from ``vla_oracle.c`` (built on first use)."""
    global _default
    if _default is None or rebuild:
        stale = (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)
        if rebuild or stale:
            build()
        _default = Oracle(LIB)
    return _default


def vla_forward(*args, **kwargs) -> OracleResult:
    return load().forward(*args, **kwargs)


def linear_attention_state(*args, **kwargs) -> np.ndarray:
    return load().linear_attention_state(*args, **kwargs)
