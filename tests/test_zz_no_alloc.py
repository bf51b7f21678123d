"""The no-allocation entry point (vla_forward_noalloc) against vla_forward.

vla_forward_noalloc is for callers that cannot allocate device memory (a
device budget already reserved in full by another runtime, loops that must not
call the allocator, callers without an allocator): its status record lives in
a static device array instead of a caller-provided workspace. Two calls in a
row must each match vla_forward within the parity tolerance (and the fp64
oracle, directly), and the second call must start from a cleared status even
though the first one left an error in the shared record.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, assert_close, errors, rel_heads, rel_rows
from sherman_morrison_memory_gb300 import VLA_ERR_NONFINITE, VLA_OK, _binding, vla_forward
from sherman_morrison_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _lib():
    lib = _binding.load_library()
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.vla_forward_noalloc.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, cf, vp, vp, vp,
                                        vp, vp, vp, vp, vp, ctypes.POINTER(ci)]
    lib.vla_forward_noalloc.restype = ci
    return lib


def _call_noalloc(lib, q, k, v, u):
    B, H, T, d = q.shape
    dev = q.device
    o = torch.empty((B, H, T, d), dtype=torch.float32, device=dev)
    S = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    A = torch.empty_like(S)
    zk = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    status = ctypes.c_int(-1)
    dt = 1 if q.dtype == torch.bfloat16 else 0
    st = lib.vla_forward_noalloc(P(q), P(k), P(v), P(u), dt, B, H, T, d, 0.1, 1e-4, None, None, None,
                                 P(o), P(S), P(A), P(zk),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(status))
    return st, status.value, (o, S, A, zk)


def _host_inputs(seed, dtype="bf16", B=2, H=3, T=77, d=96):
    arrs = W.normal(B, H, T, d, seed=seed)
    return [W.to_bf16_values(a) if dtype == "bf16" else a for a in arrs]


def _inputs(seed, dtype="bf16", B=2, H=3, T=77, d=96):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return [torch.from_numpy(a).cuda().to(tdt) for a in _host_inputs(seed, dtype, B, H, T, d)]


def _close(a, b):
    o1, S1, A1, z1 = (x.cpu().numpy().astype(np.float64) for x in a)
    o2, S2, A2, z2 = (x.cpu().numpy().astype(np.float64) for x in b)
    errs = {"o": rel_rows(o1, o2), "S": rel_heads(S1, S2), "A": rel_heads(A1, A2), "zk": rel_heads(z1, z2)}
    assert all(e <= TOL for e in errs.values()), errs


def test_noalloc_matches_vla_forward_twice():
    lib = _lib()
    orc = oracle.load()
    torch.cuda.synchronize()
    for seed, dtype, d in ((31, "bf16", 96), (32, "f32", 64)):
        q, k, v, u = _inputs(seed, dtype, d=d)
        ref_o, (ref_S, ref_A, ref_zk) = vla_forward(q, k, v, u, check=True)
        st, dev_st, out = _call_noalloc(lib, q, k, v, u)
        assert st == VLA_OK and dev_st == VLA_OK, (st, dev_st)
        _close(out, (ref_o, ref_S, ref_A, ref_zk))
        # and directly against the fp64 oracle on the same input bits
        fp64 = orc.forward(*_host_inputs(seed, dtype, d=d), lambda0=0.1, eps=1e-4)
        o, S, A, zk = out
        assert_close(errors((o, (S, A, zk)), fp64), what=f"noalloc vs oracle d={d} {dtype}")


def test_noalloc_status_is_cleared_between_calls():
    lib = _lib()
    q, k, v, u = _inputs(33, "f32", d=64)
    qn = q.clone()
    qn[0, 0, 5, 7] = float("nan")
    st, dev_st, _ = _call_noalloc(lib, qn, k, v, u)      # leaves NONFINITE in the shared record
    assert st == VLA_OK and dev_st == VLA_ERR_NONFINITE
    st, dev_st, out = _call_noalloc(lib, q, k, v, u)     # must start from a zero record
    assert st == VLA_OK and dev_st == VLA_OK
    ref_o, (ref_S, ref_A, ref_zk) = vla_forward(q, k, v, u, check=True)
    _close(out, (ref_o, ref_S, ref_A, ref_zk))
