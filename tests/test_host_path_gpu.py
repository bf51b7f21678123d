"""vla_forward_host (host buffers in and out, copies overlapped with the
kernels) against the fp64 oracle and against vla_forward on device buffers.

The host path cuts the sequence into chunks and carries the state (S, A,
z^key) from launch to launch; the cases below span several chunks with a
ragged last one, chunk lengths that are and are not multiples of the chunked
kernel's 16 tokens, a carried-in initial state, page-locked and pageable host
memory, the fixed-A variant and T = 0. Tolerance: parity_util.TOL against the
oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, assert_close, errors, rel_heads, rel_rows
from sherman_morrison_memory_gb300 import VLA_ALGO_CHUNKED, VLA_ALGO_PER_TOKEN, VLA_OK, _binding, vla_forward
from sherman_morrison_memory_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def _inputs(B, H, T, d, dtype, seed):
    arrs = W.normal(B, H, T, d, seed=seed)
    if dtype == "bf16":
        arrs = tuple(W.to_bf16_values(a) for a in arrs)
    return arrs


def _host(arrs, dtype, pin=True):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    xs = [torch.from_numpy(np.ascontiguousarray(a)).to(tdt) for a in arrs]
    return [x.pin_memory() for x in xs] if pin else xs


def _dev_run(arrs, dtype, **kw):
    return vla_forward(*[x.cuda() for x in _host(arrs, dtype, pin=False)], check=True, **kw)


def _agree(host_out, dev_out, tol=1e-4):
    ho, (hS, hA, hz) = host_out
    do, (dS, dA, dz) = dev_out
    e = {"o": rel_rows(ho.numpy(), do.cpu().numpy()), "S": rel_heads(hS.numpy(), dS.cpu().numpy()),
         "A": rel_heads(hA.numpy(), dA.cpu().numpy()), "zk": rel_heads(hz.numpy(), dz.cpu().numpy())}
    assert_close(e, tol=tol, what="host path vs device path")


@pytest.mark.parametrize("algo", [0, VLA_ALGO_PER_TOKEN, VLA_ALGO_CHUNKED])
@pytest.mark.parametrize("d,dtype,T,chunk", [(64, "f32", 300, 64), (96, "bf16", 200, 48), (32, "f32", 129, 16),
                                             (128, "bf16", 90, 40)])
def test_chunks_match_oracle(orc, d, dtype, T, chunk, algo):
    if algo == VLA_ALGO_CHUNKED and d > 96:
        pytest.skip("the chunked kernel covers d <= 96")
    arrs = _inputs(2, 3, T, d, dtype, seed=d + T)
    out = vla_forward(*_host(arrs, dtype), chunk_tokens=chunk, algo=algo, check=True)
    assert out[0].device.type == "cpu"
    assert_close(errors(out, orc.forward(*arrs)), what=f"host path d={d} T={T} chunk={chunk}")
    _agree(out, _dev_run(arrs, dtype, algo=algo))


@pytest.mark.parametrize("pin", [True, False])
def test_automatic_chunks_long_sequence(orc, pin):
    # T = 2048 -> automatic chunks of 128, 512, 512, 512, 256, 128 tokens
    arrs = _inputs(1, 4, 2048, 96, "bf16", seed=21)
    out = vla_forward(*_host(arrs, "bf16", pin=pin), check=True)
    assert_close(errors(out, orc.forward(*arrs)), what="automatic chunks")
    _agree(out, _dev_run(arrs, "bf16"))


def test_carried_state_and_pageable_memory(orc):
    d, T = 64, 150
    arrs = _inputs(1, 2, 2 * T, d, "f32", seed=22)
    first = tuple(a[:, :, :T] for a in arrs)
    second = tuple(np.ascontiguousarray(a[:, :, T:]) for a in arrs)
    o1, st1 = vla_forward(*_host(first, "f32", pin=False), chunk_tokens=64, check=True)
    o2, st2 = vla_forward(*_host(second, "f32", pin=False), state=st1, chunk_tokens=50, check=True)
    ref = orc.forward(*arrs)
    errs = errors((torch.cat([o1, o2], dim=2), st2), ref)
    assert_close(errs, what="two host calls with carried state, pageable memory")


def test_fixed_a_without_u(orc):
    # the fixed-A variant is the recurrence with u = 0 (A stays at A0)
    arrs = _inputs(1, 2, 100, 96, "bf16", seed=23)
    q, k, v, _ = _host(arrs, "bf16")
    out = vla_forward(q, k, v, None, fixed_a=True, chunk_tokens=32, check=True)
    ref = orc.forward(arrs[0], arrs[1], arrs[2], np.zeros_like(arrs[3]))
    assert_close(errors(out, ref), what="fixed A host path")
    _agree(out, vla_forward(*[x.cuda() for x in (q, k, v)], None, fixed_a=True, check=True))


def test_zero_tokens_copies_state(orc):
    d = 32
    rng = np.random.default_rng(24)
    S0 = rng.standard_normal((1, 2, d, d)).astype(np.float32)
    A0 = np.broadcast_to(np.eye(d, dtype=np.float32) * 3, (1, 2, d, d)).copy()
    zk0 = rng.random((1, 2, d)).astype(np.float32)
    e = torch.empty((1, 2, 0, d), dtype=torch.float32)
    o, (S, A, zk) = vla_forward(e, e, e, e, state=tuple(torch.from_numpy(x) for x in (S0, A0, zk0)), check=True)
    torch.cuda.synchronize()
    assert o.shape == (1, 2, 0, d)
    assert np.array_equal(S.numpy(), S0) and np.array_equal(A.numpy(), A0) and np.array_equal(zk.numpy(), zk0)


def test_workspace_size_and_arguments():
    lib = _binding.load_library()
    assert lib.vla_forward_host_workspace_bytes(1, 8, 16, 4096, 96, 0) > 3 * 4 * 128 * 1024 * 96 * 2
    assert lib.vla_forward_host_workspace_bytes(1, 1, 1, 10, 48, 0) == 0
    vp = ctypes.c_void_p
    ws = torch.zeros(1 << 16, dtype=torch.int32, device="cuda")
    small = ctypes.c_size_t(256)
    st = lib.vla_forward_host(vp(1), vp(1), vp(1), vp(1), 1, 1, 1, 10, 64, 0.1, 1e-4, None, None, None,
                              vp(1), vp(1), vp(1), None, 0, vp(ws.data_ptr()), small, None, None)
    assert st == _binding.VLA_ERR_INVALID_ARG  # workspace too small, rejected before any copy
    st = lib.vla_forward_host(vp(1), vp(1), vp(1), vp(1), 1, 1, 1, 10, 64, 0.1, 1e-4, None, None, None,
                              vp(1), vp(1), vp(1), None, -1, vp(ws.data_ptr()), small, None, None)
    assert st == _binding.VLA_ERR_INVALID_ARG  # negative chunk length
    assert _binding.vla_get_last_device_status("cuda")[0] == VLA_OK


def test_back_to_back_calls_of_different_shapes(orc):
    """Two calls enqueued one after the other, each with its own staging
    buffers from the caching allocator, before any synchronisation."""
    arrs_a = _inputs(1, 2, 120, 64, "f32", seed=25)
    arrs_b = _inputs(2, 2, 333, 96, "bf16", seed=26)
    oa = vla_forward(*_host(arrs_a, "f32"), chunk_tokens=32)
    ob = vla_forward(*_host(arrs_b, "bf16"), chunk_tokens=100)
    torch.cuda.synchronize()
    assert_close(errors(oa, orc.forward(*arrs_a)), what="first of two calls")
    assert_close(errors(ob, orc.forward(*arrs_b)), what="second of two calls")
    assert TOL == 2e-3


@pytest.mark.parametrize("pin_in,pin_out", [(True, True), (True, False), (False, True), (False, False)])
def test_output_written_in_place_or_copied(orc, pin_in, pin_out):
    """Page-locked (mapped) host o is written by the kernels directly; pageable
    o is copied out chunk by chunk. Both give the same result."""
    B, H, T, d = 1, 3, 170, 64
    arrs = _inputs(B, H, T, d, "bf16", seed=27)
    shapes = [(B, H, T, d), (B, H, d, d), (B, H, d, d), (B, H, d)]
    out = tuple(torch.full(sh, float("nan"), dtype=torch.float32, pin_memory=pin_out) for sh in shapes)
    res = vla_forward(*_host(arrs, "bf16", pin=pin_in), out=out, chunk_tokens=48, check=True)
    assert all(r is x for r, x in zip((res[0],) + tuple(res[1]), out))
    assert_close(errors(res, orc.forward(*arrs)), what=f"pin_in={pin_in} pin_out={pin_out}")
