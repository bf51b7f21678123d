"""Parity of the CUDA backward pass (vla_backward, through the C ABI) with the
fp64 oracle's reverse-mode gradient.

Cases span several 64-token checkpoint segments and a ragged tail, every
supported head dimension (d = 128 through the split reverse sweep, which is
also checked at d <= 96 against the oracle and the single-kernel sweep), both
input dtypes, with and without an initial state, each upstream seed alone,
T = 0, and sampled heads of the d = 96, T = 4096 workload. Tolerance: 2e-3 relative (parity_util.TOL), per token
(rows of dq, dk, dv, du) and per head (dS0, dA0, dzk0), as for the forward.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_close, rel_heads, rel_rows
from sherman_morrison_memory_gb300 import (VLA_ERR_NONFINITE, VLA_ERR_TIMEOUT, VLA_OK, VLAError,
                                           vla_backward, vla_get_last_device_status)
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


def _seeds(B, H, T, d, seed, with_o=True, with_state=True):
    rng = np.random.default_rng(1000 + seed)
    gO = rng.standard_normal((B, H, T, d)).astype(np.float32) if with_o else None
    gst = None
    if with_state:
        gst = (rng.standard_normal((B, H, d, d)).astype(np.float32),
               rng.standard_normal((B, H, d, d)).astype(np.float32),
               rng.standard_normal((B, H, d)).astype(np.float32))
    return gO, gst


def _warm_state(orc, B, H, d, seed):
    """A reachable initial state: the oracle's state after 30 tokens, in fp32."""
    warm = orc.forward(*W.normal(B, H, 30, d, seed=seed))
    return tuple(np.asarray(x, dtype=np.float32) for x in (warm.S, warm.A, warm.zk))


def _dev(x, dtype=torch.float32):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda().to(dtype)


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def _run(orc, arrs, dtype, gO, gst, state=None, lambda0=0.1, eps=1e-4, split=False):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v, u = (_dev(a, tdt) for a in arrs)
    grads, dstate = vla_backward(q, k, v, u, lambda0, eps, None if state is None else tuple(_dev(x) for x in state),
                                 _dev(gO), None if gst is None else tuple(_dev(x) for x in gst), check=True,
                                 split=split)
    st = (None, None, None) if state is None else tuple(_f64(x) for x in state)
    gs = (None, None, None) if gst is None else tuple(_f64(x) for x in gst)
    ref = orc.backward(*(_f64(a) for a in arrs), lambda0, eps, *st, _f64(gO), *gs)
    return grads, dstate, ref


def _errors(grads, dstate, ref):
    dq, dk, dv, du = (x.cpu().numpy() for x in grads)
    dS0, dA0, dzk0 = (x.cpu().numpy() for x in dstate)
    return dict(dq=rel_rows(dq, ref["dq"]), dk=rel_rows(dk, ref["dk"]), dv=rel_rows(dv, ref["dv"]),
                du=rel_rows(du, ref["du"]), dS0=rel_heads(dS0, ref["dS0"]), dA0=rel_heads(dA0, ref["dA0"]),
                dzk0=rel_heads(dzk0, ref["dzk0"]))


@pytest.mark.parametrize("d", [32, 64, 96])
@pytest.mark.parametrize("T", [1, 37, 129])
def test_small_f32(orc, d, T):
    arrs = _inputs(1, 2, T, d, "f32", seed=d + T)
    gO, gst = _seeds(1, 2, T, d, seed=d + T)
    assert_close(_errors(*_run(orc, arrs, "f32", gO, gst)), what=f"backward f32 d={d} T={T}")


@pytest.mark.parametrize("d", [32, 64, 96])
def test_bf16_with_initial_state(orc, d):
    """Initial state carried in; 200 tokens = three checkpoint segments + tail."""
    B, H, T = 1, 2, 200
    arrs = _inputs(B, H, T, d, "bf16", seed=d)
    state = _warm_state(orc, B, H, d, seed=d + 1)
    gO, gst = _seeds(B, H, T, d, seed=d)
    assert_close(_errors(*_run(orc, arrs, "bf16", gO, gst, state=state)), what=f"backward bf16+state d={d}")


@pytest.mark.parametrize("which", ["o_only", "state_only"])
def test_single_upstream_seed(orc, which):
    B, H, T, d = 2, 2, 100, 64
    arrs = _inputs(B, H, T, d, "f32", seed=5)
    gO, gst = _seeds(B, H, T, d, seed=5, with_o=which == "o_only", with_state=which == "state_only")
    assert_close(_errors(*_run(orc, arrs, "f32", gO, gst)), what=f"backward {which}")


def test_lambda_and_eps(orc):
    arrs = _inputs(1, 2, 80, 32, "f32", seed=6)
    gO, gst = _seeds(1, 2, 80, 32, seed=6)
    assert_close(_errors(*_run(orc, arrs, "f32", gO, gst, lambda0=0.7, eps=0.5)), what="backward lambda/eps")


def test_long_sequence_bf16(orc):
    B, H, T, d = 2, 2, 1000, 96
    arrs = _inputs(B, H, T, d, "bf16", seed=7)
    gO, gst = _seeds(B, H, T, d, seed=7)
    assert_close(_errors(*_run(orc, arrs, "bf16", gO, gst)), what="backward T=1000")


@pytest.mark.parametrize("d,split", [(64, False), (64, True), (128, False)])
def test_zero_tokens_passes_state_gradient_through(orc, d, split):
    """T = 0: the forward is the identity on the state, so dState0 = dState_T."""
    B, H = 1, 3
    arrs = tuple(np.zeros((B, H, 0, d), np.float32) for _ in range(4))
    _, gst = _seeds(B, H, 0, d, seed=8, with_o=False)
    grads, dstate, ref = _run(orc, arrs, "f32", None, gst, split=split)
    assert all(g.shape == (B, H, 0, d) for g in grads)
    for got, want in zip(dstate, gst):
        np.testing.assert_array_equal(got.cpu().numpy(), want)
    assert_close(_errors(grads, dstate, ref), what="backward T=0")


def test_workload_d96_sampled_heads(orc):
    """The d = 96, T = 4096 bf16 workload in its full launch (128 heads); the
    oracle checks two sampled heads."""
    w = W.WORKLOADS[3]
    arrs = W.make(w)
    B, H, T, d = w.B, w.H, w.T, w.d
    q, k, v, u = (_dev(a, torch.bfloat16) for a in arrs)
    rng = np.random.default_rng(9)
    gO = rng.standard_normal((B, H, T, d)).astype(np.float32)
    grads, dstate = vla_backward(q, k, v, u, 0.1, 1e-4, None, _dev(gO), check=True)
    heads = [0, B * H - 1, 77]
    flat = lambda x: x.reshape((B * H,) + x.shape[2:])[heads][None]
    ref = orc.backward(*(flat(a).astype(np.float64) for a in arrs), 0.1, 1e-4, gO=flat(gO).astype(np.float64))
    pick = lambda x: flat(x.cpu().numpy())
    dq, dk, dv, du = (pick(x) for x in grads)
    dS0, dA0, dzk0 = (pick(x) for x in dstate)
    errs = dict(dq=rel_rows(dq, ref["dq"]), dk=rel_rows(dk, ref["dk"]), dv=rel_rows(dv, ref["dv"]),
                du=rel_rows(du, ref["du"]), dS0=rel_heads(dS0, ref["dS0"]), dA0=rel_heads(dA0, ref["dA0"]),
                dzk0=rel_heads(dzk0, ref["dzk0"]))
    assert_close(errs, what="backward d96 workload")
    for g in grads + dstate:
        assert torch.isfinite(g).all()


def test_workload4_cut_d128_sampled_heads(orc):
    """The backward bench line's d = 128 configuration in its full launch: the
    long-context workload cut to 4096 tokens (B=1, H=32, bf16 inputs, the
    bench's seeded dL/do), on the taped cluster-pair forward and the
    cluster-pair sweep; the oracle checks two sampled heads, every token."""
    import dataclasses
    w = dataclasses.replace(W.WORKLOADS[4], T=4096)
    arrs = W.make(w)
    gO = W.upstream_grad(w)
    B, H, T, d = w.B, w.H, w.T, w.d
    q, k, v, u = (_dev(a, torch.bfloat16) for a in arrs)
    grads, dstate = vla_backward(q, k, v, u, w.lambda0, w.eps, None, _dev(gO), check=True)
    heads = [0, B * H - 1]
    flat = lambda x: x.reshape((B * H,) + x.shape[2:])[heads][None]
    ref = orc.backward(*(flat(a).astype(np.float64) for a in arrs), w.lambda0, w.eps,
                       gO=flat(gO).astype(np.float64))
    pick = lambda x: flat(x.cpu().numpy())
    dq, dk, dv, du = (pick(x) for x in grads)
    dS0, dA0, dzk0 = (pick(x) for x in dstate)
    errs = dict(dq=rel_rows(dq, ref["dq"]), dk=rel_rows(dk, ref["dk"]), dv=rel_rows(dv, ref["dv"]),
                du=rel_rows(du, ref["du"]), dS0=rel_heads(dS0, ref["dS0"]), dA0=rel_heads(dA0, ref["dA0"]),
                dzk0=rel_heads(dzk0, ref["dzk0"]))
    assert_close(errs, what="backward d128 workload cut to T=4096")
    for g in grads + dstate:
        assert torch.isfinite(g).all()


@pytest.mark.parametrize("split", [False, True])
def test_two_streams_at_once(orc, split):
    """Two calls on two streams with no ordering between them: each has its
    own tape (the call's buffer from the caching allocator), so both results
    are the oracle's; split=True runs the cluster-pair sweep."""
    cases = []
    for seed in (31, 32):
        arrs = _inputs(1, 2, 129, 64, "bf16", seed=seed)
        gO, gst = _seeds(1, 2, 129, 64, seed=seed)
        cases.append((arrs, gO, gst))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    dev_in = [([_dev(a, torch.bfloat16) for a in arrs], _dev(gO), tuple(_dev(x) for x in gst))
              for arrs, gO, gst in cases]
    torch.cuda.synchronize()
    res = []
    for (x, g, gs), st in zip(dev_in, streams):
        with torch.cuda.stream(st):
            res.append(vla_backward(*x, 0.1, 1e-4, None, g, gs, split=split))
    torch.cuda.synchronize()
    for (arrs, gO, gst), (grads, dstate) in zip(cases, res):
        ref = orc.backward(*(_f64(a) for a in arrs), 0.1, 1e-4, None, None, None, _f64(gO),
                           *(_f64(x) for x in gst))
        assert_close(_errors(grads, dstate, ref), what="backward on two streams")


@pytest.mark.parametrize("tensor", [0, 1, 2, 3])
def test_nonfinite_input_is_reported(tensor):
    arrs = [np.array(a) for a in _inputs(1, 1, 40, 64, "f32", seed=12)]
    arrs[tensor][0, 0, 7, 3] = np.nan
    q, k, v, u = (_dev(a) for a in arrs)
    gO, _ = _seeds(1, 1, 40, 64, seed=12, with_state=False)
    vla_backward(q, k, v, u, 0.1, 1e-4, None, _dev(gO))
    with pytest.raises(VLAError) as ei:
        vla_backward(q, k, v, u, 0.1, 1e-4, None, _dev(gO), check=True)
    assert ei.value.status == VLA_ERR_NONFINITE


def test_nonfinite_then_clean_call_succeeds(orc):
    arrs = [np.array(a) for a in _inputs(1, 1, 40, 32, "f32", seed=13)]
    bad = [a.copy() for a in arrs]
    bad[1][0, 0, 3, 1] = np.inf
    gO, _ = _seeds(1, 1, 40, 32, seed=13, with_state=False)
    with pytest.raises(VLAError):
        vla_backward(*(_dev(a) for a in bad), 0.1, 1e-4, None, _dev(gO), check=True)
    assert_close(_errors(*_run(orc, arrs, "f32", gO, None)), what="backward after a non-finite call")


@pytest.mark.parametrize("T", [1, 2, 3, 16, 37, 64, 65, 129])
def test_d128_small_f32(orc, T):
    """d = 128: the taped cluster-pair forward, then the split reverse sweep
    on a cluster pair. T = 2, 3: the A side's first wait is for a token the
    S side reaches only at its end; T = 16, 64, 65: exactly one chunk, one
    checkpoint interval, and one token past it (a second checkpoint slot)."""
    B, H, d = 1, 2, 128
    arrs = _inputs(B, H, T, d, "f32", seed=20 + T)
    gO, gst = _seeds(B, H, T, d, seed=20 + T)
    assert_close(_errors(*_run(orc, arrs, "f32", gO, gst)), what=f"backward d=128 T={T}")


def test_d128_bf16_with_initial_state(orc):
    B, H, T, d = 2, 2, 150, 128
    arrs = _inputs(B, H, T, d, "bf16", seed=24)
    gO, gst = _seeds(B, H, T, d, seed=24)
    state = _warm_state(orc, B, H, d, seed=25)
    assert_close(_errors(*_run(orc, arrs, "bf16", gO, gst, state=state)), what="backward d=128 bf16 state")


def test_d128_long_sequence_bf16(orc):
    """Many 64-token checkpoint segments at d = 128."""
    B, H, T, d = 1, 2, 1000, 128
    arrs = _inputs(B, H, T, d, "bf16", seed=26)
    gO, gst = _seeds(B, H, T, d, seed=26)
    assert_close(_errors(*_run(orc, arrs, "bf16", gO, gst)), what="backward d=128 T=1000")


@pytest.mark.parametrize("d", [32, 64, 96])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_sweep(orc, d, dtype):
    """The split reverse sweep (S side, then A side) at the head dimensions the
    single-kernel sweep also covers: both match the oracle, and each other."""
    B, H, T = 1, 3, 129
    arrs = _inputs(B, H, T, d, dtype, seed=30 + d)
    gO, gst = _seeds(B, H, T, d, seed=30 + d)
    state = _warm_state(orc, B, H, d, seed=31 + d)
    g_split, s_split, ref = _run(orc, arrs, dtype, gO, gst, state=state, split=True)
    assert_close(_errors(g_split, s_split, ref), what=f"split backward d={d} {dtype}")
    g_one, s_one, _ = _run(orc, arrs, dtype, gO, gst, state=state)
    for a, b in zip(g_split, g_one):
        assert rel_rows(a.cpu().numpy(), b.cpu().numpy().astype(np.float64)) <= 2e-3
    for a, b in zip(s_split, s_one):
        assert rel_heads(a.cpu().numpy(), b.cpu().numpy().astype(np.float64)) <= 2e-3


def test_split_single_upstream_seeds(orc):
    """Only dL/do, then only the state seeds, through the split sweep."""
    B, H, T, d = 1, 2, 70, 128
    arrs = _inputs(B, H, T, d, "f32", seed=40)
    for with_o in (True, False):
        gO, gst = _seeds(B, H, T, d, seed=40, with_o=with_o, with_state=not with_o)
        assert_close(_errors(*_run(orc, arrs, "f32", gO, gst)), what=f"backward d=128 seeds o={with_o}")


@pytest.mark.parametrize("d", [64, 128])
def test_split_wait_runs_out_and_is_reported(orc, d):
    """The split sweep's one wait (its A side waits for the S side's
    progress) is bounded: with the S side publishing nothing (test hook) it
    runs out after the limit and the call reports VLA_ERR_TIMEOUT, without a
    hang or a fault; a normal call afterwards is the oracle's again."""
    arrs = _inputs(1, 2, 70, d, "f32", seed=d + 5)
    gO, _ = _seeds(1, 2, 70, d, seed=d + 5, with_state=False)
    dev_in = [_dev(a) for a in arrs]
    with pytest.raises(VLAError) as ei:
        vla_backward(*dev_in, 0.1, 1e-4, None, _dev(gO), check=True, split=True, wait_limit_us=2000,
                     test_stall_producer=True)
    assert ei.value.status == VLA_ERR_TIMEOUT
    assert_close(_errors(*_run(orc, arrs, "f32", gO, None, split=True)), what=f"split sweep after a timeout d={d}")


def test_split_nonfinite_input_is_reported():
    arrs = [np.array(a) for a in _inputs(1, 1, 40, 128, "f32", seed=41)]
    arrs[1][0, 0, 9, 5] = np.nan
    gO, _ = _seeds(1, 1, 40, 128, seed=41, with_state=False)
    with pytest.raises(VLAError) as ei:
        vla_backward(*(_dev(a) for a in arrs), 0.1, 1e-4, None, _dev(gO), check=True)
    assert ei.value.status == VLA_ERR_NONFINITE
