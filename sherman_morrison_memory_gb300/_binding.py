"""ctypes binding of libvla_gb300.so (C ABI in include/vla.h).

Argument marshalling only: shapes, dtypes and devices are checked, outputs
and the status workspace are allocated with torch, and the C entry points are
called on the current CUDA stream. All arithmetic happens in the library.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))

VLA_OK = 0
VLA_ERR_INVALID_ARG = 1
VLA_ERR_UNSUPPORTED = 2
VLA_ERR_CUDA = 3
VLA_ERR_TIMEOUT = 4
VLA_ERR_NONFINITE = 5
VLA_ALGO_AUTO = 0
VLA_ALGO_PER_TOKEN = 1
VLA_ALGO_CHUNKED = 2
VLA_ALGO_DECODE = 3
VLA_ALGO_CHUNKED_PAIR = 4
VLA_ALGO_CHUNKED_ROWS = 5
VLA_ALGO_SEGMENTED = 6

_DTYPES = {torch.float32: 0, torch.bfloat16: 1}

_lock = threading.Lock()
_LIB = None
_WORKSPACES = {}


class VLAError(RuntimeError):
    def __init__(self, status: int, where: str, detail=None):
        self.status = status
        self.detail = detail
        msg = f"{where}: {vla_status_string(status)} (status {status})"
        if detail is not None and detail[0] >= 0:
            msg += f"; role={detail[0]} head={detail[1]} token={detail[2]}"
        super().__init__(msg)


class _Options(ctypes.Structure):
    _fields_ = [("wait_limit_us", ctypes.c_uint), ("test_stall_producer", ctypes.c_int),
                ("trace", ctypes.c_void_p), ("algo", ctypes.c_int), ("fixed_a", ctypes.c_int),
                ("scratch", ctypes.c_void_p), ("scratch_bytes", ctypes.c_size_t)]


def library_path() -> str:
    return os.path.join(_PKG, "_build", "libvla_gb300.so")


def load_library():
    """Load libvla_gb300.so; raises if it has not been built."""
    global _LIB
    with _lock:
        if _LIB is not None:
            return _LIB
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library not built: {path} is missing. "
                "Build it with `python -m sherman_morrison_memory_gb300.build`.")
        lib = ctypes.CDLL(path)
        vp, cp, ci, cf = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fwd_args = [vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, cf, vp, vp, vp, vp, vp, vp, vp, vp,
                    ctypes.c_size_t, vp]
        lib.vla_forward.argtypes = fwd_args
        lib.vla_forward.restype = ci
        lib.vla_forward_ex.argtypes = fwd_args + [ctypes.POINTER(_Options)]
        lib.vla_forward_ex.restype = ci
        lib.vla_workspace_bytes.argtypes = [ci, ci, ci, ci]
        lib.vla_workspace_bytes_ex.argtypes = [ci, ci, ci, ci, ci]
        lib.vla_workspace_bytes_ex.restype = ctypes.c_size_t
        lib.vla_workspace_bytes.restype = ctypes.c_size_t
        lib.vla_workspace_reset.argtypes = [vp, vp]
        lib.vla_workspace_reset.restype = ci
        lib.vla_get_last_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
        lib.vla_get_last_device_status.restype = ci
        lib.vla_status_string.argtypes = [ci]
        lib.vla_status_string.restype = ctypes.c_char_p
        lib.vla_linear_attention_state.argtypes = [vp, vp, ci, ci, ci, ci, ci, vp, vp]
        lib.vla_linear_attention_state.restype = ci
        lib.vla_backward_workspace_bytes.argtypes = [ci, ci, ci, ci]
        lib.vla_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.vla_backward.argtypes = ([vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, cf, vp, vp, vp, vp, vp, vp, vp]
                                     + [vp] * 7 + [vp, ctypes.c_size_t, vp])
        lib.vla_backward.restype = ci
        lib.vla_backward_split.argtypes = lib.vla_backward.argtypes
        lib.vla_backward_split.restype = ci
        lib.vla_backward_ex.argtypes = lib.vla_backward.argtypes + [ci, ctypes.POINTER(_Options)]
        lib.vla_backward_ex.restype = ci
        lib.vla_forward_host_workspace_bytes.argtypes = [ci, ci, ci, ci, ci, ci]
        lib.vla_forward_host_workspace_bytes.restype = ctypes.c_size_t
        lib.vla_forward_host.argtypes = (fwd_args[:18] + [ci, vp, ctypes.c_size_t, vp, ctypes.POINTER(_Options)])
        lib.vla_forward_host.restype = ci
        lib.vla_forward_noalloc.argtypes = fwd_args[:18] + [vp, ctypes.POINTER(ci)]
        lib.vla_forward_noalloc.restype = ci
        lib.vla_probe_ffma.argtypes = [ci, ci, ci, ci, vp, vp]
        lib.vla_probe_ffma.restype = ci
        lib.vla_probe_ffma_flop.argtypes = [ci, ci, ci, ci]
        lib.vla_probe_ffma_flop.restype = ctypes.c_double
        del cp
        _LIB = lib
        return lib


def vla_status_string(status: int) -> str:
    try:
        return load_library().vla_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def vla_workspace_bytes(B: int = 1, H: int = 1, T: int = 1, d: int = 32) -> int:
    """Device workspace bytes vla_forward needs for B x H heads of T tokens at head dimension d."""
    return int(load_library().vla_workspace_bytes(int(B), int(H), int(T), int(d)))


def vla_probe_ffma(blocks: int, threads: int, iters: int, packed: bool, sink: torch.Tensor, stream=None) -> float:
    """Enqueue the FP32 FMA throughput probe (include/vla_probe.h) on the
    current stream of sink's device; returns the FLOP the call performs."""
    lib = load_library()
    if sink.dtype != torch.float32 or not sink.is_cuda or sink.numel() < blocks * threads:
        raise ValueError("sink must be a CUDA float32 tensor of at least blocks * threads elements")
    st = lib.vla_probe_ffma(int(blocks), int(threads), int(iters), int(bool(packed)), _ptr(sink),
                            ctypes.c_void_p(_stream_handle(sink.device, stream)))
    if st != VLA_OK:
        raise VLAError(st, "vla_probe_ffma")
    return float(lib.vla_probe_ffma_flop(int(blocks), int(threads), int(iters), int(bool(packed))))


def _stream_handle(device: torch.device, stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


_STATUS_BYTES = 256


def _workspace(device: torch.device) -> torch.Tensor:
    """The device's status record (shared by the calls on it, so that the
    status is sticky until vla_get_last_device_status reads it; the kernels OR
    their error bits into it atomically, so calls on several streams may share
    it). Make one call on a device before capturing a CUDA graph there."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    ws = _WORKSPACES.get(idx)
    if ws is None:
        ws = torch.zeros(_STATUS_BYTES // 4, dtype=torch.int32, device=torch.device("cuda", idx))
        _WORKSPACES[idx] = ws
    return ws


def _on_stream(stream):
    """Allocate for `stream`: the caching allocator hands a block freed there
    to later work only once the work queued on that stream before the free
    has run, so a call's own buffers need no other lifetime management."""
    return contextlib.nullcontext() if stream is None else torch.cuda.stream(stream)


def _call_buffer(device: torch.device, nbytes: int, zero_status: bool) -> torch.Tensor:
    """Device memory of one call (the segmented path's buffers, a backward
    tape, a host-path staging area), 512-byte aligned by the caching
    allocator; its status record zeroed if asked."""
    buf = torch.empty((int(nbytes) + 3) // 4, dtype=torch.int32, device=device)
    if zero_status:
        buf[:_STATUS_BYTES // 4].zero_()
    return buf


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_state(x, shape, device, name):
    if x is None:
        return None
    if x.dtype != torch.float32 or tuple(x.shape) != shape:
        raise ValueError(f"{name} must be float32 of shape {shape}, got {x.dtype} {tuple(x.shape)}")
    if x.device != device:
        x = x.to(device, non_blocking=True)
    return x.contiguous()


def vla_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, u: torch.Tensor,
                lambda0: float = 0.1, eps: float = 1e-4, state=None, *, out=None, stream=None,
                check: bool = False, wait_limit_us: int = 0, test_stall_producer: bool = False,
                algo: int = 0, fixed_a: bool = False, chunk_tokens: int = 0):
    """VLA forward recurrence (§3.3 eq. 9-11) over all heads.

    Returns ``(o, (S, A, zk))``: o [B,H,T,d] float32, S and A [B,H,d,d], zk [B,H,d].
    ``state`` = (S0, A0, zk0), each optional, continues a previous call.
    ``out`` = (o, S, A, zk) preallocated outputs on the inputs' device.
    CPU inputs run on the current CUDA device through vla_forward_host:
    ``chunk_tokens`` tokens per launch (0 = automatic), the host<->device
    copies overlapped with the kernels; synchronise the stream before reading
    page-locked host outputs.
    ``check=True`` synchronises and raises on an in-kernel failure.
    ``algo`` selects the kernel: VLA_ALGO_AUTO (0), VLA_ALGO_PER_TOKEN (1),
    VLA_ALGO_CHUNKED (2, the tensor-core chunked kernel, d <= 96),
    VLA_ALGO_DECODE (3, short sequences with a carried state),
    VLA_ALGO_CHUNKED_PAIR (4, the chunked kernel on a cluster of two CTAs per
    head: A-pass and S-pass on separate SMs; any d), VLA_ALGO_CHUNKED_ROWS (5,
    a cluster of 1 + NS CTAs per head with S's rows split over NS of them) or
    VLA_ALGO_SEGMENTED (6, the sequence's two halves side by side; d <= 96,
    T >= 32). The segmented path's buffers (vla_workspace_bytes_ex) are
    the call's own, from torch's caching allocator on the call's stream, so
    calls on different streams may overlap and a call may be captured in a
    CUDA graph (after one eager call on the device).
    ``fixed_a=True`` runs the fixed-A variant (§3.5 ablation): A stays at its
    initial value, u is not read (it may be None).
    """
    if q.device.type == "cpu":
        return _forward_host(q, k, v, u, lambda0, eps, state, out=out, check=check, algo=algo, fixed_a=fixed_a,
                             chunk_tokens=chunk_tokens, stream=stream)
    lib = load_library()
    if u is None and not fixed_a:
        raise ValueError("u is required unless fixed_a=True")
    for name, x in (("k", k), ("v", v), ("u", u)):
        if x is None:
            continue
        if x.shape != q.shape or x.dtype != q.dtype or x.device != q.device:
            raise ValueError(f"{name} must match q in shape, dtype and device")
    if q.dim() != 4:
        raise ValueError("q, k, v, u must be [B, H, T, d]")
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported input dtype {q.dtype} (float32 or bfloat16)")
    q, k, v = (x.contiguous() for x in (q, k, v))
    u = None if u is None else u.contiguous()
    B, H, T, d = q.shape
    dev = q.device
    S0 = A0 = zk0 = None
    if state is not None:
        S0, A0, zk0 = state
        S0 = _check_state(S0, (B, H, d, d), dev, "S0")
        A0 = _check_state(A0, (B, H, d, d), dev, "A0")
        zk0 = _check_state(zk0, (B, H, d), dev, "zk0")
    ws = _workspace(dev)
    nbytes = int(lib.vla_workspace_bytes_ex(B, H, T, d, int(algo)))
    with torch.cuda.device(dev), _on_stream(stream):
        if out is None:
            o = torch.empty((B, H, T, d), dtype=torch.float32, device=dev)
            S = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
            A = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
            zk = torch.empty((B, H, d), dtype=torch.float32, device=dev)
        else:
            o, S, A, zk = out
        scratch = _call_buffer(dev, nbytes, False) if nbytes > _STATUS_BYTES else None
        sh = _stream_handle(dev, stream)
        args = (_ptr(q), _ptr(k), _ptr(v), _ptr(u), _DTYPES[q.dtype], B, H, T, d,
                float(lambda0), float(eps), _ptr(S0), _ptr(A0), _ptr(zk0),
                _ptr(o), _ptr(S), _ptr(A), _ptr(zk), _ptr(ws), ws.numel() * 4, ctypes.c_void_p(sh))
        if wait_limit_us or test_stall_producer or algo or fixed_a or scratch is not None:
            opts = _Options(int(wait_limit_us), 1 if test_stall_producer else 0, None, int(algo),
                            1 if fixed_a else 0, _ptr(scratch), 0 if scratch is None else scratch.numel() * 4)
            st = lib.vla_forward_ex(*args, ctypes.byref(opts))
        else:
            st = lib.vla_forward(*args)
    if st != VLA_OK:
        raise VLAError(st, "vla_forward")
    if check:
        st, detail = vla_get_last_device_status(dev, stream)
        if st != VLA_OK:
            raise VLAError(st, "vla_forward (device)", detail)
    return o, (S, A, zk)


def _forward_host(q, k, v, u, lambda0, eps, state, out=None, check=False, algo=0, fixed_a=False,
                  chunk_tokens=0, stream=None):
    """Host buffers in, host buffers out, through vla_forward_host: the
    sequence runs in chunks on the current CUDA device, with the copies of
    chunk j+1's inputs and chunk j-1's outputs overlapped with chunk j's
    kernel. ``out`` may hold preallocated host outputs (o, S, A, zk); new
    outputs are page-locked when q is. Like torch's non-blocking copies, the
    call returns once the work is enqueued: synchronise the stream before
    reading page-locked outputs (``check=True`` does)."""
    lib = load_library()
    if u is None and not fixed_a:
        raise ValueError("u is required unless fixed_a=True")
    for name, x in (("k", k), ("v", v), ("u", u)):
        if x is None:
            continue
        if x.shape != q.shape or x.dtype != q.dtype or x.device != q.device:
            raise ValueError(f"{name} must match q in shape, dtype and device")
    if q.dim() != 4 or q.dtype not in _DTYPES:
        raise ValueError("q, k, v, u must be [B, H, T, d] float32 or bfloat16")
    q, k, v = (x.contiguous() for x in (q, k, v))
    u = None if u is None else u.contiguous()
    B, H, T, d = q.shape
    cpu = torch.device("cpu")
    S0 = A0 = zk0 = None
    if state is not None:
        S0, A0, zk0 = state
        S0 = _check_state(S0, (B, H, d, d), cpu, "S0")
        A0 = _check_state(A0, (B, H, d, d), cpu, "A0")
        zk0 = _check_state(zk0, (B, H, d), cpu, "zk0")
    shapes = [(B, H, T, d), (B, H, d, d), (B, H, d, d), (B, H, d)]
    if out is None:
        pin = q.is_pinned()
        res = [torch.empty(sh, dtype=torch.float32, pin_memory=pin) for sh in shapes]
    else:
        res = list(out)
        for x, sh in zip(res, shapes):
            if (tuple(x.shape) != sh or x.dtype != torch.float32 or x.device.type != "cpu"
                    or not x.is_contiguous()):
                raise ValueError(f"out tensors must be contiguous float32 host tensors {sh}")
    o, S, A, zk = res
    dev = torch.device("cuda", torch.cuda.current_device())
    nbytes = int(lib.vla_forward_host_workspace_bytes(_DTYPES[q.dtype], B, H, T, d, int(chunk_tokens)))
    if nbytes == 0:
        raise ValueError("unsupported sizes for vla_forward_host")
    with torch.cuda.device(dev), _on_stream(stream):
        ws = _call_buffer(dev, nbytes, True)
        sh = _stream_handle(dev, stream)
        opts = _Options(0, 0, None, int(algo), 1 if fixed_a else 0)
        st = lib.vla_forward_host(_ptr(q), _ptr(k), _ptr(v), _ptr(u), _DTYPES[q.dtype], B, H, T, d,
                                  float(lambda0), float(eps), _ptr(S0), _ptr(A0), _ptr(zk0),
                                  _ptr(o), _ptr(S), _ptr(A), _ptr(zk), int(chunk_tokens), _ptr(ws),
                                  ws.numel() * 4, ctypes.c_void_p(sh), ctypes.byref(opts))
        if st != VLA_OK:
            raise VLAError(st, "vla_forward_host")
        if check:
            detail = (ctypes.c_int * 3)()
            st = lib.vla_get_last_device_status(_ptr(ws), ctypes.c_void_p(sh), detail)
            if st != VLA_OK:
                raise VLAError(st, "vla_forward_host (device)", (detail[0], detail[1], detail[2]))
    return o, (S, A, zk)


def vla_get_last_device_status(device=None, stream=None) -> Tuple[int, tuple]:
    """Synchronise the stream, read and clear the device status record.

    Returns (status, (role, head, token))."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ws = _workspace(dev)
    detail = (ctypes.c_int * 3)()
    with torch.cuda.device(dev):
        st = lib.vla_get_last_device_status(_ptr(ws), ctypes.c_void_p(_stream_handle(dev, stream)), detail)
    return int(st), (detail[0], detail[1], detail[2])


def _backward_host(q, k, v, u, lambda0, eps, state, grad_o, grad_state, out, check, split):
    """Host buffers in, host buffers out: H2D copies, the kernel, D2H copies,
    all on the current stream of the current CUDA device."""
    dev = torch.device("cuda", torch.cuda.current_device())
    to = lambda x: None if x is None else x.to(dev, non_blocking=True)
    dq_, dk_, dv_, du_ = (to(x) for x in (q, k, v, u))
    dstate = None if state is None else tuple(to(x) for x in state)
    dgs = None if grad_state is None else tuple(to(x) for x in grad_state)
    grads, dst = vla_backward(dq_, dk_, dv_, du_, lambda0, eps, dstate, to(grad_o), dgs, check=check, split=split)
    pin = q.is_pinned()
    outs = []
    for i, x in enumerate(grads + dst):
        h = out[i] if out is not None else torch.empty(x.shape, dtype=x.dtype, pin_memory=pin)
        h.copy_(x, non_blocking=h.is_pinned())
        outs.append(h)
    return tuple(outs[:4]), tuple(outs[4:])


def vla_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, u: torch.Tensor,
                 lambda0: float = 0.1, eps: float = 1e-4, state=None, grad_o=None, grad_state=None, *,
                 out=None, stream=None, check: bool = False, split: bool = False, wait_limit_us: int = 0,
                 test_stall_producer: bool = False):
    """Gradient of a scalar loss through vla_forward (reverse mode, §3.3 eq. 9-11).

    ``grad_o`` = dL/do [B,H,T,d] and ``grad_state`` = (dL/dS_T, dL/dA_T,
    dL/dz^key_T) (each optional, None = zero); ``state`` = the forward's
    optional initial (S0, A0, zk0). Returns ``((dq, dk, dv, du), (dS0, dA0,
    dzk0))``, float32 on the inputs' device. d in {32, 64, 96, 128}.
    ``split=True`` runs the reverse sweep split by state, as a cluster of two
    CTAs per head (vla_backward_split; the path d = 128 always takes).
    ``wait_limit_us`` bounds the split sweep's wait for its S side's progress;
    ``test_stall_producer=True`` (testing only) makes that wait run out, so
    that the call records VLA_ERR_TIMEOUT (vla_backward_ex).
    ``out`` may hold the seven result tensors (float32, contiguous, on the
    inputs' device). CPU inputs run on the current CUDA device with
    host<->device copies. ``check=True`` synchronises and raises on an
    in-kernel failure.
    """
    if q.device.type == "cpu":
        if wait_limit_us or test_stall_producer:
            raise ValueError("wait_limit_us and test_stall_producer apply to device inputs")
        return _backward_host(q, k, v, u, lambda0, eps, state, grad_o, grad_state, out, check, split)
    lib = load_library()
    for name, x in (("k", k), ("v", v), ("u", u)):
        if x.shape != q.shape or x.dtype != q.dtype or x.device != q.device:
            raise ValueError(f"{name} must match q in shape, dtype and device")
    if q.dim() != 4 or q.dtype not in _DTYPES or q.device.type != "cuda":
        raise ValueError("q, k, v, u must be [B, H, T, d] float32 or bfloat16 CUDA tensors")
    q, k, v, u = (x.contiguous() for x in (q, k, v, u))
    B, H, T, d = q.shape
    dev = q.device
    S0 = A0 = zk0 = None
    if state is not None:
        S0, A0, zk0 = state
        S0 = _check_state(S0, (B, H, d, d), dev, "S0")
        A0 = _check_state(A0, (B, H, d, d), dev, "A0")
        zk0 = _check_state(zk0, (B, H, d), dev, "zk0")
    gO = None if grad_o is None else _check_state(grad_o, (B, H, T, d), dev, "grad_o")
    gS = gA = gzk = None
    if grad_state is not None:
        gS, gA, gzk = grad_state
        gS = _check_state(gS, (B, H, d, d), dev, "dS_T")
        gA = _check_state(gA, (B, H, d, d), dev, "dA_T")
        gzk = _check_state(gzk, (B, H, d), dev, "dzk_T")
    shapes = [(B, H, T, d)] * 4 + [(B, H, d, d), (B, H, d, d), (B, H, d)]
    if out is None:
        with torch.cuda.device(dev), _on_stream(stream):
            res = [torch.empty(sh, dtype=torch.float32, device=dev) for sh in shapes]
    else:
        res = list(out)
        if len(res) != 7:
            raise ValueError("out must hold (dq, dk, dv, du, dS0, dA0, dzk0)")
        for x, sh in zip(res, shapes):
            if (tuple(x.shape) != sh or x.dtype != torch.float32 or x.device != dev or not x.is_contiguous()):
                raise ValueError(f"out tensors must be contiguous float32 {sh} on {dev}")
    outs = res[:4]
    dS0, dA0, dzk0 = res[4:]
    nbytes = int(lib.vla_backward_workspace_bytes(B, H, T, d))
    if nbytes == 0:
        raise ValueError("sizes overflow the backward workspace")
    with torch.cuda.device(dev), _on_stream(stream):
        ws = _call_buffer(dev, nbytes, True)
        sh = _stream_handle(dev, stream)
        args = (_ptr(q), _ptr(k), _ptr(v), _ptr(u), _DTYPES[q.dtype], B, H, T, d, float(lambda0), float(eps),
                _ptr(S0), _ptr(A0), _ptr(zk0), _ptr(gO), _ptr(gS), _ptr(gA), _ptr(gzk), *(_ptr(x) for x in outs),
                _ptr(dS0), _ptr(dA0), _ptr(dzk0), _ptr(ws), ws.numel() * 4, ctypes.c_void_p(sh))
        if wait_limit_us or test_stall_producer:
            opts = _Options(int(wait_limit_us), 1 if test_stall_producer else 0, None, 0, 0)
            st = lib.vla_backward_ex(*args, 1 if split else 0, ctypes.byref(opts))
        else:
            st = (lib.vla_backward_split if split else lib.vla_backward)(*args)
    if st != VLA_OK:
        raise VLAError(st, "vla_backward_split" if split else "vla_backward")
    if check:
        detail = (ctypes.c_int * 3)()
        with torch.cuda.device(dev):
            st = lib.vla_get_last_device_status(_ptr(ws), ctypes.c_void_p(_stream_handle(dev, stream)), detail)
        if st != VLA_OK:
            raise VLAError(st, "vla_backward (device)", (detail[0], detail[1], detail[2]))
    return tuple(outs), (dS0, dA0, dzk0)


def vla_linear_attention_state(k: torch.Tensor, v: torch.Tensor, stream=None) -> torch.Tensor:
    """S = sum_t v_t phi(k_t)^T per head (plain cumulative linear attention)."""
    lib = load_library()
    if k.shape != v.shape or k.dtype != v.dtype or k.dim() != 4:
        raise ValueError("k, v must be matching [B, H, T, d] tensors")
    k, v = k.contiguous(), v.contiguous()
    B, H, T, d = k.shape
    with torch.cuda.device(k.device), _on_stream(stream):
        S = torch.empty((B, H, d, d), dtype=torch.float32, device=k.device)
        st = lib.vla_linear_attention_state(_ptr(k), _ptr(v), _DTYPES[k.dtype], B, H, T, d, _ptr(S),
                                            ctypes.c_void_p(_stream_handle(k.device, stream)))
    if st != VLA_OK:
        raise VLAError(st, "vla_linear_attention_state")
    return S
