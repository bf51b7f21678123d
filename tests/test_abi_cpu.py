"""The C ABI without a GPU: the library loads, exports every entry point that
the headers under include/ declare, and rejects bad arguments before any CUDA
work."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vla.h")
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    from sherman_morrison_memory_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from sherman_morrison_memory_gb300 import _binding
    return _binding.load_library()


def declared_functions(headers=None):
    names = set()
    for h in headers or HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(vla_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("vla_forward", "vla_forward_ex", "vla_workspace_bytes", "vla_workspace_reset",
              "vla_get_last_device_status", "vla_status_string", "vla_linear_attention_state"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    assert len(HEADERS) >= 2
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared under include/ but not exported"
    assert "vla_probe_ffma" in declared_functions() and "vla_forward_noalloc" in declared_functions()


def test_probe_arguments(lib):
    """The FFMA probe's FLOP count and its argument checks (no launch)."""
    assert lib.vla_probe_ffma_flop(152, 256, 1000, 0) == 2.0 * 32 * 1000 * 152 * 256
    assert lib.vla_probe_ffma_flop(152, 256, 1000, 1) == 2.0 * 32 * 1000 * 152 * 256
    for bad in ((0, 256, 10), (1, 48, 10), (1, 2048, 10), (1, 256, 0)):
        assert lib.vla_probe_ffma_flop(*bad, 0) == 0.0
        assert lib.vla_probe_ffma(*bad, 0, ctypes.c_void_p(FAKE), None) == 1
    assert lib.vla_probe_ffma(1, 32, 1, 0, None, None) == 1
    assert lib.vla_probe_ffma(1, 32, 1, 0, ctypes.c_void_p(FAKE + 2), None) == 1


def test_noalloc_rejects_before_any_device_work(lib):
    """Argument errors of the no-allocation entry point come back before it
    touches a device, and its device-status output carries the same error."""
    vp = ctypes.c_void_p
    for (dtype, B, d, want) in ((1, 1, 48, 2), (7, 1, 64, 1), (1, -1, 64, 1)):
        st = ctypes.c_int(-7)
        r = lib.vla_forward_noalloc(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), dtype, B, 1, 4, d, 0.1, 1e-4,
                                    None, None, None, vp(FAKE), vp(FAKE), vp(FAKE), None, None, ctypes.byref(st))
        assert r == want and st.value == want


def test_status_strings(lib):
    for s in range(6):
        assert lib.vla_status_string(s)


def test_workspace_bytes(lib):
    """The status record's 256 bytes for every valid shape; 0 for invalid sizes."""
    for shape in ((1, 1, 1, 32), (8, 16, 4096, 96), (1, 32, 65536, 128), (64, 8, 1024, 64), (1, 1, 0, 64)):
        assert lib.vla_workspace_bytes(*shape) == 256
    for shape in ((-1, 1, 4, 64), (1, -1, 4, 64), (1, 1, -4, 64), (1, 1, 4, 48), (1, 1, 4, 0)):
        assert lib.vla_workspace_bytes(*shape) == 0


def test_segmented_workspace_bytes(lib):
    """The segmented path's buffers: reported for few heads of a long sequence
    at d <= 96 (no device here: 152 SMs assumed), per algo on request."""
    al = lambda x: (x + 255) // 256 * 256
    B, H, T, d = 4, 8, 4096, 64
    # the cut: past T / 2 by 0.0117 T + 136 tokens at d = 64, rounded down to 16 tokens
    BH, L1 = B * H, T - int(0.5 * T + 0.0117 * T + 136) // 16 * 16
    expect = (256 + al(BH * 16 * d * d * 4) + al(BH * 16 * d * 4) + al(BH * d * d * 4) + al(BH * d * 4)
              + al(d * d * 4) + 5 * al(BH * d * d * 4) + 2 * al(BH * d * 4) + al(BH * L1 * d * 4) + al(L1 * d * 4))
    # (the plan: prefix partials over 16 slices of the first half, the cut's A and z^key, the
    #  identity, then S_L, A and z^key scratch, G_T, Pi_T, A and z^key scratch of the
    #  transition, Pi_t phi_t / den_t, the transition's zero v rows)
    assert lib.vla_workspace_bytes_ex(B, H, T, d, 6) == expect
    assert lib.vla_workspace_bytes(B, H, T, d) == expect          # few heads, long sequence: segmented
    assert lib.vla_workspace_bytes(B, H, 1000, d) == 256          # shorter than the automatic choice's limit
    assert lib.vla_workspace_bytes(8, 16, 4096, 96) == 256        # more heads than fit three CTAs each
    assert lib.vla_workspace_bytes_ex(B, H, T, d, 2) == 256
    assert lib.vla_workspace_bytes_ex(1, 32, 65536, 128, 6) == 0  # d = 128 has no segmented path
    assert lib.vla_workspace_bytes_ex(1, 1, 31, 64, 6) == 0       # too short to cut
    assert lib.vla_workspace_bytes_ex(B, H, T, d, 7) == 0


FAKE = 1 << 20  # an aligned non-null address that the validation paths never dereference


def _call(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, u=FAKE, dtype=1, B=1, H=1, T=4, d=64, lambda0=0.1, eps=1e-4,
             S0=None, A0=None, zk0=None, o=FAKE, S=FAKE, A=FAKE, zk=None, ws=FAKE, wsb=256)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.vla_forward(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["u"]), a["dtype"], a["B"], a["H"], a["T"],
                           a["d"], a["lambda0"], a["eps"], vp(a["S0"]), vp(a["A0"]), vp(a["zk0"]), vp(a["o"]),
                           vp(a["S"]), vp(a["A"]), vp(a["zk"]), vp(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=48), 2), (dict(d=256), 2), (dict(d=0), 2),
    (dict(B=-1), 1), (dict(T=-3), 1), (dict(dtype=7), 1),
    (dict(lambda0=0.0), 1), (dict(lambda0=-1.0), 1), (dict(lambda0=float("inf")), 1),
    (dict(eps=0.0), 1), (dict(eps=float("nan")), 1),
    (dict(ws=None), 1), (dict(ws=FAKE + 4), 1), (dict(wsb=8), 1),
    (dict(q=None), 1), (dict(o=None), 1), (dict(S=None), 1), (dict(A=None), 1),
    (dict(k=FAKE + 2), 1), (dict(o=FAKE + 8), 1), (dict(S=FAKE + 4), 1),
    (dict(zk=FAKE + 2), 1), (dict(A0=FAKE + 1), 1),
    (dict(B=1 << 20, H=1 << 12), 1),
])
def test_argument_errors(lib, kw, status):
    assert _call(lib, **kw) == status


def test_empty_batch_is_a_no_op(lib):
    assert _call(lib, B=0) == 0
    assert _call(lib, H=0, q=None, o=None) == 0


def test_linear_attention_argument_errors(lib):
    vp = ctypes.c_void_p
    assert lib.vla_linear_attention_state(vp(FAKE), vp(FAKE), 0, 1, 1, 4, 40, vp(FAKE), None) == 2
    assert lib.vla_linear_attention_state(vp(FAKE), vp(FAKE), 5, 1, 1, 4, 64, vp(FAKE), None) == 1
    assert lib.vla_linear_attention_state(vp(FAKE), vp(FAKE), 0, 1, 1, 4, 64, None, None) == 1


def test_status_read_rejects_null(lib):
    d = (ctypes.c_int * 3)()
    assert lib.vla_get_last_device_status(None, None, d) == 1
    assert list(d) == [-1, -1, -1]


@pytest.mark.parametrize("algo,d,fixed,status", [
    (7, 64, 0, 1), (-1, 64, 0, 1), (2, 128, 0, 2),
    (1, 64, 1, 2), (2, 128, 1, 2), (6, 128, 0, 2), (6, 64, 0, 1),
])
def test_algo_argument_errors(lib, algo, d, fixed, status):
    """VLA_ALGO_* outside {0, ..., 6} is an argument error; the chunked kernel
    and the segmented path report d = 128 as unsupported; the segmented path
    with a 256-byte workspace (or T < 32) is an argument error; the fixed-A
    variant does not run on the per-token kernel. All are decided before any
    CUDA call."""
    from sherman_morrison_memory_gb300 import _binding
    vp = ctypes.c_void_p
    opts = _binding._Options(0, 0, None, algo, fixed)
    st = lib.vla_forward_ex(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1, 1, 1, 4, d, ctypes.c_float(0.1),
                            ctypes.c_float(1e-4), None, None, None, vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE),
                            ctypes.c_size_t(256), None, ctypes.byref(opts))
    assert st == status


@pytest.mark.parametrize("scratch_off,scratch_bytes", [(16, 1 << 30), (0, 256), (0, 0)])
def test_segmented_scratch_argument_errors(lib, scratch_off, scratch_bytes):
    """The segmented path's own buffers (vla_options.scratch) must be 256-byte
    aligned and hold vla_workspace_bytes_ex(..., VLA_ALGO_SEGMENTED) bytes,
    whatever the workspace holds; both are checked before any CUDA call."""
    from sherman_morrison_memory_gb300 import _binding
    vp = ctypes.c_void_p
    opts = _binding._Options(0, 0, None, 6, 0, vp(FAKE + scratch_off), scratch_bytes)
    st = lib.vla_forward_ex(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1, 1, 1, 64, 64, ctypes.c_float(0.1),
                            ctypes.c_float(1e-4), None, None, None, vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE),
                            ctypes.c_size_t(1 << 30), None, ctypes.byref(opts))
    assert st == 1
    assert lib.vla_workspace_bytes_ex(1, 1, 64, 64, 6) > 256


def test_u_may_be_null_only_for_fixed_a(lib):
    from sherman_morrison_memory_gb300 import _binding
    vp = ctypes.c_void_p
    opts = _binding._Options(0, 0, None, 0, 0)
    st = lib.vla_forward_ex(vp(FAKE), vp(FAKE), vp(FAKE), None, 1, 1, 1, 4, 64, ctypes.c_float(0.1),
                            ctypes.c_float(1e-4), None, None, None, vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE),
                            ctypes.c_size_t(256), None, ctypes.byref(opts))
    assert st == 1


def test_backward_workspace_bytes(lib):
    """Status record + tape (3d + 8 floats per head-token) + S, A, z^key
    checkpoints every 64 tokens plus one more slot (2 d^2 + d floats each) +
    the forward's final S, A, z^key (2 d^2 + d floats per head), each part
    256-byte aligned."""
    al = lambda x: (x + 255) // 256 * 256
    assert lib.vla_backward_workspace_bytes(1, 1, 64, 32) == (256 + al(64 * 104 * 4) + al(2 * (2 * 32 * 32 + 32) * 4)
                                                             + al((2 * 32 * 32 + 32) * 4))
    assert lib.vla_backward_workspace_bytes(2, 3, 65, 96) == (256 + al(6 * 65 * 296 * 4)
                                                             + al(6 * 3 * (2 * 96 * 96 + 96) * 4)
                                                             + al(6 * (2 * 96 * 96 + 96) * 4))
    assert lib.vla_backward_workspace_bytes(1, 1, 0, 64) > 0
    assert lib.vla_backward_workspace_bytes(-1, 1, 4, 64) == 0
    assert lib.vla_backward_workspace_bytes(1 << 30, 1 << 30, 4, 64) == 0


def _bw_call(lib, split=False, ex=False, **kw):
    """vla_backward / vla_backward_split, or with ex=True the same call
    through vla_backward_ex (options with a wait limit)."""
    a = dict(q=FAKE, k=FAKE, v=FAKE, u=FAKE, dtype=1, B=1, H=1, T=4, d=64, lambda0=0.1, eps=1e-4,
             S0=None, A0=None, zk0=None, gO=FAKE, gS=None, gA=None, gzk=None,
             dq=FAKE, dk=FAKE, dv=FAKE, du=FAKE, dS0=FAKE, dA0=FAKE, dzk0=FAKE, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    vp = ctypes.c_void_p
    p = lambda n: vp(a[n])
    args = (p("q"), p("k"), p("v"), p("u"), a["dtype"], a["B"], a["H"], a["T"], a["d"], a["lambda0"], a["eps"],
            p("S0"), p("A0"), p("zk0"), p("gO"), p("gS"), p("gA"), p("gzk"), p("dq"), p("dk"), p("dv"), p("du"),
            p("dS0"), p("dA0"), p("dzk0"), p("ws"), a["wsb"], None)
    if ex:
        from sherman_morrison_memory_gb300 import _binding
        opts = _binding._Options(5000, 0, None, 0, 0)
        return lib.vla_backward_ex(*args, 1 if split else 0, ctypes.byref(opts))
    return (lib.vla_backward_split if split else lib.vla_backward)(*args)


@pytest.mark.parametrize("ex", [False, True])
@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("kw,status", [
    (dict(d=160), 2), (dict(d=48), 2), (dict(d=0), 2),
    (dict(B=-1), 1), (dict(T=-1), 1), (dict(dtype=4), 1),
    (dict(lambda0=0.0), 1), (dict(eps=float("inf")), 1),
    (dict(ws=None), 1), (dict(ws=FAKE + 8), 1), (dict(wsb=1024), 1),
    (dict(q=None), 1), (dict(dq=None), 1), (dict(du=None), 1),
    (dict(k=FAKE + 4), 1), (dict(dv=FAKE + 8), 1), (dict(gO=FAKE + 4), 1),
    (dict(dS0=FAKE + 2), 1), (dict(S0=FAKE + 1), 1),
    (dict(B=1 << 30, H=1 << 30), 1),
])
def test_backward_argument_errors(lib, kw, status, split, ex):
    assert _bw_call(lib, split, ex, **kw) == status


@pytest.mark.parametrize("ex", [False, True])
@pytest.mark.parametrize("split", [False, True])
def test_backward_empty_batch_is_a_no_op(lib, split, ex):
    assert _bw_call(lib, split, ex, B=0) == 0
    assert _bw_call(lib, split, ex, B=0, d=128) == 0


def _host_call(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, u=FAKE, dtype=1, B=1, H=1, T=4, d=64, lambda0=0.1, eps=1e-4,
             S0=None, A0=None, zk0=None, o=FAKE, S=FAKE, A=FAKE, zk=None, chunk=0, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    vp = ctypes.c_void_p
    p = lambda n: vp(a[n])
    return lib.vla_forward_host(p("q"), p("k"), p("v"), p("u"), a["dtype"], a["B"], a["H"], a["T"], a["d"],
                                a["lambda0"], a["eps"], p("S0"), p("A0"), p("zk0"), p("o"), p("S"), p("A"),
                                p("zk"), a["chunk"], p("ws"), a["wsb"], None, None)


def test_host_workspace_bytes(lib):
    """Status record, S, A, z^key, three input slots (q, k, v, u of one chunk)
    and three output slots (o of one chunk), each part 256-byte aligned. The
    automatic chunk is about T/4 tokens, a multiple of 16, at least 256."""
    al = lambda x: (x + 255) // 256 * 256
    def expect(es, BH, T, d, tc):
        return (256 + 2 * al(BH * d * d * 4) + al(BH * d * 4) + 3 * 4 * al(BH * tc * d * es)
                + 3 * al(BH * tc * d * 4))
    assert lib.vla_forward_host_workspace_bytes(1, 8, 16, 4096, 96, 0) == expect(2, 128, 4096, 96, 1024)
    assert lib.vla_forward_host_workspace_bytes(0, 1, 32, 65536, 128, 0) == expect(4, 32, 65536, 128, 16384)
    assert lib.vla_forward_host_workspace_bytes(0, 2, 3, 1100, 64, 0) == expect(4, 6, 1100, 64, 288)
    assert lib.vla_forward_host_workspace_bytes(0, 2, 3, 300, 64, 0) == expect(4, 6, 300, 64, 256)
    assert lib.vla_forward_host_workspace_bytes(0, 2, 3, 100, 64, 0) == expect(4, 6, 100, 64, 100)
    assert lib.vla_forward_host_workspace_bytes(1, 2, 3, 300, 32, 64) == expect(2, 6, 300, 32, 64)
    assert lib.vla_forward_host_workspace_bytes(1, 2, 3, 0, 32, 0) == expect(2, 6, 0, 32, 0)
    assert lib.vla_forward_host_workspace_bytes(1, 1, 1, 4, 48, 0) == 0
    assert lib.vla_forward_host_workspace_bytes(1, 1, 1, 4, 64, -1) == 0
    assert lib.vla_forward_host_workspace_bytes(2, 1, 1, 4, 64, 0) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(d=48), 2), (dict(d=0), 2),
    (dict(B=-1), 1), (dict(T=-1), 1), (dict(dtype=3), 1), (dict(chunk=-5), 1),
    (dict(lambda0=0.0), 1), (dict(eps=float("nan")), 1),
    (dict(ws=None), 1), (dict(ws=FAKE + 16), 1), (dict(wsb=4096), 1),
    (dict(q=None), 1), (dict(u=None), 1), (dict(o=None), 1), (dict(S=None), 1), (dict(A=None), 1),
    (dict(B=1 << 20, H=1 << 12), 1),
])
def test_host_argument_errors(lib, kw, status):
    """vla_forward_host rejects these before any CUDA call or copy."""
    assert _host_call(lib, **kw) == status


def test_host_empty_batch_is_a_no_op(lib):
    assert _host_call(lib, B=0) == 0
