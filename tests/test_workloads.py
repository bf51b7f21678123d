"""The seeded input generators: shapes, determinism and the structure each
workload promises (bf16 rounding, the value clip, the recall layout)."""
import numpy as np

from sherman_morrison_memory_gb300 import workloads as W


def test_deterministic_and_shaped():
    a = W.normal(1, 2, 5, 8, seed=3)
    b = W.normal(1, 2, 5, 8, seed=3)
    for x, y in zip(a, b):
        assert x.shape == (1, 2, 5, 8) and x.dtype == np.float32
        assert np.array_equal(x, y)


def test_vclip():
    q, k, v, u = W.normal(2, 2, 64, 96, seed=0, vclip=4.0)
    n = np.linalg.norm(v.astype(np.float64), axis=-1)
    assert n.max() <= 4.0 * (1 + 1e-6) and n.min() > 0


def test_bf16_values_are_bf16():
    w = W.WORKLOADS[3]
    q, k, v, u = W.make(w, B=1, H=1, T=16)
    for x in (q, k, v, u):
        bits = x.view(np.uint32)
        assert np.all(bits & 0xFFFF == 0)


def test_recall_structure():
    q, k, v, u = W.recall(2, 3, 64, 16, seed=1)
    assert np.array_equal(q, k)
    assert np.all(v[:, :, 32:] == 0)
    assert np.allclose(np.linalg.norm(k, axis=-1), 1.0, atol=1e-6)
    for b in range(2):
        for h in range(3):
            first = {tuple(x) for x in k[b, h, :32]}
            assert len(first) <= 48
            assert all(tuple(x) in first for x in k[b, h, 32:])
    assert np.abs(u - k).max() > 0


def test_workload_table():
    assert W.WORKLOADS[3].d == 96 and W.WORKLOADS[3].T == 4096
    assert W.WORKLOADS[3].head_tokens == 8 * 16 * 4096
