"""The pins have teeth: each plausible mistake, planted in a temporary copy of
the oracle's C source (never in the oracle itself), must make at least one pin
fail.

Each mutant is a textual replacement in ``oracle/vla_oracle.c``; the copy is
compiled with gcc into a temporary directory and the pins run against it.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

# (name, original text, replacement): dropped terms, wrong signs, wrong
# operands or indices, transposed outer products, missing normalisations.
MUTANTS = [
    ("A update sign", "A[i * d + j] -= z[i] * z[j] / delta", "A[i * d + j] += z[i] * z[j] / delta"),
    ("delta drops the 1", "double delta = 1.0;", "double delta = 0.0;"),
    ("A update not divided by delta", "A[i * d + j] -= z[i] * z[j] / delta", "A[i * d + j] -= z[i] * z[j]"),
    ("A_0 = lambda0 I", "1.0 / lambda0 : 0.0", "lambda0 : 0.0"),
    ("gate uses u instead of k", "s += A[i * d + j] * kh[j];", "s += A[i * d + j] * uh[j];"),
    ("gate not normalised", "unit(a, alpha, d);", "memcpy(alpha, a, sizeof(double) * d);"),
    ("u not normalised", "unit(x, uh, d);", "memcpy(uh, x, sizeof(double) * d);"),
    ("k not normalised", "unit(x, kh, d);", "memcpy(kh, x, sizeof(double) * d);"),
    ("residual sign", "e[i] = (double)vt[i] - s;", "e[i] = (double)vt[i] + s;"),
    ("residual drops S k", "e[i] = (double)vt[i] - s;", "e[i] = (double)vt[i];"),
    ("S k with transposed S", "s += S[i * d + j] * kh[j];", "s += S[j * d + i] * kh[j];"),
    ("write transposed", "S[i * d + j] += e[i] * alpha[j];", "S[i * d + j] += e[j] * alpha[i];"),
    ("write along k instead of alpha", "S[i * d + j] += e[i] * alpha[j];", "S[i * d + j] += e[i] * kh[j];"),
    ("key sum uses q", "zk[j] += phi((double)kt[j]);", "zk[j] += phi((double)qt[j]);"),
    ("key sum uses normalised k", "zk[j] += phi((double)kt[j]);", "zk[j] += phi(kh[j]);"),
    ("phi without +1", "x > 0.0 ? x + 1.0 : exp(x)", "x > 0.0 ? x : exp(x)"),
    ("no eps floor", "if (den < eps) den = eps;", ""),
    ("readout with transposed S", "s += S[i * d + j] * pq[j];", "s += S[j * d + i] * pq[j];"),
    ("readout without normaliser", "o[(size_t)t * d + i] = s / den;", "o[(size_t)t * d + i] = s;"),
    ("linear attention transposed", "S[i * d + j] += (double)vt[i] * phi((double)kt[j]);",
     "S[i * d + j] += (double)vt[j] * phi((double)kt[i]);"),
    # backward pass
    ("backward gate without the unit-norm projection", "(gal[j] - alpha[j] * ag) / n", "gal[j] / n"),
    ("backward z adjoint without the transpose", "gz[i] = -(s1 + s2) / delta;", "gz[i] = -(2.0 * s1) / delta;"),
    ("backward normaliser sign", "const double gden = cl[t] ? 0.0 : -go_o / den;",
     "const double gden = cl[t] ? 0.0 : go_o / den;"),
    ("backward residual with S_t", "s += Sp[i * d + j] * ge[i];", "s += S[i * d + j] * ge[i];"),
    ("backward drops the key-sum path", "tmp[j] + gzk[j] * dphi(k[(size_t)t * d + j])", "tmp[j]"),
    ("backward delta adjoint dropped", "gz[j] += gdelta * ut[j];", ""),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    # an anchor shared by the forward and the backward's own forward pass is
    # mutated everywhere (the same mistake in both)
    assert source.count(old) >= 1, f"mutation anchor not in oracle source: {old!r}"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = oracle.build(str(src), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
        except (FloatingPointError, ValueError, ZeroDivisionError, OverflowError,
                __import__("numpy").linalg.LinAlgError):
            caught.append(pin.__name__)
    assert caught, f"mutant '{name}' passed every pin"
