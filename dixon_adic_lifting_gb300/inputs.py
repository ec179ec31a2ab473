"""Seeded synthetic inputs for the exact solver.

This module only draws integers and arranges them; it holds none of the
solver's arithmetic (no modular reduction, no elimination, no bounds), so
that both the CUDA path and the CPU oracle can be fed from it without
sharing any of the method.

Workloads follow the exact-solve card (kernels hub):
  * "24-bit integer entries" of its §Measured table (uniform in [-2^23, 2^23));
  * the order-30 Pascal system of its figure caption (A_ij = C(i+j, i));
  * the planted-integer-solution and scaled-Hilbert systems of §Correctness.
Random draws use numpy's PCG64 generator: ``Generator(PCG64(seed)).integers
(lo, hi)`` with ``hi`` exclusive.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


def _rng(*seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(list(seed)))


def uniform(n: int, c: int, lo: int, hi: int, seed: int, attempt: int = 0):
    """A int64 [n, n] and b int64 [n, c], i.i.d. uniform in [lo, hi)."""
    g = _rng(seed, attempt)
    A = g.integers(lo, hi, size=(n, n), dtype=np.int64)
    b = g.integers(lo, hi, size=(n, c), dtype=np.int64)
    return A, b


def pascal(n: int = 30) -> np.ndarray:
    """Symmetric Pascal matrix A_ij = C(i+j, i), 0-based (unimodular)."""
    return np.array([[math.comb(i + j, i) for j in range(n)] for i in range(n)], dtype=np.int64)


def pascal_system(n: int = 30, c: int = 1, seed: int = 0):
    """Pascal A with b uniform in [-2^23, 2^23)."""
    g = _rng(seed, 7)
    b = g.integers(-(1 << 23), 1 << 23, size=(n, c), dtype=np.int64)
    return pascal(n), b


def make_rank_deficient(A: np.ndarray, seed: int) -> np.ndarray:
    """Copy of A whose last row is the sum of two other (seeded, distinct) rows."""
    n = A.shape[0]
    g = _rng(seed, 255)
    i, j = g.choice(n - 1, size=2, replace=False)
    S = A.copy()
    S[n - 1] = A[i] + A[j]
    return S


def planted(n: int, c: int, seed: int, abits: int = 23, xbits: int = 20):
    """A uniform with |A| < 2^abits and b = A x* for an integer x* (|x*| < 2^xbits).

    Returns (A, b, x*); b is computed with Python ints and must fit int64."""
    g = _rng(seed, 11)
    A = g.integers(-(1 << abits), 1 << abits, size=(n, n), dtype=np.int64)
    X = g.integers(-(1 << xbits), 1 << xbits, size=(n, c), dtype=np.int64)
    Ai = [[int(v) for v in row] for row in A]
    Xi = [[int(v) for v in row] for row in X]
    B = [[sum(Ai[i][k] * Xi[k][j] for k in range(n)) for j in range(c)] for i in range(n)]
    if any(abs(v) >= (1 << 63) for row in B for v in row):
        raise ValueError("planted right-hand side does not fit int64")
    return A, np.array(B, dtype=np.int64), X


def scaled_hilbert(n: int) -> np.ndarray:
    """A_ij = L / (i + j + 1) with L = lcm(1 .. 2n-1): the Hilbert matrix made integral."""
    L = 1
    for k in range(1, 2 * n):
        L = L * k // math.gcd(L, k)
    A = [[L // (i + j + 1) for j in range(n)] for i in range(n)]
    if n * max(max(r) for r in A) >= (1 << 63):
        raise ValueError("scaled Hilbert matrix out of the int64 range")
    return np.array(A, dtype=np.int64)


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    c: int
    description: str


# The systems the solver is measured and checked on: the five test
# configurations, the rest of the card's §Measured grid (24-bit entries),
# one each of its planted and scaled-Hilbert systems (§Correctness), and a
# half-size n = 4096, c = 64 system (a profiling case of a few GB).
_U24 = "A, b uniform in [-2^23, 2^23)"
WORKLOADS = {
    "n32_c1_int8": Workload("n32_c1_int8", 32, 1,
                            "A, b uniform in [-127, 127]; A redrawn until invertible modulo every odd prime < 256"),
    "pascal30": Workload("pascal30", 30, 1,
                         "order-30 Pascal A_ij = C(i+j, i); b uniform in [-2^23, 2^23)"),
    "n128_c1_24bit": Workload("n128_c1_24bit", 128, 1, _U24),
    "n256_c1_24bit": Workload("n256_c1_24bit", 256, 1, _U24),
    "n512_c1_24bit": Workload("n512_c1_24bit", 512, 1, _U24),
    "n1024_c1_24bit": Workload("n1024_c1_24bit", 1024, 1, _U24),
    "n256_c16_24bit": Workload("n256_c16_24bit", 256, 16, _U24),
    "n512_c16_24bit": Workload("n512_c16_24bit", 512, 16, _U24),
    "n2048_c64_16bit": Workload("n2048_c64_16bit", 2048, 64, "A, b uniform in [-2^15, 2^15)"),
    "n4096_c64_16bit": Workload("n4096_c64_16bit", 4096, 64, "A, b uniform in [-2^15, 2^15)"),
    "hilbert21": Workload("hilbert21", 21, 1,
                          "scaled Hilbert A_ij = lcm(1..41) / (i + j + 1); b uniform in [-2^23, 2^23)"),
    "planted256": Workload("planted256", 256, 1,
                           "A uniform in [-2^23, 2^23), b = A x* for integer x* uniform in [-2^20, 2^20)"),
}


def workload(name: str, seed: int = 0, attempt: int = 0):
    """(A, b) for a named workload.  ``attempt`` selects the redraw for the
    n=32 case (the accepted attempt index per seed is stored with the tests)."""
    if name == "n32_c1_int8":
        return uniform(32, 1, -127, 128, seed, attempt)
    if name == "pascal30":
        return pascal_system(30, 1, seed)
    if name in ("n2048_c64_16bit", "n4096_c64_16bit"):
        w = WORKLOADS[name]
        return uniform(w.n, w.c, -(1 << 15), 1 << 15, seed)
    if name == "hilbert21":
        g = _rng(seed, 21)
        return scaled_hilbert(21), g.integers(-(1 << 23), 1 << 23, size=(21, 1), dtype=np.int64)
    if name == "planted256":
        A, b, _ = planted(256, 1, seed)
        return A, b
    if name in WORKLOADS and name.endswith("_24bit"):
        w = WORKLOADS[name]
        return uniform(w.n, w.c, -(1 << 23), 1 << 23, seed)
    raise KeyError(name)
