"""The named workloads beyond the five test configurations, on the GPU: the
rest of the exact-solve card's §Measured grid (n = 128 and 512 at c = 1,
n = 256 and 512 at c = 16, 24-bit entries) and one each of the planted and
scaled-Hilbert systems of its §Correctness.

Small cases are compared with the CPU oracle entry by entry.  The others are
pinned by what determines the canonical solution for a nonsingular A: the
exact identity A N = b d (Python-int products, formed in float64 over 16-bit
slices), d > 0 and gcd(d, every N) = 1; nonsingularity holds since some prime
did not divide det A.  The planted system must come back as its integer x*
over d = 1."""

import math

import numpy as np
import pytest

from dixon_adic_lifting_gb300 import api, inputs
from oracle import exact

from helpers import exact_matmul_cols

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


def solve_on_device(torch, A, b):
    return api.solve_device(torch.as_tensor(A, device="cuda"), torch.as_tensor(b, device="cuda"))


def numerators(s):
    raw = s.num_limbs.reshape(s.n * s.c, s.limbs)
    flat = [int.from_bytes(row.tobytes(), "little", signed=True) for row in raw]
    return [[flat[i * s.c + j] for j in range(s.c)] for i in range(s.n)]


def assert_canonical(A, b, N, d):
    n, c = A.shape[0], b.shape[1]
    assert d > 0
    AN = exact_matmul_cols(A, [[N[i][j] for i in range(n)] for j in range(c)])
    for j in range(c):
        for i in range(n):
            assert AN[j][i] == int(b[i, j]) * d, (i, j)
    assert math.gcd(d, *[v for row in N for v in row]) == 1


@pytest.mark.parametrize("name", ["hilbert21", "n128_c1_24bit"])
def test_workload_matches_oracle(torch_cuda, name):
    A, b = inputs.workload(name, seed=0)
    s = solve_on_device(torch_cuda, A, b)
    assert s is not None and s.primes_used >= 1
    assert (numerators(s), s.d) == exact.solve(A.tolist(), b.tolist())


@pytest.mark.parametrize("name", ["n512_c1_24bit", "n256_c16_24bit", "n512_c16_24bit"])
def test_workload_canonical(torch_cuda, name):
    A, b = inputs.workload(name, seed=0)
    w = inputs.WORKLOADS[name]
    assert A.shape == (w.n, w.n) and b.shape == (w.n, w.c)
    s = solve_on_device(torch_cuda, A, b)
    assert s is not None and s.primes_used >= 1
    assert (s.n, s.c) == (w.n, w.c)
    assert_canonical(A, b, numerators(s), s.d)


def test_planted256_returns_x_star(torch_cuda):
    A, b, X = inputs.planted(256, 1, seed=0)
    A2, b2 = inputs.workload("planted256", seed=0)
    assert np.array_equal(A, A2) and np.array_equal(b, b2)
    s = solve_on_device(torch_cuda, A, b)
    assert s is not None and s.d == 1
    assert numerators(s) == X.tolist()


def test_hilbert21_denominator_is_large(torch_cuda):
    """The scaled Hilbert system is badly conditioned: its canonical
    denominator is far above the entry size, and the lift must run past the
    first few digits before it can stop."""
    A, b = inputs.workload("hilbert21", seed=0)
    s = solve_on_device(torch_cuda, A, b)
    N, d = exact.solve(A.tolist(), b.tolist())
    assert s.d == d and d.bit_length() > 40
    assert s.m >= 2
