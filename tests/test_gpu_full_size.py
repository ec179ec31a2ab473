"""Full-size n = 4096, c = 64 (16-bit entries) on the GPU.

The CPU oracle cannot solve this size, so the result is pinned by the exact
identity A N = b d on sampled columns (products formed exactly with 16-bit
slices in float64), gcd(d, all N) = 1 (scanned entry by entry until the
running gcd reaches 1), and nonsingularity (a good prime exists); with A
nonsingular these determine the canonical solution uniquely."""

import math

import numpy as np
import pytest

from dixon_adic_lifting_gb300 import api, inputs

from helpers import exact_matmul_cols

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def c5():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    A, b = inputs.workload("n4096_c64_16bit", seed=0)
    At = torch.as_tensor(A, device="cuda")
    bt = torch.as_tensor(b, device="cuda")
    s = api.solve_device(At, bt, timing=True)
    return A, b, s


def column_numerators(s, col):
    W = s.limbs
    raw = s.num_limbs.reshape(s.n * s.c, W)[col::s.c]
    return [int.from_bytes(row.tobytes(), "little", signed=True) for row in raw]


def gcd_with_all_numerators(s):
    """gcd(d, N_0, N_1, ...) over every entry, stopping once it reaches 1."""
    W = s.limbs
    raw = s.num_limbs.reshape(s.n * s.c, W)
    g = s.d
    for k in range(raw.shape[0]):
        g = math.gcd(g, int.from_bytes(raw[k].tobytes(), "little", signed=True))
        if g == 1:
            break
    return g


@pytest.mark.parametrize("col", [0, 37])
def test_n4096_c64_identity_on_columns(c5, col):
    A, b, s = c5
    assert s.primes_used >= 1
    d = s.d
    N = column_numerators(s, col)
    AN = exact_matmul_cols(A, [N])[0]
    for i in range(A.shape[0]):
        assert AN[i] == int(b[i, col]) * d, i
    assert gcd_with_all_numerators(s) == 1


def test_n4096_c64_phases_reported(c5):
    _, _, s = c5
    assert s.m > 400 and all(t >= 0 for t in s.phase_ms)
    print("n4096 c64 phases ms:", [round(t, 1) for t in s.phase_ms], "m", s.m, "primes", s.primes_used)


def test_n512_c64_many_entries_exact_on_columns():
    """32768 entries: the one-thread-per-entry CRT, the tcgen05 product and the
    int32 residual GEMM together; exact identity on three columns."""
    import torch

    A, b = inputs.uniform(512, 64, -(1 << 15), 1 << 15, seed=512)
    s = api.solve_device(torch.as_tensor(A, device="cuda"), torch.as_tensor(b, device="cuda"))
    d = s.d
    for col in (0, 31, 63):
        N = column_numerators(s, col)
        AN = exact_matmul_cols(A, [N])[0]
        assert all(AN[i] == int(b[i, col]) * d for i in range(512)), col
    assert gcd_with_all_numerators(s) == 1
