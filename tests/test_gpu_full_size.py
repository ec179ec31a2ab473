"""Full-size n = 4096, c = 64 (16-bit entries) on the GPU.

The CPU oracle cannot solve this size, so the result is pinned by what fixes
the canonical solution uniquely for a nonsingular A (exact-solve card,
§Correctness: the exact residual at larger sizes):
  * A N = b d on EVERY column: exactly (Python ints from 16-bit slices in
    float64) on two columns, and modulo six primes just below 2^24 on all 64
    columns (numerators reduced from their limbs on the host);
  * gcd(d, all N) = 1 (scanned entry by entry until the running gcd is 1);
  * nonsingularity (a good prime exists, so det A != 0).
The lift itself is pinned at full size too: the first steps' digits satisfy
r_i - A x_i = P' r_{i+1} exactly with balanced digits (the unique digits)."""

import math

import numpy as np
import pytest

from dixon_adic_lifting_gb300 import api, inputs

from helpers import check_identity_mod_primes, check_lift_by_residuals_wide, exact_matmul_cols

pytestmark = pytest.mark.gpu

PRIMES = (3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37, 41, 43, 47, 53, 59, 61, 67, 71, 73, 79, 83, 89, 97, 101, 103,
          107, 109, 113, 127, 131, 137, 139, 149, 151, 157, 163, 167, 173, 179, 181, 191, 193, 197, 199, 211, 223,
          227, 229, 233, 239, 241, 251)


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


def test_n4096_c64_identity_on_every_column(c5):
    A, b, s = c5
    assert s.primes_used >= 1
    check_identity_mod_primes(A, b, s.num_limbs, s.limbs, s.d)


@pytest.mark.parametrize("col", [0, 37])
def test_n4096_c64_exact_identity_on_columns(c5, col):
    A, b, s = c5
    d = s.d
    N = column_numerators(s, col)
    AN = exact_matmul_cols(A, [N])[0]
    for i in range(A.shape[0]):
        assert AN[i] == int(b[i, col]) * d, i


def test_n4096_c64_minimal(c5):
    _, _, s = c5
    assert gcd_with_all_numerators(s) == 1


def test_n4096_c64_phases_reported(c5):
    _, _, s = c5
    assert s.m > 400 and all(t >= 0 for t in s.phase_ms)
    print("n4096 c64 phases ms:", [round(t, 1) for t in s.phase_ms], "m", s.m, "primes", s.primes_used)


def test_n4096_c64_lift_first_steps_by_residuals():
    """The full-size lift kernels (tcgen05 product over all good primes, CRT
    digit, tcgen05 residual with two 8-bit limbs of A) on the first three
    steps: balanced digits with r_i - A x_i = P' r_{i+1} exactly."""
    import torch

    A, b = inputs.workload("n4096_c64_16bit", seed=0)
    At = torch.as_tensor(A, device="cuda")
    bt = torch.as_tensor(b, device="cuda")
    B, good = api.inverse_mod_device(At)
    D = api.lift_device(At, bt, B, good, 3)
    del B
    g = good.cpu().numpy()
    gp = [q for j, q in enumerate(PRIMES) if g[j]]
    assert len(gp) >= 40
    check_lift_by_residuals_wide(A, b, D.cpu().numpy(), gp, 3)


def test_n512_c64_many_entries_exact_on_columns():
    """32768 entries: the one-thread-per-entry CRT, the tcgen05 product and the
    int32 residual GEMM together; exact identity on three columns and modulo
    primes on all 64."""
    import torch

    A, b = inputs.uniform(512, 64, -(1 << 15), 1 << 15, seed=512)
    s = api.solve_device(torch.as_tensor(A, device="cuda"), torch.as_tensor(b, device="cuda"))
    d = s.d
    for col in (0, 31, 63):
        N = column_numerators(s, col)
        AN = exact_matmul_cols(A, [N])[0]
        assert all(AN[i] == int(b[i, col]) * d for i in range(512)), col
    check_identity_mod_primes(A, b, s.num_limbs, s.limbs, s.d)
    assert gcd_with_all_numerators(s) == 1
