"""The vectorised checks the full-size GPU tests rely on, pinned on the CPU
against plain Python integers and the oracle, with planted mistakes that
each check must catch."""

import random

import numpy as np
import pytest

from oracle import dixon_model as dm
from oracle import exact

from helpers import (CHECK_PRIMES, check_identity_mod_primes, check_lift_by_residuals_wide, digits_to_limbs,
                     limbs_mod_primes)


def to_limbs(values, W):
    out = np.zeros((len(values), W), dtype=np.uint64)
    mask = (1 << (64 * W)) - 1
    for k, v in enumerate(values):
        out[k] = np.frombuffer((v & mask).to_bytes(8 * W, "little"), dtype=np.uint64)
    return out


def test_limbs_mod_primes_matches_python_ints():
    rng = random.Random(5)
    for W in (1, 2, 7, 40):
        vals = [rng.randrange(-(1 << (64 * W - 1)), 1 << (64 * W - 1)) for _ in range(300)]
        vals += [0, 1, -1, (1 << (64 * W - 1)) - 1, -(1 << (64 * W - 1))]
        got = limbs_mod_primes(to_limbs(vals, W), CHECK_PRIMES, block=64)
        for t, p in enumerate(CHECK_PRIMES):
            assert got[t].tolist() == [v % p for v in vals], (W, p)


def solved_system(n, c, lo, hi, seed):
    rng = random.Random(seed)
    A = [[rng.randrange(lo, hi) for _ in range(n)] for _ in range(n)]
    b = [[rng.randrange(lo, hi) for _ in range(c)] for _ in range(n)]
    N, d = exact.solve(A, b)
    return np.array(A, dtype=np.int64), np.array(b, dtype=np.int64), N, d


def test_identity_mod_primes_accepts_the_solution_and_catches_a_wrong_entry():
    A, b, N, d = solved_system(9, 4, -(1 << 15), 1 << 15, 3)
    flat = [N[i][j] for i in range(9) for j in range(4)]
    W = max(v.bit_length() for v in flat + [d]) // 64 + 2
    check_identity_mod_primes(A, b, to_limbs(flat, W), W, d)
    for k in (0, 17, 35):
        bad = list(flat)
        bad[k] += 1
        with pytest.raises(AssertionError):
            check_identity_mod_primes(A, b, to_limbs(bad, W), W, d)
    with pytest.raises(AssertionError):
        check_identity_mod_primes(A, b, to_limbs(flat, W), W, d + 1)


def test_wide_lift_check_accepts_model_digits_and_catches_planted_mistakes():
    rng = random.Random(11)
    n, c = 12, 5
    A = [[rng.randrange(-(1 << 15), 1 << 15) for _ in range(n)] for _ in range(n)]
    b = [[rng.randrange(-(1 << 15), 1 << 15) for _ in range(c)] for _ in range(n)]
    gp, Bs = dm.good_primes(A)
    digits, _ = dm.lift(A, b, gp, 3, Bs)
    D = digits_to_limbs(digits)
    An, bn = np.array(A, dtype=np.int64), np.array(b, dtype=np.int64)
    check_lift_by_residuals_wide(An, bn, D, gp, 3)
    P = 1
    for q in gp:
        P *= q
    # a digit off by one, a digit outside the balanced range (x + P: same residue mod P),
    # and a digit in the last step checked
    for step, entry, delta in ((0, 0, 1), (1, 7, P), (2, n * c - 1, -1)):
        bad = [[list(row) for row in x] for x in digits]
        r, col = divmod(entry, c)
        bad[step][r][col] += delta
        with pytest.raises(AssertionError):
            check_lift_by_residuals_wide(An, bn, digits_to_limbs(bad), gp, 3)
