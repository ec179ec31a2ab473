"""Pins of the CPU oracle to things other than itself (CPU only).

Each check is chosen so that a plausible mistake in the oracle (a dropped
term, a wrong sign or index, a transposed operand) fails: Cramer's rule by
brute-force Leibniz determinants, closed-form inverses of the Pascal and
Hilbert matrices, planted integer solutions, hand-solved systems, library
routines (sympy) on the special cases they cover, and the defining
congruences of every intermediate of the Dixon model.
"""

import itertools
import json
import math
import os
import random
from fractions import Fraction

import pytest

from dixon_adic_lifting_gb300 import inputs
from oracle import dixon_model as dm
from oracle import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def check_canonical(A, b, N, d):
    """A N == b d exactly, d > 0, gcd(d, all N) == 1."""
    n, c = len(A), len(b[0])
    assert d > 0
    for i in range(n):
        for j in range(c):
            assert sum(int(A[i][k]) * N[k][j] for k in range(n)) == int(b[i][j]) * d
    g = d
    for row in N:
        for v in row:
            g = math.gcd(g, v)
    assert g == 1


def leibniz_det(M):
    n = len(M)
    total = 0
    for perm in itertools.permutations(range(n)):
        inv = sum(1 for a in range(n) for b_ in range(a + 1, n) if perm[a] > perm[b_])
        p = 1
        for i in range(n):
            p *= M[i][perm[i]]
        total += -p if inv % 2 else p
    return total


def rand_matrix(rng, n, c, lo, hi):
    A = [[rng.randrange(lo, hi) for _ in range(n)] for _ in range(n)]
    b = [[rng.randrange(lo, hi) for _ in range(c)] for _ in range(n)]
    return A, b


def to_fracs(N, d):
    return [[Fraction(v, d) for v in row] for row in N]


# ---------------------------------------------------------------- exact.py
def test_hand_examples():
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        r = exact.solve(case["A"], case["b"])
        if case["N"] is None:
            assert r is None, case["name"]
        else:
            assert r == (case["N"], case["d"]), case["name"]


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_cramer_leibniz(n):
    rng = random.Random(1000 + n)
    for trial in range(6):
        c = 1 + trial % 3
        A, b = rand_matrix(rng, n, c, -50, 51)
        det = leibniz_det(A)
        r = exact.solve(A, b)
        if det == 0:
            assert r is None
            continue
        N, d = r
        check_canonical(A, b, N, d)
        X = to_fracs(N, d)
        for j in range(c):
            for k in range(n):
                Ak = [row[:k] + [b[i][j]] + row[k + 1:] for i, row in enumerate(A)]
                assert X[k][j] == Fraction(leibniz_det(Ak), det)
        assert exact.determinant(A) == det


def pascal_inverse(n):
    # Pascal = L L^T with L_ij = C(i, j); inverse entries are signed sums of binomial products.
    return [[(-1) ** (i + j) * sum(math.comb(k, i) * math.comb(k, j) for k in range(max(i, j), n))
             for j in range(n)] for i in range(n)]


def test_pascal_closed_form():
    n = 30
    A = inputs.pascal(n).tolist()
    Ai = pascal_inverse(n)
    # the closed form really is the inverse
    for i in range(n):
        for j in range(n):
            assert sum(A[i][k] * Ai[k][j] for k in range(n)) == (1 if i == j else 0)
    _, b = inputs.pascal_system(n, 2, seed=3)
    b = b.tolist()
    N, d = exact.solve(A, b)
    assert d == 1  # unimodular: integer solution
    for i in range(n):
        for j in range(2):
            assert N[i][j] == sum(Ai[i][k] * b[k][j] for k in range(n))
    assert exact.determinant(A) == 1


def hilbert_inverse(n):
    return [[(-1) ** (i + j) * (i + j + 1) * math.comb(n + i, n - j - 1) * math.comb(n + j, n - i - 1)
             * math.comb(i + j, i) ** 2 for j in range(n)] for i in range(n)]


@pytest.mark.parametrize("n", [2, 5, 9, 12])
def test_scaled_hilbert_closed_form(n):
    A = inputs.scaled_hilbert(n).tolist()
    L = A[0][0]  # A_00 = L / 1
    Hi = hilbert_inverse(n)
    rng = random.Random(n)
    b = [[rng.randrange(-1000, 1001)] for _ in range(n)]
    N, d = exact.solve(A, b)
    check_canonical(A, b, N, d)
    X = to_fracs(N, d)
    for i in range(n):
        assert X[i][0] == Fraction(sum(Hi[i][k] * b[k][0] for k in range(n)), L)


def test_planted_integer_solution():
    A, b, X = inputs.planted(12, 3, seed=5)
    N, d = exact.solve(A.tolist(), b.tolist())
    assert d == 1 and N == X.tolist()


def test_diagonal_and_triangular():
    rng = random.Random(7)
    n = 7
    diag = [rng.choice([-1, 1]) * rng.randrange(1, 40) for _ in range(n)]
    A = [[diag[i] if i == j else 0 for j in range(n)] for i in range(n)]
    b = [[rng.randrange(-99, 100)] for _ in range(n)]
    N, d = exact.solve(A, b)
    assert to_fracs(N, d) == [[Fraction(b[i][0], diag[i])] for i in range(n)]
    # lower triangular: forward substitution by hand
    T = [[(rng.randrange(-9, 10) if j < i else (diag[i] if i == j else 0)) for j in range(n)] for i in range(n)]
    x = []
    for i in range(n):
        x.append((Fraction(b[i][0]) - sum(T[i][j] * x[j] for j in range(i))) / T[i][i])
    N, d = exact.solve(T, b)
    assert to_fracs(N, d) == [[v] for v in x]


def test_rank_deficient_is_singular():
    A, b = inputs.uniform(16, 1, -(1 << 23), 1 << 23, seed=9)
    S = inputs.make_rank_deficient(A, seed=9)
    assert exact.solve(S.tolist(), b.tolist()) is None
    assert exact.determinant(S.tolist()) == 0
    assert dm.solve(S.tolist(), b.tolist()) is None


def test_against_sympy_lusolve():
    sympy = pytest.importorskip("sympy")
    rng = random.Random(11)
    for n in (3, 6, 10):
        A, b = rand_matrix(rng, n, 2, -1000, 1001)
        X = sympy.Matrix(A).LUsolve(sympy.Matrix(b))
        N, d = exact.solve(A, b)
        F = to_fracs(N, d)
        for i in range(n):
            for j in range(2):
                assert F[i][j] == Fraction(int(X[i, j].p), int(X[i, j].q))


# ---------------------------------------------------------------- dixon_model.py
def test_prime_set():
    sympy = pytest.importorskip("sympy")
    assert dm.PRIMES == list(sympy.primerange(3, 256))
    assert len(dm.PRIMES) == 53
    P = math.prod(dm.PRIMES)
    assert P % 2 == 1 and P.bit_length() == 334
    assert abs(math.log2(P) - 333.88) < 0.01


def test_balanced_residue():
    for q in dm.PRIMES:
        h = (q - 1) // 2
        seen = set()
        for v in range(-3 * q, 3 * q):
            r = dm.bal(v, q)
            assert -h <= r <= h and (v - r) % q == 0
            seen.add(r)
        assert seen == set(range(-h, h + 1))


def test_inverse_mod_definition():
    rng = random.Random(13)
    for q in (3, 5, 7, 101, 251):
        for n in (1, 2, 5, 9):
            for _ in range(4):
                A = [[rng.randrange(-300, 300) for _ in range(n)] for _ in range(n)]
                B = dm.inverse_mod(A, q)
                det = exact.determinant(A)
                if det % q == 0:
                    assert B is None
                    continue
                for i in range(n):
                    for j in range(n):
                        assert sum(A[i][k] * B[k][j] for k in range(n)) % q == (1 if i == j else 0)
                        assert 0 <= B[i][j] < q


def test_garner_exhaustive_small():
    primes = [3, 5, 7]
    P = 105
    got = []
    for v in itertools.product(*(range(q) for q in primes)):
        x = dm.garner_balanced(list(v), primes)
        assert -(P - 1) // 2 <= x <= (P - 1) // 2
        assert all((x - vv) % q == 0 for vv, q in zip(v, primes))
        got.append(x)
    assert sorted(got) == list(range(-(P - 1) // 2, (P - 1) // 2 + 1))


def test_garner_full_modulus_against_sympy_crt():
    crt = pytest.importorskip("sympy.ntheory.modular").crt
    P = math.prod(dm.PRIMES)
    rng = random.Random(17)
    for _ in range(200):
        v = [rng.randrange(q) for q in dm.PRIMES]
        x = dm.garner_balanced(v, dm.PRIMES)
        u = int(crt(dm.PRIMES, v)[0])  # library CRT in [0, P)
        assert x == (u if u <= (P - 1) // 2 else u - P)


def test_hadamard_bounds_hold():
    rng = random.Random(19)
    for n in (2, 4, 7, 10):
        A, b = rand_matrix(rng, n, 2, -1000, 1001)
        N2, D2 = dm.hadamard_squares(A, b)
        det = exact.determinant(A)
        assert det * det <= D2
        r = exact.solve_numerators(A, b)
        if r is None:
            continue
        dp, Y = r
        for row in Y:
            for y in row:
                assert y * y <= N2


def test_hadamard_numerator_bound_carries_the_b_term():
    """N_H = prod_i sqrt(||a_i||^2 + max_k b_ik^2) must include b: with A = I_4
    the Cramer numerators are b itself while prod_i ||a_i|| = 1; and for a dense
    4 x 4 system with 40-bit entries and 62-bit b, the bound without b asks for
    one step although P' <= 2 |N| d (one step cannot determine the fraction),
    so only the bound with b gives enough steps for the model to match the
    oracle."""
    A = [[int(i == j) for j in range(4)] for i in range(4)]
    b = [[(1 << 40) - 3], [-(1 << 40) + 5], [(1 << 39) + 1], [-(1 << 40) + 7]]
    N2, D2 = dm.hadamard_squares(A, b)
    assert D2 == 1
    dp, Y = exact.solve_numerators(A, b)
    assert dp == 1 and [row[0] for row in Y] == [row[0] for row in b]
    assert all(y * y <= N2 for row in Y for y in row)

    rng = random.Random(41)
    A = [[rng.randrange(-(1 << 40), 1 << 40) for _ in range(4)] for _ in range(4)]
    b = [[rng.randrange(-(1 << 62), 1 << 62)] for _ in range(4)]
    N, d = exact.solve(A, b)
    gp, _ = dm.good_primes(A)
    P = math.prod(gp)
    N2, D2 = dm.hadamard_squares(A, b)
    assert all(v * v <= N2 for row in N for v in row)
    assert dm.steps_needed(P, D2, D2) == 1          # what a bound without b would ask for
    assert P <= 2 * max(abs(v) for row in N for v in row) * d
    res = dm.solve(A, b)
    assert res is not None and (res[0], res[1]) == (N, d) and res[2]["m"] >= 2


def test_steps_needed_is_minimal():
    P = math.prod(dm.PRIMES)
    for N2, D2 in ((1, 1), (10 ** 50, 10 ** 80), (2 ** 600, 2 ** 700), (2 ** 5000, 3 ** 4000)):
        m = dm.steps_needed(P, N2, D2)
        assert P ** (2 * m) > 4 * N2 * D2
        assert m == 1 or P ** (2 * (m - 1)) <= 4 * N2 * D2


def test_rational_reconstruction_roundtrip():
    rng = random.Random(23)
    M = math.prod(dm.PRIMES) ** 3
    Nb = Db = math.isqrt(M // 2) - 1
    for _ in range(300):
        den = rng.randrange(1, Db + 1)
        num = rng.randrange(-Nb, Nb + 1)
        g = math.gcd(num, den)
        num, den = num // g, den // g
        u = num * pow(den, -1, M) % M if math.gcd(den, M) == 1 else None
        if u is None:
            continue
        assert dm.rational_reconstruct(u, M, Nb, Db) == (num, den)


def test_model_lift_identities_and_end_to_end():
    rng = random.Random(29)
    for n, c, lo, hi in ((1, 1, -9, 10), (3, 2, -100, 101), (8, 1, -(1 << 23), 1 << 23), (12, 3, -127, 128)):
        A, b = rand_matrix(rng, n, c, lo, hi)
        ref = exact.solve(A, b)
        res = dm.solve(A, b)
        if ref is None:
            assert res is None
            continue
        N, d, info = res
        assert (N, d) == ref
        P, m, digits = info["P"], info["m"], info["digits"]
        for x in digits:
            for row in x:
                for v in row:
                    assert abs(v) <= (P - 1) // 2
        M = P ** m
        X = [[sum(digits[t][i][j] * P ** t for t in range(m)) for j in range(c)] for i in range(n)]
        for i in range(n):
            for j in range(c):
                assert (sum(A[i][k] * X[k][j] for k in range(n)) - b[i][j]) % M == 0


def test_model_residual_stays_in_one_limb():
    # |r_{i+1}| <= |r_i| / P + n max|A| / 2: with n max|A| < 2^63 the residual fits int64.
    A, b = inputs.uniform(24, 2, -(1 << 23), 1 << 23, seed=31)
    A[0, 0] = (1 << 63) // 24 - 1  # push n max|A| to the range edge
    gp, Bs = dm.good_primes(A.tolist())
    _, residuals = dm.lift(A.tolist(), b.tolist(), gp, 4, Bs)
    for r in residuals:
        for row in r:
            for v in row:
                assert -(1 << 63) <= v < (1 << 63)


def test_model_pascal_and_hilbert_end_to_end():
    A, b = inputs.pascal_system(30, 1, seed=0)
    N, d, info = dm.solve(A.tolist(), b.tolist())
    assert (N, d) == exact.solve(A.tolist(), b.tolist()) and d == 1
    H = inputs.scaled_hilbert(8).tolist()
    hb = [[i - 3] for i in range(8)]
    N, d, _ = dm.solve(H, hb)
    assert (N, d) == exact.solve(H, hb)


def test_all_primes_dividing_det_is_a_known_deviation():
    """A nonsingular diagonal A whose determinant is divisible by every odd
    prime < 256: the method (and the CUDA library) reports it singular while
    the exact solver does not -- the documented limitation of the reading that
    'no usable prime' means singular."""
    A = all_primes_diagonal()
    b = [[1] for _ in range(len(A))]
    assert exact.solve(A, b) is not None
    assert dm.solve(A, b) is None


def all_primes_diagonal():
    groups = [[] for _ in range(8)]
    for i, q in enumerate(dm.PRIMES):
        groups[i % 8].append(q)
    diag = [math.prod(g) for g in groups]
    n = len(diag)
    assert n * max(diag) < 1 << 63
    return [[diag[i] if i == j else 0 for j in range(n)] for i in range(n)]
