"""Exact rational solution of A x = b by Bareiss elimination (Python ints).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What it computes (exact-solve card, §API): for integer A [n, n] and
b [n, c], the exact solution X = A^{-1} b over the rationals, or ``None``
when A is singular over Q.  The result is returned in canonical form
(N, d): d is the least positive integer with d X integral (the lcm of the
reduced denominators) and N = d X.  Two solvers agree bitwise exactly when
their canonical forms are equal (§Correctness compares bitwise against an
exact Gaussian-elimination oracle and uses the identity A @ N == d * b).

Algorithm: Bareiss' fraction-free elimination on [A | b] with the first
nonzero pivot at or below the diagonal, then fraction-free
back-substitution, which yields the Cramer numerators det'(A) * x as
integers; dividing out their common gcd with det' gives (N, d).
"""

from __future__ import annotations

from math import gcd
from typing import List, Optional, Sequence, Tuple

Matrix = List[List[int]]


def _as_rows(M) -> Matrix:
    return [[int(v) for v in row] for row in M]


def bareiss_upper(A: Sequence[Sequence[int]], b: Sequence[Sequence[int]]):
    """Fraction-free forward elimination of the augmented matrix [A | b].

    Returns (U, swaps) where U is the n x (n + c) augmented upper-triangular
    result (U[k][k] is the k-th leading principal minor of the row-permuted
    A) and ``swaps`` the number of row exchanges, or None when some column
    has no nonzero pivot candidate (A singular over Q).
    """
    n = len(A)
    M = [list(map(int, A[i])) + list(map(int, b[i])) for i in range(n)]
    w = len(M[0]) if n else 0
    prev = 1
    swaps = 0
    for k in range(n):
        p = k
        while p < n and M[p][k] == 0:
            p += 1
        if p == n:
            return None
        if p != k:
            M[k], M[p] = M[p], M[k]
            swaps += 1
        pk = M[k][k]
        rowk = M[k]
        for i in range(k + 1, n):
            rowi = M[i]
            f = rowi[k]
            for j in range(k + 1, w):
                num = pk * rowi[j] - f * rowk[j]
                q, r = divmod(num, prev)
                assert r == 0, "Bareiss division must be exact"
                rowi[j] = q
            rowi[k] = 0
        prev = pk
    return M, swaps


def solve_numerators(A, b) -> Optional[Tuple[int, Matrix]]:
    """(det', Y) with Y = det' * X integral, det' = det of the row-permuted A
    (= +-det A), or None if A is singular."""
    A = _as_rows(A)
    b = _as_rows(b)
    n = len(A)
    c = len(b[0]) if n else 0
    res = bareiss_upper(A, b)
    if res is None:
        return None
    U, _ = res
    det = U[n - 1][n - 1]
    Y = [[0] * c for _ in range(n)]
    for col in range(c):
        for i in range(n - 1, -1, -1):
            s = det * U[i][n + col]
            for j in range(i + 1, n):
                s -= U[i][j] * Y[j][col]
            q, r = divmod(s, U[i][i])
            assert r == 0, "fraction-free back-substitution must divide exactly"
            Y[i][col] = q
    return det, Y


def canonical(det: int, Y: Matrix) -> Tuple[Matrix, int]:
    """(N, d) from X = Y / det: d = |det| / g, N = sign(det) * Y / g with
    g = gcd(det, all Y)."""
    g = abs(det)
    for row in Y:
        for v in row:
            g = gcd(g, v)
    s = 1 if det > 0 else -1
    d = abs(det) // g
    N = [[s * (v // g) for v in row] for row in Y]
    return N, d


def solve(A, b) -> Optional[Tuple[Matrix, int]]:
    """Canonical exact solution (N, d) of A x = b, or None if A is singular."""
    r = solve_numerators(A, b)
    if r is None:
        return None
    return canonical(*r)


def solve_fractions(A, b):
    """[n][c] nested lists of fractions.Fraction, or None (the card's §API shape)."""
    from fractions import Fraction

    r = solve(A, b)
    if r is None:
        return None
    N, d = r
    return [[Fraction(v, d) for v in row] for row in N]


def determinant(A) -> int:
    """det A by Bareiss (0 when singular)."""
    A = _as_rows(A)
    n = len(A)
    if n == 0:
        return 1
    res = bareiss_upper(A, [[] for _ in range(n)])
    if res is None:
        return 0
    U, swaps = res
    return (-1) ** swaps * U[n - 1][n - 1]
