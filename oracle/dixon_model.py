"""Dixon p-adic lifting written out with Python ints, step by step.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Follows the exact-solve card (kernels hub), §Method, in its order and
notation:

  * modulus P = prod q_j over the odd primes q_j < 256 (squarefree, odd);
  * B = A^{-1} mod P, held as B_j = A^{-1} mod q_j, each computed by
    Gauss-Jordan on the augmented matrix [A | I] mod q_j;
  * r_0 = b;  x_i = B r_i mod P  (per prime, then balanced Garner CRT into
    one digit in [-(P-1)/2, (P-1)/2]);  r_{i+1} = (r_i - A x_i) / P;
  * stop when P^m exceeds twice the Hadamard bound on numerator and
    denominator; then x mod P^m = sum_i x_i P^i;
  * rational reconstruction of each component, common denominator.

Readings where the card is silent (kept identical in the CUDA library's
documentation): primes whose Gauss-Jordan finds no pivot (q_j | det A) are
dropped and P is the product of the remaining ones; when every prime is
dropped the system is reported singular; the pivot is the lowest-index
nonzero candidate row; residues and digits are balanced (symmetric) and
Garner runs over the primes in ascending order; the Hadamard bounds are
D_H = prod_i ||a_i||_2 over the rows of A and
N_H = prod_i sqrt(||a_i||^2 + max_k b_ik^2), so that every Cramer numerator
of every column of b is bounded by N_H.

Every intermediate here (B_j, each digit x_i, each residual r_i) is unique
given A, b and the prime set, so the CUDA stages are compared with it
element by element.
"""

from __future__ import annotations

from math import gcd, isqrt
from typing import List, Optional, Sequence, Tuple

Matrix = List[List[int]]


def odd_primes_below(limit: int = 256) -> List[int]:
    """Odd primes q < limit, by trial division."""
    out = []
    for q in range(3, limit, 2):
        if all(q % p for p in range(3, isqrt(q) + 1, 2)):
            out.append(q)
    return out


PRIMES = odd_primes_below(256)


def bal(v: int, q: int) -> int:
    """Balanced (symmetric) residue of v mod odd q, in [-(q-1)/2, (q-1)/2]."""
    r = v % q
    return r - q if r > (q - 1) // 2 else r


def inverse_mod(A: Sequence[Sequence[int]], q: int) -> Optional[Matrix]:
    """A^{-1} mod q by Gauss-Jordan on the augmented matrix [A | I] (entries in
    [0, q)), or None when A is singular mod q (no pivot in some column)."""
    n = len(A)
    M = [[int(v) % q for v in A[i]] + [1 if j == i else 0 for j in range(n)] for i in range(n)]
    for k in range(n):
        p = k
        while p < n and M[p][k] == 0:
            p += 1
        if p == n:
            return None
        M[k], M[p] = M[p], M[k]
        inv = pow(M[k][k], q - 2, q)  # q prime: Fermat
        M[k] = [(v * inv) % q for v in M[k]]
        rowk = M[k]
        for i in range(n):
            if i != k and M[i][k]:
                f = M[i][k]
                M[i] = [(a - f * bk) % q for a, bk in zip(M[i], rowk)]
    return [row[n:] for row in M]


def hadamard_squares(A, b) -> Tuple[int, int]:
    """(N_H^2, D_H^2) as exact integers:
    D_H^2 = prod_i ||a_i||^2,  N_H^2 = prod_i (||a_i||^2 + max_k b_ik^2)."""
    D2 = 1
    N2 = 1
    for i in range(len(A)):
        s = sum(int(v) * int(v) for v in A[i])
        bm = max((int(v) * int(v) for v in b[i]), default=0)
        D2 *= s
        N2 *= s + bm
    return N2, D2


def steps_needed(P: int, N2: int, D2: int) -> int:
    """Least m >= 1 with P^m > 2 N_H D_H, i.e. P^(2m) > 4 N_H^2 D_H^2."""
    target = 4 * N2 * D2
    m = 1
    Pm2 = P * P
    while Pm2 <= target:
        m += 1
        Pm2 *= P * P
    return m


def garner_balanced(residues: Sequence[int], primes: Sequence[int]) -> int:
    """The unique x in [-(P-1)/2, (P-1)/2] with x = residues[j] mod primes[j]:
    balanced mixed-radix (Garner) digits a_k in [-(q_k-1)/2, (q_k-1)/2],
    x = a_0 + a_1 q_0 + a_2 q_0 q_1 + ... (primes taken in the given order)."""
    x = 0
    Q = 1
    for v, q in zip(residues, primes):
        a = bal((v - x) * pow(Q % q, q - 2, q), q)
        x += a * Q
        Q *= q
    return x


def matvec(A, X) -> Matrix:
    n = len(A)
    c = len(X[0])
    return [[sum(int(A[i][k]) * X[k][j] for k in range(n)) for j in range(c)] for i in range(n)]


def lift(A, b, primes: Sequence[int], m: int, Bs: Optional[List[Matrix]] = None):
    """Run m Dixon steps.  Returns (digits, residuals): digits[i] is the n x c
    matrix x_i, residuals[i] the n x c matrix r_i (residuals[0] = b)."""
    n = len(A)
    c = len(b[0])
    A = [[int(v) for v in row] for row in A]
    if Bs is None:
        Bs = [inverse_mod(A, q) for q in primes]
    P = 1
    for q in primes:
        P *= q
    r = [[int(v) for v in row] for row in b]
    digits, residuals = [], [r]
    for _ in range(m):
        per_prime = []
        for B, q in zip(Bs, primes):
            rq = [[bal(v, q) for v in row] for row in r]
            per_prime.append([[bal(sum(B[i][k] * rq[k][j] for k in range(n)), q) for j in range(c)]
                              for i in range(n)])
        x = [[garner_balanced([pp[i][j] for pp in per_prime], primes) for j in range(c)] for i in range(n)]
        Ax = matvec(A, x)
        nxt = []
        for i in range(n):
            row = []
            for j in range(c):
                t, rem = divmod(r[i][j] - Ax[i][j], P)
                assert rem == 0, "r_i - A x_i must be divisible by P"
                row.append(t)
            nxt.append(row)
        digits.append(x)
        residuals.append(nxt)
        r = nxt
    return digits, residuals


def rational_reconstruct(u: int, M: int, Nb: int, Db: int) -> Optional[Tuple[int, int]]:
    """Wang's rational reconstruction: the fraction num/den (den > 0,
    |num| <= Nb, den <= Db, num = den * u mod M), unique when 2 Nb Db < M;
    None when none exists.  Extended Euclid on (M, u) stopped at the first
    remainder <= Nb."""
    r0, r1 = M, u % M
    t0, t1 = 0, 1
    while r1 > Nb:
        qt = r0 // r1
        r0, r1 = r1, r0 - qt * r1
        t0, t1 = t1, t0 - qt * t1
    if t1 == 0:
        return None
    num, den = (r1, t1) if t1 > 0 else (-r1, -t1)
    if den > Db or gcd(num, den) != 1:
        return None
    return num, den


def good_primes(A, primes: Sequence[int] = PRIMES):
    """(primes q_j not dividing det A, their inverses B_j), ascending."""
    gp, Bs = [], []
    for q in primes:
        B = inverse_mod(A, q)
        if B is not None:
            gp.append(q)
            Bs.append(B)
    return gp, Bs


def solve(A, b, primes: Sequence[int] = PRIMES):
    """End-to-end Dixon solve.  Returns (N, d, info) in canonical form, or None
    when every prime divides det A (singular over Q)."""
    A = [[int(v) for v in row] for row in A]
    b = [[int(v) for v in row] for row in b]
    n = len(A)
    c = len(b[0])
    gp, Bs = good_primes(A, primes)
    if not gp:
        return None
    P = 1
    for q in gp:
        P *= q
    N2, D2 = hadamard_squares(A, b)
    m = steps_needed(P, N2, D2)
    digits, _ = lift(A, b, gp, m, Bs)
    M = P ** m
    Nb, Db = isqrt(N2), isqrt(D2)
    fr = [[None] * c for _ in range(n)]
    d = 1
    for i in range(n):
        for j in range(c):
            X = 0
            for t in range(m - 1, -1, -1):
                X = X * P + digits[t][i][j]
            rr = rational_reconstruct(X % M, M, Nb, Db)
            assert rr is not None, "reconstruction must exist under the Hadamard bound"
            fr[i][j] = rr
            d = d * rr[1] // gcd(d, rr[1])
    N = [[fr[i][j][0] * (d // fr[i][j][1]) for j in range(c)] for i in range(n)]
    info = {"primes": gp, "P": P, "m": m, "digits": digits}
    return N, d, info
