"""Test helpers shared by the CPU and GPU tests (no method arithmetic of the
library; conversions and exact checks only)."""

import math

import numpy as np


def digits_to_limbs(digits, P=None):
    """Model digits (list over steps of n x c lists of Python ints) ->
    uint64 [m, n*c, 6] little-endian two's complement limbs."""
    m = len(digits)
    n = len(digits[0])
    c = len(digits[0][0])
    out = np.zeros((m, n * c, 6), dtype=np.uint64)
    mask = (1 << 384) - 1
    for i in range(m):
        for r in range(n):
            for col in range(c):
                v = digits[i][r][col] & mask
                raw = v.to_bytes(48, "little")
                out[i, r * c + col] = np.frombuffer(raw, dtype=np.uint64)
    return out


def bits_bounds(N2, D2):
    """(num_bits, den_bits) with 2^num_bits >= N_H and 2^den_bits >= D_H."""
    return math.isqrt(N2).bit_length(), math.isqrt(D2).bit_length()


def steps_for_bits(P, num_bits, den_bits):
    m = 1
    while P ** m <= 2 ** (num_bits + den_bits + 1):
        m += 1
    return m


def check_identity(A, b, N, d):
    """A N == b d exactly (Python ints) and gcd(d, N) == 1."""
    n, c = len(A), len(b[0])
    assert d > 0
    Ai = [[int(v) for v in row] for row in A]
    for j in range(c):
        col = [N[k][j] for k in range(n)]
        for i in range(n):
            assert sum(a * x for a, x in zip(Ai[i], col)) == int(b[i][j]) * d, (i, j)
    g = d
    for row in N:
        for v in row:
            g = math.gcd(g, v)
    assert g == 1


def exact_matmul_cols(A, X):
    """Exact A @ X for an int64 numpy A [n, n] and X a list of columns of Python
    ints (any size), via float64 BLAS on 16-bit slices of X offset to be
    non-negative (each partial sum stays below 2^53).  Returns a list of
    columns of Python ints."""
    A = np.asarray(A, dtype=np.int64)
    n = A.shape[0]
    amax = int(np.abs(A).max()) if n else 0
    w = 16
    if amax.bit_length() + w + n.bit_length() > 52:
        if 17 + w + n.bit_length() > 52:
            Ai = A.tolist()
            return [[sum(int(a) * x for a, x in zip(row, col)) for row in Ai] for col in X]
        # A = A0 + 2^16 A1 with 0 <= A0 < 2^16 (both exact in int64)
        A0 = A & 0xFFFF
        A1 = (A - A0) >> 16
        P0, P1 = exact_matmul_cols(A0, X), exact_matmul_cols(A1, X)
        return [[u + (v << 16) for u, v in zip(c0, c1)] for c0, c1 in zip(P0, P1)]
    Af = A.astype(np.float64)
    rows = [int(v) for v in A.sum(axis=1)]
    out = []
    for col in X:
        mn = min(col)
        off = -mn if mn < 0 else 0
        shifted = [x + off for x in col]
        nchunks = max(1, (max(shifted).bit_length() + w - 1) // w)
        mask = (1 << w) - 1
        C = np.array([[(v >> (w * t)) & mask for t in range(nchunks)] for v in shifted], dtype=np.float64)
        S = Af @ C  # exact: entries < 2^52
        Si = S.astype(np.int64)
        res = []
        for i in range(n):
            acc = 0
            for t in range(nchunks - 1, -1, -1):
                acc = (acc << w) + int(Si[i, t])
            res.append(acc - off * rows[i])
        out.append(res)
    return out


def det_mod_q(A, q):
    """det A mod q by Gaussian elimination over GF(q) (numpy int64)."""
    M = np.asarray(A, dtype=np.int64) % q
    n = M.shape[0]
    det = 1
    for k in range(n):
        piv = np.nonzero(M[k:, k])[0]
        if piv.size == 0:
            return 0
        p = k + int(piv[0])
        if p != k:
            M[[k, p]] = M[[p, k]]
            det = -det
        det = det * int(M[k, k]) % q
        inv = pow(int(M[k, k]), q - 2, q)
        f = (M[k + 1:, k] * inv) % q
        M[k + 1:] = (M[k + 1:] - np.outer(f, M[k])) % q
    return det % q
