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


def _as_u64(raw):
    """The same 64-bit words as a contiguous uint64 array (int64 words are
    reinterpreted, not converted)."""
    raw = np.ascontiguousarray(raw)
    return raw.view(np.uint64) if raw.dtype == np.int64 else raw.astype(np.uint64, copy=False)


def limbs_mod_primes(raw, primes, block=4096):
    """Residues modulo each p in `primes` of the signed integers held as rows of
    little-endian two's complement 64-bit limbs (raw uint64 [count, W]).

    Each row is read as 16-bit chunks h_t (value = sum_t h_t 2^(16 t) - s 2^(64 W),
    s the sign bit), and sum_t h_t (2^(16 t) mod p) is one float64 matrix product:
    exact while 4 W (2^16 - 1)(p - 1) < 2^53.  Returns int64 [len(primes), count]
    in [0, p)."""
    raw = _as_u64(raw)
    count, W = raw.shape
    T = 4 * W
    assert all(T * 0xFFFF * (p - 1) < (1 << 53) for p in primes), "chunk sums would not be exact"
    Wt = np.array([[pow(2, 16 * t, p) for p in primes] for t in range(T)], dtype=np.float64)
    top = np.array([pow(2, 64 * W, p) for p in primes], dtype=np.int64)
    pv = np.array(primes, dtype=np.int64)
    out = np.empty((len(primes), count), dtype=np.int64)
    for s in range(0, count, block):
        blk = raw[s:s + block]
        H = blk.view(np.uint16).reshape(blk.shape[0], T).astype(np.float64)
        S = (H @ Wt).astype(np.int64) % pv  # [rows, primes]
        neg = (blk[:, W - 1] >> np.uint64(63)).astype(np.int64)
        out[:, s:s + block] = ((S - neg[:, None] * top[None, :]) % pv).T
    return out


def signed_chunks16(raw):
    """Rows of little-endian two's complement uint64 limbs [count, W] -> int64
    [count, 4 W] 16-bit chunks with value = sum_t chunk_t 2^(16 t): chunks
    below the top are in [0, 2^16), the top chunk is signed."""
    raw = _as_u64(raw)
    ch = raw.view(np.uint16).reshape(raw.shape[0], 4 * raw.shape[1]).astype(np.int64)
    ch[:, -1] = raw.view(np.int16).reshape(raw.shape[0], 4 * raw.shape[1])[:, -1]
    return ch


def combine_chunks16(S):
    """sum_t S[..., t] 2^(16 t) as a numpy object array of Python ints."""
    acc = S[..., -1].astype(object)
    for t in range(S.shape[-1] - 2, -1, -1):
        acc = acc * 65536 + S[..., t].astype(object)
    return acc


def check_lift_by_residuals_wide(A, b, D, good_primes, steps):
    """Vectorised form of the lift identity for many entries: every digit x_i
    (D uint64 [m, n*c, 6], entry (r, col) at r*c + col) is balanced,
    r_i - A x_i is divisible by P, and r_{i+1} = (r_i - A x_i) / P fits a
    signed 64-bit word; r_0 = b.  A x_i is formed exactly from 16-bit chunks
    of x_i in float64 (needs 2^(bits(A) + 16) n < 2^53)."""
    A = np.asarray(A, dtype=np.int64)
    n, c = A.shape[0], b.shape[1]
    amax = int(np.abs(A).max())
    assert (amax << 16) * n < (1 << 53), "entries of A too wide for the float64 chunk product"
    P = math.prod(good_primes)
    half = (P - 1) // 2
    Af = A.astype(np.float64)
    r = np.asarray(b, dtype=np.int64).astype(object)  # [n, c]
    for i in range(steps):
        ch = signed_chunks16(D[i])                       # [n*c, 24]
        x = combine_chunks16(ch).reshape(n, c)
        assert all(abs(v) <= half for v in x.flat), i
        Xk = ch.reshape(n, c * ch.shape[1]).astype(np.float64)
        S = (Af @ Xk).astype(np.int64).reshape(n, c, ch.shape[1])
        AX = combine_chunks16(S)
        T = r - AX
        q = T // P
        rem = T - q * P
        assert all(v == 0 for v in rem.flat), i
        assert all(-(1 << 63) <= v < (1 << 63) for v in q.flat), i
        r = q


# six primes just below 2^24: residue sums of 16-bit chunks stay exact in float64
CHECK_PRIMES = (16777213, 16777199, 16777183, 16777153, 16777141, 16777139)


def check_identity_mod_primes(A, b, num_limbs, W, d, primes=CHECK_PRIMES):
    """(A N - b d) mod p == 0 for every entry of every column and each p, with
    N given as limbs (num_limbs: n*c rows of W little-endian two's complement
    uint64 limbs, entry (i, j) at row i*c + j).  A N mod p is one float64
    product, exact while |A| (p - 1) n < 2^53."""
    A = np.asarray(A, dtype=np.int64)
    b = np.asarray(b, dtype=np.int64)
    n, c = A.shape[0], b.shape[1]
    amax = int(np.abs(A).max())
    assert all(amax * (p - 1) * n < (1 << 53) for p in primes), "A too wide for the float64 product"
    res = limbs_mod_primes(np.asarray(num_limbs).reshape(n * c, W), primes)  # [primes, n*c]
    Af = A.astype(np.float64)
    for t, p in enumerate(primes):
        Np = res[t].reshape(n, c).astype(np.float64)
        AN = (Af @ Np).astype(np.int64) % p
        bd = (b % p) * (d % p) % p
        bad = np.argwhere(AN != bd)
        assert bad.size == 0, (p, bad[:5].tolist())


def det_mod_q_gpu(A, q):
    """det A mod q by Gaussian elimination over GF(q), the same steps as
    det_mod_q on int64 CUDA tensors (for large n; test infrastructure)."""
    import torch

    M = torch.as_tensor(np.asarray(A, dtype=np.int64) % q, device="cuda")
    n = M.shape[0]
    det = 1
    for k in range(n):
        nz = torch.nonzero(M[k:, k])
        if nz.numel() == 0:
            return 0
        p = k + int(nz[0, 0])
        if p != k:
            M[[k, p]] = M[[p, k]]
            det = -det
        piv = int(M[k, k])
        det = det * piv % q
        inv = pow(piv, q - 2, q)
        f = (M[k + 1:, k] * inv) % q
        M[k + 1:] = (M[k + 1:] - torch.outer(f, M[k])) % q
    return det % q
