"""CPU tests of the C-ABI library: it loads and exports every declared
symbol, its modular reduction matches %, its host reconstruction stage
reproduces the oracle, and argument/range errors come back as statuses.
No GPU compute is attempted here."""

import ctypes
import math

import numpy as np
import pytest

from dixon_adic_lifting_gb300 import _lib as L
from dixon_adic_lifting_gb300 import api, inputs
from oracle import dixon_model as dm
from oracle import exact

from helpers import bits_bounds, digits_to_limbs, steps_for_bits


def test_exports_every_declared_symbol(lib):
    declared = L.header_functions()
    assert len(declared) >= 16
    for name in declared:
        assert hasattr(lib, name), name
        assert name in L._SIGS, f"binding lacks {name}"
    assert lib.es_version() == 1


def test_status_strings(lib):
    for code in L.STATUS:
        assert lib.es_status_string(code)


def test_barrett_reduction_matches_mod(lib):
    # signed accumulator domain of the Gauss-Jordan update (|x| < 2^21) exhaustively,
    # both ends of the int32 lift accumulator range, and int64 residues on samples
    assert api.selftest_modular(-(1 << 21), 1 << 21, 20000) == 0
    assert api.selftest_modular(-(1 << 31), -(1 << 31) + (1 << 20), 0) == 0
    assert api.selftest_modular((1 << 31) - 256 - (1 << 20), (1 << 31) - 256, 0) == 0


def test_gauss_jordan_f32_reduction_is_exact(lib):
    """The inverse kernels reduce exact f32 integers (|x| < 2^20, and up to
    2^21 + 128 in the depth-128 update) as x - q rint(x fl(1/q)); every
    |x| <= 2^21 + 2^10 and every prime, against %."""
    assert api.selftest_gj_reduction() == 0


def model_digits(A, b, m=None):
    gp, Bs = dm.good_primes(A)
    P = math.prod(gp)
    N2, D2 = dm.hadamard_squares(A, b)
    nb, db = bits_bounds(N2, D2)
    if m is None:
        m = steps_for_bits(P, nb, db)
    digits, _ = dm.lift(A, b, gp, m, Bs)
    good = np.array([1 if q in gp else 0 for q in dm.PRIMES], dtype=np.uint8)
    return digits, good, nb, db, m


def test_bigint_selftest(lib):
    """Karatsuba products against a plain product, division and shift
    identities and the rational reconstruction's defining congruence, on
    random operands up to 1200 limbs (the reconstruction's big integers)."""
    assert api.selftest_bigint(1, 300) == 0
    assert api.selftest_bigint(2024, 300) == 0


@pytest.mark.parametrize("case", ["n5c2", "pascal30", "n24_24bit", "hilbert6", "hilbert12", "n33c5", "planted"])
def test_host_reconstruction_matches_oracle(lib, case):
    if case == "n5c2":
        A, b = inputs.uniform(5, 2, -50, 51, seed=1)
    elif case == "pascal30":
        A, b = inputs.pascal_system(30, 1, seed=0)
    elif case == "n24_24bit":
        A, b = inputs.uniform(24, 1, -(1 << 23), 1 << 23, seed=2)
    elif case.startswith("hilbert"):
        # sampled denominators miss factors that two failing components share
        k = int(case[7:])
        A = inputs.scaled_hilbert(k)
        b = np.arange(1, k + 1, dtype=np.int64).reshape(k, 1)
    elif case == "n33c5":
        A, b = inputs.uniform(33, 5, -(1 << 23), 1 << 23, seed=33)
    else:
        A, b, _ = inputs.planted(10, 3, seed=4)
    A, b = A.tolist(), b.tolist()
    ref = exact.solve(A, b)
    digits, good, nb, db, m = model_digits(A, b)
    for threads in (1, 3):
        s = api.reconstruct(digits_to_limbs(digits), len(A), len(b[0]), m, good, nb, db, threads=threads)
        assert (s.N, s.d) == ref


def test_host_reconstruction_needs_a_second_round(lib):
    # sampled components (0, 2, 4, 6 of 8) are integers; component 7 is 1/7
    A = [[7 if (i == j == 7) else (1 if i == j else 0) for j in range(8)] for i in range(8)]
    b = [[1] for _ in range(8)]
    digits, good, nb, db, m = model_digits(A, b)
    s = api.reconstruct(digits_to_limbs(digits), 8, 1, m, good, nb, db)
    assert (s.N, s.d) == exact.solve(A, b) == ([[7]] * 7 + [[1]], 7)


@pytest.mark.parametrize("threads", [1, 3])
def test_host_reconstruction_failures_in_several_columns(lib, threads):
    # the sample (one component per column, rows 0, 2, 4, 6) holds integers
    # only; row 7 is 1/7 in columns 0 and 1 and an integer in column 2
    A = [[7 if (i == j == 7) else (1 if i == j else 0) for j in range(8)] for i in range(8)]
    b = [[1, 2, 7] for _ in range(8)]
    digits, good, nb, db, m = model_digits(A, b)
    s = api.reconstruct(digits_to_limbs(digits), 8, 3, m, good, nb, db, threads=threads)
    assert (s.N, s.d) == exact.solve(A, b)
    assert s.d == 7 and s.N[7] == [1, 2, 7]


def test_host_reconstruction_large_numbers(lib):
    # numerators of ~1300 bits: exercises the Lehmer and Karatsuba paths
    A, b = inputs.uniform(44, 1, -(1 << 23), 1 << 23, seed=5)
    A, b = A.tolist(), b.tolist()
    digits, good, nb, db, m = model_digits(A, b)
    s = api.reconstruct(digits_to_limbs(digits), 44, 1, m, good, nb, db)
    assert (s.N, s.d) == exact.solve(A, b)


def test_host_reconstruction_rejects_too_few_steps(lib):
    A, b = inputs.uniform(12, 1, -(1 << 23), 1 << 23, seed=6)
    A, b = A.tolist(), b.tolist()
    digits, good, nb, db, m = model_digits(A, b)
    assert m >= 2
    with pytest.raises(api.ExactSolveError) as e:
        api.reconstruct(digits_to_limbs(digits[:m - 1]), 6, 1, m - 1, good, nb, db)
    assert e.value.status == -6  # ES_ERR_INTERNAL


def test_reconstruction_fault_injection(lib):
    A, b = inputs.uniform(3, 1, -9, 10, seed=7)
    digits, good, nb, db, m = model_digits(A.tolist(), b.tolist())
    with pytest.raises(api.ExactSolveError) as e:
        api.reconstruct(digits_to_limbs(digits), 3, 1, m, good, nb, db, fault="recon")
    assert e.value.status == -6


def test_argument_and_range_errors_without_gpu(lib):
    out = ctypes.c_void_p()
    A = np.zeros((4, 4), dtype=np.int64)
    b = np.zeros((4, 1), dtype=np.int64)
    assert lib.es_solve(A.ctypes.data, b.ctypes.data, 0, 1, None, ctypes.byref(out)) == -1
    assert lib.es_solve(A.ctypes.data, b.ctypes.data, 4, 0, None, ctypes.byref(out)) == -1
    assert lib.es_solve(None, b.ctypes.data, 4, 1, None, ctypes.byref(out)) == -1
    assert lib.es_solve(A.ctypes.data, b.ctypes.data, (1 << 17) + 1, 1, None, ctypes.byref(out)) == -2


def test_no_cpu_fallback_without_gpu(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    A, b = inputs.uniform(4, 1, -9, 10, seed=8)
    with pytest.raises(api.ExactSolveError) as e:
        api.solve(A, b)
    assert e.value.status == -7  # ES_ERR_NODEVICE


def test_named_workloads_match_their_descriptions():
    """Every named workload draws A [n, n] and b [n, c] with the declared
    shape and entry range, deterministically per seed; the planted system's
    right-hand side is A x* exactly."""
    from dixon_adic_lifting_gb300 import inputs

    ranges = {"_24bit": 1 << 23, "_16bit": 1 << 15, "_int8": 128}
    for name, w in inputs.WORKLOADS.items():
        if name == "n4096_c64_16bit":
            continue  # same generator as the n = 2048 case; 134 MB, skipped for time
        A, b = inputs.workload(name, seed=0, attempt=0)
        assert A.shape == (w.n, w.n) and b.shape == (w.n, w.c), name
        A2, b2 = inputs.workload(name, seed=0, attempt=0)
        assert np.array_equal(A, A2) and np.array_equal(b, b2), name
        for suffix, lim in ranges.items():
            if name.endswith(suffix):
                assert -lim <= A.min() and A.max() < lim and -lim <= b.min() and b.max() < lim, name
    A, b = inputs.workload("planted256", seed=0)
    _, _, X = inputs.planted(256, 1, seed=0)
    assert [[int(v)] for v in (A.astype(object) @ X.astype(object)).ravel()] == b.tolist()
    assert inputs.workload("hilbert21")[0].tolist() == inputs.scaled_hilbert(21).tolist()


@pytest.mark.parametrize("seed", range(8))
def test_host_reconstruction_random_many_columns(lib, seed):
    """Small random systems with more columns than rows or samples: the
    column-spread sample and the per-column retry rounds still give the
    oracle's canonical (N, d)."""
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(2, 7))
    c = int(rng.integers(n + 1, 3 * n + 3))
    A = rng.integers(-9, 10, size=(n, n))
    while exact.solve(A.tolist(), [[1]] * n) is None:
        A = rng.integers(-9, 10, size=(n, n))
    b = rng.integers(-20, 21, size=(n, c))
    b[:, 0] = 0  # an all-zero column: numerators 0
    A, b = A.tolist(), b.tolist()
    digits, good, nb, db, m = model_digits(A, b)
    for threads in (1, 4):
        s = api.reconstruct(digits_to_limbs(digits), n, c, m, good, nb, db, threads=threads)
        assert (s.N, s.d) == exact.solve(A, b)


@pytest.mark.parametrize("threads", [8, 16])
def test_host_reconstruction_through_the_pool_pipes(lib, threads):
    # 64 x 64, 24-bit entries: M has about 55 limbs, so every sampled run hands
    # its cofactors to a pool task (pools of 8 and more); with 16 tasks on a
    # smaller machine the low-limb servers start only after their runs and must
    # return at once
    A, b = inputs.uniform(64, 1, -(1 << 23), 1 << 23, seed=64)
    A, b = A.tolist(), b.tolist()
    digits, good, nb, db, m = model_digits(A, b)
    s = api.reconstruct(digits_to_limbs(digits), 64, 1, m, good, nb, db, threads=threads)
    assert (s.N, s.d) == exact.solve(A, b)
