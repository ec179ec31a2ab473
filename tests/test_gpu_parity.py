"""GPU parity of every CUDA stage, through the C ABI, against the CPU oracle
(bit-exact: all of this is integer work) and, where the oracle is too slow,
against properties that pin the unique result (the inverse mod q is unique;
a balanced digit with A x_i = r_i mod P is unique; a canonical (N, d) with
A N = b d and gcd 1 is unique for nonsingular A)."""

import json
import math
import os

import numpy as np
import pytest

from dixon_adic_lifting_gb300 import api, inputs
from oracle import dixon_model as dm
from oracle import exact

from helpers import bits_bounds, check_identity, det_mod_q, det_mod_q_gpu, exact_matmul_cols, steps_for_bits

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PRIMES = dm.PRIMES


@pytest.fixture(scope="module")
def torch_cuda(lib):
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


def dev(torch, a):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int64, device="cuda")


# ------------------------------------------------------------------ residues
def test_residues(torch_cuda):
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.integers(-(1 << 63), (1 << 63) - 1, 3000, dtype=np.int64),
                           np.array([-(1 << 63), (1 << 63) - 1, 0, 1, -1, 251, -251, 3 ** 39], dtype=np.int64)])
    out = api.residues_device(dev(torch_cuda, vals)).cpu().numpy()
    for j, q in enumerate(PRIMES):
        exp = [dm.bal(int(v), q) for v in vals]
        assert out[j].tolist() == exp, q


# ------------------------------------------------------------------ inverse
def model_inverse_bal(A, q):
    B = dm.inverse_mod(A, q)
    return None if B is None else [[dm.bal(v, q) for v in row] for row in B]


@pytest.mark.parametrize("n", [1, 2, 3, 7, 16, 17, 31, 32, 33, 40])
def test_inverse_vs_model(torch_cuda, n):
    A, _ = inputs.uniform(n, 1, -(1 << 23), 1 << 23, seed=100 + n)
    if n >= 3:
        A[0] *= 15  # 3 and 5 divide det A: those primes must be flagged bad
    B, good = api.inverse_mod_device(dev(torch_cuda, A))
    B = B.cpu().numpy()
    good = good.cpu().numpy()
    ld = api.padded_ld(n)
    assert B.shape == (53, n, ld)
    Al = A.tolist()
    for j, q in enumerate(PRIMES):
        exp = model_inverse_bal(Al, q)
        assert good[j] == (0 if exp is None else 1), q
        if exp is not None:
            assert B[j, :, :n].tolist() == exp, q
            assert not B[j, :, n:].any()
    if n >= 3:
        assert good[0] == 0 and good[1] == 0


def check_inverse_property(A, B, good, primes_to_check):
    n = A.shape[0]
    for j in primes_to_check:
        q = PRIMES[j]
        if good[j]:
            Aq = np.array([[dm.bal(int(v), q) for v in row] for row in A], dtype=np.float64) if n <= 64 else \
                (((A % q) + q) % q).astype(np.float64)
            Bq = B[j, :, :n].astype(np.float64)
            prod = (Aq @ Bq).astype(np.int64) % q  # exact: |entries| < 2^53
            assert np.array_equal(prod, np.eye(n, dtype=np.int64)), q
        else:
            assert (det_mod_q(A, q) if n <= 512 else det_mod_q_gpu(A, q)) == 0, q


@pytest.mark.parametrize("n", [64, 100, 256, 1024, 1025, 1100, 2000, 4096])
def test_inverse_property(torch_cuda, n):
    """A B_j = I mod q_j and the bad-prime flags; from n = 1025 to 4096 the
    panels run on thread-block clusters (1100, 2000: a partial last panel and
    rows beyond n in the cluster's last CTA)."""
    A, _ = inputs.uniform(n, 1, -(1 << 23), 1 << 23, seed=200 + n)
    A[1] *= 21  # 3 and 7 divide det A
    B, good = api.inverse_mod_device(dev(torch_cuda, A))
    B, good = B.cpu().numpy(), good.cpu().numpy()
    assert good[0] == 0 and good[2] == 0
    js = range(53) if n <= 256 else [0, 1, 2, 10, 30, 52]
    check_inverse_property(A, B, good, js)
    if n <= 256:
        for j, q in enumerate(PRIMES):
            assert bool(good[j]) == (det_mod_q(A, q) != 0), q


def test_inverse_int8_entries_and_singular_mod_small_primes(torch_cuda):
    # small entries: singular modulo several small primes is common
    for seed in range(6):
        A, _ = inputs.uniform(12, 1, -3, 4, seed=seed)
        B, good = api.inverse_mod_device(dev(torch_cuda, A))
        B, good = B.cpu().numpy(), good.cpu().numpy()
        for j, q in enumerate(PRIMES):
            exp = model_inverse_bal(A.tolist(), q)
            assert good[j] == (0 if exp is None else 1)
            if exp is not None:
                assert B[j, :, :12].tolist() == exp


# ------------------------------------------------------------------ plan
@pytest.mark.parametrize("case", [(8, 1, 23), (30, 2, 7), (64, 1, 23), (5, 3, 62)])
def test_plan_matches_exact_bounds(torch_cuda, case):
    n, c, bits = case
    lim = min(1 << bits, ((1 << 63) - 1) // n)
    A, b = inputs.uniform(n, c, -lim + 1, lim, seed=n)
    good = np.ones(53, dtype=np.uint8)
    good[3] = 0  # exercise a reduced prime set
    nb, db, m = api.plan_device(dev(torch_cuda, A), dev(torch_cuda, b), good)
    N2, D2 = dm.hadamard_squares(A.tolist(), b.tolist())
    enb, edb = bits_bounds(N2, D2)
    assert (1 << nb) ** 2 >= N2 and (1 << db) ** 2 >= D2
    assert enb - 1 <= nb <= enb + 1 and edb - 1 <= db <= edb + 1
    P = math.prod(q for j, q in enumerate(PRIMES) if good[j])
    assert P ** m > 2 ** (nb + db + 1)
    assert m == 1 or P ** (m - 1) <= 2 ** (nb + db + 2)


# ------------------------------------------------------------------ lift
def lift_gpu(torch, A, b, m):
    At, bt = dev(torch, A), dev(torch, b)
    B, good = api.inverse_mod_device(At)
    D = api.lift_device(At, bt, B, good, m)
    return api.digits_to_ints(D), good.cpu().numpy()


@pytest.mark.parametrize("case", ["n1", "n5c3", "n17", "n32_int8", "pascal30", "n40c2", "n24c17"])
def test_lift_digits_vs_model(torch_cuda, case):
    if case == "n1":
        A, b = np.array([[-6]]), np.array([[4]])
    elif case == "n5c3":
        A, b = inputs.uniform(5, 3, -50, 51, seed=1)
    elif case == "n17":
        A, b = inputs.uniform(17, 1, -(1 << 23), 1 << 23, seed=17)
    elif case == "n32_int8":
        A, b = inputs.workload("n32_c1_int8", seed=0, attempt=1)
    elif case == "pascal30":
        A, b = inputs.pascal_system(30, 1, seed=0)
    elif case == "n40c2":
        A, b = inputs.uniform(40, 2, -(1 << 23), 1 << 23, seed=40)
    else:
        A, b = inputs.uniform(24, 17, -(1 << 15), 1 << 15, seed=24)
    Al, bl = A.tolist(), b.tolist()
    gp, Bs = dm.good_primes(Al)
    m = 3
    digits, _ = dm.lift(Al, bl, gp, m, Bs)
    got, good = lift_gpu(torch_cuda, A, b, m)
    assert [q for j, q in enumerate(PRIMES) if good[j]] == gp
    n, c = len(Al), len(bl[0])
    for i in range(m):
        assert [got[i][r * c + col] for r in range(n) for col in range(c)] == \
            [digits[i][r][col] for r in range(n) for col in range(c)], i


def check_lift_by_residuals(A, b, digits, good, steps):
    """Every digit is the unique balanced x_i with A x_i = r_i (mod P), and
    r_{i+1} = (r_i - A x_i) / P exactly (Python ints)."""
    n, c = A.shape[0], b.shape[1]
    P = math.prod(q for j, q in enumerate(PRIMES) if good[j])
    r = [[int(b[i, col]) for i in range(n)] for col in range(c)]  # columns
    for i in range(steps):
        X = [[int(digits[i][k * c + col]) for k in range(n)] for col in range(c)]
        for col in range(c):
            assert all(abs(v) <= (P - 1) // 2 for v in X[col])
        AX = exact_matmul_cols(A, X)
        nxt = []
        for col in range(c):
            rc = []
            for k in range(n):
                t, rem = divmod(r[col][k] - AX[col][k], P)
                assert rem == 0, (i, col, k)
                assert -(1 << 63) <= t < (1 << 63)
                rc.append(t)
            nxt.append(rc)
        r = nxt


@pytest.mark.parametrize("n,c,bits", [(1024, 16, 7), (1030, 20, 15), (1024, 16, 23), (1100, 24, 31),
                                      (130, 16, 23), (20, 16, 40)])
def test_lift_many_columns_by_residuals(torch_cuda, n, c, bits):
    """c >= 16: the tcgen05 product; from n = 1024 with the tcgen05 residual
    update for one to four 8-bit limbs of A (bits 7, 15, 23, 31; c = 20 and
    24 leave a partial 8-column tile, n = 1030 and 1100 a partial row tile and
    K block), below it and for entries of 2^31 and more the CUDA-core update."""
    A, b = inputs.uniform(n, c, -(1 << bits) + 1, 1 << bits, seed=n + c)
    At, bt = dev(torch_cuda, A), dev(torch_cuda, b)
    B, good = api.inverse_mod_device(At)
    nb, db, m = api.plan_device(At, bt, good)
    steps = min(m, 6)
    D = api.lift_device(At, bt, B, good, steps)
    check_lift_by_residuals(A, b, api.digits_to_ints(D), good, steps)


@pytest.mark.parametrize("name,steps", [("n256_c1_24bit", None), ("n1024_c1_24bit", 6)])
def test_lift_full_size_by_residuals(torch_cuda, name, steps):
    A, b = inputs.workload(name, seed=0)
    At, bt = dev(torch_cuda, A), dev(torch_cuda, b)
    B, good = api.inverse_mod_device(At)
    nb, db, m = api.plan_device(At, bt, good)
    D = api.lift_device(At, bt, B, good, m)
    digits = api.digits_to_ints(D[: (steps or m)])
    check_lift_by_residuals(A, b, digits, good.cpu().numpy(), steps or m)


@pytest.mark.parametrize("n,bits", [(1, 23), (2, 7), (152, 23), (153, 23), (300, 40), (1000, 23), (1024, 23)])
def test_fused_lift_matches_step_kernels(torch_cuda, n, bits):
    """c = 1 and n <= 1024 run the whole lift as one cooperative launch; the
    per-step kernels (ES_FLAG_STEP_LIFT) are an independent route to the same
    unique digits, so the canonical solutions agree bit for bit."""
    A, b = inputs.uniform(n, 1, -(1 << bits), 1 << bits, seed=1000 + n)
    At, bt = dev(torch_cuda, A), dev(torch_cuda, b)
    fused = api.solve_device(At, bt, timing=2)
    step = api.solve_device(At, bt, timing=2, step_lift=True)
    assert fused.top_kernel == "k_lift_fused" and fused.top_launches == 1
    assert step.top_kernel == "k_lift_gemv" and step.top_launches == step.m
    assert fused.m == step.m and fused.top_ms > 0
    assert (fused.N, fused.d) == (step.N, step.d)
    if n <= 300:
        check_identity(A, b, fused.N, fused.d)


@pytest.mark.parametrize("n", [97, 300, 640, 1000])
def test_split_inverse_matches_one_stream(torch_cuda, n):
    """The inverse's default schedule (next 64-column block factorized on one SM
    partition while the previous block's update runs on the other) and the
    single-stream schedule are independent routes to the same unique B_j;
    the solves agree bit for bit and are exact."""
    A, b = inputs.uniform(n, 1, -(1 << 23), 1 << 23, seed=2000 + n)
    split = api.solve_canonical(A, b)
    one = api.solve_canonical(A, b, one_stream=True)
    assert (split.N, split.d) == (one.N, one.d)
    assert split.inverse_split and not one.inverse_split  # both schedules really ran
    if n <= 300:
        check_identity(A, b, split.N, split.d)


# ------------------------------------------------------------------ solve
def n32_case(seed):
    with open(os.path.join(GOLDEN, "n32_attempts.json")) as f:
        att = json.load(f)["attempts"][str(seed)]
    return inputs.workload("n32_c1_int8", seed=seed, attempt=att)


@pytest.mark.parametrize("seed", range(5))
def test_solve_n32_all_primes(torch_cuda, seed):
    A, b = n32_case(seed)
    s = api.solve_canonical(A, b)
    assert s.primes_used == 53
    assert (s.N, s.d) == exact.solve(A.tolist(), b.tolist())


def test_solve_pascal30(torch_cuda):
    A, b = inputs.workload("pascal30", seed=0)
    s = api.solve_canonical(A, b)
    with open(os.path.join(GOLDEN, "pascal30_seed0.json")) as f:
        g = json.load(f)
    assert s.d == 1 == g["d"]
    assert [row[0] for row in s.N] == [int(v) for v in g["N"]]
    assert (s.N, s.d) == exact.solve(A.tolist(), b.tolist())


def test_solve_n256_against_stored_oracle(torch_cuda):
    path = os.path.join(GOLDEN, "n256_seed0.json")
    with open(path) as f:
        g = json.load(f)
    A, b = inputs.workload("n256_c1_24bit", seed=0)
    s = api.solve_canonical(A, b)
    from tests_golden_digest import canonical_digest
    assert str(s.d) == g["regular"]["d"]
    assert [str(s.N[i][0]) for i in range(3)] == g["regular"]["N_head"]
    assert canonical_digest(s.N, s.d) == g["regular"]["digest"]
    S = inputs.make_rank_deficient(A, seed=0)
    assert g["rank_deficient"]["singular"] is True
    assert api.solve_canonical(S, b) is None


def test_solve_n1024_identity(torch_cuda):
    A, b = inputs.workload("n1024_c1_24bit", seed=0)
    s = api.solve_canonical(A, b)
    assert s.primes_used >= 1  # some prime does not divide det A: A is nonsingular
    check_identity(A, b, s.N, s.d)


@pytest.mark.parametrize("case", ["hilbert12", "hilbert21", "planted64", "n33c5", "n100", "n48_16bit_c64"])
def test_solve_various_vs_oracle(torch_cuda, case):
    if case.startswith("hilbert"):
        n = int(case[7:])
        A = inputs.scaled_hilbert(n)
        b = np.arange(1, n + 1, dtype=np.int64).reshape(n, 1)
    elif case == "planted64":
        A, b, X = inputs.planted(64, 4, seed=64)
    elif case == "n33c5":
        A, b = inputs.uniform(33, 5, -(1 << 23), 1 << 23, seed=33)
    elif case == "n100":
        A, b = inputs.uniform(100, 1, -(1 << 23), 1 << 23, seed=100)
    else:
        A, b = inputs.uniform(48, 64, -(1 << 15), 1 << 15, seed=48)
    s = api.solve_canonical(A, b)
    if case == "planted64":
        assert s.d == 1 and s.N == X.tolist()
    if case in ("n100", "n48_16bit_c64"):
        check_identity(A, b, s.N, s.d)
        g = math.gcd(*[v for row in s.N for v in row], s.d)
        assert g == 1
    else:
        assert (s.N, s.d) == exact.solve(A.tolist(), b.tolist())


def test_hand_examples(torch_cuda):
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        s = api.solve_canonical(case["A"], case["b"])
        if case["N"] is None:
            assert s is None
        else:
            assert (s.N, s.d) == (case["N"], case["d"]), case["name"]
            assert api.solve(case["A"], case["b"]) == exact.solve_fractions(case["A"], case["b"])


def test_solve_device_matches_host_and_is_deterministic(torch_cuda):
    A, b = inputs.uniform(64, 3, -(1 << 23), 1 << 23, seed=64)
    s1 = api.solve_canonical(A, b)
    s2 = api.solve_device(dev(torch_cuda, A), dev(torch_cuda, b))
    s3 = api.solve_device(dev(torch_cuda, A), dev(torch_cuda, b), threads=1, timing=True)
    assert (s1.N, s1.d) == (s2.N, s2.d) == (s3.N, s3.d)
    assert all(t >= 0 for t in s3.phase_ms) and s3.phase_ms[2] > 0


@pytest.mark.parametrize("threads", [1, 2, 5])
def test_streamed_samples_with_narrow_pools(torch_cuda, threads):
    """c = 1, n <= 1024: the fused lift streams the sampled components' digits
    to host pool tasks that assemble them while it runs.  Pools narrower than
    the task count (one thread: every task in turn on the caller, after the
    lift has ended) give the same canonical solution."""
    A, b = inputs.uniform(300, 1, -(1 << 23), 1 << 23, seed=301)
    At, bt = dev(torch_cuda, A), dev(torch_cuda, b)
    ref = api.solve_device(At, bt, timing=2)
    assert ref.top_kernel == "k_lift_fused"
    s = api.solve_device(At, bt, threads=threads)
    assert (s.N, s.d) == (ref.N, ref.d)
    check_identity(A, b, s.N, s.d)


def test_edge_cases(torch_cuda):
    # zero right-hand side
    A, _ = inputs.uniform(20, 1, -99, 100, seed=2)
    s = api.solve_canonical(A, np.zeros((20, 2), dtype=np.int64))
    assert s.d == 1 and all(v == 0 for row in s.N for v in row)
    # a zero row is singular
    Z = A.copy()
    Z[5] = 0
    assert api.solve_canonical(Z, np.ones((20, 1), dtype=np.int64)) is None
    # range edge: n * max|A| = 2^63 - 1 is allowed, 2^63 is not
    n = 7
    lim = ((1 << 63) - 1) // n
    A = np.diag([lim] * n).astype(np.int64)
    b = np.ones((n, 1), dtype=np.int64)
    s = api.solve_canonical(A, b)
    assert s.d == lim and all(row == [1] for row in s.N)
    A[0, 1] = -(lim + 1)
    with pytest.raises(api.ExactSolveError) as e:
        api.solve_canonical(A, b)
    assert e.value.status == -2
    A = np.eye(3, dtype=np.int64)
    A[2, 2] = -(1 << 63)
    with pytest.raises(api.ExactSolveError) as e:
        api.solve_canonical(A, np.ones((3, 1), dtype=np.int64))
    assert e.value.status == -2


def test_all_primes_dividing_det_reads_as_singular(torch_cuda):
    """Known deviation (prime set exhausted): a nonsingular diagonal A whose
    determinant is divisible by every odd prime < 256 is reported singular."""
    groups = [[] for _ in range(8)]
    for i, q in enumerate(PRIMES):
        groups[i % 8].append(q)
    A = np.diag([math.prod(g) for g in groups]).astype(np.int64)
    assert api.solve_canonical(A, np.ones((8, 1), dtype=np.int64)) is None
    assert exact.solve(A.tolist(), [[1]] * 8) is not None


@pytest.mark.parametrize("fault,status", [("residues", -3), ("inverse", -3), ("lift", -5), ("recon", -6),
                                          ("nomem", -4)])
def test_fault_injection_leaves_context_usable(torch_cuda, fault, status):
    A, b = inputs.uniform(16, 1, -99, 100, seed=3)
    with pytest.raises(api.ExactSolveError) as e:
        api.solve_canonical(A, b, fault=fault)
    assert e.value.status == status
    assert (api.solve_canonical(A, b).N, ) == (exact.solve(A.tolist(), b.tolist())[0], )


def test_fused_lift_expired_wait_returns_timeout(torch_cuda):
    """Device side: the fused lift's first grid barrier can never complete (its
    counter starts where arrivals wrap below the target).  Every CTA's bounded
    wait (2 s) expires, the producer lets its copies land, the kernel returns,
    the host reports ES_ERR_TIMEOUT, and the next solve on the same context
    is exact."""
    A, b = inputs.uniform(64, 1, -(1 << 20), 1 << 20, seed=64)
    s = api.solve_canonical(A, b, timing=2)
    assert s.top_kernel == "k_lift_fused" and s.m >= 2
    with pytest.raises(api.ExactSolveError) as e:
        api.solve_canonical(A, b, fault="lift_wait")
    assert e.value.status == -5
    again = api.solve_canonical(A, b)
    assert (again.N, again.d) == (s.N, s.d)
    check_identity(A, b, again.N, again.d)


def test_device_memory_cap(torch_cuda):
    A, b = inputs.uniform(64, 1, -99, 100, seed=4)
    with pytest.raises(api.ExactSolveError) as e:
        api.solve_canonical(A, b, max_device_bytes=1 << 16)
    assert e.value.status == -4


@pytest.mark.parametrize("case", ["n32", "hilbert12", "n33c5", "n64c3_int8", "diag7", "n256", "n256c16",
                                  "n256c64", "n130c127", "hilbert12c1400"])
def test_device_reconstruction_matches_host_path(torch_cuda, case):
    """The numerators on the GPU against the all-host reconstruction; from
    16384 components (n256c64; n130c127: a partial 128-component tile;
    hilbert12c1400: dense denominators) on the tensor-core product."""
    if case == "n32":
        A, b = n32_case(1)
    elif case == "hilbert12":  # sampled denominators incomplete: a second round is needed
        A = inputs.scaled_hilbert(12)
        b = np.arange(1, 13, dtype=np.int64).reshape(12, 1)
    elif case == "n33c5":
        A, b = inputs.uniform(33, 5, -(1 << 23), 1 << 23, seed=33)
    elif case == "n64c3_int8":
        A, b = inputs.uniform(64, 3, -127, 128, seed=65)
    elif case == "n256c16":
        A, b = inputs.uniform(256, 16, -(1 << 23), 1 << 23, seed=256)
    elif case == "n256c64":
        A, b = inputs.uniform(256, 64, -(1 << 15), 1 << 15, seed=257)
    elif case == "n130c127":
        A, b = inputs.uniform(130, 127, -(1 << 15), 1 << 15, seed=130)
    elif case == "hilbert12c1400":  # 16800 components whose denominators differ
        A = inputs.scaled_hilbert(12)
        b = np.random.default_rng(12).integers(-(1 << 20), 1 << 20, size=(12, 1400), dtype=np.int64)
    elif case == "diag7":  # component 7 alone carries the denominator 7
        A = np.diag([1] * 7 + [7] + [1] * 8).astype(np.int64)
        A[0, 1:] = 3
        b = np.ones((16, 1), dtype=np.int64)
    else:
        A, b = inputs.workload("n256_c1_24bit", seed=0)
    dev_s = api.solve_canonical(A, b)
    host_s = api.solve_canonical(A, b, host_recon=True)
    assert (dev_s.N, dev_s.d) == (host_s.N, host_s.d)
    if A.shape[0] <= 64:
        assert (dev_s.N, dev_s.d) == exact.solve(A.tolist(), b.tolist())
