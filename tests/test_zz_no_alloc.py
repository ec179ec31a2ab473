"""The batched modular inverse that allocates nothing, checked against the
allocating entry point.

Callers that cannot allocate device memory (inside a framework whose
caching allocator holds nearly all of it, or in loops that must not pay
cudaFree's device-wide synchronisation) use es_inverse_mod_device_noalloc,
whose working memory is a fixed array in device memory.  This file is
collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.  It passes alone in a fresh
process and after the others (the array keeps the previous call's contents,
so two calls in a row are compared)."""

import ctypes

import numpy as np
import pytest

from dixon_adic_lifting_gb300 import inputs

pytestmark = pytest.mark.gpu


def _inverse(lib, torch, fn, A):
    n = A.shape[0]
    ld = (n + 15) // 16 * 16
    At = torch.as_tensor(A, dtype=torch.int64, device="cuda")
    B = torch.full((53, n, ld), 77, dtype=torch.int8, device="cuda")
    good = torch.full((53,), 9, dtype=torch.uint8, device="cuda")
    st = fn(ctypes.c_void_p(At.data_ptr()), n, ctypes.c_void_p(B.data_ptr()), ctypes.c_void_p(good.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, B.cpu().numpy(), good.cpu().numpy()


def test_noalloc_inverse_matches_allocating_entry_point(lib):
    import torch

    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    cases = [inputs.uniform(256, 1, -(1 << 23), 1 << 23, seed=71)[0],   # the maximum size
             inputs.uniform(37, 1, -127, 128, seed=72)[0]]               # ragged, smaller: second call
    cases[1][0] *= 15  # 3 and 5 divide det A: those primes are flagged bad in both
    for A in cases:
        st_ref, B_ref, g_ref = _inverse(lib, torch, lib.es_inverse_mod_device, A)
        st, B, g = _inverse(lib, torch, lib.es_inverse_mod_device_noalloc, A)
        assert st_ref == 0 and st == 0
        assert np.array_equal(g, g_ref)
        for j in range(53):
            if g_ref[j]:
                assert np.array_equal(B[j], B_ref[j]), j  # integer result: bit-exact
    assert g[0] == 0 and g[1] == 0


def test_noalloc_accepts_any_int64_entries(lib):
    """Residues of any int64 are exact, so this entry point takes entries far
    beyond the solver's range (n max|A_ij| < 2^63), which the allocating entry
    point rejects; its inverses match the oracle's Gauss-Jordan mod q_j."""
    import torch

    from oracle import dixon_model as dm

    rng = np.random.default_rng(73)
    n = 24
    A = rng.integers(-(1 << 62), 1 << 62, size=(n, n), dtype=np.int64)
    A[0, 0], A[1, 1], A[2, 3] = np.iinfo(np.int64).min, np.iinfo(np.int64).max, -(1 << 62)
    st_ref, _, _ = _inverse(lib, torch, lib.es_inverse_mod_device, A)
    assert st_ref == -2  # ES_ERR_RANGE: outside the solver's range
    for call in range(2):  # two calls in a row through the shared array
        st, B, g = _inverse(lib, torch, lib.es_inverse_mod_device_noalloc, A)
        assert st == 0
        Al = A.tolist()
        for j, q in enumerate(dm.PRIMES):
            Bq = dm.inverse_mod(Al, q)
            assert g[j] == (0 if Bq is None else 1), (call, q)
            if Bq is not None:
                exp = np.array([[dm.bal(v, q) for v in row] for row in Bq], dtype=np.int8)
                assert np.array_equal(B[j][:, :n], exp), (call, q)


def test_noalloc_rejects_sizes_beyond_its_maximum(lib):
    import torch

    A = np.eye(257, dtype=np.int64)
    st, _, _ = _inverse(lib, torch, lib.es_inverse_mod_device_noalloc, A)
    assert st == -2  # ES_ERR_RANGE
    assert b"256" in lib.es_last_error()
