"""Python face of the exact solver: the card's ``solve(A, b)`` and the stage
entry points, all running through the C ABI of ``include/es.h``.

exact-solve card, §API: ``solve(A, b)`` returns the exact rational solution
of A x = b as ``[n][c]`` nested lists of ``fractions.Fraction``, or ``None``
when A is singular over the rationals.  This module only marshals
arguments; every step of the computation runs in the CUDA library (there is
no CPU fallback: a missing library or GPU raises).
"""

from __future__ import annotations

import ctypes
from fractions import Fraction
from typing import List, Optional, Tuple

import numpy as np

from . import _lib as L


class ExactSolveError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = L.load()
        text = lib.es_status_string(status).decode()
        detail = lib.es_last_error().decode()
        super().__init__(f"{where}: {L.STATUS.get(status, status)} ({text}){': ' + detail if detail else ''}")
        self.status = status


def _check(st: int, where: str):
    if st not in (L.ES_OK,):
        raise ExactSolveError(st, where)


class Solution:
    """Canonical exact solution x = N / d (d > 0 least, gcd(d, N) = 1).

    Holds the exported little-endian two's complement limbs ([n*c, limbs]
    numerators, [limbs] denominator); Python ints are built on first access
    of ``N`` or ``d``."""

    def __init__(self, num, den, n, c, m=0, primes_used=0, phase_ms=None, launches=0, top_launches=0, top_ms=0.0,
                 top_bytes_per_launch=0.0, top_kernel=""):
        self.num_limbs = num
        self.den_limbs = den
        self.n, self.c = n, c
        self.limbs = int(den.shape[0])
        self.m = m
        self.primes_used = primes_used
        self.phase_ms = list(phase_ms or [])
        self.launches = launches              # device kernels launched by the solve
        self.top_kernel = top_kernel          # the lift's dominant kernel (fused lift or per-step product)
        self.top_launches = top_launches      # its launches
        self.top_ms = top_ms                  # their summed CUDA-event time (timing=2 only)
        self.top_bytes_per_launch = top_bytes_per_launch
        self.inverse_split = False            # the inverse ran on two SM partitions (green contexts)
        self._N = None
        self._d = None

    @property
    def N(self) -> List[List[int]]:
        if self._N is None:
            flat = _limbs_to_ints(self.num_limbs, self.n * self.c, self.limbs, True)
            self._N = [flat[i * self.c:(i + 1) * self.c] for i in range(self.n)]
        return self._N

    @property
    def d(self) -> int:
        if self._d is None:
            self._d = _limbs_to_ints(self.den_limbs, 1, self.limbs, False)[0]
        return self._d

    def fractions(self) -> List[List[Fraction]]:
        return [[Fraction(v, self.d) for v in row] for row in self.N]


def _opts(stream=None, threads=0, timing=False, fault=None, max_device_bytes=0, host_recon=False,
          step_lift=False, one_stream=False):
    o = L.es_options()
    o.flags = ((L.FLAG_HOST_RECON if host_recon else 0) | (L.FLAG_STEP_LIFT if step_lift else 0)
               | (L.FLAG_ONE_STREAM if one_stream else 0))
    o.stream = ctypes.c_void_p(stream) if stream else None
    o.max_device_bytes = max_device_bytes
    o.fault_stage = L.FAULT[fault] if isinstance(fault, str) else int(fault or 0)
    o.threads = threads
    o.timing = int(timing) if not isinstance(timing, bool) else (1 if timing else 0)
    return o


def _limbs_to_ints(buf: np.ndarray, count: int, W: int, signed: bool) -> List[int]:
    raw = buf.view(np.uint8).tobytes()
    step = 8 * W
    return [int.from_bytes(raw[i * step:(i + 1) * step], "little", signed=signed) for i in range(count)]


class _Owner:
    """Holds an es_solution until the last array viewing its limbs is gone."""

    def __init__(self, lib, ptr):
        self._lib, self._ptr = lib, ptr

    def __del__(self):
        if self._ptr:
            self._lib.es_solution_free(self._ptr)
            self._ptr = None


class _View:
    """Array interface over limbs owned by an es_solution (no copy)."""

    def __init__(self, owner: _Owner, addr: int, count: int):
        self._owner = owner
        self.__array_interface__ = {"shape": (count,), "typestr": "<u8", "data": (addr, True), "version": 3}


def _take_solution(ptr: ctypes.c_void_p) -> Solution:
    lib = L.load()
    n, c, W = L.c_i64(), L.c_i64(), L.c_i64()
    _check(lib.es_solution_shape(ptr, ctypes.byref(n), ctypes.byref(c), ctypes.byref(W)), "es_solution_shape")
    n, c, W = n.value, c.value, W.value
    pn, pd = ctypes.c_void_p(), ctypes.c_void_p()
    _check(lib.es_solution_data(ptr, ctypes.byref(pn), ctypes.byref(pd)), "es_solution_data")
    owner = _Owner(lib, ptr)  # frees the solution with the last view (read-only arrays)
    num = np.asarray(_View(owner, pn.value or 0, n * c * W)) if n * c * W else np.zeros(0, np.uint64)
    den = np.asarray(_View(owner, pd.value or 0, W)) if W else np.zeros(0, np.uint64)
    ms = (ctypes.c_double * L.NUM_PHASES)()
    m, pu = L.c_i32(), L.c_i32()
    _check(lib.es_solution_phase_ms(ptr, ms, ctypes.byref(m), ctypes.byref(pu)), "es_solution_phase_ms")
    la, tl, tms, tb = L.c_i64(), L.c_i64(), ctypes.c_double(), ctypes.c_double()
    _check(lib.es_solution_kernels(ptr, ctypes.byref(la), ctypes.byref(tl), ctypes.byref(tms), ctypes.byref(tb)),
           "es_solution_kernels")
    top = (lib.es_solution_top_kernel(ptr) or b"").decode()
    split = bool(lib.es_solution_inverse_split(ptr))
    sol = Solution(num, den, n, c, m.value, pu.value, list(ms), la.value, tl.value, tms.value, tb.value, top)
    sol.inverse_split = split
    return sol


def _as_host_i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    a = np.asarray(x)
    if a.dtype != np.int64:
        if not np.issubdtype(a.dtype, np.integer) and a.dtype != object:
            raise TypeError("A and b must be integer arrays")
        a = a.astype(np.int64)
    return np.ascontiguousarray(a)


def solve_canonical(A, b, *, threads: int = 0, timing: bool = False, fault=None,
                    max_device_bytes: int = 0, host_recon: bool = False, step_lift: bool = False,
                    one_stream: bool = False) -> Optional[Solution]:
    """Exact solution of A x = b from host arrays (es_solve), or None if singular."""
    lib = L.load()
    A = _as_host_i64(A)
    b = _as_host_i64(b)
    if b.ndim == 1:
        b = b.reshape(-1, 1)
    if A.ndim != 2 or A.shape[0] != A.shape[1] or b.shape[0] != A.shape[0]:
        raise ValueError("A must be [n, n] and b [n, c]")
    out = ctypes.c_void_p()
    o = _opts(None, threads, timing, fault, max_device_bytes, host_recon, step_lift, one_stream)
    st = lib.es_solve(A.ctypes.data, b.ctypes.data, A.shape[0], b.shape[1], ctypes.byref(o), ctypes.byref(out))
    if st == L.ES_SINGULAR:
        return None
    _check(st, "es_solve")
    return _take_solution(out)


def solve(A, b, **kw) -> Optional[List[List[Fraction]]]:
    """The card's solve(A, b): [n][c] nested lists of Fraction, or None."""
    s = solve_canonical(A, b, **kw)
    return None if s is None else s.fractions()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def solve_device(A_t, b_t, *, stream=None, threads: int = 0, timing: bool = False, fault=None,
                 max_device_bytes: int = 0, host_recon: bool = False, step_lift: bool = False,
                 one_stream: bool = False) -> Optional[Solution]:
    """Exact solution with A, b already on the GPU (int64 CUDA tensors), es_solve_device."""
    lib = L.load()
    if b_t.dim() == 1:
        b_t = b_t.reshape(-1, 1)
    A_t = A_t.contiguous()
    b_t = b_t.contiguous()
    out = ctypes.c_void_p()
    o = _opts(_stream_handle(stream), threads, timing, fault, max_device_bytes, host_recon, step_lift, one_stream)
    st = lib.es_solve_device(A_t.data_ptr(), b_t.data_ptr(), A_t.shape[0], b_t.shape[1], ctypes.byref(o),
                             ctypes.byref(out))
    if st == L.ES_SINGULAR:
        return None
    _check(st, "es_solve_device")
    return _take_solution(out)


def residues_device(x_t, stream=None):
    """int8 [53, count] balanced residues of an int64 CUDA tensor (es_residues_device)."""
    import torch
    lib = L.load()
    x_t = x_t.contiguous().reshape(-1)
    out = torch.empty((L.NUM_PRIMES, x_t.numel()), dtype=torch.int8, device=x_t.device)
    _check(lib.es_residues_device(x_t.data_ptr(), x_t.numel(), out.data_ptr(), _stream_handle(stream)),
           "es_residues_device")
    return out


def padded_ld(n: int) -> int:
    return (n + 15) // 16 * 16


def inverse_mod_device(A_t, stream=None) -> Tuple[object, object]:
    """(B [53, n, ld] int8, good [53] uint8) = A^{-1} mod q_j (es_inverse_mod_device)."""
    import torch
    lib = L.load()
    A_t = A_t.contiguous()
    n = A_t.shape[0]
    B = torch.empty((L.NUM_PRIMES, n, padded_ld(n)), dtype=torch.int8, device=A_t.device)
    good = torch.empty(L.NUM_PRIMES, dtype=torch.uint8, device=A_t.device)
    _check(lib.es_inverse_mod_device(A_t.data_ptr(), n, B.data_ptr(), good.data_ptr(), _stream_handle(stream)),
           "es_inverse_mod_device")
    return B, good


def plan_device(A_t, b_t, good, stream=None) -> Tuple[int, int, int]:
    """(num_bits, den_bits, m) the solve would use (es_plan_device)."""
    lib = L.load()
    if b_t.dim() == 1:
        b_t = b_t.reshape(-1, 1)
    g = np.ascontiguousarray(np.asarray(good.cpu() if hasattr(good, "cpu") else good, dtype=np.uint8))
    nb, db, m = L.c_i64(), L.c_i64(), L.c_i32()
    _check(lib.es_plan_device(A_t.contiguous().data_ptr(), b_t.contiguous().data_ptr(), A_t.shape[0], b_t.shape[1],
                              g.ctypes.data, ctypes.byref(nb), ctypes.byref(db), ctypes.byref(m),
                              _stream_handle(stream)), "es_plan_device")
    return nb.value, db.value, m.value


def lift_device(A_t, b_t, B_t, good, m: int, stream=None):
    """digits uint64 [m, n*c, 6] as an int64 CUDA tensor (es_lift_device)."""
    import torch
    lib = L.load()
    if b_t.dim() == 1:
        b_t = b_t.reshape(-1, 1)
    n, c = A_t.shape[0], b_t.shape[1]
    g = np.ascontiguousarray(np.asarray(good.cpu() if hasattr(good, "cpu") else good, dtype=np.uint8))
    D = torch.empty((m, n * c, L.DIGIT_LIMBS), dtype=torch.int64, device=A_t.device)
    _check(lib.es_lift_device(A_t.contiguous().data_ptr(), b_t.contiguous().data_ptr(), n, c, B_t.data_ptr(),
                              g.ctypes.data, m, D.data_ptr(), _stream_handle(stream)), "es_lift_device")
    return D


def digits_to_ints(D) -> np.ndarray:
    """Digits tensor/array [m, nc, 6] -> object array [m, nc] of Python ints (signed)."""
    a = D.cpu().numpy() if hasattr(D, "cpu") else np.asarray(D)
    a = np.ascontiguousarray(a).view(np.uint64)
    m, nc, _ = a.shape
    flat = _limbs_to_ints(a.reshape(-1), m * nc, L.DIGIT_LIMBS, True)
    out = np.empty((m, nc), dtype=object)
    for i in range(m):
        out[i, :] = flat[i * nc:(i + 1) * nc]
    return out


def reconstruct(digits, n: int, c: int, m: int, good, num_bits: int, den_bits: int, *, threads: int = 0,
                fault=None) -> Solution:
    """Host rational reconstruction from digits [m, n*c, 6] (es_reconstruct)."""
    lib = L.load()
    d = digits.cpu().numpy() if hasattr(digits, "cpu") else np.asarray(digits)
    d = np.ascontiguousarray(d).view(np.uint64)
    g = np.ascontiguousarray(np.asarray(good.cpu() if hasattr(good, "cpu") else good, dtype=np.uint8))
    out = ctypes.c_void_p()
    o = _opts(None, threads, False, fault, 0)
    _check(lib.es_reconstruct(d.ctypes.data, n, c, m, g.ctypes.data, num_bits, den_bits, ctypes.byref(o),
                              ctypes.byref(out)), "es_reconstruct")
    return _take_solution(out)


def selftest_bigint(seed: int, rounds: int) -> int:
    """Failed checks of the host big-integer arithmetic (es_selftest_bigint; 0 = pass)."""
    return L.load().es_selftest_bigint(seed, rounds)


def selftest_modular(lo: int, hi: int, samples: int) -> int:
    """Mismatches of the library's Barrett reductions against % (host, no GPU)."""
    return L.load().es_selftest_modular(lo, hi, samples)


def selftest_gj_reduction() -> int:
    """Mismatches of the Gauss-Jordan kernels' f32 residue arithmetic against %
    over every |x| < 2^20 and every prime (host, no GPU; 0 = pass)."""
    return L.load().es_selftest_gj_reduction()
