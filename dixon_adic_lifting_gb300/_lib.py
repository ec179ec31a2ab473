"""ctypes declarations of the C ABI in ``include/es.h`` (argument marshalling only)."""

from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(os.path.dirname(_HERE), "include", "es.h")

c_i64 = ctypes.c_int64
c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p
P_i64 = ctypes.POINTER(ctypes.c_int64)
P_u64 = ctypes.POINTER(ctypes.c_uint64)
P_i32 = ctypes.POINTER(ctypes.c_int32)
P_u8 = ctypes.POINTER(ctypes.c_uint8)
P_dbl = ctypes.POINTER(ctypes.c_double)

ES_OK = 0
ES_SINGULAR = 1
STATUS = {0: "ES_OK", 1: "ES_SINGULAR", -1: "ES_ERR_ARG", -2: "ES_ERR_RANGE", -3: "ES_ERR_CUDA",
          -4: "ES_ERR_NOMEM", -5: "ES_ERR_TIMEOUT", -6: "ES_ERR_INTERNAL", -7: "ES_ERR_NODEVICE"}
NUM_PRIMES = 53
DIGIT_LIMBS = 6
NUM_PHASES = 6
FAULT = {"residues": 1, "inverse": 2, "lift": 3, "recon": 4, "nomem": 5, "lift_wait": 6}
FLAG_HOST_RECON = 1
FLAG_STEP_LIFT = 2
FLAG_ONE_STREAM = 4


class es_options(ctypes.Structure):
    _fields_ = [("stream", c_vp), ("max_device_bytes", ctypes.c_size_t), ("fault_stage", c_i32),
                ("threads", c_i32), ("timing", c_i32), ("flags", c_i32)]


_SIGS = {
    "es_solve": (c_i32, [c_vp, c_vp, c_i64, c_i64, ctypes.POINTER(es_options), ctypes.POINTER(c_vp)]),
    "es_solve_device": (c_i32, [c_vp, c_vp, c_i64, c_i64, ctypes.POINTER(es_options), ctypes.POINTER(c_vp)]),
    "es_solution_shape": (c_i32, [c_vp, P_i64, P_i64, P_i64]),
    "es_solution_export": (c_i32, [c_vp, c_vp, c_vp]),
    "es_solution_phase_ms": (c_i32, [c_vp, P_dbl, P_i32, P_i32]),
    "es_solution_kernels": (c_i32, [c_vp, P_i64, P_i64, P_dbl, P_dbl]),
    "es_solution_top_kernel": (ctypes.c_char_p, [c_vp]),
    "es_solution_inverse_split": (c_i32, [c_vp]),
    "es_solution_data": (c_i32, [c_vp, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p)]),
    "es_solution_free": (None, [c_vp]),
    "es_status_string": (ctypes.c_char_p, [c_i32]),
    "es_last_error": (ctypes.c_char_p, []),
    "es_release_workspace": (c_i32, []),
    "es_version": (c_i32, []),
    "es_residues_device": (c_i32, [c_vp, c_i64, c_vp, c_vp]),
    "es_inverse_mod_device": (c_i32, [c_vp, c_i64, c_vp, c_vp, c_vp]),
    "es_inverse_mod_device_noalloc": (c_i32, [c_vp, c_i64, c_vp, c_vp, c_vp]),
    "es_plan_device": (c_i32, [c_vp, c_vp, c_i64, c_i64, c_vp, P_i64, P_i64, P_i32, c_vp]),
    "es_lift_device": (c_i32, [c_vp, c_vp, c_i64, c_i64, c_vp, c_vp, c_i32, c_vp, c_vp]),
    "es_reconstruct": (c_i32, [c_vp, c_i64, c_i64, c_i32, c_vp, c_i64, c_i64, ctypes.POINTER(es_options),
                               ctypes.POINTER(c_vp)]),
    "es_selftest_modular": (c_i64, [c_i64, c_i64, c_i64]),
    "es_selftest_bigint": (c_i64, [ctypes.c_uint64, c_i64]),
    "es_selftest_gj_reduction": (c_i64, []),
}

_lib = None


def header_functions():
    """Names of the functions include/es.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(es_[a-z_0-9]+)\s*\(", text)))


def ensure_built():
    if not _build.up_to_date():
        _build.build()


def load():
    """The loaded library (raises if it was never built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"exact-solve library not built ({_build.LIB}); run build() first")
    lib = ctypes.CDLL(_build.LIB)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
