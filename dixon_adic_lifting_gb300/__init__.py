"""Exact rational solver for integer systems A x = b by Dixon p-adic lifting,
GB300-native (sm_103a).

The compute path is the C-ABI library built from ``csrc/`` (declared in
``include/es.h``); this package is a thin binding over it (``api``) plus the
seeded input generators (``inputs``).  Nothing here computes on the CPU in
place of the library: without the built library or a GPU the calls raise.
"""

from .api import (ExactSolveError, Solution, digits_to_ints, inverse_mod_device, lift_device, padded_ld,
                  plan_device, reconstruct, residues_device, selftest_modular, solve, solve_canonical,
                  solve_device)

__all__ = ["ExactSolveError", "Solution", "solve", "solve_canonical", "solve_device", "residues_device",
           "inverse_mod_device", "plan_device", "lift_device", "reconstruct", "digits_to_ints", "padded_ld",
           "selftest_modular"]
