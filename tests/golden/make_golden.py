"""Writes the stored expected values under tests/golden/ from the CPU oracle.

Calls only ``oracle/`` and the seeded input generators; nothing here comes
from the CUDA library.  Run from the repository root:

    python tests/golden/make_golden.py            # all fixtures
    python tests/golden/make_golden.py n32        # one of: n32 pascal n256
"""

import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from dixon_adic_lifting_gb300 import inputs  # noqa: E402
from oracle import dixon_model, exact  # noqa: E402

sys.path.insert(0, os.path.dirname(HERE))
from tests_golden_digest import canonical_digest  # noqa: E402


def n32_attempts(seeds=range(5)):
    """For each seed, the first redraw whose A is invertible modulo every odd
    prime below 256 (the n=32 workload's acceptance rule)."""
    out = {}
    for s in seeds:
        t = 0
        while True:
            A, _ = inputs.workload("n32_c1_int8", seed=s, attempt=t)
            A = A.tolist()
            if all(dixon_model.inverse_mod(A, q) is not None for q in dixon_model.PRIMES):
                out[str(s)] = t
                break
            t += 1
    return out


def solved(name, seed, A, b):
    t0 = time.time()
    r = exact.solve(A.tolist(), b.tolist())
    dt = time.time() - t0
    if r is None:
        return {"workload": name, "seed": seed, "singular": True, "oracle_seconds": round(dt, 2)}
    N, d = r
    return {
        "workload": name,
        "seed": seed,
        "singular": False,
        "oracle_seconds": round(dt, 2),
        "digest": canonical_digest(N, d),
        "d": str(d),
        "d_bits": d.bit_length(),
        "N_head": [str(N[i][0]) for i in range(min(3, len(N)))],
        "N_max_bits": max(abs(v).bit_length() for row in N for v in row),
    }


def main(which):
    if "n32" in which:
        with open(os.path.join(HERE, "n32_attempts.json"), "w") as f:
            json.dump({"_about": "accepted redraw index per seed for the n=32 workload "
                                 "(A invertible modulo all 53 odd primes < 256); written by make_golden.py",
                       "attempts": n32_attempts()}, f, indent=1)
    if "pascal" in which:
        A, b = inputs.workload("pascal30", seed=0)
        N, d = exact.solve(A.tolist(), b.tolist())
        with open(os.path.join(HERE, "pascal30_seed0.json"), "w") as f:
            json.dump({"_about": "oracle solution of the order-30 Pascal system, seed 0; written by make_golden.py",
                       "d": d, "N": [str(row[0]) for row in N]}, f, indent=1)
    if "n256" in which:
        A, b = inputs.workload("n256_c1_24bit", seed=0)
        rec = {"_about": "oracle results for the n=256, c=1 workload, seed 0, and its rank-255 variant; "
                         "written by make_golden.py",
               "regular": solved("n256_c1_24bit", 0, A, b),
               "rank_deficient": solved("n256_c1_24bit/rank255", 0, inputs.make_rank_deficient(A, seed=0), b)}
        with open(os.path.join(HERE, "n256_seed0.json"), "w") as f:
            json.dump(rec, f, indent=1)


if __name__ == "__main__":
    main(sys.argv[1:] or ["n32", "pascal", "n256"])
