"""The canonical-form digest used by the stored oracle results in tests/golden/."""

import hashlib


def canonical_digest(N, d):
    """sha256 of the canonical text form: d, then one line per row of N."""
    h = hashlib.sha256()
    h.update(f"{d}\n".encode())
    for row in N:
        h.update((",".join(str(v) for v in row) + "\n").encode())
    return h.hexdigest()
