"""CPU oracle for the exact rational solver -- TEST INFRASTRUCTURE ONLY.

Nothing in the product path may import, call or link anything here: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code, tables
or constants with the CUDA library.

Modules
  exact        -- the definition: x = A^{-1} b over Q, by fraction-free Bareiss
                  elimination and fraction-free back-substitution, returned in
                  canonical form (N, d): d the least positive common
                  denominator, N = d x.  (exact-solve card, §API and
                  §Correctness: the solution is compared bitwise against an
                  exact Gaussian-elimination oracle.)
  dixon_model  -- the method written out step by step with Python ints
                  (exact-solve card, §Method): balanced residues, inverse mod
                  each prime by Gauss-Jordan on the augmented matrix, the
                  Hadamard stop rule, the lift digits and residuals, the
                  balanced CRT digit, rational reconstruction.  Used to check
                  each CUDA stage's intermediates, which are unique.

Every function is pinned by ``tests/test_oracle_pins.py`` against closed
forms, brute force and invariants (no function is "parity unpinned").
"""
