"""CPU oracle for the Ulysses QKV front end (test infrastructure).

A plain, slow, float64 restatement of what the method computes, written from
the pages' definitions.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import it.  The product path (the CUDA library and its
binding) never imports, calls or links anything here, and the two share no
code: the only common module is the seeded input generator, which holds none
of the method's arithmetic.

Every function is pinned by `tests/test_oracle_pins.py` and
`tests/test_oracle_sage2_pins.py` to facts fixed outside the oracle itself
(closed forms, invariants, brute force on tiny inputs and the hand-written
fixtures under `tests/golden/`).  `pages_mode.py` is a diagnostic, not a parity
reference: the pages' own fp32 test-reference form, pinned by
`tests/test_oracle_pages_mode_pins.py`.  No function is "parity unpinned".
"""
from .qnre_oracle import *  # noqa: F401,F403
from .sage2_oracle import *  # noqa: F401,F403
