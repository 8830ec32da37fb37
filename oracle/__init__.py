"""fp64 CPU oracle for the Muon step (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The CUDA library and its Python
binding never import it; the two share no code.

Parity status: every function in ``muon_ref`` is pinned by ``tests/test_oracle.py``
(closed forms, invariants, a hand-written Jacobi SVD, brute force on tiny inputs);
no function is "parity unpinned".
"""
from .muon_ref import *  # noqa: F401,F403
