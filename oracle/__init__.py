"""CPU oracle for TurboQuant_prod attention scores (TEST INFRASTRUCTURE).

Plain, slow, float64 NumPy code that states what the GPU path must compute.
It is used only by ``tests/``, by ``__graft_entry__.smoke()`` and by the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  The product
library never imports, links or calls anything here, and this package never
imports the product.  Both sides take their raw random draws from ``synth``.

Every name this package exports is pinned by a ``-m "not gpu"`` test against
something other than itself: values the pages print, closed forms, special
cases that reduce to a library routine, and brute force on small inputs (see
``tests/test_oracle_pins.py``).  No exported function is "parity unpinned".
"""
from .tq_oracle import *  # noqa: F401,F403
