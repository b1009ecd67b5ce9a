"""CPU oracle for ring AllReduce: TEST INFRASTRUCTURE, not part of the product.

Only the test suite (``tests/``), ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import anything from this
package.  The CUDA library never calls it, and this package imports nothing
from the CUDA library: the two share no code.  The only module both sides
use is the seeded input generator, which holds none of the method's
arithmetic.

What is here, and what each part follows (citations name the web page by its
title and the section on it):

* ``elementops`` -- the reduction ``(+)`` applied when a chunk arrives:
  ``incoming (+) local`` for fp32 / bf16 / int32 with SUM or MAX.  Follows
  "Why AllReduce = ReduceScatter + AllGather -- NCCL Ring AllReduce" (page
  on the NCCL ring), sections 1 and 7 (partial_sum + local_chunk).
* ``ring`` -- the ring itself, simulated rank by rank and round by round
  (sections 4-6 of that page), with the NCCL primitive sequence of its
  section 8 (its restatement of Table V of "Demystifying NCCL") recorded as
  a trace and the bytes each rank sends counted (section 13).
* ``barrier`` -- a host-thread simulation of the counting barrier of
  "comm: lift the GIN scale-out ceiling by making the rail barrier a
  counting barrier" (section "Fix"), used to state what the GPU's signal
  slots must hold after a call.

Every function is pinned by ``tests/test_oracle_*.py`` to facts that do not
come from the oracle itself (the pages' worked example, closed forms,
brute-force folds through independent arithmetic, error bounds).  Nothing
here is "parity unpinned".
"""

from . import elementops, ring, barrier  # noqa: F401
