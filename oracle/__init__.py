"""CPU oracle for weight-absorbed MLA decode. TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import anything from this package. The product path (the CUDA
library and its Python binding) never imports, links or executes it, and it
never imports the product path: the two share no code. Only the seeded input
generators in ``workloads`` feed both.

Every function works in float64 and cites the passage of the pages it writes
out. See ``oracle/mla.py``.
"""
from .mla import *  # noqa: F401,F403
