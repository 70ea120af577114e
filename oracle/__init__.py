"""Float64 CPU oracle for the NVFP4 skinny-GEMM / MoE decode path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the C-ABI library and its Python binding) never
calls it, and this package never imports the product path: the two share no
code.  Inputs reach it as plain numpy arrays.
"""
from .nvfp4_oracle import *  # noqa: F401,F403
