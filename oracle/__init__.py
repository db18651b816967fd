"""Float64 CPU oracle for the CSA / HCA forward path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only code that may import it.  It
shares no code with the CUDA path (``compressed_sparse_long_05_b300``), and the
CUDA path never imports it.
"""

from . import csa_oracle, pipeline  # noqa: F401
