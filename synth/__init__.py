"""Seeded synthetic workloads for the CSA / HCA forward path.

Shared by the tests, the benchmark and the oracle checks.  It holds only sizes
(``configs``) and seeded random tensors plus the storage-format encoders that
turn them into the bytes a kernel reads (``generate``): none of the method's
arithmetic.
"""

from . import configs, generate  # noqa: F401
from .configs import get, scaled  # noqa: F401
from .generate import make_inputs  # noqa: F401
