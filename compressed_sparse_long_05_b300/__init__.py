"""B300 (sm_103a) kernels for the DeepSeek-V4 CSA / HCA attention forward.

The stages are C-ABI calls into ``lib/libcsa_b300.so`` (include/csa.h):
``csa_compress``, ``csa_index``, ``csa_topk``, ``csa_attend``, ``hca_attend``.
``path`` composes them into the prefill and decode passes of one layer.
"""

from ._lib import (BlockPool, CsaError, DecodeStepHost, Paged, attend_workspace_size,  # noqa: F401
                   csa_attend,
                   csa_attend_noalloc, csa_compress, csa_grouped_proj,
                   csa_index, csa_index_topk, csa_topk, device_error, hca_attend, lib)
from . import path  # noqa: F401
