"""KPool-DSA forward for one GB300 (sm_103a): pooled-key indexer and sparse
latent attention behind a three-call C ABI (``include/kpooldsa.h``).

``kpooldsa`` is the ctypes binding; ``build`` compiles the CUDA library in
place; ``workloads`` draws the seeded synthetic inputs.
"""
from . import kpooldsa  # noqa: F401
from .kpooldsa import (KpoolError, KpoolUnavailable, PoolLayout, dsa_index, kpool_build, make_params,  # noqa: F401
                       row_width, sparse_mla_fwd)
