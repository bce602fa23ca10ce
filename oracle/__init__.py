"""fp64 CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  The product path (the CUDA library and its Python binding) never does; it has no
CPU fallback and fails loudly when its compiled library is missing.
"""
from . import attention  # noqa: F401
