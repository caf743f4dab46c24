"""dense_tiled_matrix_gb300: the tiled dense matrix multiply C = A x B on GB300.

``libtgemm.so`` (built from ``csrc/`` by ``build.build()``) holds the CUDA
kernels and the C entry points declared in ``include/tgemm.h``; ``tgemm`` is
its Python binding and ``inputs`` the seeded synthetic input generators.
Importing this package loads nothing; the library is loaded on first call.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "tgemm", "build"]
