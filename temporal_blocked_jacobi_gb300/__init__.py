"""GB300 (sm_103a) five-point Jacobi solver for implicit 2-D diffusion.

The compute path is the C-ABI library built from csrc/ (declared in
include/jacobi.h); `temporal_blocked_jacobi_gb300.jacobi` is its thin ctypes
binding. Importing this package does not load the library, so the input
generators in `problem` can be used without a GPU.
"""

__all__ = ["problem", "jacobi"]
