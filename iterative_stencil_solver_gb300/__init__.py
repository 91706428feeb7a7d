"""libpk: persistent Jacobi 5-point Laplace/Poisson solver for one GB300 (sm_103a).

The compute runs in ``libpk.so`` (hand-written CUDA behind a C ABI declared in
``include/pk.h``); ``iterative_stencil_solver_gb300.pk`` is a thin ctypes
binding with the same names.  Importing the package does not load the
library; importing ``.pk`` does, and fails loudly when it is missing.
"""
__version__ = "0.1.0"
