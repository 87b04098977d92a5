"""FORGE tile-fused weight-gradient + optimizer step for GB300 (sm_103a).

The compute path is a C-ABI shared library of hand-written CUDA kernels
(``include/forge.h``); this package holds its sources (``csrc/``), the build step
(``build.py``), a thin ctypes binding (``api.py``) and seeded synthetic inputs
(``inputs.py``).  Importing the package does not load the library; the first
call into ``api`` does, and raises if it has not been built.
"""

__version__ = "0.1.0"
