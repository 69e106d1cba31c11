"""GB300 (sm_103a) filtered transformer backward: the hot path of Collider
("Enhancing Token Filtering Efficiency in Large Language Model Training with
Collider", arXiv 2502.00340).

The compute lives in ``libcollider.so`` (CUDA kernels behind a C ABI,
``include/collider.h``); :mod:`sparse_backward_gemm_gb300.collider` is a thin
ctypes binding with the same entry-point names.  Build the library with
``python -m sparse_backward_gemm_gb300.build``.
"""
from .collider import *  # noqa: F401,F403
