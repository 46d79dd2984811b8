"""GB300-native dense fp32 row-major matrix multiplication (SGEMM).

The compute path is the CUDA library ``libsgemm_gb300.so`` built from
``csrc/`` for sm_103a; :mod:`dense_fp32_matrix_major_gb300.sgemm` is its thin
ctypes binding. Importing the binding fails loudly when the library is
missing: there is no CPU fallback.
"""

__all__ = ["sgemm", "workloads"]
