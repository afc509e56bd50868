"""Communication-fused tensor-parallel GEMM for GB300 (sm_103a).

The compiled library is loaded on first use by :mod:`reduce_scatter_gb300.dg`.
"""
