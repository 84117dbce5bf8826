"""GEMM with a fused bias/activation epilogue for GB300 (sm_103a).

``libgemmepi.so`` (built from ``csrc/`` by ``build.py``) holds the kernels and the C ABI
declared in ``include/gemm_epi.h``; ``gemm_epi`` is its Python binding; ``workloads`` draws
the seeded synthetic inputs.  Importing the package loads nothing: the library is loaded
on the first call into ``gemm_epi``.
"""
__all__ = ["gemm_epi", "workloads", "build"]
