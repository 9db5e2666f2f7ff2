"""Batch-invariant transformer reductions for one GB300 (sm_103a).

The compute lives in ``libbi.so`` (CUDA kernels behind a C ABI, see ``include/bi.h``);
this package is its thin ctypes binding.  The shared library is loaded on first use.
"""
