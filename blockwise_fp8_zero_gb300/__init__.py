"""Block-aware ZeRO-1 optimizer step for blockwise-FP8 weights on GB300.

The compute path is libfp8z.so (hand-written sm_103a CUDA, C ABI in
include/fp8z.h); ``fp8z`` is its thin ctypes binding and ``workloads`` the
seeded synthetic input generators.  Importing the package loads nothing.
"""
