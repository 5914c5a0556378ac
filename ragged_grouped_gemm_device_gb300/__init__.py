"""Device-scheduled ragged grouped GEMM for a SwiGLU mixture-of-experts expert layer on GB300.

The compute lives in a C-ABI shared library of hand-written sm_103a CUDA kernels
(``libmoe_gg.so``, declared in ``include/moe_gg.h``); ``_lib`` is its thin ctypes binding and
``layer`` strings the calls together for one expert layer.
"""
