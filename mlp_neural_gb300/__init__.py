"""Fused FP16 MLP inference on GB300 (sm_103a).

The compute path is the C-ABI library ``libnmmlp.so`` (CUDA kernels for
sm_103a, declared in ``include/nm_mlp.h``); ``mlp_neural_gb300.nm`` is its thin
ctypes binding. Importing this package loads nothing: the library is opened
on first use, and a missing library is an error, never a fallback.
"""
