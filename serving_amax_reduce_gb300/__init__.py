"""GB300-native quantized linear layers (sm_103a).

``serving_amax_reduce_gb300.qlin`` is the thin ctypes binding over the C-ABI
library ``libqlin.so`` (built from ``csrc/``); ``inputs`` holds the seeded
synthetic workloads.  Importing the package loads nothing: the CUDA library
is loaded on first use of ``qlin`` and raises if it is missing.
"""
