"""GB300-native (sm_103a) calibration-free channel reader for MoE decoding.

The reader replaces the routed-expert gated-MLP step of one decode token:
a ternary-sketch screen of every routed channel, an exact global top-k in
output units, exact BF16 compute for the kept channels and a rank-r recovery
term for the rest.  All of it runs in hand-written CUDA kernels behind the
C ABI declared in ``include/moe_reader.h``; ``calibration_free_sparse_gb300.reader``
is the thin ctypes binding.  Importing this package does not load the CUDA
library; the binding loads it on first use and raises if it is missing.
"""

__all__ = ["reader", "synthetic"]
