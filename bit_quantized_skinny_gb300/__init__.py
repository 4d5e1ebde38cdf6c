"""Skinny-batch Q4K x bf16 matrix products on one GB300 (sm_103a).

The compute path is the CUDA library ``libqmm.so`` built from ``csrc/``; ``qmm`` is its thin
ctypes binding (argument marshalling only).  Importing this package loads nothing; the
library is loaded on first use of ``bit_quantized_skinny_gb300.qmm``.
"""
__all__ = ["qmm", "inputs"]
