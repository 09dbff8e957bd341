"""block_scaled_bit_gb300 -- fused dequantize-and-multiply small-M GEMV for one GB300 (sm_103a).

    y[M, N] = A[M, K] . deq(W)[N, K]^T,   M = 1..32

The compute path is the C-ABI CUDA library ``libbsgemv.so`` (declared in ``include/bsgemv.h``);
``block_scaled_bit_gb300.bsgemv`` is a thin ctypes binding to it (argument marshalling only) and
``block_scaled_bit_gb300.synth`` draws seeded synthetic inputs.  Importing this package loads
nothing; the library is loaded on first use of ``bsgemv`` and fails loudly if it is missing.
"""
__all__ = ["bsgemv", "synth"]
