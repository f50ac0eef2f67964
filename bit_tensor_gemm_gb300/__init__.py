"""bit_tensor_gemm_gb300 -- low-bit integer GEMM (8-, 4- and 1-bit) for GB300.

The compute path is the CUDA library ``lib/liblbgemm.so`` (C ABI in
``include/lbgemm.h``), built in-tree by ``build.build()``; ``lbgemm`` is its
Python binding and ``synth`` draws seeded synthetic operands.
"""
__all__ = ["build", "lbgemm", "synth"]
