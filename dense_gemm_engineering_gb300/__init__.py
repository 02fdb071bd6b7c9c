"""GB300 (sm_103a) dense GEMM: D = A.Bt and D = A.B, FP16/BF16 in, FP32 accumulate.

The compute path is the CUDA library built from ``csrc/`` (C ABI declared in
``include/gemm.h``); ``binding`` marshals arguments to it with ctypes.
"""
