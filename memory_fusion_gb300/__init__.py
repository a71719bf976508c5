"""GB300-native fused GEMM + row-reduce/broadcast kernels (C-ABI ``libcf``).

Importing the package loads nothing; ``memory_fusion_gb300.cf`` loads the
CUDA library on first use and raises if it is missing.
"""
__version__ = "0.1.0"
