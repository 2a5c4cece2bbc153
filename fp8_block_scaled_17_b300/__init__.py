"""Block-scaled FP8 (E4M3) quantization and GEMM for NVIDIA B300 (sm_103a).

The compute lives in ``libfp8q.so`` (CUDA, C ABI declared in include/fp8q.h);
``fp8_block_scaled_17_b300.fp8q`` is its thin Python binding.
"""
__all__ = ["fp8q", "workloads"]
