"""Block-scaled FP4 (NVFP4 / MXFP4) linear and fused-MoE layers for GB300
(sm_103a): hand-written CUDA kernels behind the C-ABI library libfp4.so.

The binding (``mxfp4_block_scaled_gb300.fp4``) loads the in-tree library on
first use and raises if it is missing; there is no fallback path.
"""
__all__ = ["fp4", "inputs"]
