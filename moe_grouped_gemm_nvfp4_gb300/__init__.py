"""NVFP4 block-scaled GEMM and MoE grouped GEMM for GB300 (sm_103a)."""
