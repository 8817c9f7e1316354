"""CPU oracle for NVFP4 quantisation, block-scaled GEMM and MoE grouped GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only the tests, the package-level smoke check and the
CPU-baseline leg of the benchmark use it.  It shares no code, tables or
constants with the CUDA library; the two meet only on the seeded inputs of
`moe_grouped_gemm_nvfp4_gb300.inputs`.

Every function is a plain, slow restatement of what the method computes,
in FP64 where the arithmetic is floating point (FP32 where the quantiser's
decisions are defined in FP32).  `sparse_ref` adds 2:4-sparse weights
(pruning, the compressed form and its tile layout); `attention_ref` decode
attention over an NVFP4 KV cache.

Parity unpinned: the accumulation order inside the tensor-core block-scaled
MMA and the FP32 summation order of the scatter-combine are not modelled;
the GEMM tolerances cover both.
"""
from .nvfp4_ref import *  # noqa: F401,F403
from .nvfp4_ref import __all__ as _dense_all
from .sparse_ref import *  # noqa: F401,F403
from .sparse_ref import __all__ as _sparse_all
from .attention_ref import *  # noqa: F401,F403
from .attention_ref import __all__ as _attention_all

__all__ = list(_dense_all) + list(_sparse_all) + list(_attention_all)
