"""gbattn: fused multi-head attention forward and backward for GB300 (sm_103a).

The computation lives in libgbattn.so (hand-written CUDA, C ABI in
include/gbattn.h and include/gbln.h); this package is its thin PyTorch binding.
"""

from .attention import (BlockMask, Fp8Operands, SeqLens, attn_bwd, attn_fwd, attn_fwd_fp8, get_status, make_params,
                        quantize_fp8)
from .layernorm import layernorm_residual

__all__ = ["attn_fwd", "attn_bwd", "BlockMask", "SeqLens", "get_status", "make_params", "layernorm_residual",
           "quantize_fp8", "attn_fwd_fp8", "Fp8Operands"]
