"""GB300 (sm_103a) routed-expert MoE layer over GGUF block-quantized weights.

The product is the CUDA library built from csrc/ with the C ABI declared in
include/moe_gb300.h; `_native` binds it with ctypes under the same names and
`layer.MoeLayer` wraps the fused call for torch-held weights.
"""
from . import _native  # noqa: F401
from ._native import *  # noqa: F401,F403
from .layer import MoeLayer  # noqa: F401
