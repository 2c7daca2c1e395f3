"""GB300-native single-GPU DeepSeek-V3-style MoE layer: a C-ABI CUDA library
(libmoe.so, include/moe.h) and its Python binding."""
from . import _abi
from ._abi import (MOE_BF16, MOE_MXFP8, MoeConfig, MoeError, MoeGrads, MoeWeights, make_config, make_grads,
                   make_weights, moe_backward, moe_forward, moe_mxfp8_weights_size, moe_quantize_weights_mxfp8,
                   moe_read_device_status, moe_route_topk, moe_route_topk_noalloc, moe_workspace_size)

__all__ = ["MOE_BF16", "MOE_MXFP8", "MoeConfig", "MoeError", "MoeGrads", "MoeWeights", "make_config",
           "make_grads", "make_weights", "moe_backward", "moe_forward", "moe_mxfp8_weights_size",
           "moe_quantize_weights_mxfp8", "moe_read_device_status", "moe_route_topk", "moe_route_topk_noalloc",
           "moe_workspace_size", "_abi"]
