"""GB300 decode-step weight stream: NVFP4 / MXFP4 / FP8 weight-streaming
products against BF16 activations, behind the C ABI of include/bws.h.

This module only marshals arguments: every step runs in libbws.so's CUDA
kernels. PyTorch provides device memory and the current stream. There is no
CPU fallback; a missing library or a CPU tensor raises.
"""
from ._lib import lib, BwsError, LIB_PATH  # noqa: F401
from .api import (  # noqa: F401
    nvfp4_quantize,
    mxfp4_quantize,
    fp8_rowwise_quantize,
    gemv_workspace_size,
    nvfp4_gemv,
    nvfp4_prepare,
    nvfp4_gemv_prepared,
    nvfp4_gate_up_silu,
    fp8_lmhead_gemv,
    fp8_lmhead_argmax,
    moe_router_topk,
    mxfp8_quantize,
    mxfp4_w4a8_gemv,
    status_word,
    hbm_read_probe,
    l2_flush,
    Workspace,
    MoeLayer,
    MoeWeights,
    mxfp4_moe_workspace_size,
    mxfp4_moe_gemv,
    mxfp4_moe_inspect,
)

from . import stack, workloads  # noqa: F401,E402

BWS_STATUS_X_TWO_BANDS = 1
BWS_STATUS_X_FLUSHED = 2
BWS_STATUS_X_ROUNDED = 8
