"""GB300-native (sm_103a) symmetric w8a8 scaled quantiser and scaled matmul.

The compute lives in the CUDA library ``libw8a8_gb300.so`` (C ABI declared in
``include/w8a8.h``); this package is a thin ctypes binding over it.
"""
from ._lib import (BF16, DYNAMIC, E4M3, FP16, FP32, INT8, INT32, PER_ROW, PER_TENSOR, REDUCE_AUTO,
                   REDUCE_CLUSTER, REDUCE_GLOBAL, STATIC, MmConfig, W8A8Error)
from .api import (Workspace, device_status, expand_shard_scales, mm_workspace_size, pick_config,
                  quant_scaled_mm, quant_workspace_size, requant_shards, scaled_dequant, scaled_mm, scaled_quant)

__all__ = [
    "E4M3", "INT8", "BF16", "FP16", "FP32", "INT32", "PER_TENSOR", "PER_ROW", "DYNAMIC", "STATIC",
    "REDUCE_AUTO", "REDUCE_GLOBAL", "REDUCE_CLUSTER",
    "MmConfig", "W8A8Error", "Workspace", "device_status", "mm_workspace_size",
    "pick_config", "quant_workspace_size", "scaled_dequant", "scaled_mm", "scaled_quant",
    "expand_shard_scales", "requant_shards", "quant_scaled_mm",
]
