"""GB300-native (sm_103a) symmetric w8a8 scaled quantiser and scaled matmul,
and decode attention over an fp8 (e4m3) KV cache.

The compute lives in the CUDA library ``libw8a8_gb300.so`` (C ABI declared in
``include/w8a8.h``); this package is a thin ctypes binding over it.
"""
from ._lib import (BF16, DYNAMIC, E4M3, FP16, FP32, INT8, INT32, PER_ROW, PER_TENSOR, REDUCE_AUTO,
                   REDUCE_CLUSTER, REDUCE_GLOBAL, STATIC, MmConfig, W8A8Error)
from .api import (Workspace, attention_workspace_size, device_status, expand_shard_scales,
                  fp8_kv_decode_attention, mm_workspace_size, pick_config, quant_scaled_mm, quant_workspace_size,
                  requant_shards, scaled_dequant, scaled_mm, scaled_quant)

__all__ = [
    "E4M3", "INT8", "BF16", "FP16", "FP32", "INT32", "PER_TENSOR", "PER_ROW", "DYNAMIC", "STATIC",
    "REDUCE_AUTO", "REDUCE_GLOBAL", "REDUCE_CLUSTER",
    "MmConfig", "W8A8Error", "Workspace", "device_status", "mm_workspace_size",
    "pick_config", "quant_workspace_size", "scaled_dequant", "scaled_mm", "scaled_quant",
    "expand_shard_scales", "requant_shards", "quant_scaled_mm", "fp8_kv_decode_attention",
    "attention_workspace_size",
]
