"""ctypes loader and prototypes for ``libw8a8_gb300.so`` (include/w8a8.h).

The library is built in-tree on first use if it is missing or older than its
sources.  There is no fallback: if the shared library cannot be built or
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

E4M3, INT8, BF16, FP16, FP32, INT32 = 0, 1, 2, 3, 4, 5
PER_TENSOR, PER_ROW = 0, 1
DYNAMIC, STATIC = 0, 1
REDUCE_AUTO, REDUCE_GLOBAL, REDUCE_CLUSTER = 0, 1, 2
ROUTES = {"auto": 0, "one_kernel": 1, "two_step": 2}

STATUS_NAMES = {
    0: "W8A8_OK",
    1: "W8A8_ERR_INVALID_ARG",
    2: "W8A8_ERR_UNSUPPORTED",
    3: "W8A8_ERR_MISALIGNED",
    4: "W8A8_ERR_WORKSPACE",
    5: "W8A8_ERR_CUDA",
    6: "W8A8_ERR_NO_DEVICE",
}

# Every symbol include/w8a8.h declares.
EXPORTS = (
    "w8a8_last_error",
    "w8a8_version",
    "w8a8_scaled_quant_workspace_size",
    "w8a8_scaled_quant",
    "w8a8_scaled_dequant",
    "w8a8_scaled_mm_workspace_size",
    "w8a8_scaled_mm",
    "w8a8_scaled_mm_pick_config",
    "w8a8_scaled_mm_config_workspace_size",
    "w8a8_scaled_mm_with_config",
    "w8a8_device_status",
    "w8a8_expand_shard_scales",
    "w8a8_requant_shards",
    "w8a8_scaled_mm_noalloc_max_scratch",
    "w8a8_scaled_mm_noalloc",
    "w8a8_debug_mm_trace",
    "w8a8_quant_scaled_mm_workspace_size",
    "w8a8_quant_scaled_mm",
    "w8a8_fp8_kv_attention_workspace_size",
    "w8a8_fp8_kv_decode_attention",
)


class MmConfig(ctypes.Structure):
    _fields_ = [("swap_ab", ctypes.c_int), ("block_n", ctypes.c_int),
                ("split_k", ctypes.c_int), ("stages", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("reduce", ctypes.c_int), ("cta_pair", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class W8A8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_needed: bool = True):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if build_if_needed else _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not found at {path}")
        lib = ctypes.CDLL(path)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.w8a8_last_error.restype = ctypes.c_char_p
        lib.w8a8_last_error.argtypes = []
        lib.w8a8_version.restype = I
        lib.w8a8_version.argtypes = []
        lib.w8a8_scaled_quant_workspace_size.restype = SZ
        lib.w8a8_scaled_quant_workspace_size.argtypes = [I64, I64, I, I]
        lib.w8a8_scaled_quant.restype = I
        lib.w8a8_scaled_quant.argtypes = [P, I, I64, I64, I64, P, I, I64, P, I, I, P, SZ, P]
        lib.w8a8_scaled_dequant.restype = I
        lib.w8a8_scaled_dequant.argtypes = [P, I, I64, I64, I64, P, I, P, I, I64, P]
        lib.w8a8_scaled_mm_workspace_size.restype = SZ
        lib.w8a8_scaled_mm_workspace_size.argtypes = [I64, I64, I64, I]
        lib.w8a8_scaled_mm.restype = I
        lib.w8a8_scaled_mm.argtypes = [P, I64, P, I64, P, I, P, I, P, I64, I64, I64, I64, I, I, P, SZ, P]
        lib.w8a8_scaled_mm_pick_config.restype = I
        lib.w8a8_scaled_mm_pick_config.argtypes = [I64, I64, I64, I, ctypes.POINTER(MmConfig)]
        lib.w8a8_scaled_mm_config_workspace_size.restype = SZ
        lib.w8a8_scaled_mm_config_workspace_size.argtypes = [I64, I64, I64, I, ctypes.POINTER(MmConfig)]
        lib.w8a8_scaled_mm_with_config.restype = I
        lib.w8a8_scaled_mm_with_config.argtypes = [P, I64, P, I64, P, I, P, I, P, I64, I64, I64, I64, I, I,
                                                   P, SZ, ctypes.POINTER(MmConfig), P]
        lib.w8a8_expand_shard_scales.restype = I
        lib.w8a8_expand_shard_scales.argtypes = [P, P, I, P, P]
        lib.w8a8_requant_shards.restype = I
        lib.w8a8_requant_shards.argtypes = [P, I, I64, I64, P, P, I, P, I64, P, P]
        lib.w8a8_scaled_mm_noalloc_max_scratch.restype = SZ
        lib.w8a8_scaled_mm_noalloc_max_scratch.argtypes = []
        lib.w8a8_scaled_mm_noalloc.restype = I
        lib.w8a8_scaled_mm_noalloc.argtypes = [P, I64, P, I64, P, I, P, I, P, I64, I64, I64, I64, I, I, P]
        lib.w8a8_debug_mm_trace.restype = I
        lib.w8a8_debug_mm_trace.argtypes = [P, SZ]
        lib.w8a8_quant_scaled_mm_workspace_size.restype = SZ
        lib.w8a8_quant_scaled_mm_workspace_size.argtypes = [I64, I64, I64, I]
        lib.w8a8_quant_scaled_mm.restype = I
        lib.w8a8_quant_scaled_mm.argtypes = [P, I, I64, P, I64, P, I, P, I64, I64, I64, I64, I, I, P, I, P, SZ, P]
        lib.w8a8_fp8_kv_attention_workspace_size.restype = SZ
        lib.w8a8_fp8_kv_attention_workspace_size.argtypes = [I64, I64, I64]
        lib.w8a8_fp8_kv_decode_attention.restype = I
        lib.w8a8_fp8_kv_decode_attention.argtypes = [P, I, I64, I64, I64, I64, P, P, I64, P, I64, I64, I64,
                                                     P, P, P, ctypes.c_float, P, I, P, SZ, P]
        lib.w8a8_device_status.restype = I
        lib.w8a8_device_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
        _lib = lib
        return lib


def check(status: int) -> None:
    if status != 0:
        msg = load().w8a8_last_error().decode(errors="replace")
        raise W8A8Error(status, msg)
