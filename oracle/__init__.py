"""CPU oracle for the w8a8 scaled quantiser and scaled matmul.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
the CPU-baseline leg of the benchmark may import this module.  The product
library never does: it shares no code, table or constant with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain C, one IEEE operation per step,
built with ``-fno-fast-math -ffp-contract=off``); this module builds it with
gcc on first use and marshals numpy arrays.  The semantics it follows, and the
reading taken wherever the pages are silent, are listed in the header of
``oracle.c``.  Sources: "[Kernel] Add w8a8 CUTLASS kernels" (feature list and
per_tensor_quantize example), "[Kernel] Support Fp8 Checkpoints (Dynamic +
Static)" (dynamic/static scales, shared merged-layer weight scale) and
"Enable scaled FP8 (e4m3fn) KV cache on ROCm (AMD GPU)" (section "Scaling
semantics").

Every function here is pinned by ``tests/test_oracle_pins.py`` against library
routines, closed forms, exact rational arithmetic and hand-worked examples.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3, INT8, BF16, FP16 = 0, 1, 2, 3
PER_TENSOR, PER_ROW = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
           "-shared", "-fPIC", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_e4m3_value.argtypes = [I]
        lib.orc_encode_e4m3.restype = ctypes.c_uint8
        lib.orc_encode_e4m3.argtypes = [ctypes.c_float]
        lib.orc_encode_int8.restype = ctypes.c_int8
        lib.orc_encode_int8.argtypes = [ctypes.c_float]
        lib.orc_f32_to_bf16.restype = ctypes.c_uint16
        lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.orc_f32_to_f16.restype = ctypes.c_uint16
        lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
        lib.orc_bf16_to_f32.restype = ctypes.c_float
        lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_f32.restype = ctypes.c_float
        lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.orc_scale_from_absmax.restype = ctypes.c_float
        lib.orc_scale_from_absmax.argtypes = [ctypes.c_float, I]
        lib.orc_absmax.restype = None
        lib.orc_absmax.argtypes = [P, I, I64, I64, I64, I, P]
        lib.orc_quant.restype = None
        lib.orc_quant.argtypes = [P, I, I64, I64, I64, P, I, I64, P, I, I]
        lib.orc_dequant.restype = None
        lib.orc_dequant.argtypes = [P, I, I64, I64, I64, P, I, P, I, I64]
        lib.orc_scaled_mm.restype = None
        lib.orc_scaled_mm.argtypes = [P, I64, P, I64, P, I, P, I, I64, I64, I64,
                                      I, I, P, P, P, P]
        lib.orc_scaled_mm_sample.restype = None
        lib.orc_scaled_mm_sample.argtypes = [P, I64, P, I64, P, I, P, I, I64, I,
                                             I, P, P, I64, P, P, P, P]
        lib.orc_requant_shards.restype = None
        lib.orc_requant_shards.argtypes = [P, I, I64, I64, P, P, I, P, I64, P]
        lib.orc_num_threads.restype = I
        lib.orc_set_num_threads.argtypes = [I]
        lib.orc_init()
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _rows_view(a: np.ndarray):
    """(rows, cols, leading dim in elements) of a 2-D array whose rows are
    contiguous (it may be a row-slice or a column-slice of a larger array)."""
    if a.ndim != 2:
        raise ValueError("expected a 2-D array")
    item = a.itemsize
    if a.shape[1] > 1 and a.strides[1] != item:
        raise ValueError("rows must be contiguous")
    ld = a.strides[0] // item if a.shape[0] > 1 else a.shape[1]
    return a.shape[0], a.shape[1], ld


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- scalars

def e4m3_value(code: int) -> float:
    """Value of an e4m3fn code (OCP definition; 0x7F / 0xFF are NaN)."""
    return _load().orc_e4m3_value(int(code))


def encode_e4m3(v) -> np.ndarray:
    """Table encoder: nearest e4m3 code of each fp32 value, ties to even,
    saturating at +-448, NaN -> 0x7F."""
    lib = _load()
    v = np.asarray(v, dtype=np.float32)
    out = np.array([lib.orc_encode_e4m3(float(x)) for x in v.ravel()], dtype=np.uint8)
    return out.reshape(v.shape)


def encode_int8(v) -> np.ndarray:
    lib = _load()
    v = np.asarray(v, dtype=np.float32)
    out = np.array([lib.orc_encode_int8(float(x)) for x in v.ravel()], dtype=np.int8)
    return out.reshape(v.shape)


def f32_to_bf16_bits(v) -> np.ndarray:
    lib = _load()
    v = np.asarray(v, dtype=np.float32)
    return np.array([lib.orc_f32_to_bf16(float(x)) for x in v.ravel()],
                    dtype=np.uint16).reshape(v.shape)


def f32_to_f16_bits(v) -> np.ndarray:
    lib = _load()
    v = np.asarray(v, dtype=np.float32)
    return np.array([lib.orc_f32_to_f16(float(x)) for x in v.ravel()],
                    dtype=np.uint16).reshape(v.shape)


def bits16_to_f32(bits, dtype: int) -> np.ndarray:
    lib = _load()
    bits = np.asarray(bits, dtype=np.uint16)
    fn = lib.orc_bf16_to_f32 if dtype == BF16 else lib.orc_f16_to_f32
    return np.array([fn(int(b)) for b in bits.ravel()], dtype=np.float32).reshape(bits.shape)


def scale_from_absmax(amax: float, q_dtype: int) -> float:
    return float(np.float32(_load().orc_scale_from_absmax(float(amax), q_dtype)))


# ---------------------------------------------------------------- arrays

def absmax(x_bits: np.ndarray, x_dtype: int, gran: int) -> np.ndarray:
    rows, cols, ld = _rows_view(x_bits)
    out = np.zeros(rows if gran == PER_ROW else 1, dtype=np.float32)
    _load().orc_absmax(_ptr(x_bits), x_dtype, rows, cols, ld, gran, _ptr(out))
    return out


def quant(x_bits: np.ndarray, x_dtype: int, q_dtype: int, gran: int,
          scale: np.ndarray | None = None):
    """Quantise a 2-D array of bf16/fp16 bit patterns.

    ``scale=None`` is the dynamic mode (scales computed from absmax and
    returned); otherwise the given fp32 scales are used (static mode).
    Returns ``(codes uint8 [rows, cols], scale float32 [rows] or [1])``.
    """
    x_bits = np.asarray(x_bits)
    if x_bits.dtype != np.uint16:
        raise TypeError("x_bits must hold 16-bit patterns (uint16)")
    rows, cols, ld = _rows_view(x_bits)
    n = rows if gran == PER_ROW else 1
    if scale is None:
        s = np.zeros(n, dtype=np.float32)
        dynamic = 1
    else:
        s = np.ascontiguousarray(np.asarray(scale, dtype=np.float32).reshape(-1))
        if s.size != n:
            raise ValueError(f"scale must have {n} entries")
        s = s.copy()
        dynamic = 0
    q = np.empty((rows, cols), dtype=np.uint8)
    _load().orc_quant(_ptr(x_bits), x_dtype, rows, cols, ld, _ptr(q), q_dtype,
                      cols, _ptr(s), gran, dynamic)
    return q, s


def dequant(q: np.ndarray, q_dtype: int, scale: np.ndarray, gran: int,
            y_dtype: int) -> np.ndarray:
    q = np.asarray(q)
    if q.dtype == np.int8:
        q = q.view(np.uint8)
    rows, cols, ld = _rows_view(q)
    s = np.ascontiguousarray(np.asarray(scale, dtype=np.float32).reshape(-1))
    y = np.empty((rows, cols), dtype=np.uint16)
    _load().orc_dequant(_ptr(q), q_dtype, rows, cols, ld, _ptr(s), gran, _ptr(y),
                        y_dtype, cols)
    return y


def _mm_operands(A, B, sa, sb):
    A = np.asarray(A)
    B = np.asarray(B)
    if A.dtype == np.int8:
        A = A.view(np.uint8)
    if B.dtype == np.int8:
        B = B.view(np.uint8)
    M, K, lda = _rows_view(A)
    N, K2, ldb = _rows_view(B)
    if K != K2:
        raise ValueError("A is [M, K] and B is stored [N, K]: K must match")
    sa = np.ascontiguousarray(np.asarray(sa, dtype=np.float32).reshape(-1))
    sb = np.ascontiguousarray(np.asarray(sb, dtype=np.float32).reshape(-1))
    a_gran = PER_ROW if sa.size == M and M > 1 else PER_TENSOR
    b_gran = PER_ROW if sb.size == N and N > 1 else PER_TENSOR
    if a_gran == PER_TENSOR and sa.size != 1:
        raise ValueError("scale_a must have 1 or M entries")
    if b_gran == PER_TENSOR and sb.size != 1:
        raise ValueError("scale_b must have 1 or N entries")
    return A, B, M, N, K, lda, ldb, sa, sb, a_gran, b_gran


def scaled_mm(A, B, sa, sb, q_dtype: int, out_dtype: int):
    """out[m, n] = round16(((float)sum_k A[m,k] B[n,k]) * sa[m|0] * sb[n|0]).

    A: [M, K] codes, B: [N, K] codes (K contiguous in both).
    Returns dict with ``acc`` (float64, exact), ``iacc`` (int64, int8 only),
    ``y`` (fp32 before the 16-bit cast) and ``out`` (16-bit bit patterns).
    """
    A, B, M, N, K, lda, ldb, sa, sb, a_gran, b_gran = _mm_operands(A, B, sa, sb)
    acc = np.empty((M, N), dtype=np.float64)
    iacc = np.empty((M, N), dtype=np.int64)
    y = np.empty((M, N), dtype=np.float32)
    out = np.empty((M, N), dtype=np.uint16)
    _load().orc_scaled_mm(_ptr(A), lda, _ptr(B), ldb, _ptr(sa), a_gran, _ptr(sb),
                          b_gran, M, N, K, q_dtype, out_dtype, _ptr(acc),
                          _ptr(iacc), _ptr(y), _ptr(out))
    return {"acc": acc, "iacc": iacc, "y": y, "out": out}


def scaled_mm_sample(A, B, sa, sb, q_dtype: int, out_dtype: int, idx_m, idx_n):
    """Like :func:`scaled_mm` for the listed (m, n) pairs only."""
    A, B, M, N, K, lda, ldb, sa, sb, a_gran, b_gran = _mm_operands(A, B, sa, sb)
    idx_m = np.ascontiguousarray(np.asarray(idx_m, dtype=np.int64))
    idx_n = np.ascontiguousarray(np.asarray(idx_n, dtype=np.int64))
    if idx_m.shape != idx_n.shape:
        raise ValueError("idx_m and idx_n must have the same length")
    if idx_m.size and (idx_m.min() < 0 or idx_m.max() >= M or idx_n.min() < 0
                       or idx_n.max() >= N):
        raise ValueError("sample index out of range")
    cnt = idx_m.size
    acc = np.empty(cnt, dtype=np.float64)
    iacc = np.empty(cnt, dtype=np.int64)
    y = np.empty(cnt, dtype=np.float32)
    out = np.empty(cnt, dtype=np.uint16)
    _load().orc_scaled_mm_sample(_ptr(A), lda, _ptr(B), ldb, _ptr(sa), a_gran,
                                 _ptr(sb), b_gran, K, q_dtype, out_dtype,
                                 _ptr(idx_m), _ptr(idx_n), cnt, _ptr(acc),
                                 _ptr(iacc), _ptr(y), _ptr(out))
    return {"acc": acc, "iacc": iacc, "y": y, "out": out}


def requant_shards(q, q_dtype: int, shard_scales, shard_rows):
    """Rewrite a row-sharded merged weight to one shared scale
    s_max = max(shard_scales): q' = encode(decode(q) * (s_i / s_max)).
    Returns (codes [rows, cols] uint8, scale [1] float32)."""
    q = np.asarray(q)
    if q.dtype == np.int8:
        q = q.view(np.uint8)
    rows, cols, ld = _rows_view(q)
    ss = np.ascontiguousarray(np.asarray(shard_scales, dtype=np.float32).reshape(-1))
    sr = np.ascontiguousarray(np.asarray(shard_rows, dtype=np.int64).reshape(-1))
    if ss.size != sr.size or ss.size < 1 or int(sr.sum()) != rows or (sr < 0).any():
        raise ValueError("shard_rows must be non-negative and sum to the number of rows")
    out = np.empty((rows, cols), dtype=np.uint8)
    smax = np.zeros(1, dtype=np.float32)
    _load().orc_requant_shards(_ptr(q), q_dtype, cols, ld, _ptr(ss), _ptr(sr), ss.size, _ptr(out), cols,
                               _ptr(smax))
    return out, smax
