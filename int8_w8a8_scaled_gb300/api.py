"""Python binding of the C ABI: torch tensors in, library calls out.

This layer only marshals arguments (pointers, sizes, strides, dtypes, the
current CUDA stream); every step of the computation runs in the CUDA
library.  Tensors must already live on the current CUDA device.

    scaled_quant(x, q, scale, per_token=True, dynamic=True)
    scaled_dequant(q, scale, y, per_token=False)
    scaled_mm(a_q, b_q, scale_a, scale_b, out)

Naming follows the pages: ``cutlass_scaled_mm_dq(a, b, scale_a, scale_b,
out_dtype)`` of "[Kernel] Add w8a8 CUTLASS kernels" (here the output tensor is
passed in, as in that page's C++ op) with B given as a [K, N] column-major
view, i.e. a [N, K] row-major tensor; the quantiser follows the "Scaling
semantics" section of "Enable scaled FP8 (e4m3fn) KV cache on ROCm".
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import _lib
from ._lib import (BF16, DYNAMIC, E4M3, FP16, FP32, INT8, INT32, PER_ROW, PER_TENSOR, STATIC,
                   MmConfig, W8A8Error, check)

__all__ = [
    "scaled_quant", "scaled_dequant", "scaled_mm", "mm_workspace_size",
    "quant_workspace_size", "pick_config", "device_status", "Workspace", "quant_scaled_mm",
    "expand_shard_scales", "requant_shards", "fp8_kv_decode_attention", "attention_workspace_size",
    "W8A8Error", "MmConfig",
]


def _qkind(t: torch.Tensor, q_dtype=None) -> int:
    if q_dtype is not None:
        return q_dtype
    if t.dtype == torch.float8_e4m3fn:
        return E4M3
    if t.dtype == torch.int8:
        return INT8
    raise TypeError(f"quantised tensors must be float8_e4m3fn or int8 (got {t.dtype}); "
                    "pass q_dtype= for a uint8 view")


def _fkind(t: torch.Tensor, wide: bool = False) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return FP16
    if wide and t.dtype == torch.float32:
        return FP32
    if wide and t.dtype == torch.int32:
        return INT32
    raise TypeError(f"expected bfloat16 or float16 (got {t.dtype})")


def _ld(t: torch.Tensor) -> int:
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("rows must be contiguous (stride(1) == 1)")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])


def _cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Workspace:
    """A zero-filled device scratch buffer reused across calls on one stream.

    The matmul's split-K counters must start at zero; the library leaves them
    at zero after each successful call, so the buffer only needs zeroing once.
    """

    def __init__(self, nbytes: int = 0, device=None):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)

    def ensure(self, nbytes: int) -> "Workspace":
        if nbytes > self.buf.numel():
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        return self

    @property
    def nbytes(self) -> int:
        return self.buf.numel()


_ws_lock = threading.Lock()
_default_ws: dict = {}


def _default_workspace(device: torch.device, nbytes: int, kind: str) -> Workspace:
    """Per (device, stream, kind) scratch; the matmul's buffer is never shared
    with the quantiser (whose absmax word would land on a counter)."""
    key = (kind, device.index, torch.cuda.current_stream(device).cuda_stream)
    with _ws_lock:
        ws = _default_ws.get(key)
        if ws is None:
            ws = _default_ws[key] = Workspace(nbytes, device)
        return ws.ensure(nbytes)


def quant_workspace_size(rows: int, cols: int, per_token: bool, dynamic: bool) -> int:
    return _lib.load().w8a8_scaled_quant_workspace_size(
        rows, cols, PER_ROW if per_token else PER_TENSOR, DYNAMIC if dynamic else STATIC)


def scaled_quant(x: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, per_token: bool = True,
                 dynamic: bool = True, workspace: torch.Tensor | None = None, q_dtype=None,
                 stream=None) -> None:
    """q = sat_round(x / scale); dynamic mode writes scale = absmax / 448
    (e4m3) or absmax / 127 (int8), per token (row) or per tensor."""
    _cuda(x, q, scale, workspace)
    lib = _lib.load()
    rows, cols = x.shape
    if tuple(q.shape) != (rows, cols):
        raise ValueError("q must have the shape of x")
    if scale.dtype != torch.float32 or not scale.is_contiguous():
        raise ValueError("scale must be a contiguous float32 tensor")
    need_scale = rows if per_token else 1
    if scale.numel() != need_scale:
        raise ValueError(f"scale must have {need_scale} elements")
    gran = PER_ROW if per_token else PER_TENSOR
    mode = DYNAMIC if dynamic else STATIC
    need = lib.w8a8_scaled_quant_workspace_size(rows, cols, gran, mode)
    if need and workspace is None:
        workspace = _default_workspace(x.device, need, "quant").buf
    check(lib.w8a8_scaled_quant(
        _ptr(x), _fkind(x), rows, cols, _ld(x), _ptr(q), _qkind(q, q_dtype), _ld(q),
        _ptr(scale), gran, mode, _ptr(workspace) if need else None,
        workspace.numel() if (need and workspace is not None) else 0, _stream(stream)))


def scaled_dequant(q: torch.Tensor, scale: torch.Tensor, y: torch.Tensor, per_token: bool = False,
                   q_dtype=None, stream=None) -> None:
    """y = round16(decode(q) * scale)."""
    _cuda(q, scale, y)
    lib = _lib.load()
    rows, cols = q.shape
    if tuple(y.shape) != (rows, cols):
        raise ValueError("y must have the shape of q")
    if scale.dtype != torch.float32 or not scale.is_contiguous():
        raise ValueError("scale must be a contiguous float32 tensor")
    check(lib.w8a8_scaled_dequant(
        _ptr(q), _qkind(q, q_dtype), rows, cols, _ld(q), _ptr(scale),
        PER_ROW if per_token else PER_TENSOR, _ptr(y), _fkind(y), _ld(y), _stream(stream)))


def _cfg(config) -> MmConfig | None:
    if config is None:
        return None
    if isinstance(config, MmConfig):
        return config
    return MmConfig(int(config.get("swap_ab", 0)), int(config.get("block_n", 0)),
                    int(config.get("split_k", 0)), int(config.get("stages", 0)),
                    int(config.get("ctas_per_sm", 0)), int(config.get("reduce", 0)),
                    int(config.get("cta_pair", 0)))


def pick_config(M: int, N: int, K: int, q_dtype: int = E4M3) -> dict:
    c = MmConfig()
    check(_lib.load().w8a8_scaled_mm_pick_config(M, N, K, q_dtype, ctypes.byref(c)))
    return c.as_dict()


def mm_workspace_size(M: int, N: int, K: int, q_dtype: int = E4M3, config=None) -> int:
    lib = _lib.load()
    c = _cfg(config)
    if c is None:
        return lib.w8a8_scaled_mm_workspace_size(M, N, K, q_dtype)
    return lib.w8a8_scaled_mm_config_workspace_size(M, N, K, q_dtype, ctypes.byref(c))


def scaled_mm(a_q: torch.Tensor, b_q: torch.Tensor, scale_a: torch.Tensor, scale_b: torch.Tensor,
              out: torch.Tensor, workspace: torch.Tensor | Workspace | None = None, config=None,
              q_dtype=None, stream=None) -> torch.Tensor:
    """out[m, n] = round16(sum_k a_q[m, k] b_q[n, k] * scale_a[m|0] * scale_b[n|0]).

    a_q: [M, K] e4m3 / int8, rows contiguous.  b_q: [N, K] (the [K, N]
    column-major weight), rows contiguous.  scale_a: [M] or [1] fp32,
    scale_b: [N] or [1] fp32.  out: [M, N] bf16 / fp16 (or float32 for the
    unrounded e4m3 result, int32 for the raw int8 accumulators).
    """
    _cuda(a_q, b_q, scale_a, scale_b, out)
    lib = _lib.load()
    M, K = a_q.shape
    N, K2 = b_q.shape
    if K != K2:
        raise ValueError("a_q is [M, K] and b_q is [N, K]: K must match")
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N]")
    for s in (scale_a, scale_b):
        if s.dtype != torch.float32 or not s.is_contiguous():
            raise ValueError("scales must be contiguous float32 tensors")
    a_gran = PER_ROW if scale_a.numel() == M and M > 1 else PER_TENSOR
    b_gran = PER_ROW if scale_b.numel() == N and N > 1 else PER_TENSOR
    if a_gran == PER_TENSOR and scale_a.numel() != 1:
        raise ValueError("scale_a must have 1 or M elements")
    if b_gran == PER_TENSOR and scale_b.numel() != 1:
        raise ValueError("scale_b must have 1 or N elements")
    qk = _qkind(a_q, q_dtype)
    if _qkind(b_q, q_dtype) != qk:
        raise TypeError("a_q and b_q must have the same element type")
    c = _cfg(config)
    need = (lib.w8a8_scaled_mm_config_workspace_size(M, N, K, qk, ctypes.byref(c)) if c is not None
            else lib.w8a8_scaled_mm_workspace_size(M, N, K, qk))
    if isinstance(workspace, Workspace):
        workspace = workspace.ensure(need).buf
    elif workspace is None and need:
        workspace = _default_workspace(a_q.device, need, "mm").buf
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (_ptr(a_q), _ld(a_q), _ptr(b_q), _ld(b_q), _ptr(scale_a), a_gran, _ptr(scale_b), b_gran,
            _ptr(out), _ld(out), M, N, K, qk, _fkind(out, wide=True), ws_ptr, ws_bytes)
    if c is None:
        check(lib.w8a8_scaled_mm(*args, _stream(stream)))
    else:
        check(lib.w8a8_scaled_mm_with_config(*args, ctypes.byref(c), _stream(stream)))
    return out


def quant_scaled_mm(x: torch.Tensor, b_q: torch.Tensor, scale_b: torch.Tensor, out: torch.Tensor,
                    scale_a_out: torch.Tensor | None = None, workspace: torch.Tensor | Workspace | None = None,
                    route: str = "auto", stream=None) -> torch.Tensor:
    """Dynamic per-token quantisation of x and the scaled matmul in one call:
    the bits of ``scaled_quant(x, ..., per_token=True, dynamic=True)``
    followed by ``scaled_mm``.

    x: [M, K] bf16 / fp16, rows contiguous.  b_q: [N, K] e4m3 / int8 (the
    operand type).  scale_b: [N] or [1] fp32.  out: [M, N] bf16 / fp16 (or
    float32 with e4m3 weights).  scale_a_out: optional [M] fp32 that receives
    the per-token scales.  route: "auto", "one_kernel" (the matmul
    quantises its own activations; decode shapes only) or "two_step".
    """
    _cuda(x, b_q, scale_b, out)
    lib = _lib.load()
    M, K = x.shape
    N, K2 = b_q.shape
    if K != K2:
        raise ValueError("x is [M, K] and b_q is [N, K]: K must match")
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N]")
    if scale_b.dtype != torch.float32 or not scale_b.is_contiguous():
        raise ValueError("scale_b must be a contiguous float32 tensor")
    b_gran = PER_ROW if scale_b.numel() == N and N > 1 else PER_TENSOR
    if b_gran == PER_TENSOR and scale_b.numel() != 1:
        raise ValueError("scale_b must have 1 or N elements")
    if scale_a_out is not None:
        _cuda(scale_a_out)
        if scale_a_out.dtype != torch.float32 or scale_a_out.numel() != M or not scale_a_out.is_contiguous():
            raise ValueError("scale_a_out must be a contiguous float32 tensor of M elements")
    qk = _qkind(b_q)
    need = lib.w8a8_quant_scaled_mm_workspace_size(M, N, K, qk)
    if isinstance(workspace, Workspace):
        workspace = workspace.ensure(need).buf
    elif workspace is None and need:
        workspace = _default_workspace(x.device, need, "mm").buf
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib.w8a8_quant_scaled_mm(_ptr(x), _fkind(x), _ld(x), _ptr(b_q), _ld(b_q), _ptr(scale_b), b_gran,
                                   _ptr(out), _ld(out), M, N, K, qk, _fkind(out, wide=True),
                                   _ptr(scale_a_out) if scale_a_out is not None else None,
                                   _lib.ROUTES[route], ws_ptr, ws_bytes, _stream(stream)))
    return out


def _shard_rows(shard_rows):
    arr = (ctypes.c_int64 * len(shard_rows))(*[int(r) for r in shard_rows])
    return arr, len(shard_rows)


def expand_shard_scales(shard_scales: torch.Tensor, shard_rows, scale_b: torch.Tensor, stream=None) -> torch.Tensor:
    """scale_b[n] = shard_scales[shard of row n]: per-shard weight scales of a
    merged layer as a per-channel vector for the fused epilogue."""
    _cuda(shard_scales, scale_b)
    arr, n = _shard_rows(shard_rows)
    check(_lib.load().w8a8_expand_shard_scales(_ptr(shard_scales), arr, n, _ptr(scale_b), _stream(stream)))
    return scale_b


def requant_shards(q: torch.Tensor, shard_scales: torch.Tensor, shard_rows, q_out: torch.Tensor,
                   scale_out: torch.Tensor, q_dtype=None, stream=None) -> None:
    """Rewrite a row-sharded merged weight to one shared scale (the largest
    shard scale, written to scale_out): q' = encode(decode(q) * s_i / s_max)."""
    _cuda(q, shard_scales, q_out, scale_out)
    arr, n = _shard_rows(shard_rows)
    rows, cols = q.shape
    if tuple(q_out.shape) != (rows, cols):
        raise ValueError("q_out must have the shape of q")
    check(_lib.load().w8a8_requant_shards(_ptr(q), _qkind(q, q_dtype), cols, _ld(q), _ptr(shard_scales), arr, n,
                                          _ptr(q_out), _ld(q_out), _ptr(scale_out), _stream(stream)))


def device_status() -> int:
    """Synchronise and read/clear the device status word (1 = a bounded
    pipeline wait timed out)."""
    v = ctypes.c_int(0)
    check(_lib.load().w8a8_device_status(ctypes.byref(v)))
    return v.value


def attention_workspace_size(batch: int, num_q_heads: int, max_seq_len: int) -> int:
    return int(_lib.load().w8a8_fp8_kv_attention_workspace_size(batch, num_q_heads, max_seq_len))


def fp8_kv_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            seq_lens: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                            out: torch.Tensor, sm_scale: float | None = None,
                            block_table: torch.Tensor | None = None, workspace=None, stream=None) -> None:
    """Decode attention reading an e4m3 KV cache with per-tensor scales
    ("Enable scaled FP8 (e4m3fn) KV cache on ROCm", "Scaling semantics").

    q, out: [batch, num_q_heads, 128] bf16 / fp16.  Without block_table the
    caches are [batch, max_seq_len, num_kv_heads, 128]; with block_table
    (int32 [batch, max_blocks]) they are [num_blocks, block_size,
    num_kv_heads, 128] (the paged cache).  Codes are float8_e4m3fn (or uint8
    views).  seq_lens: int32 [batch]; k_scale, v_scale: float32 [1].
    sm_scale defaults to 1/sqrt(128)."""
    _cuda(q, k_cache, v_cache, seq_lens, k_scale, v_scale, out)
    lib = _lib.load()
    if q.dim() != 3 or not q.is_contiguous() or tuple(out.shape) != tuple(q.shape) or not out.is_contiguous():
        raise ValueError("q and out must be contiguous [batch, num_q_heads, head_dim] tensors")
    batch, hq, d = q.shape
    if k_cache.dim() != 4 or tuple(k_cache.shape) != tuple(v_cache.shape):
        raise ValueError("k_cache and v_cache must be 4-d tensors of one shape")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    for c in (k_cache, v_cache):
        if c.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError("caches must hold float8_e4m3fn codes (or uint8 views)")
    hkv = k_cache.shape[2]
    if k_cache.shape[3] != d:
        raise ValueError("cache head_dim must equal q's")
    if seq_lens.dtype != torch.int32 or seq_lens.numel() != batch or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous int32 tensor of batch entries")
    for s_ in (k_scale, v_scale):
        if s_.dtype != torch.float32 or s_.numel() != 1:
            raise ValueError("k_scale and v_scale must be float32 tensors of one element")
    if block_table is None:
        if k_cache.shape[0] != batch:
            raise ValueError("without a block table the caches are [batch, max_seq_len, num_kv_heads, head_dim]")
        max_seq = k_cache.shape[1]
        bt, bsz, maxb, nblk = None, 0, 0, 0
    else:
        if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != batch \
                or not block_table.is_contiguous():
            raise ValueError("block_table must be a contiguous int32 [batch, max_blocks] tensor")
        _cuda(block_table)
        nblk, bsz = k_cache.shape[0], k_cache.shape[1]
        maxb = block_table.shape[1]
        max_seq = maxb * bsz
        bt = _ptr(block_table)
    need = lib.w8a8_fp8_kv_attention_workspace_size(batch, hq, max_seq)
    if isinstance(workspace, Workspace):
        wbuf = workspace.ensure(need).buf
    elif workspace is None:
        wbuf = _default_workspace(q.device, need, "attention").buf
    else:
        wbuf = workspace
    if sm_scale is None:
        sm_scale = 1.0 / float(d) ** 0.5
    check(lib.w8a8_fp8_kv_decode_attention(
        _ptr(q), _fkind(q), batch, hq, hkv, d, _ptr(k_cache), _ptr(v_cache), max_seq, bt, bsz, maxb, nblk,
        _ptr(seq_lens), _ptr(k_scale), _ptr(v_scale), float(sm_scale), _ptr(out), _fkind(out),
        _ptr(wbuf), wbuf.numel(), _stream(stream)))
