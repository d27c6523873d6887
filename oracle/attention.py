"""CPU oracle for decode attention over an fp8 (e4m3) KV cache.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only the test suite,
the package smoke check and the CPU-baseline leg of the benchmark may use it.

What it computes, in float64, straight from the definitions:
  * dequantisation, "Enable scaled FP8 (e4m3fn) KV cache on ROCm (AMD GPU)",
    section "Scaling semantics": a cached code stands for its e4m3 value
    times the tensor's scaling factor, with one per-tensor factor for K and
    one for V (the kv_scale of the paged attention kernel).  The e4m3 value
    is the exact value of the OCP e4m3fn code (``oracle.e4m3_value``).
  * attention: the pages name the kernel (paged attention) but not its
    arithmetic; the plain reading is textbook scaled-dot-product attention
    of one query token per sequence over the cached tokens t < seq_len,
    s_t = sm_scale * q . K_t, out = sum_t softmax(s)_t V_t, with query head h
    reading KV head h // (num_q_heads // num_kv_heads).  An empty sequence
    gives zeros.
  * paging: token t of sequence b lives in cache row
    block_table[b, t // block_size] * block_size + t % block_size.  A
    table entry outside [0, num_blocks) marks padding: the tokens it would
    hold are not attended to (the usual -1 padding of a block table, and
    any id past the end of the cache alike).  A sequence with no attended
    token gives zeros, as an empty one does.

Pinned by ``tests/test_oracle_attention.py``: brute force with Python
scalars on tiny inputs, closed forms (one token, equal keys, a dominant
key), the paged layout against the contiguous one, padding entries against
the contiguous sequence with those tokens removed, and grouped heads against
one head at a time.
"""
from __future__ import annotations

import numpy as np

from . import BF16, FP16, bits16_to_f32, e4m3_value

_E4M3 = None


def e4m3_table() -> np.ndarray:
    """float64 value of every e4m3fn code (NaN for 0x7F / 0xFF)."""
    global _E4M3
    if _E4M3 is None:
        _E4M3 = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
    return _E4M3


def gather_rows(cache: np.ndarray, b: int, n: int, block_table=None) -> np.ndarray:
    """Rows of the attended tokens among 0..n-1 of sequence b, in token
    order: [n', num_kv_heads, head_dim].  Without a block table all n; with
    one, the tokens whose block id lies in [0, num_blocks)."""
    if block_table is None:
        return cache[b, :n]
    num_blocks, bs = cache.shape[0], cache.shape[1]
    t = np.arange(n)
    blk = np.asarray(block_table, dtype=np.int64)[b, t // bs]
    keep = (blk >= 0) & (blk < num_blocks)
    return cache[blk[keep], (t % bs)[keep]]


def fp8_kv_decode_attention(q_bits, q_dtype: int, k_codes, v_codes, seq_lens, k_scale: float,
                            v_scale: float, sm_scale: float, block_table=None) -> np.ndarray:
    """q_bits: uint16 [B, Hq, D] (bf16 or fp16 bit patterns); k/v_codes:
    uint8 [B, T, Hkv, D] or, with block_table [B, max_blocks], uint8
    [num_blocks, block_size, Hkv, D].  Returns float64 [B, Hq, D]."""
    q = bits16_to_f32(np.asarray(q_bits, dtype=np.uint16), q_dtype).astype(np.float64)
    B, Hq, D = q.shape
    Hkv = k_codes.shape[2]
    G = Hq // Hkv
    tab = e4m3_table()
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        n = int(seq_lens[b])
        if n <= 0:
            continue
        K = tab[gather_rows(k_codes, b, n, block_table)] * float(k_scale)   # [n', Hkv, D]
        V = tab[gather_rows(v_codes, b, n, block_table)] * float(v_scale)
        if K.shape[0] == 0:
            continue                      # every token is padding: zeros
        for h in range(Hq):
            g = h // G
            s = (K[:, g, :] @ q[b, h]) * float(sm_scale)                      # [n]
            w = np.exp(s - s.max())
            out[b, h] = (w @ V[:, g, :]) / w.sum()
    return out


def attention_bruteforce(q, K, V, sm_scale: float) -> list:
    """One head, Python floats only: q [D], K and V [n][D] (already
    dequantised).  For pinning the array version on tiny inputs."""
    import math
    s = [sm_scale * sum(qd * kd for qd, kd in zip(q, k)) for k in K]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    tot = sum(w)
    return [sum(wi * v[d] for wi, v in zip(w, V)) / tot for d in range(len(q))]


__all__ = ["e4m3_table", "gather_rows", "fp8_kv_decode_attention", "attention_bruteforce", "BF16", "FP16"]
