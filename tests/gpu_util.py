"""Helpers shared by the GPU parity tests (inputs come from synthetic_inputs,
expected values from the oracle; nothing here computes the method)."""
import numpy as np
import torch

import oracle
import synthetic_inputs as si

# fp8 output tolerance: |gpu - y| <= 2^-7 |y| + 1e-3 against the oracle's fp32 y.
FP8_RTOL = 2.0 ** -7
FP8_ATOL = 1e-3

QD = {"e4m3": oracle.E4M3, "int8": oracle.INT8}


def q_torch_dtype(qd):
    return torch.float8_e4m3fn if qd == oracle.E4M3 else torch.int8


def to_gpu_codes(codes: np.ndarray, qd) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(codes).view(np.uint8)).cuda()
    return t.view(q_torch_dtype(qd))


def codes_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def bits_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def out_to_f32(bits: np.ndarray, od) -> np.ndarray:
    if od == oracle.BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)


def assert_fp8_close(gpu_out_f32: np.ndarray, y: np.ndarray, what=""):
    y = y.astype(np.float64)
    g = gpu_out_f32.astype(np.float64)
    err = np.abs(g - y)
    tol = FP8_RTOL * np.abs(y) + FP8_ATOL
    bad = ~(err <= tol)
    if bad.any():
        i = np.argmax(np.where(bad, err - tol, -np.inf))
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside |gpu-y| <= 2^-7|y|+1e-3; "
                             f"worst at {np.unravel_index(i, bad.shape)}: gpu={g.flat[i]} y={y.flat[i]}")


def assert_bits16_equal(a: np.ndarray, b: np.ndarray, od, what=""):
    """Bit equality of 16-bit float patterns, NaN payloads aside."""
    fa, fb = out_to_f32(a, od), out_to_f32(b, od)
    na, nb = np.isnan(fa), np.isnan(fb)
    assert np.array_equal(na, nb), f"{what}: NaN positions differ"
    diff = (a != b) & ~na
    assert not diff.any(), f"{what}: {diff.sum()} elements differ, first at {np.argwhere(diff)[0]}"


def quantized_operand(shape, seed, qd, per_row=True, weight=False):
    """bf16 synthetic tensor -> oracle codes and scales (dynamic)."""
    if weight:
        x = si.normal(shape, seed=seed, std=0.02)
    else:
        x = si.normal_with_outliers(shape, seed=seed)
    q, s = oracle.quant(si.bits16(x), oracle.BF16, qd, oracle.PER_ROW if per_row else oracle.PER_TENSOR)
    return x, q, s
