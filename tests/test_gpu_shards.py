"""Merged-layer (QKV / gate-up) helpers on the GPU against the oracle:
per-shard scales expanded for the fused epilogue, and shards requantised to
the largest shard scale (bit-exact codes)."""
import numpy as np
import pytest
import torch

import int8_w8a8_scaled_gb300 as w8
import oracle
import synthetic_inputs as si
from gpu_util import assert_fp8_close, bits_np, codes_np, out_to_f32, q_torch_dtype, to_gpu_codes

pytestmark = pytest.mark.gpu

QKV_ROWS = (4096, 1024, 1024)      # Llama-3-8B q / k / v output rows


def shard_weights(qd, rows=QKV_ROWS, K=512, seed=50):
    parts, scales = [], []
    for i, r in enumerate(rows):
        x = si.normal((r, K), seed=seed + i, std=0.02 * (1 + 0.5 * i))
        q, s = oracle.quant(si.bits16(x), oracle.BF16, qd, oracle.PER_TENSOR)
        parts.append(q)
        scales.append(s[0])
    return np.concatenate(parts), np.array(scales, np.float32)


def test_expand_shard_scales():
    ss = np.array([0.5, 0.25, 3.0], np.float32)
    out = torch.empty(sum(QKV_ROWS), dtype=torch.float32, device="cuda")
    w8.expand_shard_scales(torch.from_numpy(ss).cuda(), QKV_ROWS, out)
    assert np.array_equal(out.cpu().numpy(), np.repeat(ss, QKV_ROWS))


@pytest.mark.parametrize("qd", [oracle.E4M3, oracle.INT8])
@pytest.mark.parametrize("inplace", [False, True])
def test_requant_shards_bit_exact(qd, inplace):
    q, ss = shard_weights(qd)
    want, wscale = oracle.requant_shards(q, qd, ss, QKV_ROWS)
    qg = to_gpu_codes(q, qd)
    out = qg if inplace else torch.empty_like(qg)
    so = torch.empty(1, dtype=torch.float32, device="cuda")
    w8.requant_shards(qg, torch.from_numpy(ss).cuda(), QKV_ROWS, out, so)
    torch.cuda.synchronize()
    assert so.item() == wscale[0]
    assert np.array_equal(codes_np(out), want)


@pytest.mark.parametrize("M", [1, 16, 300])
def test_merged_qkv_gemm_with_shard_scales(M):
    """One GEMM over the merged weight with the shard scales fused in the
    epilogue, and one after requantising to the shared scale; both against
    the oracle."""
    K = 512
    q, ss = shard_weights(oracle.E4M3, K=K)
    _, A, sa = (None, *oracle.quant(si.bits16(si.normal_with_outliers((M, K), seed=9)), oracle.BF16,
                                    oracle.E4M3, oracle.PER_ROW))
    N = q.shape[0]
    a_g, q_g = to_gpu_codes(A, oracle.E4M3), to_gpu_codes(q, oracle.E4M3)
    sa_g = torch.from_numpy(sa).cuda()
    # fused per-shard scales
    sb = torch.empty(N, dtype=torch.float32, device="cuda")
    w8.expand_shard_scales(torch.from_numpy(ss).cuda(), QKV_ROWS, sb)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    w8.scaled_mm(a_g, q_g, sa_g, sb, out)
    ref = oracle.scaled_mm(A, q, sa, np.repeat(ss, QKV_ROWS), oracle.E4M3, oracle.BF16)
    assert_fp8_close(out_to_f32(bits_np(out), oracle.BF16), ref["y"], "per-shard fused")
    # requantised to the shared scale
    q2 = torch.empty_like(q_g)
    s2 = torch.empty(1, dtype=torch.float32, device="cuda")
    w8.requant_shards(q_g, torch.from_numpy(ss).cuda(), QKV_ROWS, q2, s2)
    out2 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    w8.scaled_mm(a_g, q2, sa_g, s2, out2)
    torch.cuda.synchronize()
    oq2, os2 = oracle.requant_shards(q, oracle.E4M3, ss, QKV_ROWS)
    ref2 = oracle.scaled_mm(A, oq2, sa, os2, oracle.E4M3, oracle.BF16)
    assert_fp8_close(out_to_f32(bits_np(out2), oracle.BF16), ref2["y"], "requantised")


def test_shard_argument_errors():
    ss = torch.ones(3, dtype=torch.float32, device="cuda")
    out = torch.empty(8, dtype=torch.float32, device="cuda")
    with pytest.raises(w8.W8A8Error):
        w8.expand_shard_scales(ss, [1] * 17, out)       # more than 16 shards
    with pytest.raises(w8.W8A8Error):
        w8.expand_shard_scales(ss, [4, -1, 5], out)     # negative shard
