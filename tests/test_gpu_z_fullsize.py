"""Parity at the full workload sizes, in the launch configuration the
benchmark uses (the library's automatic choice): quantiser codes and scales
are compared in full, matmul outputs on sampled elements the oracle computes
one by one (whole rows, whole columns, every tile corner and random points).

Workloads: Llama-3-8B decode fp8 (M in {1, 16, 64, 256}), Llama-3-8B prefill
fp8 static (M = 4096), int8 at Llama-3-70B shapes (M = 8192) and the scaled
FP8 KV cache [65536, 8, 128].
"""
import numpy as np
import pytest
import torch

import int8_w8a8_scaled_gb300 as w8
import oracle
import synthetic_inputs as si
from gpu_util import assert_bits16_equal, assert_fp8_close, bits_np, codes_np, out_to_f32

pytestmark = pytest.mark.gpu

LLAMA8B = (("qkv", 6144, 4096, True), ("o", 4096, 4096, False),
           ("gate_up", 28672, 4096, False), ("down", 4096, 14336, False))
LLAMA70B = (("qkv", 10240, 8192), ("gate_up", 57344, 8192), ("down", 8192, 28672))


def sample_points(M, N, seed, tile_p=128):
    rng = np.random.default_rng(seed)
    rows = sorted({0, M - 1, int(rng.integers(0, M)), int(rng.integers(0, M))})
    cols = sorted({0, N - 1, int(rng.integers(0, N)), int(rng.integers(0, N))})
    pts = set()
    for r in rows:
        pts.update((r, n) for n in range(N))
    for c in cols:
        pts.update((m, c) for m in range(M))
    # tile corners on a 128 x 16 grid (every few tiles on the largest shapes)
    n_tiles = ((M + tile_p - 1) // tile_p) * ((N + 15) // 16)
    step = max(1, int(np.sqrt(n_tiles / 4096.0)) + (1 if n_tiles > 4096 else 0))
    for m0 in range(0, M, tile_p * step):
        for n0 in range(0, N, 16 * step):
            for dm, dn in ((0, 0), (min(tile_p, M - m0) - 1, 0), (0, min(16, N - n0) - 1),
                           (min(tile_p, M - m0) - 1, min(16, N - n0) - 1)):
                pts.add((m0 + dm, n0 + dn))
    for _ in range(512):
        pts.add((int(rng.integers(0, M)), int(rng.integers(0, N))))
    pts = np.array(sorted(pts), dtype=np.int64)
    return pts[:, 0], pts[:, 1]


def gpu_quant(x_cpu, qd, per_token, dynamic=True, scale=None):
    rows, cols = x_cpu.shape
    q = torch.empty(rows, cols, dtype=torch.float8_e4m3fn if qd == oracle.E4M3 else torch.int8, device="cuda")
    if scale is None:
        s = torch.zeros(rows if per_token else 1, dtype=torch.float32, device="cuda")
    else:
        s = torch.from_numpy(np.asarray(scale, np.float32)).cuda()
    w8.scaled_quant(x_cpu.cuda(), q, s, per_token=per_token, dynamic=dynamic)
    torch.cuda.synchronize()
    return q, s


def check_quant(x_cpu, q, s, qd, per_token, scale=None):
    oq, os_ = oracle.quant(si.bits16(x_cpu), oracle.BF16, qd, oracle.PER_ROW if per_token else oracle.PER_TENSOR,
                           scale=scale)
    assert np.array_equal(s.cpu().numpy(), os_), "scales differ"
    gq = codes_np(q)
    assert np.array_equal(gq, oq), f"{(gq != oq).sum()} codes differ"
    return oq, os_


@pytest.mark.parametrize("M", [1, 16, 64, 256])
def test_decode_fp8_llama8b(M):
    for j, (name, N, K, shared) in enumerate(LLAMA8B):
        wt = si.normal((N, K), seed=700 + j, std=0.02)
        x = si.normal_with_outliers((M, K), seed=800 + M + j)
        wq, sw = gpu_quant(wt, oracle.E4M3, per_token=not shared)
        aq, sa = gpu_quant(x, oracle.E4M3, per_token=True)
        owq, osw = check_quant(wt, wq, sw, oracle.E4M3, not shared)
        oaq, osa = check_quant(x, aq, sa, oracle.E4M3, True)
        out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        w8.scaled_mm(aq, wq, sa, sw, out)
        torch.cuda.synchronize()
        got = out_to_f32(bits_np(out), oracle.BF16)
        if M <= 16:
            ref = oracle.scaled_mm(oaq, owq, osa, osw, oracle.E4M3, oracle.BF16)
            assert_fp8_close(got, ref["y"], f"decode M={M} {name}")
        else:
            im, inn = sample_points(M, N, seed=M + j)
            ref = oracle.scaled_mm_sample(oaq, owq, osa, osw, oracle.E4M3, oracle.BF16, im, inn)
            assert_fp8_close(got[im, inn], ref["y"], f"decode M={M} {name}")
    assert w8.device_status() == 0


def test_prefill_fp8_static_llama8b():
    M = 4096
    for j, (name, N, K, _) in enumerate(LLAMA8B):
        wt = si.normal((N, K), seed=900 + j, std=0.02)
        wq, sw = gpu_quant(wt, oracle.E4M3, per_token=False)
        owq, osw = check_quant(wt, wq, sw, oracle.E4M3, False)
        calib = si.student_t_columns((M, K), seed=950 + j)
        _, sa = gpu_quant(calib, oracle.E4M3, per_token=False)       # static scale from calibration
        _, osa = oracle.quant(si.bits16(calib), oracle.BF16, oracle.E4M3, oracle.PER_TENSOR)
        assert sa.cpu().numpy()[0] == osa[0]
        x = si.student_t_columns((M, K), seed=980 + j)
        aq, sa2 = gpu_quant(x, oracle.E4M3, per_token=False, dynamic=False, scale=osa)
        oaq, _ = check_quant(x, aq, sa2, oracle.E4M3, False, scale=osa)
        out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        w8.scaled_mm(aq, wq, sa2, sw, out)
        torch.cuda.synchronize()
        got = out_to_f32(bits_np(out), oracle.BF16)
        im, inn = sample_points(M, N, seed=j)
        ref = oracle.scaled_mm_sample(oaq, owq, osa, osw, oracle.E4M3, oracle.BF16, im, inn)
        assert_fp8_close(got[im, inn], ref["y"], f"prefill {name}")
    assert w8.device_status() == 0


@pytest.mark.parametrize("proj", LLAMA70B, ids=[p[0] for p in LLAMA70B])
def test_int8_llama70b(proj):
    name, N, K = proj
    M = 8192
    wt = si.normal((N, K), seed=1100 + N, std=0.02)
    x = si.normal_with_outliers((M, K), seed=1200 + N)
    wq, sw = gpu_quant(wt, oracle.INT8, per_token=True)
    aq, sa = gpu_quant(x, oracle.INT8, per_token=True)
    owq, osw = check_quant(wt, wq, sw, oracle.INT8, True)
    oaq, osa = check_quant(x, aq, sa, oracle.INT8, True)
    del wt, x
    out = torch.empty(M, N, dtype=torch.float16, device="cuda")
    w8.scaled_mm(aq, wq, sa, sw, out)
    acc = torch.empty(M, N, dtype=torch.int32, device="cuda")
    w8.scaled_mm(aq, wq, sa, sw, acc)
    torch.cuda.synchronize()
    im, inn = sample_points(M, N, seed=N)
    ref = oracle.scaled_mm_sample(oaq.view(np.int8), owq.view(np.int8), osa, osw, oracle.INT8, oracle.FP16,
                                  im, inn)
    gacc = acc.cpu().numpy()[im, inn].astype(np.int64)
    assert np.array_equal(gacc, ref["iacc"]), f"{(gacc != ref['iacc']).sum()} int32 accumulators differ"
    assert_bits16_equal(bits_np(out)[im, inn], ref["out"], oracle.FP16, f"int8 {name} fp16 out")
    assert w8.device_status() == 0


@pytest.mark.parametrize("block_n", [160, 256])
def test_int8_llama70b_qkv_tile_widths(block_n):
    """Both int8 accumulator layouts at full size, many tiles per persistent
    CTA: two chunk accumulators alternating (160 columns) and one chunk
    accumulator (256 columns)."""
    name, N, K = LLAMA70B[0]
    M = 8192
    wt = si.normal((N, K), seed=1500 + block_n, std=0.02)
    x = si.normal_with_outliers((M, K), seed=1600 + block_n)
    wq, sw = gpu_quant(wt, oracle.INT8, per_token=True)
    aq, sa = gpu_quant(x, oracle.INT8, per_token=True)
    owq, osw = check_quant(wt, wq, sw, oracle.INT8, True)
    oaq, osa = check_quant(x, aq, sa, oracle.INT8, True)
    del wt, x
    cfg = {"swap_ab": 0, "block_n": block_n, "split_k": 1}
    acc = torch.empty(M, N, dtype=torch.int32, device="cuda")
    w8.scaled_mm(aq, wq, sa, sw, acc, config=cfg)
    torch.cuda.synchronize()
    im, inn = sample_points(M, N, seed=block_n)
    ref = oracle.scaled_mm_sample(oaq.view(np.int8), owq.view(np.int8), osa, osw, oracle.INT8, oracle.FP16,
                                  im, inn)
    gacc = acc.cpu().numpy()[im, inn].astype(np.int64)
    assert np.array_equal(gacc, ref["iacc"]), f"{(gacc != ref['iacc']).sum()} int32 accumulators differ ({name})"
    assert w8.device_status() == 0


def test_kv_cache_fp8_round_trip_full():
    T, H, D = 65536, 8, 128
    for j in range(2):  # K then V, each with its own per-tensor scale
        x = si.kv_with_spikes(T, H, D, seed=1300 + j).reshape(T * H, D)
        q, s = gpu_quant(x, oracle.E4M3, per_token=False)
        oq, os_ = check_quant(x, q, s, oracle.E4M3, False)
        y = torch.empty(T * H, D, dtype=torch.bfloat16, device="cuda")
        w8.scaled_dequant(q, s, y)
        torch.cuda.synchronize()
        want = oracle.dequant(oq, oracle.E4M3, os_, oracle.PER_TENSOR, oracle.BF16)
        got = bits_np(y)
        assert_bits16_equal(got, want, oracle.BF16, "kv dequant")
        # round-trip error: half an e4m3 ulp of x/s times s, plus the bf16 rounding
        xf = x.float().numpy().astype(np.float64)
        yf = out_to_f32(got, oracle.BF16).astype(np.float64)
        v = np.abs(xf / float(os_[0]))
        e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
        half_ulp = 0.5 * np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3)) * float(os_[0])
        bound = half_ulp * (1 + 2.0 ** -20) + 2.0 ** -8 * np.abs(yf) + 2.0 ** -23 * np.abs(xf)
        assert np.all(np.abs(yf - xf) <= bound)
    assert w8.device_status() == 0
