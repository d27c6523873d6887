"""GPU scaled-matmul parity against the oracle on seeded inputs.

fp8: the bf16/fp16 output must satisfy |gpu - y| <= 2^-7 |y| + 1e-3 against
the oracle's fp32 y.  int8: the int32 accumulators and the fp16/bf16 outputs
must match bit for bit.  Every kernel variant (swap / no swap, every block_n,
split-K) runs on shapes that span several tiles and ragged tails.
"""
import numpy as np
import pytest
import torch

import int8_w8a8_scaled_gb300 as w8
import oracle
import synthetic_inputs as si
from gpu_util import (assert_bits16_equal, assert_fp8_close, bits_np, codes_np, out_to_f32,
                      q_torch_dtype, quantized_operand, to_gpu_codes)

pytestmark = pytest.mark.gpu


def run_gpu(A, B, sa, sb, qd, out_dtype, config=None, lda_pad=0, ldc_pad=0):
    """Upload codes/scales and run scaled_mm; optional padded leading dims."""
    M, K = A.shape
    N = B.shape[0]
    if lda_pad:
        big = np.zeros((M, K + lda_pad), np.uint8)
        big[:, :K] = A.view(np.uint8)
        a_g = to_gpu_codes(big, qd)[:, :K]
    else:
        a_g = to_gpu_codes(A, qd)
    b_g = to_gpu_codes(B, qd)
    sa_g = torch.from_numpy(np.asarray(sa, np.float32)).cuda()
    sb_g = torch.from_numpy(np.asarray(sb, np.float32)).cuda()
    if ldc_pad:
        out_big = torch.zeros(M, N + ldc_pad, dtype=out_dtype, device="cuda")
        out = out_big[:, :N]
    else:
        out_big = None
        out = torch.empty(M, N, dtype=out_dtype, device="cuda")
    w8.scaled_mm(a_g, b_g, sa_g, sb_g, out, config=config)
    torch.cuda.synchronize()
    if out_big is not None:
        assert not out_big[:, N:].any().item(), "wrote past N into the ldc padding"
    return out


def fp8_problem(M, N, K, seed, a_per_row=True, b_per_row=True):
    _, A, sa = quantized_operand((M, K), seed, oracle.E4M3, per_row=a_per_row)
    _, B, sb = quantized_operand((N, K), seed + 1, oracle.E4M3, per_row=b_per_row, weight=True)
    return A, B, sa, sb


def int8_problem(M, N, K, seed):
    _, A, sa = quantized_operand((M, K), seed, oracle.INT8)
    _, B, sb = quantized_operand((N, K), seed + 1, oracle.INT8, weight=True)
    return A.view(np.int8), B.view(np.int8), sa, sb


FP8_CONFIGS = [
    None,
    {"swap_ab": 0, "block_n": 256, "split_k": 1},
    {"swap_ab": 0, "block_n": 128, "split_k": 1},
    {"swap_ab": 0, "block_n": 64, "split_k": 3},
    {"swap_ab": 0, "block_n": 16, "split_k": 1},
    {"swap_ab": 1, "block_n": 16, "split_k": 1},
    {"swap_ab": 1, "block_n": 16, "split_k": 5},
    {"swap_ab": 1, "block_n": 32, "split_k": 2},
    {"swap_ab": 1, "block_n": 64, "split_k": 1},
    {"swap_ab": 1, "block_n": 128, "split_k": 3},
    {"swap_ab": 1, "block_n": 256, "split_k": 1},
    {"swap_ab": 0, "block_n": 256, "split_k": 2, "stages": 2},
    {"swap_ab": 0, "block_n": 160, "split_k": 1},
    {"swap_ab": 0, "block_n": 192, "split_k": 2},
    {"swap_ab": 0, "block_n": 224, "split_k": 1},
    # split-K through the workspace (last arriver) and through a cluster
    {"swap_ab": 1, "block_n": 16, "split_k": 5, "reduce": w8.REDUCE_GLOBAL},
    {"swap_ab": 0, "block_n": 64, "split_k": 3, "reduce": w8.REDUCE_GLOBAL},
    {"swap_ab": 1, "block_n": 16, "split_k": 12},
    {"swap_ab": 1, "block_n": 32, "split_k": 8, "reduce": w8.REDUCE_CLUSTER},
    {"swap_ab": 1, "block_n": 16, "split_k": 7, "reduce": w8.REDUCE_CLUSTER},
    {"swap_ab": 0, "block_n": 256, "split_k": 2, "stages": 2, "reduce": w8.REDUCE_CLUSTER},
    {"swap_ab": 0, "block_n": 128, "split_k": 4, "reduce": w8.REDUCE_CLUSTER},
    {"swap_ab": 1, "block_n": 256, "split_k": 4},
]


def cfg_id(c):
    if c is None:
        return "auto"
    t = f"s{c['swap_ab']}_bn{c['block_n']}_k{c['split_k']}"
    if "stages" in c:
        t += f"_st{c['stages']}"
    if "reduce" in c:
        t += {w8.REDUCE_GLOBAL: "_glob", w8.REDUCE_CLUSTER: "_clus"}.get(c["reduce"], "_auto")
    return t


FP8_SHAPES = [(1, 256, 512), (32, 256, 512), (3, 100, 272), (129, 300, 1040), (300, 384, 640),
              (17, 4096, 4096)]


@pytest.mark.parametrize("cfg", FP8_CONFIGS, ids=cfg_id)
@pytest.mark.parametrize("shape", FP8_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fp8_variants(cfg, shape):
    M, N, K = shape
    A, B, sa, sb = fp8_problem(M, N, K, seed=M + N + K)
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.BF16)
    out = run_gpu(A, B, sa, sb, oracle.E4M3, torch.float32, config=cfg)
    assert_fp8_close(out.cpu().numpy(), ref["y"], f"fp32 out {shape} {cfg}")
    out16 = run_gpu(A, B, sa, sb, oracle.E4M3, torch.bfloat16, config=cfg)
    assert_fp8_close(out_to_f32(bits_np(out16), oracle.BF16), ref["y"], f"bf16 out {shape} {cfg}")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("grans", [(True, True), (True, False), (False, True), (False, False)])
def test_fp8_scale_granularities(out_dtype, grans):
    M, N, K = 70, 200, 768
    A, B, sa, sb = fp8_problem(M, N, K, seed=3, a_per_row=grans[0], b_per_row=grans[1])
    od = oracle.BF16 if out_dtype == torch.bfloat16 else oracle.FP16
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, od)
    out = run_gpu(A, B, sa, sb, oracle.E4M3, out_dtype)
    assert_fp8_close(out_to_f32(bits_np(out), od), ref["y"])


def test_fp8_per_tensor_equals_broadcast():
    M, N, K = 40, 256, 512
    A, B, _, _ = fp8_problem(M, N, K, seed=8)
    sa, sb = np.float32(0.013), np.float32(0.0007)
    for cfg in (None, {"swap_ab": 0, "block_n": 128, "split_k": 1}):
        o1 = bits_np(run_gpu(A, B, [sa], [sb], oracle.E4M3, torch.bfloat16, config=cfg))
        o2 = bits_np(run_gpu(A, B, [sa] * M, [sb] * N, oracle.E4M3, torch.bfloat16, config=cfg))
        assert np.array_equal(o1, o2)


def test_fp8_strided_submatrices():
    """Sub-matrix views (lda > K, ldc > N), the CUTLASS page's unit-test case."""
    M, N, K = 50, 130, 384
    A, B, sa, sb = fp8_problem(M, N, K, seed=9)
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.BF16)
    for cfg in (None, {"swap_ab": 0, "block_n": 64, "split_k": 1}):
        out = run_gpu(A, B, sa, sb, oracle.E4M3, torch.bfloat16, config=cfg, lda_pad=64, ldc_pad=24)
        assert_fp8_close(out_to_f32(bits_np(out), oracle.BF16), ref["y"])


def test_fp8_extreme_codes_exact_small_k():
    """All-+-448 operands: acc = +-448^2 K exactly, so fp32 output is exact."""
    M, N, K = 8, 32, 64
    A = np.full((M, K), 0x7E, np.uint8)
    A[1::2] = 0xFE
    B = np.full((N, K), 0x7E, np.uint8)
    out = run_gpu(A, B, [1.0], [1.0], oracle.E4M3, torch.float32)
    want = np.where(np.arange(M)[:, None] % 2 == 1, -1.0, 1.0) * 448.0 * 448.0 * K
    assert np.array_equal(out.cpu().numpy(), np.broadcast_to(want, (M, N)).astype(np.float32))


def test_fp8_zero_activation_rows():
    M, N, K = 9, 64, 256
    A, B, sa, sb = fp8_problem(M, N, K, seed=2)
    A[4] = 0
    A[7] = 0x80
    out = run_gpu(A, B, sa, sb, oracle.E4M3, torch.bfloat16)
    o = out.float().cpu().numpy()
    assert not o[4].any() and not o[7].any()


def test_tiny_config_end_to_end():
    """The tiny fp8 configuration: A bf16 [32, 512] N(0,1) with 1% x20
    outliers, W bf16 [256, 512] N(0, 0.02); dynamic per-token activation and
    per-channel weight e4m3 scales on the GPU; bf16 output."""
    a = si.normal_with_outliers((32, 512), seed=101)
    wt = si.normal((256, 512), seed=102, std=0.02)
    a_q = torch.empty(32, 512, dtype=torch.float8_e4m3fn, device="cuda")
    w_q = torch.empty(256, 512, dtype=torch.float8_e4m3fn, device="cuda")
    sa = torch.empty(32, dtype=torch.float32, device="cuda")
    sw = torch.empty(256, dtype=torch.float32, device="cuda")
    w8.scaled_quant(a.cuda(), a_q, sa, per_token=True, dynamic=True)
    w8.scaled_quant(wt.cuda(), w_q, sw, per_token=True, dynamic=True)
    out = torch.empty(32, 256, dtype=torch.bfloat16, device="cuda")
    w8.scaled_mm(a_q, w_q, sa, sw, out)
    torch.cuda.synchronize()
    qa, osa = oracle.quant(si.bits16(a), oracle.BF16, oracle.E4M3, oracle.PER_ROW)
    qw, osw = oracle.quant(si.bits16(wt), oracle.BF16, oracle.E4M3, oracle.PER_ROW)
    assert np.array_equal(codes_np(a_q), qa) and np.array_equal(sa.cpu().numpy(), osa)
    assert np.array_equal(codes_np(w_q), qw) and np.array_equal(sw.cpu().numpy(), osw)
    ref = oracle.scaled_mm(qa, qw, osa, osw, oracle.E4M3, oracle.BF16)
    assert_fp8_close(out_to_f32(bits_np(out), oracle.BF16), ref["y"])


INT8_CONFIGS = [
    None,
    {"swap_ab": 0, "block_n": 128, "split_k": 1},
    {"swap_ab": 0, "block_n": 64, "split_k": 2},
    {"swap_ab": 1, "block_n": 16, "split_k": 1},
    {"swap_ab": 1, "block_n": 16, "split_k": 3},
    {"swap_ab": 1, "block_n": 32, "split_k": 1},
    {"swap_ab": 1, "block_n": 128, "split_k": 2},
    {"swap_ab": 0, "block_n": 256, "split_k": 1},
    {"swap_ab": 0, "block_n": 256, "split_k": 2},
    {"swap_ab": 0, "block_n": 160, "split_k": 1},
    {"swap_ab": 0, "block_n": 160, "split_k": 2, "stages": 2},
    {"swap_ab": 1, "block_n": 16, "split_k": 3, "reduce": w8.REDUCE_GLOBAL},
    {"swap_ab": 0, "block_n": 256, "split_k": 2, "reduce": w8.REDUCE_GLOBAL},
    {"swap_ab": 1, "block_n": 32, "split_k": 8, "reduce": w8.REDUCE_CLUSTER},
    {"swap_ab": 0, "block_n": 64, "split_k": 5, "reduce": w8.REDUCE_CLUSTER},
]

INT8_SHAPES = [(1, 128, 64), (5, 100, 1040), (130, 260, 2112), (300, 128, 3072)]


@pytest.mark.parametrize("cfg", INT8_CONFIGS, ids=cfg_id)
@pytest.mark.parametrize("shape", INT8_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_int8_variants_bit_exact(cfg, shape):
    M, N, K = shape
    A, B, sa, sb = int8_problem(M, N, K, seed=M * 3 + K)
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.INT8, oracle.FP16)
    acc = run_gpu(A, B, sa, sb, oracle.INT8, torch.int32, config=cfg)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref["iacc"])
    out = run_gpu(A, B, sa, sb, oracle.INT8, torch.float16, config=cfg)
    assert_bits16_equal(bits_np(out), ref["out"], oracle.FP16, f"int8 fp16 out {shape} {cfg}")


@pytest.mark.parametrize("cfg", [None, {"swap_ab": 0, "block_n": 128, "split_k": 1},
                                 {"swap_ab": 0, "block_n": 256, "split_k": 1},
                                 {"swap_ab": 0, "block_n": 160, "split_k": 1},
                                 {"swap_ab": 1, "block_n": 16, "split_k": 4}])
def test_int8_worst_case_magnitudes_exact(cfg):
    """+-127 / -128 everywhere at a long K: every 1024-long chunk reaches
    |sum| = 2^24 (the exact-fp32 limit) and the int32 total 2^14 K."""
    M, N, K = 4, 256, 28672
    A = np.full((M, K), -128, np.int8)
    A[1] = 127
    A[2, ::2] = -128
    A[2, 1::2] = 127
    A[3] = np.random.default_rng(1).choice(np.array([-128, 127], np.int8), size=K)
    B = np.full((N, K), -128, np.int8)
    B[1::3] = 127
    ref = oracle.scaled_mm(A, B, np.ones(M, np.float32), np.ones(N, np.float32), oracle.INT8, oracle.FP16)
    acc = run_gpu(A, B, np.ones(M, np.float32), np.ones(N, np.float32), oracle.INT8, torch.int32, config=cfg)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref["iacc"])


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_int8_outputs_bit_exact(out_dtype):
    M, N, K = 64, 512, 4096
    A, B, sa, sb = int8_problem(M, N, K, seed=77)
    od = oracle.BF16 if out_dtype == torch.bfloat16 else oracle.FP16
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.INT8, od)
    out = run_gpu(A, B, sa, sb, oracle.INT8, out_dtype)
    assert_bits16_equal(bits_np(out), ref["out"], od)


def test_misaligned_pointer_is_an_error_status():
    A, B, sa, sb = fp8_problem(16, 64, 128, seed=1)
    a_g = torch.zeros(16 * 128 + 16, dtype=torch.uint8, device="cuda")
    a_view = a_g[1:1 + 16 * 128].view(16, 128).view(torch.float8_e4m3fn)
    b_g = to_gpu_codes(B, oracle.E4M3)
    out = torch.empty(16, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w8.W8A8Error) as ei:
        w8.scaled_mm(a_view, b_g, torch.ones(16, device="cuda"), torch.ones(64, device="cuda"), out)
    assert ei.value.status == 3


def test_cuda_graph_capture_and_replay():
    """Quantise + matmul captured in a CUDA graph and replayed (the CUTLASS
    page's "operation not permitted when stream is capturing" regression)."""
    M, N, K = 16, 512, 1024
    x = si.normal_with_outliers((M, K), seed=5).cuda()
    _, B, _, sb = fp8_problem(M, N, K, seed=6)
    b_g = to_gpu_codes(B, oracle.E4M3)
    sb_g = torch.from_numpy(sb).cuda()
    a_q = torch.empty(M, K, dtype=torch.float8_e4m3fn, device="cuda")
    sa = torch.empty(M, dtype=torch.float32, device="cuda")
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = w8.Workspace(w8.mm_workspace_size(M, N, K, w8.E4M3))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w8.scaled_quant(x, a_q, sa)
        w8.scaled_mm(a_q, b_g, sa, sb_g, out, workspace=ws)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        w8.scaled_quant(x, a_q, sa)
        w8.scaled_mm(a_q, b_g, sa, sb_g, out, workspace=ws)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert w8.device_status() == 0


def test_split_k_workspace_is_left_zeroed():
    M, N, K = 1, 1024, 4096
    A, B, sa, sb = fp8_problem(M, N, K, seed=12)
    cfg = {"swap_ab": 1, "block_n": 16, "split_k": 8, "reduce": w8.REDUCE_GLOBAL}
    ws = w8.Workspace(w8.mm_workspace_size(M, N, K, w8.E4M3, cfg))
    a_g, b_g = to_gpu_codes(A, oracle.E4M3), to_gpu_codes(B, oracle.E4M3)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.BF16)
    for _ in range(3):
        w8.scaled_mm(a_g, b_g, torch.from_numpy(sa).cuda(), torch.from_numpy(sb).cuda(), out,
                     workspace=ws, config=cfg)
        torch.cuda.synchronize()
        assert_fp8_close(out_to_f32(bits_np(out), oracle.BF16), ref["y"])
    tiles = (N + 127) // 128
    assert not ws.buf[: tiles * 4].any().item()  # counters back at zero


def test_no_device_timeouts_recorded():
    assert w8.device_status() == 0


def test_shared_workspace_across_shapes_and_dtypes():
    """One zero-filled workspace serves any sequence of calls: an int8 call
    (f16 planes in the scratch area) followed by split-K calls must still
    find zero arrival counters."""
    ws = w8.Workspace(1 << 20)
    seqs = [((130, 260, 2112), w8.INT8, None), ((5, 100, 1040), w8.INT8, {"swap_ab": 1, "block_n": 16, "split_k": 4}),
            ((3, 300, 1024), w8.E4M3, {"swap_ab": 1, "block_n": 16, "split_k": 3}),
            ((64, 512, 4096), w8.INT8, None), ((1, 1024, 4096), w8.E4M3, None)]
    for (M, N, K), qd, cfg in seqs * 2:
        if qd == w8.INT8:
            A, B, sa, sb = int8_problem(M, N, K, seed=M + N)
            ref = oracle.scaled_mm(A, B, sa, sb, oracle.INT8, oracle.FP16)
            a_g, b_g = to_gpu_codes(A, oracle.INT8), to_gpu_codes(B, oracle.INT8)
            acc = torch.empty(M, N, dtype=torch.int32, device="cuda")
            w8.scaled_mm(a_g, b_g, torch.from_numpy(sa).cuda(), torch.from_numpy(sb).cuda(), acc,
                         workspace=ws, config=cfg)
            torch.cuda.synchronize()
            assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref["iacc"]), (M, N, K, cfg)
        else:
            A, B, sa, sb = fp8_problem(M, N, K, seed=M + N)
            ref = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.BF16)
            a_g, b_g = to_gpu_codes(A, oracle.E4M3), to_gpu_codes(B, oracle.E4M3)
            out = torch.empty(M, N, dtype=torch.float32, device="cuda")
            w8.scaled_mm(a_g, b_g, torch.from_numpy(sa).cuda(), torch.from_numpy(sb).cuda(), out,
                         workspace=ws, config=cfg)
            torch.cuda.synchronize()
            assert_fp8_close(out.cpu().numpy(), ref["y"], f"{(M, N, K, cfg)}")
    assert not ws.buf[:65536].any().item()


@pytest.mark.parametrize("cfg", [{"swap_ab": 1, "block_n": 32, "split_k": 2},
                                 {"swap_ab": 1, "block_n": 64, "split_k": 1},
                                 {"swap_ab": 1, "block_n": 16, "split_k": 3},
                                 {"swap_ab": 0, "block_n": 64, "split_k": 1, "stages": 3},
                                 {"swap_ab": 0, "block_n": 128, "split_k": 1, "stages": 3},
                                 {"swap_ab": 0, "block_n": 224, "split_k": 1, "stages": 3}],
                         ids=lambda c: "_".join(f"{k}{v}" for k, v in c.items()))
def test_fp8_many_resident_ctas(cfg):
    """Enough work units that several persistent CTAs share each SM (each
    with its own TMEM allocation), checked element-wise."""
    M, N, K = (32, 16384, 1024) if cfg["swap_ab"] else (1024, 7168, 512)
    A, B, sa, sb = fp8_problem(M, N, K, seed=61)
    out = run_gpu(A, B, sa, sb, oracle.E4M3, torch.float32, config=cfg)
    im = np.random.default_rng(0).integers(0, M, 4000)
    inn = np.random.default_rng(1).integers(0, N, 4000)
    ref = oracle.scaled_mm_sample(A, B, sa, sb, oracle.E4M3, oracle.BF16, im, inn)
    assert_fp8_close(out.cpu().numpy()[im, inn], ref["y"], str(cfg))


def test_back_to_back_graph_of_gemms_with_overlap():
    """Several different GEMMs replayed back to back in one CUDA graph
    (programmatic dependent launch lets the next kernel's CTAs start while
    the previous one finishes); every output checked against the oracle."""
    shapes = [(16, 4096, 1024), (16, 8192, 1024), (300, 3072, 512), (1, 6144, 2048)]
    probs = [fp8_problem(M, N, K, seed=70 + i) for i, (M, N, K) in enumerate(shapes)]
    dev = [(to_gpu_codes(A, oracle.E4M3), to_gpu_codes(B, oracle.E4M3), torch.from_numpy(sa).cuda(),
            torch.from_numpy(sb).cuda(), torch.empty(A.shape[0], B.shape[0], dtype=torch.float32, device="cuda"))
           for A, B, sa, sb in probs]
    ws = w8.Workspace(max(w8.mm_workspace_size(M, N, K, w8.E4M3) for M, N, K in shapes))
    s = torch.cuda.Stream()

    def run():
        for a, b, sa, sb, out in dev:
            w8.scaled_mm(a, b, sa, sb, out, workspace=ws)
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            run()
    for _, _, _, _, out in dev:
        out.zero_()
    g.replay()
    torch.cuda.synchronize()
    for (A, B, sa, sb), (_, _, _, _, out) in zip(probs, dev):
        ref = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.BF16)
        assert_fp8_close(out.cpu().numpy(), ref["y"])
    assert w8.device_status() == 0


@pytest.mark.parametrize("qd,shape,base", [
    (oracle.E4M3, (1, 6144, 4096), {"swap_ab": 1, "block_n": 16}),
    (oracle.E4M3, (16, 4096, 14336), {"swap_ab": 1, "block_n": 32}),
    (oracle.E4M3, (50, 1000, 3008), {"swap_ab": 1, "block_n": 32}),
    (oracle.E4M3, (256, 4096, 4096), {"swap_ab": 0, "block_n": 64}),
    (oracle.E4M3, (256, 4096, 14336), {"swap_ab": 1, "block_n": 256}),
    (oracle.INT8, (7, 2048, 4096), {"swap_ab": 1, "block_n": 16}),
], ids=["M1_qkv", "M16_down", "ragged", "M256_o", "M256_down_swap", "int8_M7"])
@pytest.mark.parametrize("splits", [2, 3, 6, 8])
def test_cluster_and_global_reductions_agree_bitwise(qd, shape, base, splits):
    """Both reductions start from zero and add the slices in the order
    0..S-1, so their raw outputs (fp32 y / int32 accumulators) are the same
    bits; both are checked against the oracle on a sample."""
    M, N, K = shape
    if qd == oracle.E4M3:
        A, B, sa, sb = fp8_problem(M, N, K, seed=M + splits)
        out_dt = torch.float32
    else:
        A, B, sa, sb = int8_problem(M, N, K, seed=M + splits)
        out_dt = torch.int32
    outs = {}
    for red in (w8.REDUCE_GLOBAL, w8.REDUCE_CLUSTER):
        cfg = dict(base, split_k=splits, reduce=red)
        outs[red] = run_gpu(A, B, sa, sb, qd, out_dt, config=cfg).cpu().numpy()
    assert np.array_equal(outs[w8.REDUCE_GLOBAL].view(np.uint32), outs[w8.REDUCE_CLUSTER].view(np.uint32))
    im = np.random.default_rng(2).integers(0, M, 3000)
    inn = np.random.default_rng(3).integers(0, N, 3000)
    if qd == oracle.E4M3:
        ref = oracle.scaled_mm_sample(A, B, sa, sb, oracle.E4M3, oracle.BF16, im, inn)
        assert_fp8_close(outs[w8.REDUCE_CLUSTER][im, inn], ref["y"], f"{shape} S={splits}")
    else:
        ref = oracle.scaled_mm_sample(A, B, sa, sb, oracle.INT8, oracle.FP16, im, inn)
        assert np.array_equal(outs[w8.REDUCE_CLUSTER][im, inn].astype(np.int64), ref["iacc"])
    assert w8.device_status() == 0


def test_cluster_reduction_config_errors():
    A, B, sa, sb = fp8_problem(1, 512, 4096, seed=5)
    with pytest.raises(w8.W8A8Error):      # more slices than one portable cluster
        run_gpu(A, B, sa, sb, oracle.E4M3, torch.bfloat16,
                config={"swap_ab": 1, "block_n": 16, "split_k": 9, "reduce": w8.REDUCE_CLUSTER})
    with pytest.raises(w8.W8A8Error):
        run_gpu(A, B, sa, sb, oracle.E4M3, torch.bfloat16, config={"reduce": 7})
