"""quant_scaled_mm: dynamic per-token activation quantiser and scaled matmul
in one call.  Decode shapes run as one kernel that quantises its own
activations; the result must be the bits of the two calls (quantiser, then
matmul with the same configuration), the per-token scales must equal the
oracle's bit for bit, and the output must meet the fp8 tolerance against the
oracle.  Other shapes take the two-step route inside the call."""
import numpy as np
import pytest
import torch

import int8_w8a8_scaled_gb300 as w8
import oracle
import synthetic_inputs as si
from gpu_util import assert_fp8_close, bits_np, out_to_f32, quantized_operand, to_gpu_codes

pytestmark = pytest.mark.gpu

OUT_ORACLE = {torch.bfloat16: oracle.BF16, torch.float16: oracle.FP16}


def problem(M, N, K, seed, x_dtype=torch.bfloat16, per_channel=True):
    x = si.normal_with_outliers((M, K), seed=seed)
    if x_dtype == torch.float16:
        xg = x.to(torch.float16)
        xbits = xg.view(torch.int16).numpy().view(np.uint16)
        xkind = oracle.FP16
    else:
        xg = x
        xbits = si.bits16(x)
        xkind = oracle.BF16
    _, B, sb = quantized_operand((N, K), seed + 1, oracle.E4M3, per_row=per_channel, weight=True)
    return xg.cuda(), xbits, xkind, B, sb


def two_step(xg, b_g, sb_g, out_dtype, M, N):
    aq = torch.empty(xg.shape, dtype=torch.float8_e4m3fn, device="cuda")
    sa = torch.empty(M, dtype=torch.float32, device="cuda")
    w8.scaled_quant(xg, aq, sa, per_token=True, dynamic=True)
    out = torch.empty(M, N, dtype=out_dtype, device="cuda")
    w8.scaled_mm(aq, b_g, sa, sb_g, out)
    return out, sa


@pytest.mark.parametrize("shape", [(1, 1024, 1024), (1, 6144, 4096), (16, 4096, 14336), (5, 600, 1040),
                                   (16, 2048, 4096), (33, 512, 2048), (64, 4096, 4096), (2, 28672, 4096)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("x_dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
def test_fused_equals_two_calls_and_oracle(shape, x_dtype):
    M, N, K = shape
    xg, xbits, xkind, B, sb = problem(M, N, K, seed=M * 7 + N, x_dtype=x_dtype)
    b_g = to_gpu_codes(B, oracle.E4M3)
    sb_g = torch.from_numpy(sb).cuda()
    cfg = w8.pick_config(M, N, K, w8.E4M3)
    assert cfg["swap_ab"] == 1 and M <= cfg["block_n"]  # the one-kernel route
    for out_dtype in (torch.bfloat16, torch.float32):
        out = torch.empty(M, N, dtype=out_dtype, device="cuda")
        sa_out = torch.empty(M, dtype=torch.float32, device="cuda")
        w8.quant_scaled_mm(xg, b_g, sb_g, out, scale_a_out=sa_out, route="one_kernel")
        ref_out, ref_sa = two_step(xg, b_g, sb_g, out_dtype, M, N)
        torch.cuda.synchronize()
        assert torch.equal(sa_out, ref_sa)
        assert torch.equal(out.view(torch.int16 if out_dtype != torch.float32 else torch.int32),
                           ref_out.view(torch.int16 if out_dtype != torch.float32 else torch.int32)), (shape, out_dtype)
    # against the oracle: scales bit-exact, outputs within the fp8 tolerance (sampled)
    aq, osa = oracle.quant(xbits, xkind, oracle.E4M3, oracle.PER_ROW)
    assert np.array_equal(sa_out.cpu().numpy(), osa)
    im = np.random.default_rng(1).integers(0, M, 2000)
    inn = np.random.default_rng(2).integers(0, N, 2000)
    ref = oracle.scaled_mm_sample(aq, B, osa, sb, oracle.E4M3, oracle.BF16, im, inn)
    assert_fp8_close(out.cpu().numpy()[im, inn], ref["y"], f"fused {shape}")
    assert w8.device_status() == 0


def test_fused_per_tensor_weight_scale_and_special_rows():
    """Merged-QKV style per-tensor weight scale; an all-zero token row (scale
    1, codes 0) and a row of one repeated tiny negative value (its scale a
    tiny normal, every code -448)."""
    M, N, K = 8, 1536, 2048
    xg, xbits, xkind, B, sb = problem(M, N, K, seed=3, per_channel=False)
    xg[2].zero_()
    xg[5] = -1e-30
    xbits = xg.cpu().view(torch.int16).numpy().view(np.uint16)
    b_g = to_gpu_codes(B, oracle.E4M3)
    sb_g = torch.from_numpy(sb).cuda()
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    sa_out = torch.empty(M, dtype=torch.float32, device="cuda")
    w8.quant_scaled_mm(xg, b_g, sb_g, out, scale_a_out=sa_out, route="one_kernel")
    ref_out, ref_sa = two_step(xg, b_g, sb_g, torch.bfloat16, M, N)
    torch.cuda.synchronize()
    assert torch.equal(sa_out, ref_sa) and sa_out[2].item() == 1.0
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    aq, osa = oracle.quant(xbits, xkind, oracle.E4M3, oracle.PER_ROW)
    ref = oracle.scaled_mm(aq, B, osa, sb, oracle.E4M3, oracle.BF16)
    assert_fp8_close(out_to_f32(bits_np(out), oracle.BF16), ref["y"], "per-tensor weight scale")


@pytest.mark.parametrize("case", ["large_m", "int8", "unaligned_x"])
def test_two_step_route(case):
    """Shapes the one kernel does not take still give the two calls' bits."""
    if case == "large_m":
        M, N, K, qd = 200, 768, 1024, oracle.E4M3
    elif case == "int8":
        M, N, K, qd = 16, 640, 1024, oracle.INT8
    else:
        M, N, K, qd = 4, 512, 1008, oracle.E4M3
    x = si.normal_with_outliers((M, K + 8), seed=11).cuda()
    # unaligned_x: the first row starts 8 bytes into the buffer (not 16-byte aligned)
    xg = x[:, 4:4 + K] if case == "unaligned_x" else x[:, :K].contiguous()
    _, B, sb = quantized_operand((N, K), 12, qd, per_row=True, weight=True)
    b_g = to_gpu_codes(B, qd)
    sb_g = torch.from_numpy(sb).cuda()
    od = torch.bfloat16 if qd == oracle.E4M3 else torch.float16
    out = torch.empty(M, N, dtype=od, device="cuda")
    sa_out = torch.empty(M, dtype=torch.float32, device="cuda")
    w8.quant_scaled_mm(xg, b_g, sb_g, out, scale_a_out=sa_out)   # auto: the two-step route here
    aq = torch.empty(M, K, dtype=torch.float8_e4m3fn if qd == oracle.E4M3 else torch.int8, device="cuda")
    sa = torch.empty(M, dtype=torch.float32, device="cuda")
    w8.scaled_quant(xg, aq, sa, per_token=True, dynamic=True)
    ref = torch.empty(M, N, dtype=od, device="cuda")
    w8.scaled_mm(aq, b_g, sa, sb_g, ref)
    torch.cuda.synchronize()
    assert torch.equal(sa_out, sa)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_fused_in_cuda_graph_back_to_back():
    """Several fused calls captured in one graph and replayed twice (each
    kernel launches the next early; the activations are read only after the
    dependency wait)."""
    shapes = [(1, 6144, 4096), (1, 4096, 4096), (16, 4096, 14336), (16, 28672, 4096)]
    items = []
    for i, (M, N, K) in enumerate(shapes):
        xg, _, _, B, sb = problem(M, N, K, seed=40 + i)
        items.append((xg, to_gpu_codes(B, oracle.E4M3), torch.from_numpy(sb).cuda(),
                      torch.empty(M, N, dtype=torch.bfloat16, device="cuda")))
    ws = w8.Workspace(1 << 26)  # larger than any of the calls needs: no growth during capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for xg, b_g, sb_g, out in items:      # warm-up (lazy initialisation outside capture)
            w8.quant_scaled_mm(xg, b_g, sb_g, out, workspace=ws, route="one_kernel", stream=s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for xg, b_g, sb_g, out in items:
                w8.quant_scaled_mm(xg, b_g, sb_g, out, workspace=ws, route="one_kernel", stream=s)
    for out in (it[3] for it in items):
        out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for xg, b_g, sb_g, out in items:
        ref, _ = two_step(xg, b_g, sb_g, torch.bfloat16, xg.shape[0], b_g.shape[0])
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert w8.device_status() == 0


def test_route_one_kernel_refused_where_it_cannot_run():
    M, N, K = 100, 512, 1024      # tokens span more than one narrow tile
    xg, _, _, B, sb = problem(M, N, K, seed=21)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(w8.W8A8Error):
        w8.quant_scaled_mm(xg, to_gpu_codes(B, oracle.E4M3), torch.from_numpy(sb).cuda(), out, route="one_kernel")


@pytest.mark.parametrize("shape", [(1, 6144, 4096), (16, 4096, 4096)], ids=lambda s: "x".join(map(str, s)))
def test_auto_route_equals_both_routes(shape):
    M, N, K = shape
    xg, _, _, B, sb = problem(M, N, K, seed=31)
    b_g, sb_g = to_gpu_codes(B, oracle.E4M3), torch.from_numpy(sb).cuda()
    outs = {}
    for route in ("auto", "one_kernel", "two_step"):
        outs[route] = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        w8.quant_scaled_mm(xg, b_g, sb_g, outs[route], route=route)
    torch.cuda.synchronize()
    assert torch.equal(outs["auto"].view(torch.int16), outs["one_kernel"].view(torch.int16))
    assert torch.equal(outs["auto"].view(torch.int16), outs["two_step"].view(torch.int16))
