"""Scaled matmul on CTA pairs (tcgen05 cta_group::2, 256-row tiles) against
the oracle on seeded inputs, on shapes with several pair tiles and ragged
tails in M, N and K ("[Kernel] Add w8a8 CUTLASS kernels", feature list of
cutlass_scaled_mm_dq).  fp8: |gpu - y| <= 2^-7 |y| + 1e-3 against the
oracle's fp32 y; int8: the int32 accumulators and the fp16 outputs bit for
bit.  The 128-column tiles come first: they use 256 TMEM columns per CTA."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_bits16_equal, assert_fp8_close, out_to_f32, bits_np
from test_gpu_gemm import fp8_problem, int8_problem, run_gpu

pytestmark = pytest.mark.gpu


def pair(bn, stages=0):
    return {"swap_ab": 0, "block_n": bn, "split_k": 1, "stages": stages, "cta_pair": 1}


SHAPES = [(256, 256, 512), (300, 200, 1008), (1024, 768, 2048), (520, 1040, 4112)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_pair_fp8_block_n_128(M, N, K):
    A, B, sa, sb = fp8_problem(M, N, K, seed=M + N + K)
    out = run_gpu(A, B, sa, sb, oracle.E4M3, torch.bfloat16, config=pair(128))
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.BF16)
    assert_fp8_close(out_to_f32(bits_np(out), oracle.BF16), ref["y"], "pair 128")


@pytest.mark.parametrize("M,N,K", SHAPES[:3])
def test_pair_int8_block_n_128(M, N, K):
    K = (K + 15) // 16 * 16
    A, B, sa, sb = int8_problem(M, N, K, seed=M * 3 + N)
    acc = run_gpu(A, B, np.ones(M, np.float32), np.ones(N, np.float32), oracle.INT8, torch.int32,
                  config=pair(128))
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.INT8, oracle.FP16)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref["iacc"])
    out = run_gpu(A, B, sa, sb, oracle.INT8, torch.float16, config=pair(128))
    assert_bits16_equal(bits_np(out), ref["out"], oracle.FP16, "pair int8 128")


@pytest.mark.parametrize("bn", [256, 224, 192, 96, 64])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_pair_fp8_wide(bn, M, N, K):
    A, B, sa, sb = fp8_problem(M, N, K, seed=M + N + K + bn)
    out = run_gpu(A, B, sa, sb, oracle.E4M3, torch.bfloat16, config=pair(bn))
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.BF16)
    assert_fp8_close(out_to_f32(bits_np(out), oracle.BF16), ref["y"], f"pair {bn}")


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (300, 200, 2048), (1024, 768, 3072), (200, 512, 1040),
                                   (520, 1040, 4112)])
def test_pair_int8_block_n_256(M, N, K):
    """Three 1024-K chunks at K = 3072: the exact chunked accumulation drains
    into the int32 total between chunks on both CTAs of the pair.  K = 1040
    and 4112 end in a partial 64-deep f16 block."""
    A, B, sa, sb = int8_problem(M, N, K, seed=M * 5 + N)
    acc = run_gpu(A, B, np.ones(M, np.float32), np.ones(N, np.float32), oracle.INT8, torch.int32,
                  config=pair(256))
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.INT8, oracle.FP16)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref["iacc"])


def test_pair_per_tensor_scales_fp16_and_two_stages():
    M, N, K = 512, 512, 1024
    A, B, sa, sb = fp8_problem(M, N, K, seed=77, a_per_row=False, b_per_row=False)
    out = run_gpu(A, B, sa, sb, oracle.E4M3, torch.float16, config=pair(256, stages=2))
    ref = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.FP16)
    assert_fp8_close(out_to_f32(bits_np(out), oracle.FP16), ref["y"], "pair per-tensor")


def test_pair_rejects_split_and_swap():
    import int8_w8a8_scaled_gb300 as w8
    A, B, sa, sb = fp8_problem(256, 256, 512, seed=5)
    for bad in ({"swap_ab": 1, "block_n": 128, "split_k": 1, "cta_pair": 1},
                {"swap_ab": 0, "block_n": 128, "split_k": 3, "cta_pair": 1},
                {"swap_ab": 0, "block_n": 80, "split_k": 1, "cta_pair": 1}):
        with pytest.raises(w8.W8A8Error):
            run_gpu(A, B, sa, sb, oracle.E4M3, torch.bfloat16, config=bad)
    A8, B8, sa8, sb8 = int8_problem(256, 256, 512, seed=6)
    with pytest.raises(w8.W8A8Error):   # K halves are for e4m3 only
        run_gpu(A8, B8, sa8, sb8, oracle.INT8, torch.float16,
                config={"swap_ab": 0, "block_n": 256, "split_k": 2, "cta_pair": 1})


# K halves of the last round (split_k 2): shapes whose pair tiles leave a last
# round of at most half of the pairs, computed against the oracle on every
# fifth row (all columns, so every split tile is covered).  With 76 pairs:
# 5 x 16 = 80 tiles leave 4 (K = 1040: halves of 4 and 5 blocks, the last
# one partial; ragged M and N put a split tile in the corner), 6 x 19 = 114
# leave 38, exactly half of the pairs (K = 256: one block per half).
TAIL_SHAPES = [(1280, 4096, 1040), (1200, 4000, 1040), (1536, 4864, 256)]


def tail_cfg(bn=256):
    return {"swap_ab": 0, "block_n": bn, "split_k": 2, "cta_pair": 1}


def tail_used(M, N, K, cfg):
    import int8_w8a8_scaled_gb300 as w8
    return w8.mm_workspace_size(M, N, K, w8.E4M3, cfg) > 0


@pytest.mark.parametrize("M,N,K", TAIL_SHAPES)
def test_pair_fp8_last_round_k_halves(M, N, K):
    if not tail_used(M, N, K, tail_cfg()):
        pytest.skip("this GPU's pair count leaves no last round to split for this shape")
    A, B, sa, sb = fp8_problem(M, N, K, seed=M + N + K + 11)
    out = run_gpu(A, B, sa, sb, oracle.E4M3, torch.bfloat16, config=tail_cfg())
    rows = np.arange(0, M, 5)
    ref = oracle.scaled_mm(A[rows], B, sa[rows], sb, oracle.E4M3, oracle.BF16)
    assert_fp8_close(out_to_f32(bits_np(out), oracle.BF16)[rows], ref["y"], "pair K halves")


def test_pair_k_halves_deterministic_and_counters_reset():
    """The two halves are summed in half order whichever pair finishes
    first, and the last one resets its arrival counter: repeated calls on one
    workspace give the same bits, and raw fp32 outputs match the oracle."""
    import int8_w8a8_scaled_gb300 as w8
    M, N, K = 1280, 4096, 1040
    cfg = tail_cfg()
    if not tail_used(M, N, K, cfg):
        pytest.skip("this GPU's pair count leaves no last round to split for this shape")
    A, B, sa, sb = fp8_problem(M, N, K, seed=91, a_per_row=False, b_per_row=True)
    a_g = torch.from_numpy(A.view(np.uint8)).cuda().view(torch.float8_e4m3fn)
    b_g = torch.from_numpy(B.view(np.uint8)).cuda().view(torch.float8_e4m3fn)
    sa_g = torch.from_numpy(np.asarray(sa, np.float32)).cuda()
    sb_g = torch.from_numpy(np.asarray(sb, np.float32)).cuda()
    ws = w8.Workspace(w8.mm_workspace_size(M, N, K, w8.E4M3, cfg), torch.device("cuda"))
    outs = []
    for _ in range(3):
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        w8.scaled_mm(a_g, b_g, sa_g, sb_g, out, workspace=ws, config=cfg)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
    assert torch.equal(outs[0].view(torch.int32), outs[2].view(torch.int32))
    rows = np.arange(3, M, 7)
    ref = oracle.scaled_mm(A[rows], B, sa, sb, oracle.E4M3, oracle.BF16)   # y: fp32 before the cast
    assert_fp8_close(outs[0].cpu().numpy()[rows].astype(np.float64), ref["y"], "pair K halves fp32")
    assert w8.device_status() == 0


def test_pair_k_halves_fp16_per_tensor():
    M, N, K = 1536, 4864, 256
    if not tail_used(M, N, K, tail_cfg()):
        pytest.skip("this GPU's pair count leaves no last round to split for this shape")
    A, B, sa, sb = fp8_problem(M, N, K, seed=123, a_per_row=False, b_per_row=False)
    out = run_gpu(A, B, sa, sb, oracle.E4M3, torch.float16, config=tail_cfg())
    rows = np.arange(1, M, 5)
    ref = oracle.scaled_mm(A[rows], B, sa, sb, oracle.E4M3, oracle.FP16)
    assert_fp8_close(out_to_f32(bits_np(out), oracle.FP16)[rows], ref["y"], "pair K halves fp16")


def test_pair_no_device_timeouts():
    import int8_w8a8_scaled_gb300 as w8
    assert w8.device_status() == 0
