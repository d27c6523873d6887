"""The allocation-free scaled matmul entry point.

w8a8_scaled_mm_noalloc serves callers that cannot allocate device memory
where they run the matmul (allocator hooks, plug-ins given only operand and
output buffers, processes whose memory another runtime has reserved): it
keeps its scratch (split-K partials through the workspace, int8 operand
planes) in a fixed array the library defines in device memory.  Checked here
through the C ABI against w8a8_scaled_mm with a caller workspace, on two
calls in a row: both run the same kernel configuration with the same
deterministic split-K order, so the outputs must be the same bits (e4m3 and
int8 alike).  One shape is also checked against the oracle, within the fp8
tolerance the other matmul tests use.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from int8_w8a8_scaled_gb300 import _lib

pytestmark = pytest.mark.gpu

E4M3, INT8, BF16, FP16, PER_ROW, PER_TENSOR = 0, 1, 2, 3, 1, 0


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _problem(M, N, K, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    a = torch.randint(0, 126, (M, K), generator=g, device="cuda", dtype=torch.uint8)
    b = torch.randint(0, 126, (N, K), generator=g, device="cuda", dtype=torch.uint8)
    a[:, ::3] |= 0x80  # mixed signs
    sa = torch.rand(M, generator=g, device="cuda") * 1e-3
    sb = torch.rand(N, generator=g, device="cuda") * 1e-3
    return a, b, sa, sb


@pytest.mark.parametrize("M,N,K,qd", [(1, 4096, 4096, E4M3), (16, 6144, 4096, E4M3), (64, 4096, 14336, E4M3),
                                      (3, 300, 1040, E4M3), (16, 1024, 1024, INT8), (5, 640, 2048, INT8)])
def test_noalloc_matches_workspace_entry_point_twice(M, N, K, qd):
    lib = _lib.load()
    a, b, sa, sb = _problem(M, N, K, seed=M + N)
    if qd == INT8:
        a, b = a - 64, b - 64      # int8 codes spread over both signs
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    need = lib.w8a8_scaled_mm_workspace_size(M, N, K, qd)
    assert 0 < need <= lib.w8a8_scaled_mm_noalloc_max_scratch()  # split-K partials / int8 planes
    ws = torch.zeros(max(need, 1), dtype=torch.uint8, device="cuda")
    od = BF16 if qd == E4M3 else FP16
    tdt = torch.bfloat16 if qd == E4M3 else torch.float16
    ref = torch.empty(M, N, dtype=tdt, device="cuda")
    st = lib.w8a8_scaled_mm(_p(a), K, _p(b), K, _p(sa), PER_ROW, _p(sb), PER_ROW, _p(ref), N, M, N, K, qd, od,
                            _p(ws), need, stream)
    assert st == 0, lib.w8a8_last_error()
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        st = lib.w8a8_scaled_mm_noalloc(_p(a), K, _p(b), K, _p(sa), PER_ROW, _p(sb), PER_ROW, _p(out), N, M, N, K,
                                        qd, od, stream)
        assert st == 0, lib.w8a8_last_error()
        torch.cuda.synchronize()
        # same configuration, same slice order: the same bits
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_noalloc_matches_the_oracle():
    """M=16 tokens x the O projection [4096 x 4096] (a split-K decode shape):
    bf16 outputs within |gpu - y| <= 2^-7 |y| + 1e-3 of the oracle's fp32 y."""
    import oracle
    import synthetic_inputs as si
    lib = _lib.load()
    M, N, K = 16, 4096, 4096
    qa, sa = oracle.quant(si.bits16(si.normal_with_outliers((M, K), seed=31)), oracle.BF16, oracle.E4M3,
                          oracle.PER_ROW)
    qb, sb = oracle.quant(si.bits16(si.normal((N, K), seed=32, std=0.02)), oracle.BF16, oracle.E4M3, oracle.PER_ROW)
    assert lib.w8a8_scaled_mm_workspace_size(M, N, K, E4M3) > 0      # the fixed array is in use
    a = torch.from_numpy(qa).cuda()
    b = torch.from_numpy(qb).cuda()
    ga, gb = torch.from_numpy(sa).cuda(), torch.from_numpy(sb).cuda()
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.w8a8_scaled_mm_noalloc(_p(a), K, _p(b), K, _p(ga), PER_ROW, _p(gb), PER_ROW, _p(out), N, M, N, K,
                                    E4M3, BF16, stream)
    assert st == 0, lib.w8a8_last_error()
    torch.cuda.synchronize()
    y = oracle.scaled_mm(qa, qb, sa, sb, oracle.E4M3, oracle.BF16)["y"].astype(np.float64)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - y) <= 2.0 ** -7 * np.abs(y) + 1e-3)


def test_noalloc_runs_pair_tiles_whole_when_their_k_halves_do_not_fit():
    """The prefill down projection (M=4096, N=4096, K=14336): the automatic
    configuration runs the last round of CTA-pair tiles as K halves, whose
    partials (about 15 MB) exceed the fixed array, so the allocation-free
    entry point runs those tiles whole.  Its output is then the bits of the
    same configuration with split_k 1 through a caller workspace, and within
    the fp8 tolerance of the oracle on sampled outputs."""
    import int8_w8a8_scaled_gb300 as w8
    import oracle
    M, N, K = 4096, 4096, 14336
    lib = _lib.load()
    auto = w8.pick_config(M, N, K, w8.E4M3)
    if not (auto["cta_pair"] and auto["split_k"] == 2):
        pytest.skip("this GPU's automatic configuration takes no K halves here")
    assert lib.w8a8_scaled_mm_workspace_size(M, N, K, E4M3) > lib.w8a8_scaled_mm_noalloc_max_scratch()
    a, b, sa, sb = _problem(M, N, K, seed=77)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = lib.w8a8_scaled_mm_noalloc(_p(a), K, _p(b), K, _p(sa), PER_ROW, _p(sb), PER_ROW, _p(out), N, M, N, K,
                                    E4M3, BF16, stream)
    assert st == 0, lib.w8a8_last_error()
    whole = dict(auto, split_k=1)
    assert w8.mm_workspace_size(M, N, K, w8.E4M3, whole) == 0
    ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    w8.scaled_mm(a.view(torch.float8_e4m3fn), b.view(torch.float8_e4m3fn), sa, sb, ref, config=whole)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    rng = np.random.default_rng(5)
    im = rng.integers(0, M, 2048)
    jn = rng.integers(0, N, 2048)
    A, B = a.cpu().numpy(), b.cpu().numpy()
    y = oracle.scaled_mm_sample(A, B, sa.cpu().numpy(), sb.cpu().numpy(), oracle.E4M3, oracle.BF16, im, jn)["y"]
    got = out.float().cpu().numpy()[im, jn].astype(np.float64)
    y = y.astype(np.float64)
    assert np.all(np.abs(got - y) <= 2.0 ** -7 * np.abs(y) + 1e-3)


def test_noalloc_rejects_problems_beyond_its_array():
    lib = _lib.load()
    a, b, sa, sb = _problem(16, 64, 64, seed=1)
    out = torch.empty(16, 64, dtype=torch.float16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # int8 widens both operands into f16 planes: 2 * (8192 + 8192) * 8192
    # bytes, far beyond the fixed array; rejected before any launch
    M = N = K = 8192
    assert lib.w8a8_scaled_mm_workspace_size(M, N, K, 1) > lib.w8a8_scaled_mm_noalloc_max_scratch()
    st = lib.w8a8_scaled_mm_noalloc(_p(a), K, _p(b), K, _p(sa), PER_ROW, _p(sb), PER_ROW, _p(out), N, M, N, K,
                                    1, 3, stream)
    assert st == 4  # W8A8_ERR_WORKSPACE
    assert b"fixed array" in lib.w8a8_last_error()
