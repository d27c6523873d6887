"""The diagnostic phase trace of the scaled matmul (w8a8_debug_mm_trace):
armed, every traced CTA stamps its phases in causal order and names an SM
that exists; the traced launch gives the same output bits as an untraced
one; disarmed, the buffer is left alone.  It measures, it never changes a
result ("[Kernel] Add w8a8 CUTLASS kernels": the matmul the trace watches)."""
import ctypes

import pytest
import torch

import int8_w8a8_scaled_gb300 as w8
from int8_w8a8_scaled_gb300 import _lib

pytestmark = pytest.mark.gpu

SLOTS = 16
START, PROLOGUE, DEP, FIRST, _MMA, EPI, END, SMID = range(8)


def _operands(M, N, K, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    a = torch.randint(0, 126, (M, K), generator=g, device="cuda", dtype=torch.uint8)
    b = torch.randint(0, 126, (N, K), generator=g, device="cuda", dtype=torch.uint8)
    b[:, ::5] |= 0x80
    sa = torch.rand(M, generator=g, device="cuda") * 1e-3
    sb = torch.rand(N, generator=g, device="cuda") * 1e-3
    return (a.view(torch.float8_e4m3fn), b.view(torch.float8_e4m3fn), sa, sb)


def _arm(buf):
    lib = _lib.load()
    if buf is None:
        assert lib.w8a8_debug_mm_trace(None, 0) == 0
    else:
        assert lib.w8a8_debug_mm_trace(ctypes.c_void_p(buf.data_ptr()), buf.numel() * 8) == 0


@pytest.mark.parametrize("M,N,K", [(16, 6144, 4096), (256, 4096, 14336), (1, 28672, 4096)])
def test_trace_stamps_in_order_and_output_unchanged(M, N, K):
    a, b, sa, sb = _operands(M, N, K, seed=M + N)
    ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    w8.scaled_mm(a, b, sa, sb, ref)
    ctas = 4096
    buf = torch.zeros(ctas * SLOTS, dtype=torch.int64, device="cuda")
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    _arm(buf)
    try:
        w8.scaled_mm(a, b, sa, sb, out)
        torch.cuda.synchronize()
    finally:
        _arm(None)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    t = buf.view(ctas, SLOTS).cpu()
    ran = t[:, START] != 0
    assert ran.any()
    # the grid is one contiguous range of CTA indices starting at 0
    n = int(ran.sum())
    assert bool(ran[:n].all()) and not bool(ran[n:].any())
    t = t[:n]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert bool((t[:, SMID] >= 0).all()) and bool((t[:, SMID] < sms).all())
    for lo, hi in ((START, PROLOGUE), (PROLOGUE, DEP), (DEP, FIRST), (EPI, END), (START, END)):
        has = t[:, hi] != 0
        assert bool((t[has, lo] <= t[has, hi]).all()), (lo, hi)
    # disarmed: a later launch leaves the buffer as it was
    before = buf.clone()
    w8.scaled_mm(a, b, sa, sb, out)
    torch.cuda.synchronize()
    assert torch.equal(buf, before)
    assert w8.device_status() == 0
