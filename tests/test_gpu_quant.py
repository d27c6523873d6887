"""GPU quantiser / dequantiser parity: codes and scales bit-exact against the
oracle on the same seeded inputs (all 65536 bf16 and fp16 patterns, dynamic
and static, per-row and per-tensor, ragged, strided and unaligned layouts)."""
import numpy as np
import pytest
import torch

import int8_w8a8_scaled_gb300 as w8
import oracle
import synthetic_inputs as si
from gpu_util import assert_bits16_equal, bits_np, codes_np, q_torch_dtype

pytestmark = pytest.mark.gpu

QDS = [oracle.E4M3, oracle.INT8]


def gpu_quant(x_gpu, qd, per_token, dynamic, scale=None):
    rows, cols = x_gpu.shape
    q = torch.empty(rows, cols, dtype=q_torch_dtype(qd), device="cuda")
    if scale is None:
        s = torch.zeros(rows if per_token else 1, dtype=torch.float32, device="cuda")
    else:
        s = torch.from_numpy(np.asarray(scale, np.float32)).cuda()
    w8.scaled_quant(x_gpu, q, s, per_token=per_token, dynamic=dynamic)
    torch.cuda.synchronize()
    return codes_np(q), s.cpu().numpy()


def oracle_quant(x_cpu, qd, per_token, scale=None):
    xd = oracle.BF16 if x_cpu.dtype == torch.bfloat16 else oracle.FP16
    return oracle.quant(si.bits16(x_cpu), xd, qd, oracle.PER_ROW if per_token else oracle.PER_TENSOR,
                        scale=scale)


def all_patterns(dtype):
    return torch.arange(65536, dtype=torch.int32).to(torch.int16).view(dtype).reshape(256, 256)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("qd", QDS)
@pytest.mark.parametrize("scale", [1.0, 0.37, 2.5e-3, 7.1, 1.0e-30])
def test_sweep_all_16bit_patterns_static(dtype, qd, scale):
    x = all_patterns(dtype)
    g, _ = gpu_quant(x.cuda(), qd, per_token=False, dynamic=False, scale=[scale])
    o, _ = oracle_quant(x, qd, per_token=False, scale=np.array([scale], np.float32))
    assert np.array_equal(g, o)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("qd", QDS)
def test_sweep_all_16bit_patterns_static_per_row(dtype, qd):
    x = all_patterns(dtype)
    scales = np.geomspace(1e-3, 10.0, 256).astype(np.float32)
    g, _ = gpu_quant(x.cuda(), qd, per_token=True, dynamic=False, scale=scales)
    o, _ = oracle_quant(x, qd, per_token=True, scale=scales)
    assert np.array_equal(g, o)


@pytest.mark.parametrize("qd", QDS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("shape", [(1, 16), (3, 4096), (7, 4104), (5, 1000), (64, 28672), (2, 40000),
                                   (300, 512), (1, 7)])
def test_dynamic_per_token(qd, dtype, shape):
    x = si.normal_with_outliers(shape, seed=sum(shape), dtype=dtype)
    g, gs = gpu_quant(x.cuda(), qd, per_token=True, dynamic=True)
    o, os_ = oracle_quant(x, qd, per_token=True)
    assert np.array_equal(gs, os_)
    assert np.array_equal(g, o)


@pytest.mark.parametrize("qd", QDS)
@pytest.mark.parametrize("shape", [(1000, 1000), (1, 5), (4096, 128), (17, 4104), (1, 65536)])
def test_dynamic_per_tensor(qd, shape):
    x = si.normal_with_outliers(shape, seed=shape[0] * 7 + shape[1])
    g, gs = gpu_quant(x.cuda(), qd, per_token=False, dynamic=True)
    o, os_ = oracle_quant(x, qd, per_token=False)
    assert gs[0] == os_[0]
    assert np.array_equal(g, o)


@pytest.mark.parametrize("qd", QDS)
@pytest.mark.parametrize("per_token", [True, False])
def test_strided_views(qd, per_token):
    big = si.normal_with_outliers((40, 3000), seed=12)
    xg = big.cuda()[3:33, 104:2104]          # ld 3000 elements; rows start 16-byte aligned
    xo = big[3:33, 104:2104]
    g, gs = gpu_quant(xg, qd, per_token=per_token, dynamic=True)
    o, os_ = oracle_quant(xo.contiguous(), qd, per_token=per_token)
    assert np.array_equal(gs, os_)
    assert np.array_equal(g, o)
    # unaligned start (odd element offset) -> scalar path
    xg2 = big.cuda()[:, 1:2001]
    g2, gs2 = gpu_quant(xg2, qd, per_token=per_token, dynamic=True)
    o2, os2 = oracle_quant(big[:, 1:2001].contiguous(), qd, per_token=per_token)
    assert np.array_equal(gs2, os2)
    assert np.array_equal(g2, o2)


@pytest.mark.parametrize("qd", QDS)
def test_strided_output(qd):
    x = si.normal_with_outliers((20, 256), seed=3)
    qbig = torch.zeros(20, 512, dtype=q_torch_dtype(qd), device="cuda")
    q = qbig[:, 128:384]
    s = torch.zeros(20, dtype=torch.float32, device="cuda")
    w8.scaled_quant(x.cuda(), q, s, per_token=True, dynamic=True)
    o, os_ = oracle_quant(x, qd, per_token=True)
    big = codes_np(qbig)
    assert np.array_equal(big[:, 128:384], o)
    assert not big[:, :128].any() and not big[:, 384:].any()  # guard bands untouched
    assert np.array_equal(s.cpu().numpy(), os_)


@pytest.mark.parametrize("qd", QDS)
def test_zero_rows_and_specials(qd):
    x = si.normal((6, 64), seed=1).float()
    x[1] = 0.0
    x[2, 5] = float("nan")
    x[3, 7] = float("inf")
    x[4, :] = -0.0
    x[5, 9] = -float("inf")
    x = x.to(torch.bfloat16)
    g, gs = gpu_quant(x.cuda(), qd, per_token=True, dynamic=True)
    o, os_ = oracle_quant(x, qd, per_token=True)
    assert np.array_equal(gs, os_)
    assert gs[1] == 1.0 and gs[4] == 1.0
    assert np.array_equal(g, o)


@pytest.mark.parametrize("qd", QDS)
def test_per_tensor_equals_broadcast_per_row(qd):
    x = si.normal_with_outliers((64, 1024), seed=5).cuda()
    s = 0.0371
    a, _ = gpu_quant(x, qd, per_token=False, dynamic=False, scale=[s])
    b, _ = gpu_quant(x, qd, per_token=True, dynamic=False, scale=[s] * 64)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("qd", QDS)
@pytest.mark.parametrize("yd", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("per_token", [False, True])
def test_dequant_all_codes(qd, yd, per_token):
    codes = np.tile(np.arange(256, dtype=np.uint8), (64, 4))  # [64, 1024]
    scales = np.geomspace(1e-4, 30.0, 64).astype(np.float32) if per_token else np.array([0.0123], np.float32)
    qg = torch.from_numpy(codes).cuda().view(q_torch_dtype(qd))
    y = torch.empty(64, 1024, dtype=yd, device="cuda")
    w8.scaled_dequant(qg, torch.from_numpy(scales).cuda(), y, per_token=per_token)
    od = oracle.BF16 if yd == torch.bfloat16 else oracle.FP16
    want = oracle.dequant(codes, qd, scales, oracle.PER_ROW if per_token else oracle.PER_TENSOR, od)
    assert_bits16_equal(bits_np(y), want, od, "dequant")


def test_dequant_strided_and_odd_sizes():
    codes = np.random.default_rng(0).integers(0, 256, size=(9, 301)).astype(np.uint8)
    qbig = torch.zeros(9, 320, dtype=torch.uint8, device="cuda")
    qbig[:, 3:304] = torch.from_numpy(codes).cuda()
    q = qbig[:, 3:304].view(torch.float8_e4m3fn)
    y = torch.empty(9, 301, dtype=torch.bfloat16, device="cuda")
    s = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    w8.scaled_dequant(q, s, y, per_token=False)
    want = oracle.dequant(codes, oracle.E4M3, np.array([0.5], np.float32), oracle.PER_TENSOR, oracle.BF16)
    assert_bits16_equal(bits_np(y), want, oracle.BF16)


def test_quant_dequant_round_trip_kv_shape():
    """KV-cache round trip at a reduced size (full size is in the full-size
    tests): bit-exact codes, scale and dequant."""
    k = si.kv_with_spikes(4096, 8, 128, seed=41).reshape(-1, 128)
    g, gs = gpu_quant(k.cuda(), oracle.E4M3, per_token=False, dynamic=True)
    o, os_ = oracle_quant(k, oracle.E4M3, per_token=False)
    assert gs[0] == os_[0] and np.array_equal(g, o)
    qg = torch.from_numpy(g).cuda().view(torch.float8_e4m3fn)
    y = torch.empty_like(k, device="cuda")
    w8.scaled_dequant(qg, torch.from_numpy(gs).cuda(), y)
    want = oracle.dequant(o, oracle.E4M3, os_, oracle.PER_TENSOR, oracle.BF16)
    assert_bits16_equal(bits_np(y), want, oracle.BF16)


def test_no_device_timeouts_recorded():
    assert w8.device_status() == 0


@pytest.mark.parametrize("qd", QDS)
def test_all_bf16_patterns_under_many_scales(qd):
    """The quantiser takes the code from a reciprocal multiply where that
    provably equals the code of the IEEE quotient: every bf16 pattern under
    64 random static scales, bit-exact against the oracle."""
    rng = np.random.default_rng(17)
    scales = np.exp(rng.uniform(np.log(1e-4), np.log(30.0), 64)).astype(np.float32)
    x = all_patterns(torch.bfloat16).reshape(1, -1).repeat(64, 1)   # [64, 65536]
    g, _ = gpu_quant(x.cuda(), qd, per_token=True, dynamic=False, scale=scales)
    o, _ = oracle_quant(x, qd, per_token=True, scale=scales)
    assert np.array_equal(g, o)


def _near_decision_points(qd, dtype, seed):
    """Inputs whose quotient by a random scale lands within a few 16-bit ulps
    of every decision point of the encoder (e4m3 midpoints, int8 halves)."""
    rng = np.random.default_rng(seed)
    if qd == oracle.E4M3:
        vals = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
        mids = (vals[:-1] + vals[1:]) / 2
    else:
        mids = np.arange(-128, 128) + 0.5
    rows, scales = [], []
    for _ in range(32):
        s = np.float32(np.exp(rng.uniform(np.log(1e-3), np.log(10.0))))
        t = torch.tensor(np.concatenate([mids, -mids]) * float(s), dtype=torch.float32).to(dtype)
        bits = t.view(torch.int16).to(torch.int32)
        nb = torch.cat([bits + d for d in (-3, -2, -1, 0, 1, 2, 3)])
        rows.append(nb.to(torch.int16).view(dtype))
        scales.append(s)
    n = min(r.numel() for r in rows)
    return torch.stack([r[:n] for r in rows]), np.array(scales, np.float32)


@pytest.mark.parametrize("qd", QDS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_inputs_at_decision_points(qd, dtype):
    x, scales = _near_decision_points(qd, dtype, seed=5)
    g, _ = gpu_quant(x.cuda(), qd, per_token=True, dynamic=False, scale=scales)
    o, _ = oracle_quant(x, qd, per_token=True, scale=scales)
    assert np.array_equal(g, o)
    # the same rows through the flat per-tensor kernel, one scale at a time
    for i in range(0, 32, 8):
        xi = x[i:i + 1].repeat(64, 1)
        g1, _ = gpu_quant(xi.cuda(), qd, per_token=False, dynamic=False, scale=[scales[i]])
        o1, _ = oracle_quant(xi, qd, per_token=False, scale=np.array([scales[i]], np.float32))
        assert np.array_equal(g1, o1)


def _patterns_up_to(dtype, amax):
    """Every 16-bit pattern whose magnitude is <= amax (NaNs included: the
    absmax ignores them), padded with zeros to 65536, plus amax itself."""
    allp = all_patterns(dtype).reshape(-1)
    f = allp.float()
    keep = (f.abs() <= amax) | torch.isnan(f)
    row = torch.zeros(65536, dtype=dtype)
    sel = allp[keep]
    row[:sel.numel()] = sel
    row[-1] = torch.tensor(amax, dtype=torch.float32).to(dtype)
    return row


DYN_AMAX = {torch.bfloat16: [1.0, 0.37, 448.0, 2.5e-3, 7.1, 1.0e-30, 3.0e38, 127.0, 65504.0, 1.5e-38],
            torch.float16: [1.0, 0.37, 448.0, 2.5e-3, 7.1, 65504.0, 127.0, 6.1e-5, 3.0e-7]}


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("qd", QDS)
def test_dynamic_rows_of_every_pattern_below_their_absmax(dtype, qd):
    """Dynamic per-row scales with every representable input at or below each
    row's absmax: the codes of the whole sweep bit-exact against the oracle
    (the quotient of a dynamic scale never leaves the code range)."""
    x = torch.stack([_patterns_up_to(dtype, a) for a in DYN_AMAX[dtype]])
    g, gs = gpu_quant(x.cuda(), qd, per_token=True, dynamic=True)
    o, os_ = oracle_quant(x, qd, per_token=True)
    assert np.array_equal(gs, os_)
    assert np.array_equal(g, o)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("qd", QDS)
@pytest.mark.parametrize("amax", [0.37, 448.0, 65504.0])
def test_dynamic_tensor_of_every_pattern_below_its_absmax(dtype, qd, amax):
    x = _patterns_up_to(dtype, amax).reshape(256, 256)
    g, gs = gpu_quant(x.cuda(), qd, per_token=False, dynamic=True)
    o, os_ = oracle_quant(x, qd, per_token=False)
    assert gs[0] == os_[0]
    assert np.array_equal(g, o)
