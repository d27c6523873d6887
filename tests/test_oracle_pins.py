"""Pins for the CPU oracle: it is checked here against things other than
itself -- library routines (torch's float8_e4m3fn / bfloat16 casts, numpy's
float16 and rint), exact rational arithmetic, closed forms and hand-worked
examples from the source pages (tests/golden/worked_examples.json).

Each test is chosen so that a plausible slip in the oracle (a wrong rounding
tie, a dropped sign, a swapped operand, a wrong scale order) fails it.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


# ---------------------------------------------------------------- helpers

def torch_e4m3_values(codes):
    """Library decode of e4m3fn codes."""
    t = torch.tensor(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy().astype(np.float64)


def torch_e4m3_encode(v):
    """The pages' own quantiser expression: clamp to the finite range, then
    cast (torch's cast rounds to nearest even)."""
    t = torch.from_numpy(np.asarray(v, dtype=np.float32))
    t = t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def all_bf16_patterns():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def e4m3_ulp(v):
    v = abs(float(v))
    if v < 2.0 ** -6:
        return 2.0 ** -9
    return 2.0 ** (math.floor(math.log2(v)) - 3)


def arithmetic_e4m3_encode(v):
    """Second, independent encoder: frexp-based round-half-even on the
    significand, written without the value table."""
    v = float(v)
    if math.isnan(v):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if a >= 448.0:
        return sign | 0x7E
    if a < 2.0 ** -6:  # subnormal range, quantum 2^-9
        n = a / 2.0 ** -9
        r = round(n)  # Python rounds half to even
        if r == 8:
            return sign | 0x08
        return sign | int(r)
    m, e = math.frexp(a)  # a = m * 2^e, m in [0.5, 1)
    sig = m * 16.0  # in [8, 16): 1 implicit + 3 fraction bits
    r = round(sig)
    if r == 16:
        r = 8
        e += 1
    exp_field = e - 1 + 7
    code = (exp_field << 3) | (int(r) - 8)
    if code > 0x7E:
        code = 0x7E
    return sign | code


# ---------------------------------------------------------------- e4m3 table

def test_e4m3_table_matches_library_decode():
    codes = np.arange(256)
    ours = np.array([oracle.e4m3_value(c) for c in codes])
    lib = torch_e4m3_values(codes)
    nan_ours = np.isnan(ours)
    assert np.array_equal(nan_ours, np.isnan(lib))
    assert set(np.nonzero(nan_ours)[0]) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan_ours], lib[~nan_ours])
    # signs of zero
    assert math.copysign(1.0, oracle.e4m3_value(0x80)) < 0


def test_e4m3_spot_values():
    # MAXNORM = 448 is printed on the KV-cache page (Scaling semantics).
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0xFE) == -448.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6   # smallest normal
    assert oracle.e4m3_value(0x01) == 2.0 ** -9   # smallest subnormal
    assert oracle.e4m3_value(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_value(0x38) == 1.0
    assert math.isnan(oracle.e4m3_value(0x7F))


# ---------------------------------------------------------------- encoders

@pytest.mark.parametrize("scale", [1.0, 0.37, 2.5e-3, 7.1, 1.0e-30])
def test_e4m3_quant_sweep_all_bf16_matches_page_expression(scale):
    """All 65536 bf16 patterns, static per-tensor scale: the oracle equals the
    clamp-then-cast expression of the CUTLASS review thread, computed by
    torch (x / s in fp32, clamp to +-448, RNE cast)."""
    bits = all_bf16_patterns().reshape(256, 256)
    q, _ = oracle.quant(bits, oracle.BF16, oracle.E4M3, oracle.PER_TENSOR,
                        scale=np.array([scale], np.float32))
    x = torch.from_numpy(bf16_bits_to_f32(bits))
    v = (x / torch.tensor(np.float32(scale))).numpy()
    ref = torch_e4m3_encode(v)
    nan = np.isnan(v)
    assert np.all(q[nan] == 0x7F)  # NaN reading: canonical positive NaN
    assert np.array_equal(q[~nan], ref[~nan])


def test_e4m3_two_encoders_agree_on_sweep():
    bits = all_bf16_patterns()
    vals = bf16_bits_to_f32(bits)
    table = oracle.encode_e4m3(vals)
    arith = np.array([arithmetic_e4m3_encode(v) for v in vals], dtype=np.uint8)
    assert np.array_equal(table, arith)


def test_e4m3_midpoints_tie_to_even():
    # every midpoint between adjacent finite codes, both signs
    vals, expect = [], []
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_value(c), oracle.e4m3_value(c + 1)
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        vals += [mid, -mid]
        expect += [even, even | 0x80]
    vals = np.array(vals, dtype=np.float32)
    assert np.all(vals.astype(np.float64) == np.array(
        [(oracle.e4m3_value(c) + oracle.e4m3_value(c + 1)) / 2 * s
         for c in range(0, 0x7E) for s in (1, -1)]))  # midpoints exact in fp32
    assert np.array_equal(oracle.encode_e4m3(vals), np.array(expect, dtype=np.uint8))


def test_e4m3_saturation_and_specials():
    v = np.array([448.0, 449.0, 464.0, 480.0, 1e30, np.inf, -np.inf, np.nan,
                  -np.nan, 0.0, -0.0, -1e-30], dtype=np.float32)
    got = oracle.encode_e4m3(v)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F, 0x7F,
                         0x00, 0x80, 0x80]


@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.3])
def test_int8_quant_sweep_matches_numpy(scale):
    bits = all_bf16_patterns().reshape(256, 256)
    q, _ = oracle.quant(bits, oracle.BF16, oracle.INT8, oracle.PER_TENSOR,
                        scale=np.array([scale], np.float32))
    v = bf16_bits_to_f32(bits) / np.float32(scale)
    with np.errstate(invalid="ignore"):
        ref = np.clip(np.rint(v.astype(np.float64)), -128, 127)
    ref = np.where(np.isnan(v), 0, ref).astype(np.int8).view(np.uint8)
    assert np.array_equal(q, ref)


# ---------------------------------------------------------------- 16-bit floats

def test_bf16_decode_all_patterns():
    bits = all_bf16_patterns()
    ours = oracle.bits16_to_f32(bits, oracle.BF16)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    m = ~np.isnan(lib)
    assert np.array_equal(ours[m].view(np.uint32), lib[m].view(np.uint32))


def test_fp16_decode_all_patterns():
    bits = all_bf16_patterns()
    ours = oracle.bits16_to_f32(bits, oracle.FP16)
    lib = bits.view(np.float16).astype(np.float32)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    m = ~np.isnan(lib)
    assert np.array_equal(ours[m].view(np.uint32), lib[m].view(np.uint32))


def _special_f32():
    rng = np.random.default_rng(5)
    raw = rng.integers(0, 2 ** 32, size=40000, dtype=np.uint64).astype(np.uint32)
    vals = raw.view(np.float32)
    # values near bf16/fp16 rounding boundaries and ranges
    base = rng.standard_normal(20000).astype(np.float32) * np.float32(1000)
    extra = np.array([0.0, -0.0, np.inf, -np.inf, 65504, 65519.99, 65520, 65536,
                      6.0e-8, 5.96e-8, 2.98e-8, 2.99e-8, 1e-40, -1e-45, 3.4e38,
                      3.3961e38, 3.3963e38], dtype=np.float32)
    halfway = (np.arange(1, 3000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    return np.concatenate([vals, base, extra, halfway])


def test_bf16_rounding_matches_torch():
    v = _special_f32()
    ours = oracle.f32_to_bf16_bits(v)
    lib = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(v)
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.all((ours[nan] & 0x7F80) == 0x7F80) and np.all(ours[nan] & 0x7F)


def test_fp16_rounding_matches_numpy():
    v = _special_f32()
    ours = oracle.f32_to_f16_bits(v)
    with np.errstate(over="ignore"):
        lib = v.astype(np.float16).view(np.uint16)
    nan = np.isnan(v)
    assert np.array_equal(ours[~nan], lib[~nan])


# ---------------------------------------------------------------- scale semantics

@pytest.mark.parametrize("q_dtype,qmax,code_max", [(oracle.E4M3, 448.0, 0x7E),
                                                   (oracle.INT8, 127.0, 127)])
def test_dynamic_absmax_element_hits_qmax(q_dtype, qmax, code_max):
    """Scaling semantics (KV-cache page): scale = absmax / 448, so the absmax
    element lands on the largest code (+-448, or +-127 for int8)."""
    x = si.normal_with_outliers((48, 300), seed=11)
    x[5].zero_()
    bits = si.bits16(x)
    q, s = oracle.quant(bits, oracle.BF16, q_dtype, oracle.PER_ROW)
    xf = x.float().numpy()
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(s[amax > 0], (amax[amax > 0] / np.float32(qmax)).astype(np.float32))
    assert s[5] == 1.0 and np.all(q[5] == 0)   # zero row: scale 1.0, codes 0
    for i in range(48):
        if amax[i] == 0:
            continue
        j = int(np.argmax(np.abs(xf[i])))
        code = int(q[i, j])
        if q_dtype == oracle.E4M3:
            assert code & 0x7F == code_max and (code >> 7) == (xf[i, j] < 0)
        else:
            assert abs(np.int8(np.uint8(code))) == code_max
    if q_dtype == oracle.E4M3:
        vals = torch_e4m3_values(q.ravel())
        assert np.all(np.abs(vals) <= 448)


def test_scale_from_absmax_closed_form():
    assert oracle.scale_from_absmax(448.0, oracle.E4M3) == 1.0
    assert oracle.scale_from_absmax(3.5, oracle.E4M3) == 2.0 ** -7
    assert oracle.scale_from_absmax(127.0, oracle.INT8) == 1.0
    assert oracle.scale_from_absmax(0.0, oracle.E4M3) == 1.0  # no scale -> 1.0


def test_per_tensor_dynamic_equals_static_with_same_scale():
    x = si.normal_with_outliers((64, 96), seed=3)
    bits = si.bits16(x)
    qd, sd = oracle.quant(bits, oracle.BF16, oracle.E4M3, oracle.PER_TENSOR)
    amax = np.abs(x.float().numpy()).max()
    assert sd[0] == np.float32(amax) / np.float32(448.0)
    qs, _ = oracle.quant(bits, oracle.BF16, oracle.E4M3, oracle.PER_TENSOR, scale=sd)
    assert np.array_equal(qd, qs)


@pytest.mark.parametrize("q_dtype", [oracle.E4M3, oracle.INT8])
def test_per_tensor_equals_broadcast_per_row(q_dtype):
    x = si.normal_with_outliers((40, 72), seed=4)
    bits = si.bits16(x)
    s = np.float32(0.0371)
    q1, _ = oracle.quant(bits, oracle.BF16, q_dtype, oracle.PER_TENSOR, scale=np.array([s]))
    q2, _ = oracle.quant(bits, oracle.BF16, q_dtype, oracle.PER_ROW,
                         scale=np.full(40, s, np.float32))
    assert np.array_equal(q1, q2)
    y1 = oracle.dequant(q1, q_dtype, np.array([s]), oracle.PER_TENSOR, oracle.BF16)
    y2 = oracle.dequant(q2, q_dtype, np.full(40, s, np.float32), oracle.PER_ROW, oracle.BF16)
    assert np.array_equal(y1, y2)


def test_round_trip_bound_e4m3():
    """quant -> dequant error is at most half an e4m3 ulp of x/s, times s
    (plus fp32 rounding), for |x/s| <= 448."""
    x = si.normal_with_outliers((64, 512), seed=21)
    bits = si.bits16(x)
    q, s = oracle.quant(bits, oracle.BF16, oracle.E4M3, oracle.PER_ROW)
    xf = x.float().numpy().astype(np.float64)
    d = torch_e4m3_values(q.ravel()).reshape(q.shape)
    deq32 = (d.astype(np.float32) * s[:, None]).astype(np.float64)
    v = np.abs(xf / s[:, None].astype(np.float64))
    ulp = np.vectorize(e4m3_ulp)(v)
    bound = 0.5 * ulp * s[:, None] * (1 + 2.0 ** -20) + 2.0 ** -23 * np.abs(xf)
    assert np.all(np.abs(deq32 - xf) <= bound)
    # the oracle's bf16 dequant is the fp32 value rounded once more
    y = oracle.dequant(q, oracle.E4M3, s, oracle.PER_ROW, oracle.BF16)
    yb = torch.from_numpy(y.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.all(np.abs(yb - deq32) <= 2.0 ** -8 * np.abs(deq32))  # bf16 unit roundoff


# ---------------------------------------------------------------- golden

def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _f32_to_bf16_bits_torch(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("case", _golden()["quant_cases"], ids=lambda c: c["name"])
def test_golden_quant(case):
    qd = oracle.E4M3 if case["q_dtype"] == "e4m3" else oracle.INT8
    gran = oracle.PER_ROW if case["gran"] == "per_row" else oracle.PER_TENSOR
    bits = _f32_to_bf16_bits_torch(case["x"]).reshape(1, -1)
    scale = None if case["mode"] == "dynamic" else np.array(case["scale"], np.float32)
    q, s = oracle.quant(bits, oracle.BF16, qd, gran, scale=scale)
    assert list(s) == case["scale"]
    if qd == oracle.E4M3:
        assert list(q.ravel()) == case["codes"]
    else:
        assert list(q.ravel().view(np.int8)) == case["codes"]
    y = oracle.dequant(q, qd, s, gran, oracle.BF16)
    want = _f32_to_bf16_bits_torch(case["dequant_bf16"])
    assert np.array_equal(y.ravel(), want)


@pytest.mark.parametrize("case", _golden()["mm_cases"], ids=lambda c: c["name"])
def test_golden_mm(case):
    qd = oracle.E4M3 if case["q_dtype"] == "e4m3" else oracle.INT8
    if qd == oracle.E4M3:
        A = np.array(case["A_codes"], np.uint8)
        B = np.array(case["B_codes"], np.uint8)
        assert np.array_equal(torch_e4m3_values(A), np.array(case["A_values"]))
        assert np.array_equal(torch_e4m3_values(B), np.array(case["B_values"]))
    else:
        A = np.array(case["A_codes"], np.int8)
        B = np.array(case["B_codes"], np.int8)
    for od, key in ((oracle.BF16, "out_bf16"), (oracle.FP16, "out_fp16")):
        if key not in case:
            continue
        r = oracle.scaled_mm(A, B, case["scale_a"], case["scale_b"], qd, od)
        assert np.array_equal(r["acc"], np.array(case["acc"], np.float64))
        assert np.array_equal(r["y"], np.array(case["y"], np.float32))
        want = np.array(case[key], np.float32)
        if od == oracle.BF16:
            got = torch.from_numpy(r["out"].view(np.int16)).view(torch.bfloat16).float().numpy()
        else:
            got = r["out"].view(np.float16).astype(np.float32)
        assert np.array_equal(got, want)


# ---------------------------------------------------------------- GEMM

def _finite_e4m3_codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    # force some extremes, subnormals and signed zeros
    flat = c.reshape(-1)
    picks = rng.integers(0, flat.size, size=max(1, flat.size // 8))
    flat[picks] = rng.choice(np.array([0x7E, 0xFE, 0x01, 0x81, 0x80, 0x00, 0x07], np.uint8),
                             size=picks.size)
    return c


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (3, 5, 7, 1), (8, 6, 16, 2),
                                        (16, 16, 16, 3), (5, 9, 33, 4)])
def test_fp8_mm_exact_rational(M, N, K, seed):
    rng = np.random.default_rng(seed)
    A = _finite_e4m3_codes(rng, (M, K))
    B = _finite_e4m3_codes(rng, (N, K))
    sa = (rng.random(M) * 0.01 + 1e-4).astype(np.float32)
    sb = (rng.random(N) * 0.02 + 1e-5).astype(np.float32)
    r = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.BF16)
    Av = [[Fraction(float(v)) for v in row] for row in torch_e4m3_values(A)]
    Bv = [[Fraction(float(v)) for v in row] for row in torch_e4m3_values(B)]
    for m in range(M):
        for n in range(N):
            exact = sum(Av[m][k] * Bv[n][k] for k in range(K))
            assert Fraction(r["acc"][m, n]) == exact
            # epilogue: three roundings of an exact product, each <= 2^-24 rel.
            full = exact * Fraction(float(sa[m])) * Fraction(float(sb[n]))
            err = abs(Fraction(float(r["y"][m, n])) - full)
            assert err <= abs(full) * Fraction(3, 2 ** 24) * Fraction(1001, 1000)
    # 16-bit output is one RNE of y (library cast)
    want = torch.from_numpy(r["y"]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r["out"], want)


@pytest.mark.parametrize("M,N,K,seed", [(2, 3, 5, 0), (7, 4, 64, 1), (4, 4, 1000, 2)])
def test_int8_mm_exact_integer(M, N, K, seed):
    rng = np.random.default_rng(seed)
    A = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    B = rng.integers(-128, 128, size=(N, K)).astype(np.int8)
    sa = (rng.random(M) * 0.05).astype(np.float32)
    sb = (rng.random(N) * 0.05).astype(np.float32)
    r = oracle.scaled_mm(A, B, sa, sb, oracle.INT8, oracle.FP16)
    exact = [[sum(int(A[m, k]) * int(B[n, k]) for k in range(K)) for n in range(N)]
             for m in range(M)]
    assert np.array_equal(r["iacc"], np.array(exact, np.int64))
    want = r["y"].astype(np.float16).view(np.uint16)
    assert np.array_equal(r["out"], want)


def test_int8_extremes_long_k_no_overflow():
    K = 28672
    A = np.full((2, K), -128, np.int8)
    A[1] = 127
    B = np.full((2, K), -128, np.int8)
    B[1] = 127
    r = oracle.scaled_mm(A, B, np.ones(2, np.float32), np.ones(2, np.float32),
                         oracle.INT8, oracle.FP16)
    assert r["iacc"][0, 0] == 128 * 128 * K
    assert r["iacc"][0, 1] == -128 * 127 * K
    assert r["iacc"][1, 1] == 127 * 127 * K
    assert abs(r["iacc"]).max() < 2 ** 31


def test_fp8_all_max_closed_form():
    K = 4096
    A = np.full((2, K), 0x7E, np.uint8)
    A[1] = 0xFE
    B = np.full((1, K), 0x7E, np.uint8)
    r = oracle.scaled_mm(A, B, [1.0], [1.0], oracle.E4M3, oracle.BF16)
    assert r["acc"][0, 0] == 448.0 * 448.0 * K
    assert r["acc"][1, 0] == -448.0 * 448.0 * K


def test_fp8_one_hot_b_selects_columns():
    """B = one-hot rows of 1.0 (code 0x38): out[m, n] = round(dec(A[m, k_n]) * sa * sb)."""
    rng = np.random.default_rng(9)
    M, K, N = 6, 32, 5
    A = _finite_e4m3_codes(rng, (M, K))
    ks = rng.choice(K, size=N, replace=False)
    B = np.zeros((N, K), np.uint8)
    B[np.arange(N), ks] = 0x38
    sa = np.float32(0.75)
    sb = (rng.random(N) + 0.5).astype(np.float32)
    r = oracle.scaled_mm(A, B, [sa], sb, oracle.E4M3, oracle.BF16)
    a = torch.from_numpy(torch_e4m3_values(A[:, ks]).astype(np.float32))
    ref = (a * torch.tensor(sa)) * torch.from_numpy(sb)[None, :]
    want = ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r["out"], want)


def test_operand_order_matters():
    """A transposed-operand slip would swap the roles of the two scales; use
    distinct per-token and per-channel scales to catch it."""
    rng = np.random.default_rng(2)
    A = _finite_e4m3_codes(rng, (3, 16))
    B = _finite_e4m3_codes(rng, (4, 16))
    sa = np.array([1.0, 2.0, 4.0], np.float32)
    sb = np.array([1.0, 8.0, 64.0, 512.0], np.float32)
    r = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.FP16)
    exact = torch_e4m3_values(A) @ torch_e4m3_values(B).T
    assert np.array_equal(r["acc"], exact)  # small exact case: float64 matmul exact
    assert np.allclose(r["y"], exact * sa[:, None] * sb[None, :], rtol=1e-6)


def test_sample_equals_full():
    rng = np.random.default_rng(7)
    A = _finite_e4m3_codes(rng, (9, 48))
    B = _finite_e4m3_codes(rng, (11, 48))
    sa = rng.random(9).astype(np.float32)
    sb = rng.random(11).astype(np.float32)
    full = oracle.scaled_mm(A, B, sa, sb, oracle.E4M3, oracle.BF16)
    im = rng.integers(0, 9, 30)
    inn = rng.integers(0, 11, 30)
    smp = oracle.scaled_mm_sample(A, B, sa, sb, oracle.E4M3, oracle.BF16, im, inn)
    assert np.array_equal(smp["out"], full["out"][im, inn])
    assert np.array_equal(smp["acc"], full["acc"][im, inn])


def test_strided_views():
    """Leading dimensions larger than the row length (sub-matrices)."""
    rng = np.random.default_rng(8)
    big_a = _finite_e4m3_codes(rng, (10, 80))
    big_b = _finite_e4m3_codes(rng, (12, 96))
    A = big_a[2:7, 16:48]
    B = big_b[1:9, 32:64]
    r1 = oracle.scaled_mm(A, B, [0.5], [0.25], oracle.E4M3, oracle.BF16)
    r2 = oracle.scaled_mm(np.ascontiguousarray(A), np.ascontiguousarray(B), [0.5],
                          [0.25], oracle.E4M3, oracle.BF16)
    assert np.array_equal(r1["out"], r2["out"])
    x = si.normal((20, 64), seed=1)
    bits = si.bits16(x)
    q1, s1 = oracle.quant(bits[3:15, 8:40], oracle.BF16, oracle.E4M3, oracle.PER_ROW)
    q2, s2 = oracle.quant(np.ascontiguousarray(bits[3:15, 8:40]), oracle.BF16,
                          oracle.E4M3, oracle.PER_ROW)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_fp16_input_quant():
    x = si.normal_with_outliers((16, 64), seed=6, dtype=torch.float16)
    bits = si.bits16(x)
    q, s = oracle.quant(bits, oracle.FP16, oracle.E4M3, oracle.PER_ROW)
    xf = x.float()
    ref = torch_e4m3_encode((xf / torch.from_numpy(s)[:, None]).numpy())
    assert np.array_equal(q, ref)


# ---------------------------------------------------------------- merged-layer shards

def _shards(seed, qd=oracle.E4M3):
    rows = (48, 16, 16)                      # e.g. q / k / v row blocks
    parts, scales = [], []
    for i, r in enumerate(rows):
        x = si.normal((r, 64), seed=seed + i, std=0.02 * (1 + i))
        q, s = oracle.quant(si.bits16(x), oracle.BF16, qd, oracle.PER_TENSOR)
        parts.append(q)
        scales.append(s[0])
    return np.concatenate(parts), np.array(scales, np.float32), np.array(rows)


def test_requant_shards_matches_page_expression():
    """w_scale = max(shard scales); w_i' = (s_i / w_scale) * w_i, cast back
    to e4m3 (torch's clamp-then-cast as the library reference)."""
    q, ss, rows = _shards(31)
    out, smax = oracle.requant_shards(q, oracle.E4M3, ss, rows)
    assert smax[0] == ss.max()
    row0 = 0
    for i, r in enumerate(rows):
        ratio = torch.tensor(np.float32(ss[i]) / np.float32(smax[0]))
        v = torch.from_numpy(torch_e4m3_values(q[row0:row0 + r]).astype(np.float32)) * ratio
        want = v.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(out[row0:row0 + r], want)
        row0 += r


def test_requant_shards_max_shard_unchanged_and_error_bound():
    q, ss, rows = _shards(37)
    out, smax = oracle.requant_shards(q, oracle.E4M3, ss, rows)
    imax = int(np.argmax(ss))
    starts = np.concatenate([[0], np.cumsum(rows)])
    sl = slice(starts[imax], starts[imax + 1])
    assert np.array_equal(out[sl], q[sl])          # ratio 1: codes unchanged
    before = torch_e4m3_values(q) * np.repeat(ss, rows)[:, None]
    after = torch_e4m3_values(out) * float(smax[0])
    v = np.abs(before / float(smax[0]))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    half_ulp = 0.5 * np.where(v < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3)) * float(smax[0])
    assert np.all(np.abs(after - before) <= half_ulp * (1 + 2.0 ** -20) + 2.0 ** -22 * np.abs(before))


def test_requant_shards_power_of_two_ratio_is_exact():
    q = np.array([[0x38, 0x40, 0xB0, 0x50, 0x01, 0x7E]], np.uint8)   # 1, 2, -0.5, 8, 2^-9, 448
    out, smax = oracle.requant_shards(np.concatenate([q, q]), oracle.E4M3,
                                      np.array([0.5, 1.0], np.float32), [1, 1])
    assert smax[0] == 1.0
    assert list(torch_e4m3_values(out[0])) == [0.5, 1.0, -0.25, 4.0, 0.0, 224.0]  # 2^-10 ties to 0
    assert np.array_equal(out[1], q[0])


def test_requant_shards_int8():
    q, ss, rows = _shards(41, qd=oracle.INT8)
    out, smax = oracle.requant_shards(q, oracle.INT8, ss, rows)
    row0 = 0
    for i, r in enumerate(rows):
        ratio = np.float32(ss[i]) / np.float32(smax[0])
        v = q[row0:row0 + r].view(np.int8).astype(np.float32) * ratio
        want = np.clip(np.rint(v.astype(np.float64)), -128, 127).astype(np.int8).view(np.uint8)
        assert np.array_equal(out[row0:row0 + r], want)
        row0 += r


def test_per_shard_scales_equal_expanded_per_channel():
    """A per-shard weight scale is a per-output-channel scale that is constant
    over each shard: the fused-epilogue reading of the merged layer."""
    rng = np.random.default_rng(3)
    A = _finite_e4m3_codes(rng, (5, 64))
    B, ss, rows = _shards(43)
    sa = (rng.random(5) * 0.01).astype(np.float32)
    per_channel = np.repeat(ss, rows).astype(np.float32)
    full = oracle.scaled_mm(A, B, sa, per_channel, oracle.E4M3, oracle.BF16)
    starts = np.concatenate([[0], np.cumsum(rows)])
    for i in range(len(rows)):
        part = oracle.scaled_mm(A, B[starts[i]:starts[i + 1]], sa, [ss[i]], oracle.E4M3, oracle.BF16)
        assert np.array_equal(full["out"][:, starts[i]:starts[i + 1]], part["out"])
