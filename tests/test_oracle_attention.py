"""Pins of the fp8-KV decode attention oracle ("Enable scaled FP8 (e4m3fn) KV
cache on ROCm (AMD GPU)", section "Scaling semantics": dequantised value =
decode(code) * scaling_factor, per-tensor factors for K and V), against
things other than itself: brute force with Python scalars, closed forms, and
layout / head-grouping invariances."""
import math

import numpy as np
import pytest

import oracle
from oracle import attention as oa


def random_case(B, Hq, Hkv, T, D, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    q_bits = oracle.f32_to_bf16_bits(q)
    # codes of finite e4m3 values only (not 0x7F / 0xFF), both signs
    k = rng.integers(0, 0x7F, (B, T, Hkv, D), dtype=np.uint8) | (rng.integers(0, 2, (B, T, Hkv, D), dtype=np.uint8) << 7)
    v = rng.integers(0, 0x7F, (B, T, Hkv, D), dtype=np.uint8) | (rng.integers(0, 2, (B, T, Hkv, D), dtype=np.uint8) << 7)
    return q_bits, k, v


def test_e4m3_table_spot_values():
    t = oa.e4m3_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0      # MAXNORM of the scaling semantics
    assert t[0x08] == 2.0 ** -6 and t[0x01] == 2.0 ** -9 and t[0x00] == 0.0
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert t[0x38] == 1.0


def test_bruteforce_agrees_on_tiny_inputs():
    B, Hq, Hkv, T, D = 2, 4, 2, 5, 8
    q_bits, k, v = random_case(B, Hq, Hkv, T, D, seed=1)
    lens = np.array([5, 3], np.int32)
    ks, vs, sm = 0.03125, 0.0078125, 0.35
    got = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, lens, ks, vs, sm)
    q = oracle.bits16_to_f32(q_bits, oracle.BF16)
    tab = [oracle.e4m3_value(c) for c in range(256)]
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            K = [[tab[int(c)] * ks for c in k[b, t, g]] for t in range(lens[b])]
            V = [[tab[int(c)] * vs for c in v[b, t, g]] for t in range(lens[b])]
            ref = oa.attention_bruteforce([float(x) for x in q[b, h]], K, V, sm)
            np.testing.assert_allclose(got[b, h], ref, rtol=1e-12, atol=1e-15)


def test_single_token_returns_its_value_row():
    """softmax over one token is 1: the output is that token's dequantised V."""
    B, Hq, Hkv, T, D = 1, 2, 1, 4, 16
    q_bits, k, v = random_case(B, Hq, Hkv, T, D, seed=2)
    out = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, np.array([1], np.int32), 0.5, 0.25, 1.0)
    want = oa.e4m3_table()[v[0, 0, 0]] * 0.25
    for h in range(Hq):
        np.testing.assert_array_equal(out[0, h], want)


def test_equal_keys_average_the_values():
    """Identical keys give uniform weights: the output is the mean of V."""
    B, Hq, Hkv, T, D = 1, 1, 1, 7, 16
    q_bits, k, v = random_case(B, Hq, Hkv, T, D, seed=3)
    k[:] = k[0, 0]
    out = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, np.array([T], np.int32), 1.0, 2.0, 0.7)
    want = (oa.e4m3_table()[v[0, :, 0]] * 2.0).mean(axis=0)
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-14, atol=1e-14)


def test_dominant_key_selects_its_value():
    """A key whose score exceeds all others by ~1000 takes all the weight."""
    B, Hq, Hkv, T, D = 1, 1, 1, 6, 16
    q = np.zeros((B, Hq, D), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((B, T, Hkv, D), np.uint8)                 # zero keys ...
    k[0, 4, 0, 0] = 0x7E                                    # ... except token 4: k[0] = 448
    _, _, v = random_case(B, Hq, Hkv, T, D, seed=4)
    out = oa.fp8_kv_decode_attention(oracle.f32_to_bf16_bits(q), oracle.BF16, k, v, np.array([T], np.int32),
                                     1.0, 1.0, 2.5)
    np.testing.assert_allclose(out[0, 0], oa.e4m3_table()[v[0, 4, 0]], rtol=1e-12, atol=1e-300)


def test_empty_sequence_gives_zeros_and_length_masks_the_tail():
    B, Hq, Hkv, T, D = 2, 2, 2, 6, 8
    q_bits, k, v = random_case(B, Hq, Hkv, T, D, seed=5)
    out = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, np.array([0, 3], np.int32), 1.0, 1.0, 0.5)
    assert np.all(out[0] == 0.0)
    v2 = v.copy()
    v2[1, 3:] = 0x7E      # tokens past the length do not matter
    k2 = k.copy()
    k2[1, 3:] = 0x7E
    out2 = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k2, v2, np.array([0, 3], np.int32), 1.0, 1.0, 0.5)
    np.testing.assert_array_equal(out[1], out2[1])


def test_paged_layout_equals_contiguous():
    """Scatter each sequence's tokens into shuffled blocks of 4: the result
    through the block table equals the contiguous one exactly."""
    B, Hq, Hkv, T, D, bs = 3, 4, 2, 12, 8, 4
    q_bits, k, v = random_case(B, Hq, Hkv, T, D, seed=6)
    lens = np.array([12, 5, 9], np.int32)
    nb = B * (T // bs)
    perm = np.random.default_rng(7).permutation(nb)
    table = perm.reshape(B, T // bs).astype(np.int32)
    kp = np.zeros((nb, bs, Hkv, D), np.uint8)
    vp = np.zeros((nb, bs, Hkv, D), np.uint8)
    for b in range(B):
        for j in range(T // bs):
            kp[table[b, j]] = k[b, j * bs:(j + 1) * bs]
            vp[table[b, j]] = v[b, j * bs:(j + 1) * bs]
    a = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, lens, 0.125, 0.5, 0.3)
    p = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, kp, vp, lens, 0.125, 0.5, 0.3, block_table=table)
    np.testing.assert_array_equal(a, p)


@pytest.mark.parametrize("G", [2, 4])
def test_grouped_heads_equal_one_head_at_a_time(G):
    """Query head h reads KV head h // G: the same as giving each query head
    its own copy of that KV head."""
    B, Hkv, T, D = 2, 2, 5, 8
    Hq = Hkv * G
    q_bits, k, v = random_case(B, Hq, Hkv, T, D, seed=8 + G)
    lens = np.array([5, 4], np.int32)
    grouped = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, lens, 0.25, 0.25, 0.4)
    k1 = np.repeat(k, G, axis=2)
    v1 = np.repeat(v, G, axis=2)
    single = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k1, v1, lens, 0.25, 0.25, 0.4)
    np.testing.assert_array_equal(grouped, single)


def test_scales_enter_linearly():
    """v_scale multiplies the output; k_scale acts like sm_scale."""
    B, Hq, Hkv, T, D = 1, 2, 1, 6, 8
    q_bits, k, v = random_case(B, Hq, Hkv, T, D, seed=9)
    lens = np.array([6], np.int32)
    a = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, lens, 0.5, 1.0, 0.25)
    b = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, lens, 0.25, 4.0, 0.5)
    np.testing.assert_allclose(b, 4.0 * a, rtol=1e-13, atol=1e-300)


def _scatter_paged(k, v, bs, table, nb):
    B, T = k.shape[:2]
    kp = np.zeros((nb, bs) + k.shape[2:], np.uint8)
    vp = np.zeros((nb, bs) + v.shape[2:], np.uint8)
    for b in range(B):
        for j in range(T // bs):
            if 0 <= table[b, j] < nb:
                kp[table[b, j]] = k[b, j * bs:(j + 1) * bs]
                vp[table[b, j]] = v[b, j * bs:(j + 1) * bs]
    return kp, vp


@pytest.mark.parametrize("pad_id", [-1, -7, 10_000])
def test_padding_block_ids_drop_their_tokens(pad_id):
    """A block-table entry outside [0, num_blocks) (the -1 padding of a paged
    cache, or an id past its end) holds no tokens: the result equals the
    contiguous sequence with that block's tokens removed, checked against
    brute force over the remaining tokens."""
    B, Hq, Hkv, T, D, bs = 2, 4, 2, 16, 8, 4
    q_bits, k, v = random_case(B, Hq, Hkv, T, D, seed=11)
    lens = np.array([16, 11], np.int32)
    nb = B * (T // bs)
    table = np.random.default_rng(12).permutation(nb).reshape(B, T // bs).astype(np.int32)
    table[0, 1] = pad_id                 # tokens 4..7 of sequence 0
    table[1, 2] = pad_id                 # tokens 8..10 of sequence 1 (ragged tail)
    kp, vp = _scatter_paged(k, v, bs, table, nb)
    ks, vs, sm = 0.0625, 0.25, 0.3
    got = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, kp, vp, lens, ks, vs, sm, block_table=table)
    q = oracle.bits16_to_f32(q_bits, oracle.BF16)
    tab = [oracle.e4m3_value(c) for c in range(256)]
    kept = {0: [t for t in range(16) if not 4 <= t < 8], 1: [t for t in range(11) if t < 8]}
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            K = [[tab[int(c)] * ks for c in k[b, t, g]] for t in kept[b]]
            V = [[tab[int(c)] * vs for c in v[b, t, g]] for t in kept[b]]
            ref = oa.attention_bruteforce([float(x) for x in q[b, h]], K, V, sm)
            np.testing.assert_allclose(got[b, h], ref, rtol=1e-12, atol=1e-15)
    # and the contiguous oracle over the compacted sequences agrees exactly
    kc = np.zeros_like(k)
    vc = np.zeros_like(v)
    for b in range(B):
        kc[b, :len(kept[b])] = k[b, kept[b]]
        vc[b, :len(kept[b])] = v[b, kept[b]]
    compact = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, kc, vc, np.array([len(kept[0]), len(kept[1])], np.int32),
                                         ks, vs, sm)
    np.testing.assert_array_equal(got, compact)


def test_all_blocks_padding_gives_zeros():
    B, Hq, Hkv, T, D, bs = 1, 2, 1, 8, 8, 4
    q_bits, k, v = random_case(B, Hq, Hkv, T, D, seed=13)
    table = np.array([[-1, 5]], np.int32)      # 2 blocks exist: id 5 is past the end
    kp, vp = _scatter_paged(k, v, bs, np.array([[0, 1]], np.int32), 2)
    out = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, kp, vp, np.array([8], np.int32), 1.0, 1.0, 0.5,
                                     block_table=table)
    assert np.all(out == 0.0)


def test_uniform_weights_count_every_token_exactly():
    """Equal (zero) keys give every token weight 1/n; V marks dim d with 1.0
    on tokens [4d, 4d + 4): every output is exactly 4/n (a closed form that a
    dropped or repeated token changes)."""
    B, Hq, Hkv, D = 1, 2, 1, 8
    T = 4 * D
    q_bits, _, _ = random_case(B, Hq, Hkv, T, D, seed=14)
    k = np.zeros((B, T, Hkv, D), np.uint8)
    v = np.zeros((B, T, Hkv, D), np.uint8)
    for d in range(D):
        v[0, 4 * d:4 * d + 4, 0, d] = 0x38           # e4m3 1.0
    out = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, np.array([T], np.int32), 1.0, 0.5, 0.9)
    np.testing.assert_array_equal(out, np.full((B, Hq, D), 4.0 / T * 0.5))
