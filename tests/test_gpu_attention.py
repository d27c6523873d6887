"""Decode attention over an fp8 (e4m3) KV cache: the CUDA path against the
oracle ("Enable scaled FP8 (e4m3fn) KV cache on ROCm", section "Scaling
semantics": K and V dequantised as decode(code) * per-tensor scale inside the
attention).

The caches are seeded bf16 KV with rare spikes, quantised per tensor by the
oracle on the CPU; both sides read the same codes.  Tolerance: the kernel
computes in fp32 (exact code decoding, fp32 dot products and sums, exp2) and
rounds the output to bf16 / fp16, so |gpu - ref| <= 2^-8 |ref| + 2^-14 r,
where r is the same attention over |V| (the softmax-weighted mean of |V|,
the scale of the fp32 rounding in the sums): half an output ulp is
2^-9 |ref|, and fp32 score and sum errors stay near 1e-6 r.  A dropped or
repeated token moves an output by about r / T, above the bound for every
length tested but the 65536-token one."""
import numpy as np
import pytest
import torch

import int8_w8a8_scaled_gb300 as w8
import oracle
import synthetic_inputs as si
from oracle import attention as oa
from gpu_util import bits_np, out_to_f32

pytestmark = pytest.mark.gpu


def kv_codes(B, T, Hkv, D, seed):
    """Seeded bf16 K and V [B, T, Hkv, D] quantised per tensor (oracle)."""
    out = []
    for j in range(2):
        x = si.kv_with_spikes(B * T, Hkv, D, seed=seed + j)
        codes, s = oracle.quant(si.bits16(x).reshape(B * T, Hkv * D), oracle.BF16, oracle.E4M3, oracle.PER_TENSOR)
        out.append((codes.reshape(B, T, Hkv, D), np.float32(s[0])))
    return out


def run_case(B, Hq, Hkv, T, lens, seed, q_dtype=torch.bfloat16, out_dtype=torch.bfloat16, paged_bs=0,
             check_b=None, pad=()):
    """pad: (sequence, block index, id) entries written into the block table
    after the cache is laid out: ids outside [0, num_blocks) are padding."""
    D = 128
    (k, ks), (v, vs) = kv_codes(B, T, Hkv, D, seed)
    q = si.normal((B, Hq, D), seed=seed + 7, dtype=q_dtype)
    qkind = oracle.BF16 if q_dtype == torch.bfloat16 else oracle.FP16
    lens = np.asarray(lens, np.int32)
    table = None
    kc, vc = k, v
    if paged_bs:
        nbps = T // paged_bs
        nb = B * nbps + 3                      # a few blocks no sequence uses
        perm = np.random.default_rng(seed).permutation(nb)[:B * nbps]
        table = perm.reshape(B, nbps).astype(np.int32)
        kc = np.zeros((nb, paged_bs, Hkv, D), np.uint8)
        vc = np.zeros((nb, paged_bs, Hkv, D), np.uint8)
        for b in range(B):
            for j in range(nbps):
                kc[table[b, j]] = k[b, j * paged_bs:(j + 1) * paged_bs]
                vc[table[b, j]] = v[b, j * paged_bs:(j + 1) * paged_bs]
        for b, j, blk in pad:
            table[b, j] = blk
    dev = "cuda"
    out = torch.empty(B, Hq, D, dtype=out_dtype, device=dev)
    w8.fp8_kv_decode_attention(q.to(dev), torch.from_numpy(kc).to(dev), torch.from_numpy(vc).to(dev),
                               torch.from_numpy(lens).to(dev), torch.tensor([ks], device=dev),
                               torch.tensor([vs], device=dev), out,
                               block_table=None if table is None else torch.from_numpy(table).to(dev))
    torch.cuda.synchronize()
    okind = oracle.BF16 if out_dtype == torch.bfloat16 else oracle.FP16
    got = out_to_f32(bits_np(out), okind).astype(np.float64)
    bsel = list(range(B)) if check_b is None else check_b
    qb = si.bits16(q)[bsel]
    if table is None:
        ref = oa.fp8_kv_decode_attention(qb, qkind, k[bsel], v[bsel], lens[bsel], ks, vs, 1.0 / np.sqrt(D))
        # the same weights over |V| (clearing an e4m3 code's sign bit gives |value|)
        r_abs = oa.fp8_kv_decode_attention(qb, qkind, k[bsel], v[bsel] & 0x7F, lens[bsel], ks, vs, 1.0 / np.sqrt(D))
    else:
        ref = oa.fp8_kv_decode_attention(qb, qkind, kc, vc, lens[bsel], ks, vs, 1.0 / np.sqrt(D),
                                         block_table=table[bsel])
        r_abs = oa.fp8_kv_decode_attention(qb, qkind, kc, vc & 0x7F, lens[bsel], ks, vs, 1.0 / np.sqrt(D),
                                           block_table=table[bsel])
    err = np.abs(got[bsel] - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * r_abs
    bad = err > bound
    assert not bad.any(), f"{int(bad.sum())} outputs off; worst {float((err - bound).max())}"
    for b in bsel:
        if lens[b] == 0:
            assert np.all(got[b] == 0.0)
    return got, ref


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_grouped_heads_ragged_lengths(G):
    Hkv = 2
    # one token, a chunk boundary, a ragged tail, the maximum length
    run_case(B=4, Hq=Hkv * G, Hkv=Hkv, T=600, lens=[1, 256, 333, 600], seed=100 + G)


def test_paged_cache_and_empty_sequence():
    run_case(B=3, Hq=8, Hkv=2, T=512, lens=[512, 0, 77], seed=200, paged_bs=16)


@pytest.mark.parametrize("pad_id", [-1, 1 << 20])
def test_paged_cache_padding_entries(pad_id):
    """Block-table entries outside the cache (-1 padding, or an id past its
    end) hold no tokens, on the GPU as in the oracle: a whole middle block,
    the block of a ragged tail, and every block of one sequence."""
    nbps = 512 // 16
    pad = [(0, 5, pad_id), (1, 77 // 16, pad_id)] + [(2, j, pad_id) for j in range(nbps)]
    run_case(B=3, Hq=8, Hkv=2, T=512, lens=[512, 77, 300], seed=210, paged_bs=16, pad=pad)


@pytest.mark.parametrize("bs,T", [(8, 512), (48, 480), (32, 512)])
def test_paged_block_sizes(bs, T):
    """Block sizes that are not a multiple of 16 take per-lane copies; 32 and
    48 take the bulk-tensor copies of 16-token blocks inside a cache block."""
    run_case(B=3, Hq=8, Hkv=2, T=T, lens=[T, T - 37, 100], seed=220 + bs, paged_bs=bs,
             pad=[(1, 2, -1)])


def test_query_not_8_byte_aligned():
    """A query view that starts 2 bytes into its storage takes the scalar
    query loads; the result equals the aligned query's bit for bit."""
    B, Hq, Hkv, T, D = 2, 8, 2, 200, 128
    (k, ks), (v, vs) = kv_codes(B, T, Hkv, D, 230)
    dev = "cuda"
    q = si.normal((B, Hq, D), seed=231).to(dev)
    store = torch.empty(B * Hq * D + 1, dtype=torch.bfloat16, device=dev)
    qu = store[1:].view(B, Hq, D)
    qu.copy_(q)
    assert qu.data_ptr() % 8 != 0
    kc, vc = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    lens = torch.tensor([200, 77], dtype=torch.int32, device=dev)
    ksc, vsc = torch.tensor([ks], device=dev), torch.tensor([vs], device=dev)
    outs = [torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    w8.fp8_kv_decode_attention(q, kc, vc, lens, ksc, vsc, outs[0])
    w8.fp8_kv_decode_attention(qu, kc, vc, lens, ksc, vsc, outs[1])
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_fp16_query_and_output():
    run_case(B=2, Hq=8, Hkv=2, T=300, lens=[300, 129], seed=300, q_dtype=torch.float16, out_dtype=torch.float16)


def test_llama3_8b_decode_shape_sampled():
    """16 sequences x 4096 tokens, 32 query / 8 KV heads (the benchmark's
    shape), every output of four sequences checked."""
    run_case(B=16, Hq=32, Hkv=8, T=4096, lens=[4096] * 15 + [1000], seed=400, check_b=[0, 7, 14, 15])


def test_long_single_sequence():
    """One sequence of 65536 tokens: 8 KV heads x 128 (the KV-cache tensor
    of the quantiser benchmark), many chunks combined."""
    run_case(B=1, Hq=32, Hkv=8, T=65536, lens=[65536], seed=500)


def _long_case_inputs(T, Hkv, Hq, D):
    dev = "cuda"
    lens = torch.tensor([T], dtype=torch.int32, device=dev)
    ks = torch.tensor([2.0 ** -3], device=dev)
    vs = torch.tensor([2.0 ** -4], device=dev)
    return dev, lens, ks, vs


def test_long_sequence_counts_every_token_exactly():
    """65536 tokens, all keys zero: every token weighs 1/65536.  V marks dim
    d of every KV head with 1.0 on tokens [512 d, 512 d + 512), so every
    output is exactly 512/65536 * v_scale, a value that a dropped or repeated
    token (or chunk) changes.  The fp32 sums of ones are exact, so the GPU
    must match the oracle bit for bit."""
    B, T, Hkv, Hq, D = 1, 65536, 8, 32, 128
    dev, lens, ks, vs = _long_case_inputs(T, Hkv, Hq, D)
    k = np.zeros((B, T, Hkv, D), np.uint8)
    v = np.zeros((B, T, Hkv, D), np.uint8)
    for d in range(D):
        v[0, 512 * d:512 * (d + 1), :, d] = 0x38          # e4m3 1.0
    q = si.normal((B, Hq, D), seed=700)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    w8.fp8_kv_decode_attention(q.to(dev), torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), lens, ks, vs,
                               out)
    torch.cuda.synchronize()
    ref = oa.fp8_kv_decode_attention(si.bits16(q), oracle.BF16, k, v, np.array([T], np.int32), 2.0 ** -3,
                                     2.0 ** -4, 1.0 / np.sqrt(D))
    assert np.all(ref == 2.0 ** -7 * 2.0 ** -4)
    got = out_to_f32(bits_np(out), oracle.BF16).astype(np.float64)
    np.testing.assert_array_equal(got, ref)


def test_long_sequence_dominant_key_per_head():
    """65536 tokens; query head h is one-hot on dim d_h and only token t_h has
    a key on that dim (448): its score leads every other by more than 200, so
    head h returns token t_h's value row exactly.  The t_h sit on the first
    and last tokens and on both sides of 64/128/256/512-token boundaries."""
    B, T, Hkv, Hq, D = 1, 65536, 8, 32, 128
    G = Hq // Hkv
    dev, lens, ks, vs = _long_case_inputs(T, Hkv, Hq, D)
    rng = np.random.default_rng(701)
    k = np.zeros((B, T, Hkv, D), np.uint8)
    v = rng.integers(0, 0x7F, (B, T, Hkv, D), dtype=np.uint8) | (rng.integers(0, 2, (B, T, Hkv, D), dtype=np.uint8) << 7)
    spots = [0, T - 1, 63, 64, 127, 128, 255, 256, 511, 512, 4095, 4096, 30000, 32767, 32768, 65535 - 256,
             65535 - 255, 1, 1000, 2047, 2048, 8191, 8192, 16383, 16384, 40000, 50000, 60000, 65000, 65280, 12345, 777]
    qf = np.zeros((B, Hq, D), np.float32)
    t_of = {}
    for h in range(Hq):
        g, j = divmod(h, G)
        d = 16 * j + 3
        t = spots[h]
        k[0, t, g, d] = 0x7E                                  # 448
        qf[0, h, d] = 4.0                                     # score 4 * 448 / 8 / sqrt(128) ~ 19.8 ...
        t_of[h] = (t, g)
    qf *= 16.0                                                # ... x16: ~317 above every other token
    q_bits = oracle.f32_to_bf16_bits(qf)
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
    w8.fp8_kv_decode_attention(q.to(dev), torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), lens, ks, vs,
                               out)
    torch.cuda.synchronize()
    got = out_to_f32(bits_np(out), oracle.BF16).astype(np.float64)
    ref = oa.fp8_kv_decode_attention(q_bits, oracle.BF16, k, v, np.array([T], np.int32), 2.0 ** -3, 2.0 ** -4,
                                     1.0 / np.sqrt(D))
    tab = oa.e4m3_table()
    for h in range(Hq):
        t, g = t_of[h]
        want = tab[v[0, t, g]] * 2.0 ** -4                   # exact in bf16
        # the oracle (fp64) keeps the other tokens' weights of ~1e-138
        np.testing.assert_allclose(ref[0, h], want, rtol=1e-12, atol=1e-120)
        np.testing.assert_array_equal(got[0, h], want, err_msg=f"head {h} (token {t})")


def test_graph_capture_and_determinism():
    """Same inputs twice inside one CUDA graph: identical bits (no atomics)."""
    B, Hq, Hkv, T, D = 4, 16, 4, 1024, 128
    (k, ks), (v, vs) = kv_codes(B, T, Hkv, D, 600)
    dev = "cuda"
    q = si.normal((B, Hq, D), seed=601).to(dev)
    kc, vc = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    lens = torch.tensor([1024, 999, 1, 512], dtype=torch.int32, device=dev)
    ksc, vsc = torch.tensor([ks], device=dev), torch.tensor([vs], device=dev)
    outs = [torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ws = w8.Workspace(w8.attention_workspace_size(B, Hq, T))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        w8.fp8_kv_decode_attention(q, kc, vc, lens, ksc, vsc, outs[0], workspace=ws, stream=s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for o in outs:
                w8.fp8_kv_decode_attention(q, kc, vc, lens, ksc, vsc, o, workspace=ws, stream=s)
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_argument_errors():
    dev = "cuda"
    q = torch.zeros(2, 6, 128, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(2, 16, 4, 128, dtype=torch.uint8, device=dev)
    lens = torch.ones(2, dtype=torch.int32, device=dev)
    sc = torch.ones(1, device=dev)
    out = torch.empty_like(q)
    with pytest.raises(w8.W8A8Error):    # 6 query heads over 4 KV heads
        w8.fp8_kv_decode_attention(q, kc, kc, lens, sc, sc, out)
    q64 = torch.zeros(2, 8, 64, dtype=torch.bfloat16, device=dev)
    kc64 = torch.zeros(2, 16, 4, 64, dtype=torch.uint8, device=dev)
    with pytest.raises(w8.W8A8Error):    # head_dim 64
        w8.fp8_kv_decode_attention(q64, kc64, kc64, lens, sc, sc, torch.empty_like(q64))


def test_workspace_shared_across_shapes():
    """One workspace serves calls of any shape in turn (it holds only each
    call's own partial results): every call gives the bits of a call with a
    fresh workspace."""
    torch.manual_seed(0)
    shapes = [(4, 32, 8, 1000), (2, 8, 2, 3000), (6, 16, 4, 700), (4, 32, 8, 1000)]
    ws = w8.Workspace(max(w8.attention_workspace_size(B, Hq, T) for B, Hq, _, T in shapes))
    for i, (B, Hq, Hkv, T) in enumerate(shapes):
        g = torch.Generator(device="cuda")
        g.manual_seed(100 + i)
        kc = torch.randint(0, 126, (B, T, Hkv, 128), generator=g, device="cuda", dtype=torch.uint8)
        vc = torch.randint(0, 126, (B, T, Hkv, 128), generator=g, device="cuda", dtype=torch.uint8)
        q = torch.randn(B, Hq, 128, generator=g, device="cuda").to(torch.bfloat16)
        lens = torch.randint(1, T + 1, (B,), generator=g, device="cuda", dtype=torch.int32)
        sc = torch.full((1,), 0.05, device="cuda")
        out = torch.empty(B, Hq, 128, dtype=torch.bfloat16, device="cuda")
        ref = torch.empty_like(out)
        w8.fp8_kv_decode_attention(q, kc, vc, lens, sc, sc, out, workspace=ws)
        w8.fp8_kv_decode_attention(q, kc, vc, lens, sc, sc, ref,
                                   workspace=w8.Workspace(w8.attention_workspace_size(B, Hq, T)))
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (B, Hq, Hkv, T)
    assert w8.device_status() == 0

