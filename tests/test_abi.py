"""Host-only checks of the C ABI: the library builds, loads and exports every
symbol include/w8a8.h declares; invalid arguments come back as status codes
(validated before any CUDA call, so nothing here touches a GPU)."""
import ctypes
import os
import re

import pytest

import int8_w8a8_scaled_gb300 as w8
from int8_w8a8_scaled_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "w8a8.h")


def header_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"W8A8_API\s+[\w\s\*]+?\b(w8a8_\w+)\s*\(", text)))


def test_header_declares_expected_symbols():
    assert header_symbols() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    for name in header_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_last_error():
    lib = _lib.load()
    assert lib.w8a8_version() >= 100
    assert isinstance(lib.w8a8_last_error(), bytes)


FAKE = ctypes.c_void_p(0x7F0000000000)      # never dereferenced: validation fails first
FAKE_ODD = ctypes.c_void_p(0x7F0000000001)


def mm(lib, a=FAKE, lda=64, b=FAKE, ldb=64, sa=FAKE, ag=0, sb=FAKE, bg=0, out=FAKE, ldc=64,
       M=4, N=64, K=64, qd=w8.E4M3, od=w8.BF16, ws=None, wsb=0):
    return lib.w8a8_scaled_mm(a, lda, b, ldb, sa, ag, sb, bg, out, ldc, M, N, K, qd, od, ws, wsb, None)


@pytest.mark.parametrize("kw,status", [
    (dict(a=None), 1), (dict(b=None), 1), (dict(sa=None), 1), (dict(sb=None), 1), (dict(out=None), 1),
    (dict(qd=7), 1), (dict(od=9), 1), (dict(ag=3), 1), (dict(M=0), 1), (dict(N=-1), 1), (dict(K=0), 1),
    (dict(lda=32), 1), (dict(ldc=10), 1),
    (dict(od=w8.INT32), 2), (dict(qd=w8.INT8, od=w8.FP32), 2),
    (dict(qd=w8.INT8, K=131072, lda=131072, ldb=131072), 2), (dict(qd=w8.INT8, K=40, lda=48, ldb=48), 2),
    (dict(a=FAKE_ODD), 3), (dict(lda=72), 3), (dict(ldb=88), 3),
])
def test_scaled_mm_rejects_bad_arguments(kw, status):
    lib = _lib.load()
    assert mm(lib, **kw) == status
    assert lib.w8a8_last_error()


def test_b_not_k_major_is_a_status_not_a_crash():
    """The CUTLASS review thread: passing B with the wrong layout used to end
    in "misaligned address".  Here a row stride that is not a 16-byte
    multiple is rejected with W8A8_ERR_MISALIGNED."""
    lib = _lib.load()
    assert mm(lib, M=8, N=8192, K=4096, lda=4096, ldb=4097, ldc=8192) == 3


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), 1), (dict(xd=w8.E4M3), 1), (dict(qd=w8.BF16), 1), (dict(rows=0), 1),
    (dict(ldx=3), 1), (dict(gran=5), 1), (dict(mode=4), 1), (dict(x=FAKE_ODD), 3),
    (dict(gran=0, mode=0), 4),
])
def test_scaled_quant_rejects_bad_arguments(kw, status):
    lib = _lib.load()
    a = dict(x=FAKE, xd=w8.BF16, rows=4, cols=64, ldx=64, q=FAKE, qd=w8.E4M3, ldq=64, scale=FAKE,
             gran=1, mode=0, ws=None, wsb=0)
    a.update(kw)
    st = lib.w8a8_scaled_quant(a["x"], a["xd"], a["rows"], a["cols"], a["ldx"], a["q"], a["qd"], a["ldq"],
                               a["scale"], a["gran"], a["mode"], a["ws"], a["wsb"], None)
    assert st == status


def test_scaled_dequant_rejects_bad_arguments():
    lib = _lib.load()
    assert lib.w8a8_scaled_dequant(None, 0, 4, 4, 4, FAKE, 0, FAKE, w8.BF16, 4, None) == 1
    assert lib.w8a8_scaled_dequant(FAKE, 0, 4, 4, 4, FAKE, 0, FAKE, w8.E4M3, 4, None) == 1
    assert lib.w8a8_scaled_dequant(FAKE, 0, 4, 4, 4, FAKE, 0, FAKE_ODD, w8.BF16, 4, None) == 3


def test_workspace_sizes():
    assert w8.quant_workspace_size(10, 10, per_token=False, dynamic=True) == 16
    assert w8.quant_workspace_size(10, 10, per_token=True, dynamic=True) == 0
    assert w8.quant_workspace_size(10, 10, per_token=False, dynamic=False) == 0
    # no split, fp8: no workspace (gate-up at M=4096: 1792 pair tiles over 76
    # pairs, a last round of 44 tiles, more than half: the tiles run whole)
    assert w8.pick_config(4096, 28672, 4096, w8.E4M3)["split_k"] == 1
    assert w8.mm_workspace_size(4096, 28672, 4096, w8.E4M3) == 0
    # CTA pairs whose last round keeps at most half of the pairs busy run its
    # tiles as K halves where K is long enough to pay for the exchange (the
    # down projection, K = 14336): 256 tiles of 256 x 256 over 76 pairs leave
    # 28; two halves x two CTAs x 128 x 256 fp32 each, after the counter region
    c = w8.pick_config(4096, 4096, 14336, w8.E4M3)
    assert (c["cta_pair"], c["block_n"], c["split_k"]) == (1, 256, 2)
    assert w8.mm_workspace_size(4096, 4096, 14336, w8.E4M3) == 65536 + 28 * 4 * 128 * 256 * 4
    # the same tiles whole: no workspace
    whole = dict(c, split_k=1)
    assert w8.mm_workspace_size(4096, 4096, 14336, w8.E4M3, whole) == 0
    # at K = 4096 the halves do not pay: whole tiles, no workspace
    assert w8.pick_config(4096, 4096, 4096, w8.E4M3)["split_k"] == 1
    assert w8.mm_workspace_size(4096, 4096, 4096, w8.E4M3) == 0
    # int8 pairs take no K halves: only the f16 operand planes
    i8 = {"swap_ab": 0, "block_n": 256, "split_k": 2, "cta_pair": 1}
    assert w8.mm_workspace_size(4096, 4096, 4096, w8.INT8, i8) == w8.mm_workspace_size(4096, 4096, 4096, w8.INT8,
                                                                                       dict(i8, split_k=1))
    # int8 widens both operands to f16 planes
    assert w8.mm_workspace_size(512, 256, 1024, w8.INT8) >= (512 + 256) * 1024 * 2
    # split-K through the workspace: partials + counters
    cfg = {"swap_ab": 1, "block_n": 16, "split_k": 4, "reduce": w8.REDUCE_GLOBAL}
    assert w8.mm_workspace_size(1, 4096, 4096, w8.E4M3, cfg) >= 32 * 4 * 128 * 16 * 4
    # split-K through a thread-block cluster: the same partials, no counters used
    for red in (w8.REDUCE_AUTO, w8.REDUCE_CLUSTER):
        cfg = {"swap_ab": 1, "block_n": 16, "split_k": 4, "reduce": red}
        assert w8.mm_workspace_size(1, 4096, 4096, w8.E4M3, cfg) >= 32 * 4 * 128 * 16 * 4
    # more slices than one portable cluster: the workspace reduction
    cfg = {"swap_ab": 1, "block_n": 16, "split_k": 16}
    assert w8.mm_workspace_size(1, 4096, 4096, w8.E4M3, cfg) >= 32 * 16 * 128 * 16 * 4


@pytest.mark.parametrize("M,N,K,bn,tail", [
    (4096, 4096, 14336, 256, 28),   # 256 tiles over 76 pairs: a last round of 28 <= 38
    (1280, 4096, 1040, 256, 4),     # 80 tiles: 4 left
    (1536, 4864, 256, 256, 38),     # 114 tiles: 38 left, exactly half of the pairs
    (1536, 5120, 256, 256, 0),      # 120 tiles: 44 left, more than half: whole tiles
    (4096, 4864, 4096, 256, 0),     # 304 tiles: four full rounds
    (1280, 4096, 128, 256, 0),      # one K block: nothing to halve
    (1024, 4096, 4096, 256, 0),     # 64 tiles: fewer tiles than pairs, one round
    (4096, 4096, 14336, 224, 0),    # 304 tiles of 224 columns: four full rounds
])
def test_pair_k_halves_workspace(M, N, K, bn, tail):
    """Host rule of the CTA-pair K halves (split_k 2) on a 152-SM GB300 (76
    pairs): the tiles of a last round that keeps at most half of the pairs
    busy are split, and each needs two halves x two CTAs x 128 x block_n
    fp32 after the 64 KiB counter region; otherwise no workspace."""
    cfg = {"swap_ab": 0, "block_n": bn, "split_k": 2, "cta_pair": 1}
    want = 65536 + tail * 4 * 128 * bn * 4 if tail else 0
    assert w8.mm_workspace_size(M, N, K, w8.E4M3, cfg) == want


@pytest.mark.parametrize("M", [1, 16, 64, 256, 4096])
def test_pick_config_regimes(M):
    c = w8.pick_config(M, 4096, 4096, w8.E4M3)
    assert c["swap_ab"] == (1 if M <= 64 else 0)    # decode regime: weights on the 128-row side
    assert c["block_n"] in (16, 32, 64, 128, 160, 192, 224, 256)
    assert c["split_k"] >= 1
    assert c["split_k"] <= 8 and c["reduce"] == w8.REDUCE_AUTO   # splits fit one cluster
    if M >= 4096:
        assert c["block_n"] >= 128   # many tiles: wide tile, no split-K (K halves of the last round only)
    # 256-row tiles on CTA pairs for large-M e4m3 only
    assert c["cta_pair"] == (1 if M >= 1024 else 0)
    if c["cta_pair"]:
        assert c["block_n"] in (192, 224, 256) and c["swap_ab"] == 0 and c["split_k"] in (1, 2)
    c8 = w8.pick_config(M, 4096, 4096, w8.INT8)
    assert c8["block_n"] <= 128 or (c8["block_n"] in (160, 256) and not c8["swap_ab"])
    assert c8["cta_pair"] == 0


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(kc=None), 1), (dict(lens=None), 1), (dict(out=None), 1),
    (dict(qd=w8.E4M3), 1), (dict(od=w8.INT8), 1), (dict(hd=64), 1), (dict(hq=12), 1), (dict(hq=24, hkv=8), 1),
    (dict(batch=0), 1), (dict(maxseq=0), 1),
    (dict(bt=FAKE, bs=16, maxb=2, nblk=8), 1),          # max_blocks * block_size < max_seq_len
    (dict(kc=FAKE_ODD), 3), (dict(ws=None), 4), (dict(wsb=16), 4),
])
def test_attention_rejects_bad_arguments(kw, status):
    """w8a8_fp8_kv_decode_attention validates everything before any CUDA call."""
    lib = _lib.load()
    a = dict(q=FAKE, qd=w8.BF16, batch=2, hq=32, hkv=8, hd=128, kc=FAKE, vc=FAKE, maxseq=4096, bt=None, bs=0,
             maxb=0, nblk=0, lens=FAKE, ks=FAKE, vs=FAKE, out=FAKE, od=w8.BF16, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    st = lib.w8a8_fp8_kv_decode_attention(a["q"], a["qd"], a["batch"], a["hq"], a["hkv"], a["hd"], a["kc"], a["vc"],
                                          a["maxseq"], a["bt"], a["bs"], a["maxb"], a["nblk"], a["lens"], a["ks"],
                                          a["vs"], 0.088, a["out"], a["od"], a["ws"], a["wsb"], None)
    assert st == status
    assert lib.w8a8_last_error()


def test_attention_workspace_size():
    # 64-token chunks at most: [batch, q heads, chunks, 132 floats]
    assert w8.attention_workspace_size(16, 32, 4096) == 16 * 32 * 64 * 132 * 4
    assert w8.attention_workspace_size(1, 8, 1) == 8 * 1 * 132 * 4
    assert w8.attention_workspace_size(0, 8, 10) == 0
    # a product beyond 2^62 bytes is refused, not wrapped around
    assert w8.attention_workspace_size(65535, 65535, 1 << 30) == 0
    lib = _lib.load()
    st = lib.w8a8_fp8_kv_decode_attention(FAKE, w8.BF16, 65535, 65535, 65535, 128, FAKE, FAKE, 1 << 30, None, 0, 0, 0,
                                          FAKE, FAKE, FAKE, 0.088, FAKE, w8.BF16, FAKE, 1 << 40, None)
    assert st == 1
