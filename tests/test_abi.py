"""The C ABI library builds, loads and exports every entry point declared in
include/fp8bs.h; argument validation and path selection work without a GPU
(these calls return before any CUDA call)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def L():
    from fp8_block_scaled_02_gb300 import build
    build.build()
    import fp8_block_scaled_02_gb300 as pkg
    return pkg.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("fp8bs_quantize", "fp8bs_gemv", "fp8bs_gemv_ex", "fp8bs_gemv_ws", "fp8bs_gemv_ws_bytes",
                 "fp8bs_gemv_batch", "fp8bs_gemv_batch_ex",
                 "mxfp8_gemv_batch", "mxfp8_gemv_batch_ex", "mxfp8_quantize", "mxfp8_gemv",
                 "mxfp8_gemv_ex", "fp8row_quantize", "fp8tensor_quantize", "fp8row_gemv", "fp8row_gemv_ex",
                 "fp8tensor_gemv", "fp8tensor_gemv_ex", "fp8act_quantize", "w8a8_gemm", "w8a8_gemm_ex",
                 "fp8bs_moe_gemv", "fp8kv_append", "fp8kv_decode_attention", "fp8bs_select_path", "fp8bs_strerror",
                 "fp8bs_check_device_error", "fp8bs_debug_wait_expiry", "fp8bs_debug_encode_f32",
                 "fp8bs_version"):
        assert want in names, names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    from fp8_block_scaled_02_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(declared_functions()) <= exported


def test_version_and_strerror(L):
    assert L.fp8bs_version() == 106
    import fp8_block_scaled_02_gb300 as pkg
    for st in range(-7, 1):
        assert pkg.strerror(st) and pkg.strerror(st) != "unknown status"
    assert pkg.strerror(-99) == "unknown status"


P = ctypes.c_void_p


def test_quantize_validation(L):
    w, c, s = P(0x10000), P(0x20000), P(0x30000)
    assert L.fp8bs_quantize(w, 0, 10, 128, c, s, None) == -2
    assert L.fp8bs_quantize(w, 10, -1, 128, c, s, None) == -2
    assert L.fp8bs_quantize(w, 10, 10, 64, c, s, None) == -3
    assert L.fp8bs_quantize(None, 10, 10, 128, c, s, None) == -1
    assert L.fp8bs_quantize(w, 10, 10, 128, None, s, None) == -1
    assert L.fp8bs_quantize(w, 10, 10, 128, c, None, None) == -1
    assert L.fp8bs_quantize(P(0x10001), 10, 10, 128, c, s, None) == -4
    assert L.fp8bs_quantize(w, 10, 10, 128, c, P(0x30002), None) == -4
    assert L.mxfp8_quantize(w, 0, 10, c, s, None) == -2
    assert L.mxfp8_quantize(w, 10, 10, None, s, None) == -1
    assert L.mxfp8_quantize(P(0x10001), 10, 10, c, s, None) == -4


def test_gemv_validation(L):
    x, c, s, y = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    assert L.fp8bs_gemv(x, -1, c, s, 10, 10, y, None) == -2
    assert L.fp8bs_gemv(x, 1, c, s, 0, 10, y, None) == -2
    assert L.fp8bs_gemv(x, 1, c, s, 10, 0, y, None) == -2
    assert L.fp8bs_gemv(x, 1, c, s, 1 << 31, 10, y, None) == -2
    assert L.fp8bs_gemv(None, 0, None, None, 10, 10, None, None) == 0   # m == 0: no-op
    assert L.fp8bs_gemv(None, 1, c, s, 10, 10, y, None) == -1
    assert L.fp8bs_gemv(x, 1, c, s, 10, 10, None, None) == -1
    assert L.fp8bs_gemv(P(0x10001), 1, c, s, 10, 10, y, None) == -4
    assert L.fp8bs_gemv(x, 1, c, P(0x30002), 10, 10, y, None) == -4
    assert L.fp8bs_gemv_ex(x, 1, c, s, 10, 10, y, 9, None) == -7
    # an explicit path that cannot take the shape is refused before launch
    assert L.fp8bs_gemv_ex(x, 1, c, s, 10, 10, y, 1, None) == -7    # decode needs k % 16 == 0
    assert L.fp8bs_gemv_ex(x, 1, P(0x20001), s, 10, 32, y, 1, None) == -7  # decode needs aligned codes
    assert L.mxfp8_gemv_ex(x, 40, c, s, 10, 24, y, 2, None) == -7   # the MX prefill needs k % 16 == 0
    assert L.mxfp8_gemv(x, 1, c, None, 10, 32, y, None) == -1


def batch(*ops):
    from fp8_block_scaled_02_gb300 import GemvOp
    arr = (GemvOp * max(1, len(ops)))()
    for i, o in enumerate(ops):
        arr[i] = GemvOp(*o)
    return ctypes.cast(arr, ctypes.c_void_p)


def test_gemv_batch_validation(L):
    good = (0x10000, 0x20000, 0x30000, 0x40000, 128, 256)
    for f, fx in ((L.fp8bs_gemv_batch, L.fp8bs_gemv_batch_ex), (L.mxfp8_gemv_batch, L.mxfp8_gemv_batch_ex)):
        assert f(None, 0, 1, None) == 0                                   # empty batch: no-op
        assert f(None, 2, 1, None) == -1                                  # no op array
        assert f(batch(good, good), -1, 1, None) == -2
        assert f(batch(good, good), 2, -1, None) == -2
        assert f(batch(good, (0x10000, 0x20000, 0x30000, 0x40000, 0, 256)), 2, 1, None) == -2
        assert f(batch(good, (0x10000, None, 0x30000, 0x40000, 128, 256)), 2, 1, None) == -1
        assert f(batch(good, (0x10001, 0x20000, 0x30000, 0x40000, 128, 256)), 2, 1, None) == -4
        assert f(batch(good, (None, None, None, None, 128, 256)), 2, 0, None) == 0   # m == 0: no-op
        assert fx(batch(good), 1, 1, 9, None) == -7
        # the decode path needs k % 16 == 0 and 16-byte aligned x and codes
        assert fx(batch(good, (0x10000, 0x20000, 0x30000, 0x40000, 128, 200)), 2, 1, 1, None) == -7
        assert fx(batch(good, (0x10008, 0x20000, 0x30000, 0x40000, 128, 256)), 2, 1, 1, None) == -7
    # block scales must be 4-byte aligned; the prefill path needs k % 16 == 0
    assert L.fp8bs_gemv_batch(batch(good, (0x10000, 0x20000, 0x30002, 0x40000, 128, 256)), 2, 1, None) == -4
    assert L.mxfp8_gemv_batch_ex(batch((0x10000, 0x20000, 0x30000, 0x40000, 128, 200)), 1, 40, 2, None) == -7


def test_gemv_ws_validation(L):
    x, c, s, y, w = P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000)
    need = L.fp8bs_gemv_ws_bytes(16, 4096)
    assert need == 2 * 16 * 4096 + 128 * 32               # f16 copy of x + one factor per (row slot, K block)
    assert L.fp8bs_gemv_ws_bytes(0, 4096) == 0
    assert L.fp8bs_gemv_ws_bytes(100, 4096) == L.fp8bs_gemv_ws_bytes(32, 4096)  # decode chunks of 32 rows
    assert L.fp8bs_gemv_ws_bytes(-1, 4096) == -2 and L.fp8bs_gemv_ws_bytes(1, 0) == -2
    assert L.fp8bs_gemv_ws(x, 16, c, s, 256, 4096, y, None, need, None) == -1        # decode path needs it
    assert L.fp8bs_gemv_ws(x, 16, c, s, 256, 4096, y, P(0x50008), need, None) == -4  # 16-byte aligned
    assert L.fp8bs_gemv_ws(x, 16, c, s, 256, 4096, y, w, need - 1, None) == -2       # too small
    assert L.fp8bs_gemv_ws(x, -1, c, s, 256, 4096, y, w, need, None) == -2
    assert L.fp8bs_gemv_ws(None, 0, None, None, 256, 4096, None, None, 0, None) == 0  # m == 0: no-op
    assert L.fp8bs_gemv_ws(x, 16, c, P(0x30002), 256, 4096, y, w, need, None) == -4


def test_rowwise_validation(L):
    w, c, s, x, y = P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000)
    for q in (L.fp8row_quantize, L.fp8tensor_quantize):
        assert q(w, 0, 10, c, s, None) == -2
        assert q(w, 10, 1 << 31, c, s, None) == -2
        assert q(None, 10, 10, c, s, None) == -1
        assert q(w, 10, 10, None, s, None) == -1
        assert q(w, 10, 10, c, None, None) == -1
        assert q(P(0x10001), 10, 10, c, s, None) == -4
        assert q(w, 10, 10, c, P(0x30002), None) == -4
    for g, gx in ((L.fp8row_gemv, L.fp8row_gemv_ex), (L.fp8tensor_gemv, L.fp8tensor_gemv_ex)):
        assert g(x, -1, c, s, 10, 10, y, None) == -2
        assert g(None, 0, None, None, 10, 10, None, None) == 0
        assert g(x, 1, c, None, 10, 10, y, None) == -1
        assert g(x, 1, c, P(0x30002), 10, 10, y, None) == -4
        assert gx(x, 1, c, s, 10, 10, y, 9, None) == -7
        assert gx(x, 1, c, s, 10, 10, y, 1, None) == -7   # decode needs k % 16 == 0
        assert gx(x, 40, c, s, 10, 24, y, 2, None) == -7  # prefill needs k % 16 == 0


def test_w8a8_validation(L):
    x, c, s, y, w, t = P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000), P(0x60000)
    assert L.fp8act_quantize(x, 0, 10, c, s, None) == -2
    assert L.fp8act_quantize(None, 1, 10, c, s, None) == -1
    assert L.fp8act_quantize(x, 1, 10, c, P(0x30001), None) == -4
    assert L.w8a8_gemm(c, -1, s, w, t, 10, 10, y, None) == -2
    assert L.w8a8_gemm(None, 0, None, None, None, 10, 10, None, None) == 0
    assert L.w8a8_gemm(c, 1, None, w, t, 10, 10, y, None) == -1
    assert L.w8a8_gemm(c, 1, s, w, None, 10, 10, y, None) == -1
    assert L.w8a8_gemm(c, 1, P(0x30002), w, t, 10, 10, y, None) == -4
    assert L.w8a8_gemm_ex(c, 1, s, w, t, 10, 10, y, 9, None) == -7
    assert L.w8a8_gemm_ex(c, 1, s, w, t, 10, 24, y, 1, None) == -7    # decode needs k % 16 == 0
    assert L.w8a8_gemm_ex(c, 40, s, P(0x50008), t, 10, 32, y, 2, None) == -7  # prefill needs aligned codes


def test_moe_validation(L):
    x, i, c, s, y = P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000)
    f = L.fp8bs_moe_gemv
    assert f(x, 1, i, 0, c, s, 8, 128, 128, y, None) == -2          # topk < 1
    assert f(x, 1, i, 9, c, s, 8, 128, 128, y, None) == -2          # topk > experts
    assert f(x, 1, i, 2, c, s, 1025, 128, 128, y, None) == -2       # too many experts
    assert f(x, 1, i, 2, c, s, 1024, 1 << 21, 128, y, None) == -2   # E * n >= 2^31
    assert f(None, 0, None, 2, None, None, 8, 128, 128, None, None) == 0
    assert f(x, 1, None, 2, c, s, 8, 128, 128, y, None) == -1
    assert f(x, 1, P(0x20002), 2, c, s, 8, 128, 128, y, None) == -4
    assert f(x, 1, i, 2, c, s, 8, 128, 120, y, None) == -7          # k % 16 != 0


def test_moe_ws_validation(L):
    x, i, c, s, y, w = P(0x10000), P(0x20000), P(0x30000), P(0x40000), P(0x50000), P(0x60000)
    f = L.fp8bs_moe_gemv_ws
    need = L.fp8bs_moe_gemv_ws_bytes(64, 12, 256, 4096)
    assert need > 2 * 64 * 12 * 4096 and L.fp8bs_moe_gemv_ws_bytes(32, 12, 256, 4096) == 0  # m <= 32: decode path
    assert L.fp8bs_moe_gemv_ws_bytes(64, 0, 256, 4096) == -2 and L.fp8bs_moe_gemv_ws_bytes(64, 2, 2000, 4096) == -2
    assert f(x, 64, i, 12, c, s, 256, 2048, 4096, y, None, need, None) == -1      # grouped path needs it
    assert f(x, 64, i, 12, c, s, 256, 2048, 4096, y, P(0x60010), need, None) == -4  # 256-byte aligned
    assert f(x, 64, i, 12, c, s, 256, 2048, 4096, y, w, need - 1, None) == -2
    assert f(x, 64, i, 0, c, s, 256, 2048, 4096, y, w, need, None) == -2
    assert f(x, 64, i, 12, c, s, 256, 2048, 4004, y, w, need, None) == -7        # k % 16 != 0
    assert f(None, 0, None, 12, None, None, 256, 2048, 4096, None, None, 0, None) == 0


@pytest.mark.parametrize("m,topk,e,k", [(64, 12, 256, 4096), (512, 12, 256, 4096), (2048, 12, 256, 4096),
                                        (33, 1, 1, 16), (300, 6, 6, 256), (40, 2, 1024, 7168)])
def test_moe_ws_bytes_cover_every_region(L, m, topk, e, k):
    """The workspace holds, for P = m * topk routed pairs: the x copy (2 P k
    bytes), the pair order (4 P), the per-expert offsets, one 16-byte record
    per tile of either size (at most ceil(P / tile) + min(E, P) tiles) and,
    for the decode tiles, one fp32 factor per (tile, 128-column K block,
    row of 32): a library that reserved less would let a kernel write past
    the caller's buffer."""
    p = m * topk
    cdiv = lambda a, b: -(-a // b)
    dec_tiles = cdiv(p, 32) + min(e, p)
    gemm_tiles = cdiv(p, 128) + min(e, p)
    floor = 2 * p * k + 4 * p + 5 * 4 * e + 16 * (dec_tiles + gemm_tiles) + 4 * dec_tiles * cdiv(k, 128) * 32
    got = L.fp8bs_moe_gemv_ws_bytes(m, topk, e, k)
    assert got >= floor, (got, floor)
    assert got <= floor + 9 * 256 + 4 * e, (got, floor)   # no more than region alignment beyond it


def test_kv_validation(L):
    x, sl, s, c = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    a = L.fp8kv_append
    assert a(x, 4, 8, 64, sl, s, c, 1024, None) == -2            # head_dim must be 128
    assert a(x, 0, 8, 128, None, None, None, 1024, None) == 0
    assert a(None, 4, 8, 128, sl, s, c, 1024, None) == -1
    assert a(P(0x10008), 4, 8, 128, sl, s, c, 1024, None) == -4  # x 16-byte aligned
    q, k, v, ks, vs, bt, lens, o = (P(0x10000 * i) for i in range(1, 9))
    f = L.fp8kv_decode_attention
    ok = dict(q=q, k=k, v=v, ks=ks, vs=vs, bt=bt, mb=4, lens=lens, b=2, hq=32, hkv=8, d=128, page=16, nb=64,
              ml=64, sm=0.088, o=o)

    def call(**kw):
        a_ = dict(ok, **kw)
        return f(a_["q"], a_["k"], a_["v"], a_["ks"], a_["vs"], a_["bt"], a_["mb"], a_["lens"], a_["b"], a_["hq"],
                 a_["hkv"], a_["d"], a_["page"], a_["nb"], a_["ml"], ctypes.c_float(a_["sm"]), a_["o"], None)
    assert call(d=64) == -2
    assert call(hq=30) == -2                 # not a multiple of the kv heads
    assert call(hq=80) == -2                 # more than 8 query heads per kv head
    assert call(page=24) == -2
    assert call(ml=65) == -2                 # beyond the block table
    assert call(sm=float("nan")) == -2
    assert call(b=0, q=None) == 0
    assert call(q=None) == -1
    assert call(q=P(0x10008)) == -4


def test_encode_probe_validation(L):
    c = P(0x10000)
    f = L.fp8bs_debug_encode_f32
    assert f(0, 16, None, None) == -1
    assert f(0, 0, c, None) == -2
    assert f(0, 6, c, None) == -2                     # not a multiple of 4
    assert f(0xFFFFFFF0, 32, c, None) == -2           # runs past 2^32
    assert f(0, 16, P(0x10002), None) == -4           # codes not 4-byte aligned


def test_select_path(L):
    a16, c16 = P(0x10000), P(0x20000)
    assert L.fp8bs_select_path(1, 100, 4096, a16, c16, 0) == 1          # decode
    assert L.fp8bs_select_path(32, 100, 4096, a16, c16, 0) == 1
    assert L.fp8bs_select_path(33, 100, 4096, a16, c16, 0) == 2         # prefill
    assert L.fp8bs_select_path(4096, 100, 4096, a16, c16, 1) == 2       # MX: tensor cores too
    assert L.fp8bs_select_path(1, 100, 4100, a16, c16, 0) == 3          # k % 16 != 0 -> generic
    assert L.fp8bs_select_path(1, 100, 4096, P(0x10008), c16, 0) == 3   # x not 16-byte aligned
    assert L.fp8bs_select_path(0, 100, 4096, a16, c16, 0) == -2
