"""Pins for the oracle's per-row and per-tensor FP8 quantizers and their
fp64 GEMV (CPU only).

FreeToken PR #389 ("load-time per-tensor FP8 dense projections") quantizes
each weight to e4m3 with one fp32 scale (per tensor) and lists a per-row
W8A16 route beside it.  The scale rule is the block rule applied to a row
or to the whole tensor, so the pins tie these functions to the block
quantizer where the two must agree (a weight that is one tile, a row that
is one tile), plus the invariants that hold at any size: the amax element
encodes to +-448, an all-zero row takes s = 1, a row whose amax is 448 is
the plain e4m3 cast, and each code is the nearest e4m3 value of w/s.  The
GEMV is pinned against numpy's float64 matmul on an independently built
dequantized weight, exact one-hot columns, and the block GEMV when the
scales are constant per 128-row tile.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import bitwise_e4m3_encode, e4m3_values_torch
from fp8_block_scaled_02_gb300 import inputs


def bits_of(t):
    return inputs.bf16_bits(t)


def f32_of_bits(b):
    return (np.asarray(b).astype(np.uint32) << 16).view(np.float32)


def e4m3_ulp(v):
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    return np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)


# ------------------------------------------------------------- quantizers
@pytest.mark.parametrize("n,k", [(1, 1), (7, 100), (130, 128), (3, 5)])
def test_row_equals_block_when_a_row_is_one_tile(n, k):
    """With k <= 128 a single row is a whole 128x128 tile of the 1-row
    weight, so per-row quantization must equal block quantization row by
    row."""
    w = bits_of(inputs.gaussian_bf16((n, k), 0.02, 60 + n + k))
    codes, scales = oracle.row_quantize(w)
    assert codes.shape == (n, k) and scales.shape == (n,)
    for r in range(n):
        cb, sb = oracle.block_quantize(w[r:r + 1])
        assert np.array_equal(codes[r:r + 1], cb)
        assert scales[r].view(np.uint32) == sb[0, 0].view(np.uint32)


@pytest.mark.parametrize("n,k", [(1, 1), (128, 128), (77, 13)])
def test_tensor_equals_block_when_the_weight_is_one_tile(n, k):
    w = bits_of(inputs.gaussian_bf16((n, k), 0.02, 70 + n + k))
    codes, scale = oracle.tensor_quantize(w)
    cb, sb = oracle.block_quantize(w)
    assert scale.shape == (1,)
    assert np.array_equal(codes, cb)
    assert scale[0].view(np.uint32) == sb[0, 0].view(np.uint32)


def test_tensor_equals_row_when_every_row_shares_the_amax():
    w = bits_of(inputs.gaussian_bf16((40, 700), 0.02, 71))
    rng = np.random.default_rng(3)
    cols = rng.integers(0, 700, 40)
    signs = rng.choice([0x3E00, 0xBE00], 40)   # +-0.125, above every N(0, 0.02^2) sample here
    w[np.arange(40), cols] = signs
    ct, st = oracle.tensor_quantize(w)
    cr, sr = oracle.row_quantize(w)
    assert np.all(sr == st[0])
    assert np.array_equal(ct, cr)


def test_row_scale_formula_and_amax_element():
    w = bits_of(inputs.lm_head_weight(2, shape=(64, 1000)))
    codes, scales = oracle.row_quantize(w)
    wf = np.abs(f32_of_bits(w))
    amax = wf.max(axis=1)
    assert np.array_equal(scales, amax / np.float32(448.0))
    arg = wf.argmax(axis=1)
    assert np.all(codes[np.arange(64), arg] & 0x7F == 0x7E)


def test_tensor_scale_formula_and_amax_element():
    w = bits_of(inputs.lm_head_weight(2, shape=(64, 1000)))
    codes, scale = oracle.tensor_quantize(w)
    wf = np.abs(f32_of_bits(w))
    assert scale[0] == wf.max() / np.float32(448.0)
    r, c = np.unravel_index(np.argmax(wf), wf.shape)
    assert codes[r, c] & 0x7F == 0x7E
    # every other row's largest code is at most 448
    assert np.all(codes & 0x7F <= 0x7E)


def test_zero_row_and_zero_tensor():
    w = bits_of(inputs.gaussian_bf16((4, 300), 0.02, 72))
    w[2] = 0
    w[2, 17] = 0x8000
    codes, scales = oracle.row_quantize(w)
    assert scales[2] == 1.0 and codes[2, 17] == 0x80 and np.all(np.delete(codes[2], 17) == 0)
    z = np.zeros((3, 9), dtype=np.uint16)
    cz, sz = oracle.tensor_quantize(z)
    assert sz[0] == 1.0 and np.all(cz == 0)


def test_row_with_amax_448_is_plain_cast():
    """s = 448/448 = 1 exactly, so the codes are the e4m3 cast of w, which
    an independent bit-arithmetic encoder computes."""
    rng = np.random.default_rng(6)
    v = np.float32(rng.uniform(-448, 448, (3, 500)))
    v[:, 11] = 448.0
    wb = bits_of(torch.from_numpy(v).to(torch.bfloat16))
    codes, scales = oracle.row_quantize(wb)
    assert np.all(scales == 1.0)
    assert np.array_equal(codes, bitwise_e4m3_encode(f32_of_bits(wb)))
    ct, st = oracle.tensor_quantize(wb)
    assert st[0] == 1.0 and np.array_equal(ct, codes)


def test_codes_are_nearest_to_the_fp32_quotient():
    """Each code is within half an e4m3 ulp of the binary32 quotient w/s
    (the per-element bound of the block form, with the row scale)."""
    w = bits_of(inputs.heavy_tail_weight(7, shape=(32, 640), frac=0.01))
    codes, scales = oracle.row_quantize(w)
    table = oracle.e4m3_decode_table()
    q = (f32_of_bits(w) / scales[:, None]).astype(np.float64)
    assert np.all(np.abs(q - table[codes]) <= 0.5 * e4m3_ulp(q))


def test_rows_api_matches_full():
    w = bits_of(inputs.gaussian_bf16((50, 260), 0.02, 73))
    c, s = oracle.row_quantize(w)
    rows = [49, 0, 17]
    cr, sr = oracle.row_quantize(w, rows=rows)
    assert np.array_equal(cr, c[rows]) and np.array_equal(sr, s[rows])
    ct, st = oracle.tensor_quantize(w)
    ctr, str_ = oracle.tensor_quantize(w, rows=rows)
    assert np.array_equal(ctr, ct[rows]) and st[0] == str_[0]


# ------------------------------------------------------------------- GEMV
SHAPES = [(1, 1, 1), (3, 1, 7), (2, 130, 300), (4, 320, 704), (5, 64, 33)]


@pytest.mark.parametrize("m,n,k", SHAPES)
@pytest.mark.parametrize("mode", ["row", "tensor"])
def test_gemv_vs_numpy_dequant_matmul(m, n, k, mode):
    w = bits_of(inputs.gaussian_bf16((n, k), 0.02, n * 5 + k))
    x = bits_of(inputs.activations(m, k, 51 + m))
    codes, scales = (oracle.row_quantize if mode == "row" else oracle.tensor_quantize)(w)
    y = oracle.row_gemv(x, codes, scales)
    s = np.broadcast_to(scales.astype(np.float64), (n,))
    deq = e4m3_values_torch()[codes] * s[:, None]
    ref = f32_of_bits(x).astype(np.float64) @ deq.T
    assert y.shape == (m, n)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_one_hot_is_exact():
    w = bits_of(inputs.gaussian_bf16((70, 300), 0.02, 74))
    codes, scales = oracle.row_quantize(w)
    table = e4m3_values_torch()
    for kk in (0, 127, 128, 299):
        x = np.zeros((1, 300), dtype=np.uint16)
        x[0, kk] = 0x3F80  # 1.0
        y = oracle.row_gemv(x, codes, scales)
        assert np.array_equal(y[0], table[codes[:, kk]] * scales.astype(np.float64))


def test_row_gemv_equals_block_gemv_with_tile_constant_scales():
    """Per-row scales that are constant over each 128-row tile are the block
    scales broadcast along K: the two GEMVs must agree to rounding."""
    n, k = 300, 400
    rng = np.random.default_rng(8)
    codes = rng.integers(0, 256, (n, k), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10
    tile_s = np.float32(rng.uniform(1e-4, 1e-3, 3))
    row_s = np.repeat(tile_s, 128)[:n].astype(np.float32)
    block_s = np.repeat(tile_s[:, None], 4, 1).astype(np.float32)
    x = bits_of(inputs.activations(3, k, 9))
    yr = oracle.row_gemv(x, codes, row_s)
    yb = oracle.block_gemv(x, codes, block_s)
    assert np.allclose(yr, yb, rtol=1e-13, atol=1e-13 * np.abs(yb).max())


def test_tensor_scale_broadcasts():
    w = bits_of(inputs.gaussian_bf16((20, 90), 0.02, 75))
    codes, scale = oracle.tensor_quantize(w)
    x = bits_of(inputs.activations(2, 90, 10))
    y1 = oracle.row_gemv(x, codes, scale)
    y2 = oracle.row_gemv(x, codes, np.full(20, scale[0], dtype=np.float32))
    assert np.array_equal(y1, y2)


def test_zero_input_gives_zero():
    w = bits_of(inputs.gaussian_bf16((9, 40), 0.02, 76))
    codes, scales = oracle.row_quantize(w)
    y = oracle.row_gemv(np.zeros((2, 40), dtype=np.uint16), codes, scales)
    assert np.all(y == 0)


def test_row_subset_matches_full():
    w = bits_of(inputs.gaussian_bf16((60, 130), 0.02, 77))
    codes, scales = oracle.row_quantize(w)
    x = bits_of(inputs.activations(3, 130, 11))
    full = oracle.row_gemv(x, codes, scales)
    rows = [59, 3, 3, 0]
    assert np.array_equal(oracle.row_gemv(x, codes, scales, rows=rows), full[:, rows])
