"""Pins for the oracle's W8A8 GEMV (CPU only).

FreeToken PR #389 quantizes the activations dynamically per tensor (an amax
pass, then the cast) and multiplies them with the per-tensor e4m3 weight,
scaled by both scales.  The activation quantizer is the (pinned) per-tensor
quantizer applied to x; the GEMV is pinned against numpy's float64 matmul of
independently decoded codes, exact one-hot products, and the per-tensor
W8A16 GEMV when x is already on the e4m3 grid times its scale (then the
activation cast is exact and both must agree).
"""
import numpy as np
import pytest

import oracle
from conftest import e4m3_values_torch
from fp8_block_scaled_02_gb300 import inputs


def bits_of(t):
    return inputs.bf16_bits(t)


@pytest.mark.parametrize("m,n,k", [(1, 1, 1), (3, 5, 7), (4, 130, 300), (17, 64, 256)])
def test_w8a8_vs_numpy(m, n, k):
    wc, sw = oracle.tensor_quantize(bits_of(inputs.gaussian_bf16((n, k), 0.02, n + k)))
    xc, sx = oracle.act_quantize(bits_of(inputs.activations(m, k, m + 3)))
    y = oracle.w8a8_gemv(xc, sx, wc, sw)
    t = e4m3_values_torch()
    ref = (t[xc] @ t[wc].T) * float(sx[0]) * float(sw[0])
    assert y.shape == (m, n)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_one_hot_product_is_exact():
    t = e4m3_values_torch()
    wc = np.arange(256, dtype=np.uint8).reshape(256, 1)
    wc[(wc[:, 0] & 0x7F) == 0x7F] = 0
    xc = np.array([[0x38]], dtype=np.uint8)   # 1.0
    y = oracle.w8a8_gemv(xc, np.float32(0.5), wc, np.float32(0.25))
    assert np.array_equal(y[0], t[wc[:, 0]] * 0.125)


def test_act_quantize_is_the_per_tensor_rule():
    x = bits_of(inputs.activations(8, 300, 4))
    xc, sx = oracle.act_quantize(x)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    assert sx[0] == np.abs(xf).max() / np.float32(448.0)
    assert np.all(xc & 0x7F <= 0x7E)


def test_equals_w8a16_when_x_is_on_the_grid():
    """x = dec(code) * sx exactly (bf16-representable): quantizing x gives
    the same codes back, and W8A8 equals the per-tensor W8A16 GEMV."""
    rng = np.random.default_rng(5)
    t = e4m3_values_torch()
    codes = rng.integers(0, 0x70, (3, 200)).astype(np.uint8) | (rng.integers(0, 2, (3, 200)) << 7).astype(np.uint8)
    codes[0, 0] = 0x7E   # amax 448 -> sx = 2^-4 exactly
    sx = np.float32(2.0 ** -4)
    xf = (t[codes] * float(sx)).astype(np.float32)
    xb = (xf.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((xb.astype(np.uint32) << 16).view(np.float32), xf)
    xc, sx2 = oracle.act_quantize(xb)
    assert sx2[0] == sx and np.array_equal(xc, codes)
    wc, sw = oracle.tensor_quantize(bits_of(inputs.gaussian_bf16((40, 200), 0.02, 6)))
    y8 = oracle.w8a8_gemv(xc, sx2, wc, sw)
    y16 = oracle.row_gemv(xb, wc, sw)
    assert np.allclose(y8, y16, rtol=1e-13, atol=1e-13 * np.abs(y16).max())


def test_zero_activations():
    xc, sx = oracle.act_quantize(np.zeros((2, 50), dtype=np.uint16))
    assert sx[0] == 1.0 and np.all(xc == 0)
    wc, sw = oracle.tensor_quantize(bits_of(inputs.gaussian_bf16((9, 50), 0.02, 7)))
    assert np.all(oracle.w8a8_gemv(xc, sx, wc, sw) == 0)


def test_row_subset_matches_full():
    wc, sw = oracle.tensor_quantize(bits_of(inputs.gaussian_bf16((30, 64), 0.02, 8)))
    xc, sx = oracle.act_quantize(bits_of(inputs.activations(2, 64, 9)))
    full = oracle.w8a8_gemv(xc, sx, wc, sw)
    assert np.array_equal(oracle.w8a8_gemv(xc, sx, wc, sw, rows=[29, 0, 7]), full[:, [29, 0, 7]])
