"""Pins for the oracle's fp64 W8A16 GEMV (CPU only).

InfiniLM PR #586 and FreeToken PR #389 (Testing) check the FP8 linear
against a plain linear on the *dequantized* weight; here the dequantized
weight is built independently (torch's float8_e4m3fn decode times the block
scale) and multiplied with numpy's float64 matmul.  One-hot inputs pin the
indexing and the scale lookup exactly, including ragged edge tiles.
"""
import numpy as np
import pytest

import oracle
from conftest import e4m3_values_torch
from fp8_block_scaled_02_gb300 import inputs


def f32_of_bits(b):
    return (np.asarray(b).astype(np.uint32) << 16).view(np.float32)


def dequant_block_independent(codes, scales):
    table = e4m3_values_torch()
    n, k = codes.shape
    s = np.repeat(np.repeat(scales.astype(np.float64), 128, 0), 128, 1)[:n, :k]
    return table[codes] * s


def dequant_mx_independent(codes, e8m0):
    table = e4m3_values_torch()
    n, k = codes.shape
    s = np.ldexp(1.0, np.repeat(e8m0.astype(np.int64) - 127, 32, 1)[:, :k])
    return table[codes] * s


SHAPES = [(1, 1, 1), (1, 5, 1), (3, 1, 7), (2, 130, 300), (4, 320, 704), (1, 129, 128), (5, 64, 33)]


@pytest.mark.parametrize("m,n,k", SHAPES)
def test_block_gemv_vs_numpy_dequant_matmul(m, n, k):
    w = inputs.bf16_bits(inputs.gaussian_bf16((n, k), 0.02, n * 7 + k))
    x = inputs.bf16_bits(inputs.activations(m, k, 31 + m))
    codes, scales = oracle.block_quantize(w)
    y = oracle.block_gemv(x, codes, scales)
    ref = f32_of_bits(x).astype(np.float64) @ dequant_block_independent(codes, scales).T
    assert y.shape == (m, n)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("m,n,k", SHAPES)
def test_mx_gemv_vs_numpy_dequant_matmul(m, n, k):
    w = inputs.bf16_bits(inputs.gaussian_bf16((n, k), 0.02, n * 3 + k))
    x = inputs.bf16_bits(inputs.activations(m, k, 41 + m))
    codes, e8m0 = oracle.mx_quantize(w)
    y = oracle.mx_gemv(x, codes, e8m0)
    ref = f32_of_bits(x).astype(np.float64) @ dequant_mx_independent(codes, e8m0).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_one_hot_is_exact_on_ragged_tiles():
    """x = e_k picks column k exactly: y[n] = dec(q[n,k]) * s[n//128, k//128]."""
    w = inputs.bf16_bits(inputs.tiny_ragged_weight(0))
    n, k = w.shape
    codes, scales = oracle.block_quantize(w)
    table = e4m3_values_torch()
    for col in (0, 127, 128, 600, 703):
        x = np.zeros((1, k), dtype=np.uint16)
        x[0, col] = 0x3F80  # 1.0
        y = oracle.block_gemv(x, codes, scales)[0]
        want = table[codes[:, col]] * scales[np.arange(n) // 128, col // 128].astype(np.float64)
        assert np.array_equal(y, want)


def test_mx_one_hot_is_exact():
    w = inputs.bf16_bits(inputs.heavy_tail_weight(5, shape=(50, 70), frac=0.02))
    codes, e8m0 = oracle.mx_quantize(w)
    table = e4m3_values_torch()
    for col in (0, 31, 32, 69):
        x = np.zeros((1, 70), dtype=np.uint16)
        x[0, col] = 0xC000  # -2.0
        y = oracle.mx_gemv(x, codes, e8m0)[0]
        want = -2.0 * table[codes[:, col]] * np.ldexp(1.0, e8m0[:, col // 32].astype(np.int64) - 127)
        assert np.array_equal(y, want)


def test_zero_input_gives_zero():
    w = inputs.bf16_bits(inputs.gaussian_bf16((70, 90), 0.02, 1))
    codes, scales = oracle.block_quantize(w)
    y = oracle.block_gemv(np.zeros((3, 90), dtype=np.uint16), codes, scales)
    assert np.all(y == 0)


def test_scale_doubling_changes_only_its_tile():
    """Doubling scales[bn, bk] adds exactly the contribution of tile
    (bn, bk) once more (pins the scale layout [N/128, K/128])."""
    w = inputs.bf16_bits(inputs.gaussian_bf16((300, 260), 0.02, 2))
    x = inputs.bf16_bits(inputs.activations(2, 260, 3))
    codes, scales = oracle.block_quantize(w)
    y0 = oracle.block_gemv(x, codes, scales)
    s2 = scales.copy()
    s2[1, 2] *= 2
    y1 = oracle.block_gemv(x, codes, s2)
    dq = dequant_block_independent(codes, scales)
    part = f32_of_bits(x)[:, 256:260].astype(np.float64) @ dq[128:256, 256:260].T
    assert np.allclose(y1[:, 128:256] - y0[:, 128:256], part, rtol=1e-12, atol=1e-15)
    assert np.array_equal(y1[:, :128], y0[:, :128]) and np.array_equal(y1[:, 256:], y0[:, 256:])


def test_row_subset_matches_full():
    w = inputs.bf16_bits(inputs.gaussian_bf16((200, 150), 0.02, 12))
    x = inputs.bf16_bits(inputs.activations(3, 150, 13))
    codes, scales = oracle.block_quantize(w)
    full = oracle.block_gemv(x, codes, scales)
    rows = [199, 0, 128, 57]
    assert np.array_equal(oracle.block_gemv(x, codes, scales, rows=rows), full[:, rows])
    e_codes, e8m0 = oracle.mx_quantize(w)
    fullmx = oracle.mx_gemv(x, e_codes, e8m0)
    assert np.array_equal(oracle.mx_gemv(x, e_codes, e8m0, rows=rows), fullmx[:, rows])


def test_linearity_in_x():
    w = inputs.bf16_bits(inputs.gaussian_bf16((64, 256), 0.02, 14))
    codes, scales = oracle.block_quantize(w)
    x = np.zeros((2, 256), dtype=np.uint16)
    x[0, :128] = inputs.bf16_bits(inputs.activations(1, 128, 15))[0]
    x[1, 128:] = inputs.bf16_bits(inputs.activations(1, 128, 16))[0]
    xs = x[0] | x[1]  # disjoint supports: the bf16 sum is exact
    y = oracle.block_gemv(np.stack([x[0], x[1], xs]), codes, scales)
    assert np.allclose(y[0] + y[1], y[2], rtol=1e-13, atol=1e-15)
