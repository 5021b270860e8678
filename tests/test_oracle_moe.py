"""Pins for the oracle's grouped MoE GEMV (CPU only).

Each (token, slot) output is the block GEMV of that token with the selected
expert's weight (Atlas quantize_fp8_bs.rs module notes: routed experts as
block-FP8 weights with [N/128, K/128] fp32 scales).  Pinned against numpy's
float64 matmul of independently dequantized expert weights, invariance
under relabelling the experts, and out-of-range ids giving zero rows.
"""
import numpy as np

import oracle
from conftest import e4m3_values_torch
from fp8_block_scaled_02_gb300 import inputs


def experts(e, n, k, seed):
    codes, scales = [], []
    for i in range(e):
        c, s = oracle.block_quantize(inputs.bf16_bits(inputs.gaussian_bf16((n, k), 0.02, seed + i)))
        codes.append(c)
        scales.append(s)
    return np.stack(codes), np.stack(scales)


def test_vs_numpy_dequant():
    E, n, k, m, topk = 5, 130, 260, 3, 2
    codes, scales = experts(E, n, k, 10)
    x = inputs.bf16_bits(inputs.activations(m, k, 4))
    ids = np.array([[4, 0], [1, 3], [2, 4]], dtype=np.int32)
    y = oracle.moe_gemv(x, ids, codes, scales)
    t = e4m3_values_torch()
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for ti in range(m):
        for j in range(topk):
            e = ids[ti, j]
            s = np.repeat(np.repeat(scales[e].astype(np.float64), 128, 0), 128, 1)[:n, :k]
            ref = (t[codes[e]] * s) @ xf[ti]
            assert np.allclose(y[ti, j], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_relabelling_experts_is_invariant():
    E, n, k = 4, 64, 128
    codes, scales = experts(E, n, k, 20)
    x = inputs.bf16_bits(inputs.activations(2, k, 5))
    ids = np.array([[0, 3], [2, 1]], dtype=np.int32)
    perm = np.array([2, 0, 3, 1])          # new label of old expert i is perm[i]
    inv = np.argsort(perm)
    y1 = oracle.moe_gemv(x, ids, codes, scales)
    y2 = oracle.moe_gemv(x, perm[ids].astype(np.int32), codes[inv], scales[inv])
    assert np.array_equal(y1, y2)


def test_out_of_range_ids_give_zero_rows():
    codes, scales = experts(2, 32, 64, 30)
    x = inputs.bf16_bits(inputs.activations(2, 64, 6))
    y = oracle.moe_gemv(x, np.array([[0, 7], [-1, 1]], dtype=np.int32), codes, scales)
    assert np.all(y[0, 1] == 0) and np.all(y[1, 0] == 0) and np.any(y[0, 0] != 0)


def test_row_subset_matches_full():
    codes, scales = experts(3, 200, 128, 40)
    x = inputs.bf16_bits(inputs.activations(2, 128, 7))
    ids = np.array([[2, 0], [1, 2]], dtype=np.int32)
    full = oracle.moe_gemv(x, ids, codes, scales)
    rows = [199, 0, 128]
    assert np.array_equal(oracle.moe_gemv(x, ids, codes, scales, rows=rows), full[:, :, rows])
