"""The GEMV acceptance test (oracle/tolerance.py) is tight enough to catch the
mistakes a block-FP8 or MXFP8 GEMV kernel plausibly makes (CPU only).

Each case builds a kernel-like result in numpy -- fp32 partial sums per K block
(block scales) or per 32-element group (MX), the scale applied to the fp32
partial, one bf16 rounding at the end -- once correctly and once with one
planted mistake, and checks that the acceptance test passes the first and
rejects the second, against the oracle's fp64 result.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import inputs
from oracle import tolerance


def to_bf16_bits(y64: np.ndarray) -> np.ndarray:
    return inputs.bf16_bits(torch.from_numpy(np.ascontiguousarray(y64, dtype=np.float32)).to(torch.bfloat16))


def x_f32(xb):
    return (xb.astype(np.uint32) << 16).view(np.float32)


def kernel_like_block(xb, codes, scales, bug=None):
    """fp32 partial per (row, K block) x scale, fp32 sum, bf16 rounding; `bug`
    plants one mistake."""
    table = oracle.e4m3_decode_table().astype(np.float32)
    x = x_f32(xb)
    m, k = x.shape
    n = codes.shape[0]
    nb, kb_n = scales.shape
    deq = table[codes]                                     # unscaled weights, fp32
    y = np.zeros((m, n), dtype=np.float32)
    for kb in range(kb_n):
        if bug == "drop_last_block" and kb == kb_n - 1:
            continue
        c0, c1 = kb * 128, min(k, kb * 128 + 128)
        xs = x[:, c0:c1]
        if bug == "x_rows_shifted":
            xs = np.roll(xs, 1, axis=0)
        part = xs @ deq[:, c0:c1].T                        # fp32 partial [m, n]
        for rb in range(nb):
            r0, r1 = rb * 128, min(n, rb * 128 + 128)
            s = scales[rb, kb]
            if bug == "next_k_block_scale":
                s = scales[rb, (kb + 1) % kb_n]
            elif bug == "next_row_block_scale":
                s = scales[(rb + 1) % nb, kb]
            elif bug == "transposed_scale_grid":
                s = scales.T.reshape(nb, kb_n)[rb, kb]     # same buffer read with the other stride
            elif bug == "scale_applied_twice":
                s = s * s
            elif bug == "sign_of_one_block" and kb == 1:
                s = -s
            y[:, r0:r1] += np.float32(s) * part[:, r0:r1]
    return to_bf16_bits(y)


def kernel_like_mx(xb, codes, e8m0, bug=None):
    table = oracle.e4m3_decode_table().astype(np.float32)
    x = x_f32(xb)
    m, k = x.shape
    deq = table[codes]
    groups = e8m0.shape[1]
    y = np.zeros((m, codes.shape[0]), dtype=np.float32)
    for g in range(groups):
        c0, c1 = g * 32, min(k, g * 32 + 32)
        part = x[:, c0:c1] @ deq[:, c0:c1].T
        E = e8m0[:, g].astype(np.int64)
        if bug == "next_group_exponent":
            E = e8m0[:, (g + 1) % groups].astype(np.int64)
        elif bug == "bias_126":
            E = E + 1
        y += np.ldexp(np.float32(1.0), (E - 127))[None, :].astype(np.float32) * part
    return to_bf16_bits(y)


@pytest.fixture(scope="module")
def block_case():
    w = inputs.bf16_bits(inputs.gaussian_bf16((384, 704), 0.02, 5))   # 3 x 6 tiles, ragged K
    xb = inputs.bf16_bits(inputs.activations(4, 704, 6))
    codes, scales = oracle.block_quantize(w)
    y64 = oracle.block_gemv(xb, codes, scales)
    wmax = tolerance.block_wmax_rows(codes, scales, np.arange(codes.shape[0]), oracle.e4m3_decode_table())
    return xb, codes, scales, y64, wmax


@pytest.fixture(scope="module")
def mx_case():
    w = inputs.bf16_bits(inputs.gaussian_bf16((256, 704), 0.02, 7))
    xb = inputs.bf16_bits(inputs.activations(4, 704, 8))
    codes, e8m0 = oracle.mx_quantize(w)
    y64 = oracle.mx_gemv(xb, codes, e8m0)
    wmax = tolerance.mx_wmax_rows(codes, e8m0, oracle.e4m3_decode_table())
    return xb, codes, e8m0, y64, wmax


def test_correct_block_kernel_passes(block_case):
    xb, codes, scales, y64, wmax = block_case
    st = tolerance.gemv_errors(kernel_like_block(xb, codes, scales), y64, xb, wmax)
    assert tolerance.gemv_ok(st), st


@pytest.mark.parametrize("bug", ["drop_last_block", "x_rows_shifted", "next_k_block_scale",
                                 "next_row_block_scale", "transposed_scale_grid", "scale_applied_twice",
                                 "sign_of_one_block"])
def test_block_kernel_mistakes_fail(block_case, bug):
    xb, codes, scales, y64, wmax = block_case
    st = tolerance.gemv_errors(kernel_like_block(xb, codes, scales, bug), y64, xb, wmax)
    assert not tolerance.gemv_ok(st), (bug, st)


def test_correct_mx_kernel_passes(mx_case):
    xb, codes, e8m0, y64, wmax = mx_case
    st = tolerance.gemv_errors(kernel_like_mx(xb, codes, e8m0), y64, xb, wmax)
    assert tolerance.gemv_ok(st), st


@pytest.mark.parametrize("bug", ["next_group_exponent", "bias_126"])
def test_mx_kernel_mistakes_fail(mx_case, bug):
    xb, codes, e8m0, y64, wmax = mx_case
    st = tolerance.gemv_errors(kernel_like_mx(xb, codes, e8m0, bug), y64, xb, wmax)
    assert not tolerance.gemv_ok(st), (bug, st)
