"""Pins for the oracle's block-FP8 and MXFP8 quantizers (CPU only).

The checks come from what the pages and the format fix: hand-worked
examples (tests/golden/worked_examples.json), the amax-to-448 invariant,
the zero-tile and amax==448 special cases, the per-element error bound, the
~2.25% round-trip error FreeToken PR #636 reports, block locality (a tile's
codes depend on that tile alone), and the MX exponent's defining inequality.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import bitwise_e4m3_encode
from fp8_block_scaled_02_gb300 import inputs


def bits_of(t: torch.Tensor) -> np.ndarray:
    return inputs.bf16_bits(t)


def f32_of_bits(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def e4m3_ulp(v):
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    return np.ldexp(1.0, np.maximum(ex - 1, -6) - 3)


# ------------------------------------------------------------------ block
def test_worked_example_block(golden):
    ex = golden["block_tile_2x2"]
    w = np.array(ex["w_bf16_bits"], dtype=np.uint16)
    codes, scales = oracle.block_quantize(w)
    assert codes.tolist() == ex["codes"]
    assert scales.shape == (1, 1)
    assert int(scales.view(np.uint32)[0, 0]) == ex["scale_f32_bits"]


@pytest.mark.parametrize("n,k", [(1, 1), (128, 128), (129, 257), (320, 704), (300, 33)])
def test_scale_grid_shape(n, k):
    w = bits_of(inputs.gaussian_bf16((n, k), 0.02, 11))
    codes, scales = oracle.block_quantize(w)
    assert codes.shape == (n, k)
    assert scales.shape == (math.ceil(n / 128), math.ceil(k / 128))


def _tiles(n, k):
    for bn in range(math.ceil(n / 128)):
        for bk in range(math.ceil(k / 128)):
            yield bn, bk, slice(bn * 128, min(n, bn * 128 + 128)), slice(bk * 128, min(k, bk * 128 + 128))


def test_amax_element_maps_to_448_and_scale_formula():
    w = bits_of(inputs.tiny_ragged_weight(0))
    n, k = w.shape
    codes, scales = oracle.block_quantize(w)
    wf = f32_of_bits(w)
    for bn, bk, rs, cs in _tiles(n, k):
        tile = np.abs(wf[rs, cs])
        amax = tile.max()
        assert scales[bn, bk] == np.float32(amax) / np.float32(448.0)
        r, c = np.unravel_index(np.argmax(tile), tile.shape)
        assert codes[rs, cs][r, c] & 0x7F == 0x7E


def test_block_scale_every_bf16_amax():
    """Exhaustive over the tile maximum: one ragged 1 x 128 tile per positive
    finite bf16 amax (with its negation and a smaller element beside it).
    s is the IEEE fp32 quotient amax / 448; the codes are the independent
    encoder's codes of the IEEE fp32 quotients w / s; and whenever s is a
    normal fp32 value the amax element encodes to exactly +-448."""
    amax_bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)
    t = amax_bits.size
    w = np.zeros((1, 128 * t), dtype=np.uint16)
    w[0, 0::128] = amax_bits
    w[0, 1::128] = amax_bits | 0x8000
    w[0, 2::128] = amax_bits >> 3
    codes, scales = oracle.block_quantize(w)
    amax = (amax_bits << 16).view(np.float32)
    s = amax / np.float32(448.0)                                      # IEEE fp32 division
    assert scales.shape == (1, t) and np.array_equal(scales[0].view(np.uint32), s.view(np.uint32))
    for col in (0, 1, 2):
        wv = (w[0, col::128].astype(np.uint32) << 16).view(np.float32)
        assert np.array_equal(codes[0, col::128], bitwise_e4m3_encode(wv / s))
    normal = s >= np.float32(2.0 ** -126)
    assert np.all(codes[0, 0::128][normal] == 0x7E) and np.all(codes[0, 1::128][normal] == 0xFE)


def test_tiny_ragged_outliers_set_their_tiles():
    w = bits_of(inputs.tiny_ragged_weight(0))
    codes, scales = oracle.block_quantize(w)
    for r, c, v in inputs.tiny_ragged_outliers(0):
        assert scales[r // 128, c // 128] == np.float32(1.5) / np.float32(448.0)
        assert codes[r, c] == (0x7E if v > 0 else 0xFE)


def test_zero_tile_and_negative_zero():
    w = bits_of(inputs.gaussian_bf16((256, 256), 0.02, 3))
    w[:128, 128:] = 0
    w[0, 130] = 0x8000  # -0.0
    codes, scales = oracle.block_quantize(w)
    assert scales[0, 1] == 1.0
    assert np.all(codes[:128, 128:][w[:128, 128:] == 0] == 0x00)
    assert codes[0, 130] == 0x80


def test_tile_with_amax_448_is_plain_cast():
    rng = np.random.default_rng(5)
    v = np.float32(rng.uniform(-448, 448, (128, 128)))
    v[17, 3] = 448.0
    w = (torch.from_numpy(v).to(torch.bfloat16))
    wb = bits_of(w)
    codes, scales = oracle.block_quantize(wb)
    assert scales[0, 0] == 1.0
    f = f32_of_bits(wb)
    assert np.array_equal(codes, bitwise_e4m3_encode(f))


def test_per_element_error_bound():
    w = bits_of(inputs.lm_head_weight(2, shape=(256, 384)))
    codes, scales = oracle.block_quantize(w)
    table = oracle.e4m3_decode_table()
    wf = f32_of_bits(w).astype(np.float64)
    s = np.repeat(np.repeat(scales, 128, 0), 128, 1)[:256, :384].astype(np.float64)
    q = (f32_of_bits(w) / s.astype(np.float32)).astype(np.float64)  # fp32 quotient
    dq = table[codes]
    assert np.all(np.abs(q - dq) <= 0.5 * e4m3_ulp(q) + 1e-300)
    # and in weight units: <= half an e4m3 ulp times s, plus the fp32 quotient rounding
    err = np.abs(wf - dq * s)
    assert np.all(err <= 0.5 * e4m3_ulp(q) * s + 2.0 ** -24 * np.abs(wf) * 1.0001)


def test_roundtrip_relative_error_matches_page(golden):
    """FreeToken PR #636 reports ~2.25% round-trip relative error for the
    128-block quantizer; on N(0, 0.02^2) weights the mean per-element
    |w_hat - w| / |w| is that number."""
    w = bits_of(inputs.gaussian_bf16((1024, 2048), 0.02, 21))
    codes, scales = oracle.block_quantize(w)
    table = oracle.e4m3_decode_table()
    wf = f32_of_bits(w).astype(np.float64)
    s = np.repeat(np.repeat(scales, 128, 0), 128, 1).astype(np.float64)
    what = table[codes] * s
    nz = wf != 0
    rel = np.abs(what[nz] - wf[nz]) / np.abs(wf[nz])
    target = golden["roundtrip_mean_relative_error"]["value"]
    assert abs(rel.mean() - target) < 0.0025, rel.mean()
    rel_l2 = np.linalg.norm(what - wf) / np.linalg.norm(wf)
    assert 0.024 < rel_l2 < 0.029


def test_block_locality():
    """A tile's codes and scale depend only on that tile: perturbing one
    tile changes nothing elsewhere (pins the tile indexing)."""
    w = bits_of(inputs.gaussian_bf16((300, 260), 0.02, 8))
    c0, s0 = oracle.block_quantize(w)
    w2 = w.copy()
    w2[130:140, 129:131] = 0x3FC0  # 1.5 inside tile (1, 1)
    c1, s1 = oracle.block_quantize(w2)
    diff_s = np.argwhere(s0 != s1)
    assert diff_s.tolist() == [[1, 1]]
    changed = np.argwhere(c0 != c1)
    assert changed.size and np.all(changed[:, 0] // 128 == 1) and np.all(changed[:, 1] // 128 == 1)


def test_tile_api_matches_full():
    w = bits_of(inputs.gaussian_bf16((260, 300), 0.02, 9))
    c, s = oracle.block_quantize(w)
    ct, st = oracle.block_quantize_tiles(w, [(2, 2), (0, 1)])
    assert np.array_equal(ct[256:, 256:], c[256:, 256:]) and st[2, 2] == s[2, 2]
    assert np.array_equal(ct[:128, 128:256], c[:128, 128:256]) and st[0, 1] == s[0, 1]


def test_subnormal_tile():
    """A tile of bf16 subnormals: s is an fp32 subnormal (never 0) and the
    amax element still maps to 448."""
    w = np.zeros((4, 4), dtype=np.uint16)
    w[0, 0] = 0x0001          # 2^-133
    w[1, 1] = 0x8003          # -3 * 2^-133
    codes, scales = oracle.block_quantize(w)
    s = scales[0, 0]
    assert 0 < s < np.finfo(np.float32).tiny
    assert s == np.float32(3 * 2.0 ** -133) / np.float32(448)
    assert codes[1, 1] == 0xFE


# --------------------------------------------------------------------- MX
def test_worked_example_mx(golden):
    ex = golden["mx_row_3_groups"]
    w = np.zeros((1, ex["k"]), dtype=np.uint16)
    for i, b in ex["nonzero_w"].items():
        w[0, int(i)] = b
    codes, e8m0 = oracle.mx_quantize(w)
    assert e8m0[0].tolist() == ex["e8m0"]
    want = np.zeros(ex["k"], dtype=np.uint8)
    for i, c in ex["nonzero_codes"].items():
        want[int(i)] = c
    assert np.array_equal(codes[0], want)
    ex2 = golden["mx_above_448"]
    w = np.zeros((1, 32), dtype=np.uint16)
    w[0, 5] = ex2["w_bf16_bits"]
    codes, e8m0 = oracle.mx_quantize(w)
    assert e8m0[0, 0] == ex2["e8m0"] and codes[0, 5] == ex2["code"]


def _exact_ceil_log2(amax: Fraction) -> int:
    """ceil(log2(amax / 448)) by exact rational comparison."""
    r = amax / 448
    e = math.ceil(math.log2(r))  # a starting guess; the loops below make it exact
    while Fraction(2) ** e < r:
        e += 1
    while Fraction(2) ** (e - 1) >= r:
        e -= 1
    return e


def test_mx_exponent_definition_and_range():
    w = bits_of(inputs.heavy_tail_weight(5, shape=(64, 200), frac=0.01))
    codes, e8m0 = oracle.mx_quantize(w)
    wf = f32_of_bits(w).astype(np.float64)
    table = oracle.e4m3_decode_table()
    for r in range(64):
        for g in range(e8m0.shape[1]):
            grp = wf[r, g * 32:(g + 1) * 32]
            amax = np.abs(grp).max()
            E = int(e8m0[r, g])
            if amax == 0:
                assert E == 127
                continue
            e = _exact_ceil_log2(Fraction(float(amax)))
            assert E == e + 127
            ratio = amax / 2.0 ** e
            assert 224 < ratio <= 448                  # never saturates
            q = (grp / 2.0 ** e).astype(np.float32)    # exact (power of two)
            assert np.array_equal(codes[r, g * 32:(g + 1) * 32], bitwise_e4m3_encode(q))
            assert np.all(np.abs(table[codes[r, g * 32:(g + 1) * 32]]) <= 448)


def test_mx_grid_values_roundtrip_exactly():
    """w = e4m3 grid value * 2^j for a common j round-trips exactly."""
    table = oracle.e4m3_decode_table()
    rng = np.random.default_rng(3)
    for j in (-20, -3, 0, 5, 30):
        idx = rng.integers(0x08, 0x7F, 32)            # normal codes
        idx[0] = 0x7E                                  # amax = 448 * 2^j
        sgn = np.where(rng.random(32) < 0.5, -1.0, 1.0)
        v = sgn * table[idx] * 2.0 ** j
        w = torch.from_numpy(v).to(torch.bfloat16)
        wb = bits_of(w)
        assert np.array_equal(f32_of_bits(wb).astype(np.float64), v)  # exactly bf16
        codes, e8m0 = oracle.mx_quantize(wb[None, :])
        assert e8m0[0, 0] == 127 + j
        back = table[codes[0]] * 2.0 ** (int(e8m0[0, 0]) - 127)
        assert np.array_equal(back, v)


def test_mx_exponent_every_bf16_amax():
    """Exhaustive over the group maximum: for every positive finite bf16
    value as the amax of a 32-element group (the other elements smaller or
    its negation), E = clamp(ceil(log2(amax / 448)) + 127, 0, 254) by exact
    rational arithmetic; where E is not clamped, amax / 2^e lies in
    (224, 448] (the group never saturates) and the amax element's code is the
    independent bit-arithmetic encoder's code of that exact quotient, its
    negation's the same code with the sign bit set."""
    amax_bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)          # every positive finite bf16
    n = amax_bits.size
    w = np.zeros((n, 32), dtype=np.uint16)
    w[:, 13] = amax_bits
    w[:, 20] = amax_bits >> 1                                        # a smaller element of each group
    w[:, 27] = (amax_bits | 0x8000) & np.where(amax_bits > 1, 0xFFFF, 0x8000)  # -amax or -0
    codes, e8m0 = oracle.mx_quantize(w)
    vals = (amax_bits << 16).view(np.float32).astype(np.float64)
    es = np.array([_exact_ceil_log2(Fraction(float(v))) for v in vals])
    E = np.clip(es + 127, 0, 254)
    assert np.array_equal(e8m0[:, 0].astype(np.int64), E)
    free = (es + 127 >= 0) & (es + 127 <= 254)                           # E not clamped
    ratio = vals[free] * np.exp2(-es[free].astype(np.float64))            # exact: power-of-two scaling
    assert np.all((ratio > 224) & (ratio <= 448))
    want = bitwise_e4m3_encode(ratio.astype(np.float32))
    assert np.array_equal(codes[free, 13], want)
    neg = free & (amax_bits > 1)
    assert np.array_equal(codes[neg, 27], bitwise_e4m3_encode(ratio[(amax_bits > 1)[free]].astype(np.float32)) | 0x80)


@pytest.mark.parametrize("amax_bits,E", [(0x43E0, 127), (0x43E1, 128), (0x4360, 126), (0x4361, 127),
                                          (0x0000, 127), (0x0001, 0), (0x7F7F, 127 + 120)])
def test_mx_exponent_special_cases(amax_bits, E):
    """448 -> E=127; 450 -> 128; 224 -> 126; 225 -> 127; all-zero -> 127;
    the smallest bf16 subnormal clamps to E=0; the largest bf16 gives e=120."""
    w = np.zeros((1, 32), dtype=np.uint16)
    w[0, 7] = amax_bits
    _, e8m0 = oracle.mx_quantize(w)
    assert e8m0[0, 0] == E


def test_mx_group_axis_and_ragged_tail():
    w = bits_of(inputs.gaussian_bf16((3, 70), 0.02, 4))  # groups 32, 32, 6
    c0, e0 = oracle.mx_quantize(w)
    assert e0.shape == (3, 3)
    w2 = w.copy()
    w2[1, 66] = 0x4000  # 2.0 inside row 1, tail group 2
    c1, e1 = oracle.mx_quantize(w2)
    assert np.argwhere(e0 != e1).tolist() == [[1, 2]]
    changed = np.argwhere(c0 != c1)
    assert np.all(changed[:, 0] == 1) and np.all(changed[:, 1] >= 64)
    assert c1[1, 66] == 0x7E or e1[1, 2] == 127 + _exact_ceil_log2(Fraction(2))


def test_mx_rows_api_matches_full():
    w = bits_of(inputs.gaussian_bf16((40, 100), 0.02, 6))
    c, e = oracle.mx_quantize(w)
    cr, er = oracle.mx_quantize_rows(w, [39, 0, 17])
    assert np.array_equal(cr, c[[39, 0, 17]]) and np.array_equal(er, e[[39, 0, 17]])
