"""Pins for the oracle's e4m3 and bf16 codecs (CPU only).

Each check ties the oracle to something other than itself: the closed form of
the OCP E4M3 FN format, torch's float8_e4m3fn cast (an independent library),
an independent bit-arithmetic encoder, and brute-force neighbour search for
bf16 rounding.
"""
import math

import numpy as np
import pytest

import oracle
from conftest import bitwise_e4m3_encode, e4m3_values_torch


def test_decode_spot_values_closed_form(golden):
    t = oracle.e4m3_decode_table()
    assert t[0x7E] == golden["e4m3_max"]["value"] == 448.0
    assert t[0x08] == 2.0 ** -6           # smallest normal
    assert t[0x01] == 2.0 ** -9           # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9       # largest subnormal
    assert t[0x77] == 240.0
    assert t[0x38] == 1.0                 # E = 7 (bias), M = 0
    assert t[0x00] == 0.0 and not math.copysign(1, t[0x00]) < 0
    assert t[0x80] == 0.0 and math.copysign(1, t[0x80]) < 0
    assert t[0xFE] == -448.0
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])


def test_decode_structure():
    t = oracle.e4m3_decode_table()
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)                 # monotone in the code
    assert np.count_nonzero(pos > 0) == 126          # finite non-zero magnitudes
    for c in range(0x7F):
        assert t[c | 0x80] == -t[c]
    # every value is (integer with <= 4 significant bits) * 2^e, e >= -9
    for v in pos[1:]:
        m, e = math.frexp(v)
        assert (m * 16).is_integer() and e - 1 >= -9


def test_decode_matches_torch_exhaustive():
    ours = oracle.e4m3_decode_table()
    ref = e4m3_values_torch()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.signbit(ours[~both_nan]), np.signbit(ref[~both_nan]))


def _structured_f32():
    """Grid points, exact midpoints, their float32 neighbours, and a few
    points inside every interval between adjacent e4m3 magnitudes."""
    mags = oracle.e4m3_decode_table()[:0x7F]
    mags = np.append(mags, 480.0)  # virtual next point above 448
    vals = []
    for lo, hi in zip(mags[:-1], mags[1:]):
        mid = np.float32((lo + hi) / 2)
        for p in (np.float32(lo), np.float32(hi), mid):
            vals += [p, np.nextafter(p, np.float32(np.inf)), np.nextafter(p, np.float32(-np.inf))]
        vals += list(np.float32(lo + (hi - lo) * np.array([0.1, 0.3, 0.49, 0.51, 0.7, 0.9])))
    vals += [np.float32(2.0 ** e) for e in range(-149, 128)]
    vals += [np.float32(1e-45), np.float32(2.0 ** -10), np.float32(3 * 2.0 ** -11),
             np.float32(np.finfo(np.float32).max)]
    v = np.array(vals, dtype=np.float32)
    return np.concatenate([v, -v])


def test_encode_matches_bitwise_encoder_structured():
    v = _structured_f32()
    assert np.array_equal(oracle.e4m3_encode_f32(v), bitwise_e4m3_encode(v))


def test_encode_matches_bitwise_encoder_random():
    rng = np.random.default_rng(123)
    v = np.float32(np.exp(rng.uniform(np.log(2.0 ** -14), np.log(600.0), 300_000)))
    v *= np.where(rng.random(v.size) < 0.5, -1, 1).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode_f32(v), bitwise_e4m3_encode(v))


def test_encode_all_bf16_patterns_vs_torch():
    """Every finite bf16 value, cast by torch where torch's cast is defined
    the same way (|v| < 464: above that torch returns NaN instead of
    saturating)."""
    import torch
    bits = np.arange(65536, dtype=np.uint32)
    f32 = (bits << 16).view(np.float32)
    f32 = f32[np.isfinite(f32)]
    ours = oracle.e4m3_encode_f32(f32)
    ok = np.abs(f32) < 464.0
    ref = torch.from_numpy(f32[ok]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours[ok], ref)
    # saturation ("satfinite"): everything at or above 448 in magnitude -> +-448
    big = np.abs(f32) >= 448.0
    assert np.all((ours[big] & 0x7F) == 0x7E)
    assert np.array_equal(ours[big] >> 7, np.signbit(f32[big]).astype(np.uint8))


def test_encode_structured_vs_torch():
    import torch
    v = _structured_f32()
    ok = np.abs(v) < 464.0
    ref = torch.from_numpy(v[ok]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode_f32(v[ok]), ref)


def test_encode_ties_to_even_and_sign_of_zero():
    # 1.5 * 2^-9 lies halfway between codes 0x01 and 0x02: even code wins
    assert oracle.e4m3_encode(1.5 * 2.0 ** -9) == 0x02
    assert oracle.e4m3_encode(2.5 * 2.0 ** -9) == 0x02
    # halfway between 0 and the smallest subnormal rounds to 0
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(-(2.0 ** -10)) == 0x80
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-30) == 0x80
    # 464 (between 448 and the unrepresentable 480) saturates
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE


def _all_positive_bf16():
    bits = np.arange(0x0001, 0x7F80, dtype=np.uint32)
    return (bits << 16).view(np.float32).astype(np.float64), bits


def test_bf16_rounding_brute_force_neighbours():
    vals, bits = _all_positive_bf16()
    rng = np.random.default_rng(7)
    # random doubles spread over the whole bf16 range, plus exact midpoints
    xs = np.exp(rng.uniform(np.log(1e-41), np.log(3.3e38), 4000))
    mids = (vals[:-1] + vals[1:]) / 2
    xs = np.concatenate([xs, mids[rng.integers(0, len(mids), 2000)], vals[rng.integers(0, len(vals), 500)]])
    for x in xs:
        got = oracle.double_to_bf16(x)
        i = np.searchsorted(vals, x)
        cands = []
        if i < len(vals):
            cands.append((abs(vals[i] - x), bits[i]))
        if i > 0:
            cands.append((abs(vals[i - 1] - x), bits[i - 1]))
        if x < vals[0]:
            cands.append((x, 0))
        best = min(d for d, _ in cands)
        winners = [b for d, b in cands if d == best]
        want = winners[0] if len(winners) == 1 else [b for b in winners if b % 2 == 0][0]
        assert got == want, (x, hex(got), hex(want))
        assert oracle.double_to_bf16(-x) == want | 0x8000


def test_bf16_special_values():
    assert oracle.double_to_bf16(0.0) == 0x0000
    assert oracle.double_to_bf16(-0.0) == 0x8000
    assert oracle.double_to_bf16(float("inf")) == 0x7F80
    assert oracle.double_to_bf16(3.4e38) == 0x7F80        # above max + half ulp
    assert oracle.double_to_bf16(255 * 2.0 ** 120) == 0x7F7F
    assert oracle.double_to_bf16(2.0 ** -133) == 0x0001
    assert oracle.double_to_bf16(2.0 ** -134) == 0x0000   # tie -> even (0)
    assert oracle.double_to_bf16(1.5 * 2.0 ** -133) == 0x0002
    for b in (0x3F80, 0x0001, 0x7F7F, 0x3DCD, 0xC040):
        assert oracle.double_to_bf16(oracle.bf16_to_double(b)) == b


@pytest.mark.parametrize("code", range(256))
def test_every_decoded_code_reencodes_to_itself(code):
    v = oracle.e4m3_decode(code)
    if math.isnan(v):
        return
    assert oracle.e4m3_encode(v) == code


def test_encode_every_finite_f32_vs_torch():
    """Exhaustive: the oracle's brute-force encoder against torch's
    float8_e4m3fn cast on every finite binary32 value below 464 in magnitude
    (above that torch gives NaN instead of saturating), and saturation to
    +-448 with the sign kept for every finite value at or above it."""
    import torch
    from f32_sweep import FINITE, f32_slice, sweep

    def check(base):
        f, fin = f32_slice(base)
        v = f[fin]
        ours = oracle.e4m3_encode_f32(v)
        small = np.abs(v) < 464.0
        ref = torch.from_numpy(v[small]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bad = int(np.count_nonzero(ours[small] != ref))
        big = ~small
        bad += int(np.count_nonzero((ours[big] & 0x7F) != 0x7E))
        bad += int(np.count_nonzero((ours[big] >> 7) != np.signbit(v[big])))
        return bad, v.size

    threads = torch.get_num_threads()
    torch.set_num_threads(1)
    try:
        bad, checked = sweep(check)
    finally:
        torch.set_num_threads(threads)
    assert checked == FINITE
    assert bad == 0
