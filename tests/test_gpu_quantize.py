"""GPU parity: block-FP8 and MXFP8 load-time quantization vs the CPU oracle.

Codes and scales must be bit-exact.  Small and ragged cases are compared in
full; the full-size workloads (lm_head [152064, 4096], MXFP8 [18432, 7168])
are compared on sampled tiles / rows, plus properties checked over every
tile on the device.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import inputs

from gpu_helpers import bits, guard_intact, guarded_empty, lib_or_skip

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    return lib_or_skip()


def run_block(pkg, w_cpu, offset_elems=0):
    n, k = w_cpu.shape
    if offset_elems:
        buf = torch.empty(n * k + offset_elems, dtype=torch.bfloat16, device=DEV)
        w = buf[offset_elems:].view(n, k)
        w.copy_(w_cpu)
    else:
        w = w_cpu.to(DEV)
    codes, craw = guarded_empty((n, k), torch.uint8, DEV)
    scales, sraw = guarded_empty((-(-n // 128), -(-k // 128)), torch.float32, DEV)
    pkg.quantize(w, codes=codes, scales=scales)
    torch.cuda.synchronize()
    assert guard_intact(craw, n * k) and guard_intact(sraw, scales.numel() * 4)
    return codes.cpu().numpy(), scales.cpu().numpy()


def run_mx(pkg, w_cpu, offset_elems=0):
    n, k = w_cpu.shape
    if offset_elems:
        buf = torch.empty(n * k + offset_elems, dtype=torch.bfloat16, device=DEV)
        w = buf[offset_elems:].view(n, k)
        w.copy_(w_cpu)
    else:
        w = w_cpu.to(DEV)
    codes, craw = guarded_empty((n, k), torch.uint8, DEV)
    e8m0, eraw = guarded_empty((n, -(-k // 32)), torch.uint8, DEV)
    pkg.mx_quantize(w, codes=codes, e8m0=e8m0)
    torch.cuda.synchronize()
    assert guard_intact(craw, n * k) and guard_intact(eraw, e8m0.numel())
    return codes.cpu().numpy(), e8m0.cpu().numpy()


def assert_block_equal(pkg, w_cpu, **kw):
    c, s = run_block(pkg, w_cpu, **kw)
    oc, os_ = oracle.block_quantize(bits(w_cpu))
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32)), np.argwhere(s != os_)[:5]
    bad = np.argwhere(c != oc)
    assert bad.size == 0, (bad[:5], c[tuple(bad[0])], oc[tuple(bad[0])])


def assert_mx_equal(pkg, w_cpu, **kw):
    c, e = run_mx(pkg, w_cpu, **kw)
    oc, oe = oracle.mx_quantize(bits(w_cpu))
    assert np.array_equal(e, oe), np.argwhere(e != oe)[:5]
    assert np.array_equal(c, oc), np.argwhere(c != oc)[:5]


def test_tiny_ragged_block(pkg):
    assert_block_equal(pkg, inputs.tiny_ragged_weight(0))


def test_tiny_ragged_mx(pkg):
    assert_mx_equal(pkg, inputs.tiny_ragged_weight(0))


SHAPES = [(1, 1), (1, 8), (7, 5), (3, 40), (129, 257), (300, 33), (256, 1024), (128, 128), (200, 136), (64, 7168)]


@pytest.mark.parametrize("n,k", SHAPES)
def test_shapes_block(pkg, n, k):
    assert_block_equal(pkg, inputs.gaussian_bf16((n, k), 0.02, 100 + n + k))


@pytest.mark.parametrize("n,k", SHAPES)
def test_shapes_mx(pkg, n, k):
    assert_mx_equal(pkg, inputs.heavy_tail_weight(7, shape=(n, k), frac=0.01))


@pytest.mark.parametrize("offset", [1, 4])
def test_unaligned_source_takes_scalar_kernel(pkg, offset):
    w = inputs.gaussian_bf16((130, 264), 0.02, 55)
    assert_block_equal(pkg, w, offset_elems=offset)
    assert_mx_equal(pkg, w, offset_elems=offset)


def special_weight():
    """Zero tiles, -0, bf16 subnormals, the largest bf16, an exact 448 tile,
    values on rounding midpoints."""
    w = inputs.gaussian_bf16((384, 512), 0.02, 9).view(torch.int16).numpy().view(np.uint16).copy()
    w[:128, :128] = 0                     # all-zero tile
    w[5, 7] = 0x8000                      # -0 inside it
    w[128:256, :128] = 0x0001             # tile of the smallest subnormal
    w[130, 3] = 0x8005
    w[:128, 128:256] = 0x3F80             # 1.0 ...
    w[17, 200] = 0x43E0                   # ... with amax exactly 448
    w[256:, 256:384] = 0x7F7F             # largest finite bf16
    w[300, 300] = 0xFF7F
    w[256, 384:] = 0x4040                 # 3.0 rows: ties when divided
    t = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16)
    return t


def test_special_values_block(pkg):
    assert_block_equal(pkg, special_weight())


def test_special_values_mx(pkg):
    assert_mx_equal(pkg, special_weight())


def test_quotients_on_rounding_midpoints(pkg):
    """Tiles whose scale is a power of two (amax = 448 * 2^j) and whose
    entries sit exactly on e4m3 rounding midpoints (and their bf16
    neighbours) times that scale: every tie must resolve to the even code,
    exactly as the oracle's IEEE quotient does."""
    mags = oracle.e4m3_decode_table()[:0x7F]
    mids = (mags[:-1] + mags[1:]) / 2
    rng = np.random.default_rng(11)
    w = np.zeros((256, 256), dtype=np.float64)
    for bn in range(2):
        for bk in range(2):
            j = int(rng.integers(-20, 10))
            tile = rng.choice(mids, size=(128, 128)) * rng.choice([-1.0, 1.0], size=(128, 128))
            tile[0, 0] = 448.0
            w[bn * 128:(bn + 1) * 128, bk * 128:(bk + 1) * 128] = tile * 2.0 ** j
    wt = torch.from_numpy(w).to(torch.bfloat16)
    # bf16 neighbours of some entries (one ulp up/down) for near-ties
    bitsw = wt.view(torch.int16).numpy().view(np.uint16).copy()
    bitsw[1::3, ::5] += 1
    bitsw[2::3, 1::5] -= 1
    wt = torch.from_numpy(bitsw.view(np.int16)).view(torch.bfloat16)
    assert_block_equal(pkg, wt)


def test_amax_448_tile_is_plain_cast(pkg):
    w = special_weight()
    c, s = run_block(pkg, w)
    assert s[0, 1] == 1.0 and c[17, 200] == 0x7E and c[0, 128] == 0x38  # 1.0 -> 0x38


# --------------------------------------------------------- full-size cases
def _sample_tiles(nb, kb, rng, count):
    tiles = {(0, 0), (nb - 1, kb - 1), (0, kb - 1), (nb - 1, 0)}
    while len(tiles) < count:
        tiles.add((int(rng.integers(nb)), int(rng.integers(kb))))
    return sorted(tiles)


@pytest.mark.parametrize("which", ["lm_head", "mx_shape"])
def test_full_size_block_sampled_tiles(pkg, which):
    if which == "lm_head":
        w = inputs.lm_head_weight(2, device=DEV)
    else:
        w = inputs.heavy_tail_weight(5, device=DEV)
    n, k = w.shape
    codes, scales = pkg.quantize(w)
    torch.cuda.synchronize()
    nb, kb = -(-n // 128), -(-k // 128)
    # every tile: its amax element encodes to +-448 and no NaN code appears
    tiles = (codes.view(nb, 128, kb, 128) & 0x7F).amax(dim=(1, 3))
    assert int((tiles != 0x7E).sum()) == 0
    assert int(((codes & 0x7F) == 0x7F).sum()) == 0
    rng = np.random.default_rng(1)
    for bn, bk in _sample_tiles(nb, kb, rng, 48):
        wt = bits(w[bn * 128:(bn + 1) * 128, bk * 128:(bk + 1) * 128].cpu())
        oc, os_ = oracle.block_quantize(wt)
        gc = codes[bn * 128:(bn + 1) * 128, bk * 128:(bk + 1) * 128].cpu().numpy()
        assert np.array_equal(gc, oc), (bn, bk)
        assert scales[bn, bk].item() == float(os_[0, 0]), (bn, bk)


def test_full_size_mx_sampled_rows(pkg):
    w = inputs.heavy_tail_weight(5, device=DEV)
    n, k = w.shape
    codes, e8m0 = pkg.mx_quantize(w)
    torch.cuda.synchronize()
    assert int(((codes & 0x7F) == 0x7F).sum()) == 0
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 62)]))
    wr = bits(w[torch.from_numpy(rows).to(DEV)].cpu())
    oc, oe = oracle.mx_quantize(wr)
    assert np.array_equal(e8m0[torch.from_numpy(rows).to(DEV)].cpu().numpy(), oe)
    assert np.array_equal(codes[torch.from_numpy(rows).to(DEV)].cpu().numpy(), oc)


def test_encode_step_every_finite_f32_matches_oracle(pkg):
    """Exhaustive: the e4m3 encode step every quantizer applies to its fp32
    quotients, run on the GPU (fp8bs_debug_encode_f32, 2^28 patterns per
    launch), against the oracle's brute-force nearest-code encoder on every
    finite binary32 value."""
    from f32_sweep import ALL, FINITE, SLICE, f32_slice, sweep
    chunk = 1 << 28
    buf = torch.empty(chunk, dtype=torch.uint8, device=DEV)
    bad = checked = 0
    examples = []
    for c0 in range(0, ALL, chunk):
        pkg.debug_encode_f32(c0, chunk, out=buf)
        host = buf.cpu().numpy()

        def check(base, host=host, c0=c0):
            f, fin = f32_slice(base)
            got = host[base - c0:base - c0 + SLICE][fin]
            ref = oracle.e4m3_encode_f32(f[fin])
            wrong = np.nonzero(got != ref)[0]
            if wrong.size:
                i = wrong[0]
                examples.append((hex(int(f[fin][i].view(np.uint32))), int(got[i]), int(ref[i])))
            return int(wrong.size), int(ref.size)
        b, n = sweep(check, range(c0, c0 + chunk, SLICE))
        bad += b
        checked += n
    assert checked == FINITE
    assert bad == 0, examples[:5]
    assert pkg.check_device_error() == 0


def test_no_device_error(pkg):
    assert pkg.check_device_error() == 0
