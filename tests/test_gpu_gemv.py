"""GPU parity: the W8A16 GEMV / skinny GEMM vs the CPU oracle's fp64 result.

The GEMV's inputs (codes, scales, x) on every checked output come from the
seeded generators and the oracle's own quantizer, never from the CUDA path.
Exact checks: every e4m3 code decodes exactly (one-hot x), one-hot columns
of ragged tiles give bf16(fl32(dec * s)), x = 0 gives 0.  Everything else is
held to the tolerance in oracle/tolerance.py.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import PATH_DECODE, PATH_GENERIC, PATH_PREFILL, inputs

from gpu_helpers import (bits, check_block_gemv, check_mx_gemv, guard_intact, guarded_empty, install_block_rows,
                         lib_or_skip, oracle_block_rows, table)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    return lib_or_skip()


def to_dev_bits(a: np.ndarray, dtype=torch.uint8):
    return torch.from_numpy(a).to(DEV)


def bf16_dev(a_bits: np.ndarray):
    return torch.from_numpy(a_bits.view(np.int16)).view(torch.bfloat16).to(DEV)


# ------------------------------------------------------------ exact checks
@pytest.mark.parametrize("path", [PATH_DECODE, PATH_GENERIC, PATH_PREFILL])
@pytest.mark.parametrize("m", [1, 5, 8, 9, 16, 17, 32, 40, 130])
def test_every_code_decodes_exactly(pkg, path, m):
    """Row i of W holds code i at column 3 (scales 1); x = e_3, so
    y[:, i] = bf16(dec(i)) exactly for every finite code."""
    codes_list = [c for c in range(256) if c not in (0x7F, 0xFF)]
    n, k = len(codes_list), 32
    w = np.zeros((n, k), dtype=np.uint8)
    w[:, 3] = codes_list
    scales = np.ones((-(-n // 128), 1), dtype=np.float32)
    x = np.zeros((m, k), dtype=np.uint16)
    x[:, 3] = 0x3F80
    y = pkg.gemv(bf16_dev(x), to_dev_bits(w), torch.from_numpy(scales).to(DEV), path=path)
    torch.cuda.synchronize()
    # a sum that starts from +0 turns the -0 of code 0x80 into +0 (IEEE)
    want = np.array([oracle.double_to_bf16(0.0 + v) for v in table()[codes_list]], dtype=np.uint16)
    got = bits(y.cpu())
    for i in range(m):
        assert np.array_equal(got[i], want), np.argwhere(got[i] != want)[:5]


@pytest.mark.parametrize("path", [PATH_DECODE, PATH_GENERIC, PATH_PREFILL])
def test_one_hot_columns_on_ragged_tiles(pkg, path):
    w = inputs.tiny_ragged_weight(0)
    n, k = w.shape
    oc, os_ = oracle.block_quantize(bits(w))
    codes, scales = to_dev_bits(oc), torch.from_numpy(os_).to(DEV)
    cols = [0, 1, 127, 128, 300, 640, 703]
    x = np.zeros((len(cols), k), dtype=np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = 0x3F80
    y = bits(pkg.gemv(bf16_dev(x), codes, scales, path=path).cpu())
    for i, c in enumerate(cols):
        prod = (table()[oc[:, c]].astype(np.float32) * os_[np.arange(n) // 128, c // 128]).astype(np.float32)
        want = np.array([oracle.double_to_bf16(0.0 + float(v)) for v in prod], dtype=np.uint16)
        assert np.array_equal(y[i], want), (c, np.argwhere(y[i] != want)[:5])


def test_zero_input_gives_zero(pkg):
    w = inputs.gaussian_bf16((256, 512), 0.02, 3)
    oc, os_ = oracle.block_quantize(bits(w))
    for path in (PATH_DECODE, PATH_GENERIC, PATH_PREFILL):
        y = pkg.gemv(torch.zeros((4, 512), dtype=torch.bfloat16, device=DEV), to_dev_bits(oc),
                     torch.from_numpy(os_).to(DEV), path=path)
        assert int((y.view(torch.int16) & 0x7FFF).abs().sum()) == 0


# ----------------------------------------------------------- small, full
def full_block_case(pkg, w, m, path, seed=7):
    n, k = w.shape
    oc, os_ = oracle.block_quantize(bits(w))
    x = inputs.activations(m, k, seed)
    y, raw = guarded_empty((m, n), torch.bfloat16, DEV)
    pkg.gemv(x.to(DEV), to_dev_bits(oc), torch.from_numpy(os_).to(DEV), y=y, path=path)
    torch.cuda.synchronize()
    assert guard_intact(raw, m * n * 2)
    rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(-(-n // 128))}
    return check_block_gemv(y, bits(x), rows_q)


@pytest.mark.parametrize("path", [PATH_DECODE, PATH_GENERIC, PATH_PREFILL])
@pytest.mark.parametrize("m", [1, 2, 3, 4, 7, 8, 9, 15, 16, 24, 31, 32, 33, 40, 64, 100])
def test_tiny_ragged_all_m(pkg, m, path):
    full_block_case(pkg, inputs.tiny_ragged_weight(0), m, path)


SHAPES = [(1, 16), (1, 1), (5, 300), (37, 48), (128, 128), (129, 272), (300, 7), (513, 1024), (64, 4096)]


@pytest.mark.parametrize("n,k", SHAPES)
@pytest.mark.parametrize("m", [1, 8, 19, 32])
def test_small_shapes(pkg, n, k, m):
    full_block_case(pkg, inputs.gaussian_bf16((n, k), 0.02, n * 31 + k), m, 0)


@pytest.mark.parametrize("n,k", [(37, 48), (300, 7), (129, 272), (5, 1)])
@pytest.mark.parametrize("m", [1, 8, 12, 20, 33])
def test_small_shapes_mx(pkg, n, k, m):
    w = inputs.heavy_tail_weight(3, shape=(n, k), frac=0.01)
    oc, oe = oracle.mx_quantize(bits(w))
    x = inputs.activations(m, k, 5)
    for path in (0, PATH_GENERIC) if k % 16 else (0, PATH_DECODE, PATH_GENERIC):
        y = pkg.mx_gemv(x.to(DEV), to_dev_bits(oc), to_dev_bits(oe), path=path)
        check_mx_gemv(y, bits(x), np.arange(n), oc, oe)


@pytest.mark.parametrize("m", [1, 8, 16, 32, 40, 130])
def test_mx_extreme_group_exponents(pkg, m):
    """MXFP8 groups whose exponent E lies outside [3, 134] (amax below
    2^-116 or above 57344) cannot carry their scale inside a bf16 weight; a
    K block holding one takes the per-group fp32 promotion instead of the
    folded decode.  Rows with tiny groups, huge groups, a single tiny group
    among normal ones, and ordinary rows, at every path."""
    g = torch.Generator().manual_seed(21)
    w = torch.randn((256, 512), generator=g) * 0.02
    w[0:16, :] *= 2.0 ** -115          # every group tiny: E = 0
    w[16:32, 128:256] *= 2.0 ** 24     # one K block of huge groups: E > 134
    w[32:48, 32:64] *= 2.0 ** -115     # one tiny group among normal ones
    w = w.to(torch.bfloat16)
    oc, oe = oracle.mx_quantize(bits(w))
    assert oe[0:16].max() < 3 and oe[16:32, 4:8].min() > 134
    x = inputs.activations(m, 512, 31 + m)
    for path in (0, PATH_DECODE, PATH_GENERIC) + ((PATH_PREFILL,) if m > 32 else ()):
        y = pkg.mx_gemv(x.to(DEV), to_dev_bits(oc), to_dev_bits(oe), path=path)
        for rows in (np.arange(0, 16), np.arange(16, 32), np.arange(32, 48), np.arange(48, 256)):
            check_mx_gemv(y[:, torch.from_numpy(rows).to(DEV)], bits(x), np.arange(len(rows)), oc[rows], oe[rows])


@pytest.mark.parametrize("scale_e", [127, 130, 100, 140])
def test_mx_prefill_every_code_exact(pkg, scale_e):
    """The MX prefill folds 2^(E-127) into the decoded bf16 weight: with one
    exponent for every group, row i holding code i at column 3 and x = e_3,
    y[:, i] = bf16(dec(i) * 2^(E-127)) exactly (one multiply for E in
    [3, 134], two above)."""
    codes_list = [c for c in range(256) if c not in (0x7F, 0xFF)]
    n, k, m = len(codes_list), 64, 40
    w = np.zeros((n, k), dtype=np.uint8)
    w[:, 3] = codes_list
    e8m0 = np.full((n, 2), scale_e, dtype=np.uint8)
    x = np.zeros((m, k), dtype=np.uint16)
    x[:, 3] = 0x3F80
    y = pkg.mx_gemv(bf16_dev(x), to_dev_bits(w), to_dev_bits(e8m0), path=PATH_PREFILL)
    want = np.array([oracle.double_to_bf16(0.0 + v * 2.0 ** (scale_e - 127)) for v in table()[codes_list]],
                    dtype=np.uint16)
    got = bits(y.cpu())
    for i in range(m):
        assert np.array_equal(got[i], want), np.argwhere(got[i] != want)[:5]


MX_PREFILL_SHAPES = [(129, 272), (256, 1024), (520, 640), (300, 16), (1, 128), (37, 48)]


@pytest.mark.parametrize("n,k", MX_PREFILL_SHAPES)
@pytest.mark.parametrize("m", [33, 128, 130, 257])
def test_mx_prefill_small_shapes(pkg, n, k, m):
    w = inputs.heavy_tail_weight(7, shape=(n, k), frac=0.01)
    oc, oe = oracle.mx_quantize(bits(w))
    x = inputs.activations(m, k, 13 + m)
    for path in (0, PATH_PREFILL):
        y = pkg.mx_gemv(x.to(DEV), to_dev_bits(oc), to_dev_bits(oe), path=path)
        check_mx_gemv(y, bits(x), np.arange(n), oc, oe)


def test_mx_prefill_full_size_sampled(pkg):
    """The MXFP8 [18432, 7168] weight (0.1% Student-t entries) at prefill
    sizes: sampled weight rows (oracle codes installed) and sampled x rows."""
    w = inputs.heavy_tail_weight(5, device=DEV)
    n, k = w.shape
    codes, e8m0 = pkg.mx_quantize(w)
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 126)]))
    oc, oe = oracle.mx_quantize(bits(w[torch.from_numpy(rows).to(DEV)].cpu()))
    ridx = torch.from_numpy(rows).to(DEV)
    codes[ridx] = to_dev_bits(oc)
    e8m0[ridx] = to_dev_bits(oe)
    for m in (64, 512, 2048):
        x = inputs.activations(m, k, 60 + m, device=DEV)
        y = pkg.mx_gemv(x, codes, e8m0)
        torch.cuda.synchronize()
        xr = np.unique(np.concatenate([[0, m - 1], rng.integers(0, m, 14)]))
        xb = bits(x[torch.from_numpy(xr).to(DEV)].cpu())
        check_mx_gemv(y[torch.from_numpy(xr).to(DEV)], xb, rows, oc, oe)


PREFILL_SHAPES = [(129, 272), (256, 1024), (64, 4096), (300, 16), (1, 128), (520, 640)]


@pytest.mark.parametrize("n,k", PREFILL_SHAPES)
@pytest.mark.parametrize("m", [33, 128, 130, 257])
def test_prefill_small_shapes(pkg, n, k, m):
    full_block_case(pkg, inputs.gaussian_bf16((n, k), 0.02, n * 17 + k), m, PATH_PREFILL, seed=m)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("kind", ["block", "mx"])
@pytest.mark.parametrize("k", [512, 1024])
def test_prefill_split_last_wave(pkg, kind, k):
    """A call whose tile count leaves a partial last wave of at most half the
    SMs: those tiles run as a second launch split over K in clusters (their
    partial sums exchanged between the CTAs), overlapping the full waves.
    n = 2048 (16 weight tiles) and m = 256 * ceil(SMs / 16) + 1 give one more
    ragged x tile than the full waves hold, so 16 tiles are split (with
    k = 512 each split CTA runs a single K block).  Every output checked."""
    n = 2048
    m = 256 * (-(-_sms() // 16)) + 1
    tiles = 16 * (-(-m // 256))
    assert 0 < tiles % _sms() <= _sms() // 2
    w = inputs.heavy_tail_weight(11, shape=(n, k), frac=0.01) if kind == "mx" else inputs.gaussian_bf16((n, k), 0.02, 5)
    x = inputs.activations(m, k, 19)
    if kind == "mx":
        oc, oe = oracle.mx_quantize(bits(w))
        y = pkg.mx_gemv(x.to(DEV), to_dev_bits(oc), to_dev_bits(oe), path=PATH_PREFILL)
        torch.cuda.synchronize()
        check_mx_gemv(y, bits(x), np.arange(n), oc, oe)
    else:
        full_block_case(pkg, w, m, PATH_PREFILL, seed=19)
    assert pkg.check_device_error() == 0


# ------------------------------------------------------ full-size, sampled
def sampled_block_case(pkg, w_dev, ms, row_blocks, seed=11, path=0, x_rows=None):
    n, k = w_dev.shape
    codes, scales = pkg.quantize(w_dev)
    w_bits = None
    rows_q = {}
    for rb in row_blocks:
        sub = bits(w_dev[rb * 128:rb * 128 + 128].cpu())
        c, s = oracle.block_quantize(sub)
        rows_q[int(rb)] = (c, s[0])
    del w_bits
    install_block_rows(codes, scales, rows_q)
    stats = []
    for m in ms:
        x = inputs.activations(m, k, seed + m, device=DEV)
        y = pkg.gemv(x, codes, scales, path=path)
        torch.cuda.synchronize()
        xr = None if x_rows is None else x_rows(m)
        stats.append(check_block_gemv(y, bits(x.cpu()), rows_q, m_rows=xr))
    return stats


def _row_blocks(n, count, seed):
    nb = -(-n // 128)
    rng = np.random.default_rng(seed)
    return sorted(set([0, nb - 1] + list(rng.integers(0, nb, count))))


def test_lm_head_full_size(pkg):
    w = inputs.lm_head_weight(2, device=DEV)
    sampled_block_case(pkg, w, [1, 4, 8, 16, 24, 32], _row_blocks(w.shape[0], 4, 1))


@pytest.mark.parametrize("j", range(4))
def test_rotation_shapes(pkg, j):
    w = inputs.rotation_weight(0, j, device=DEV)
    sampled_block_case(pkg, w, [1, 8, 16, 32], _row_blocks(w.shape[0], 3, j))


@pytest.mark.parametrize("n,ms", [(2560, [12, 17, 24, 32]), (3072, [17, 24, 32]), (5120, [17, 32])])
def test_split_cluster_sizes(pkg, n, ms):
    """Weights of 20 / 40 / 48 / 80 row tiles: the split-K cluster size is the
    largest whose clusters all fit in one wave (not capacity / tiles, which
    gives 6 or 7 here); every split count must give the same sums."""
    w = inputs.gaussian_bf16((n, 2560), 0.02, n + 11, device=DEV)
    sampled_block_case(pkg, w, ms, _row_blocks(n, 3, n))


def test_sweep_shape_all_m(pkg):
    w = inputs.sweep_weight(0, device=DEV)
    sampled_block_case(pkg, w, list(range(1, 33)), _row_blocks(w.shape[0], 2, 5))


def test_prefill_shapes_sampled(pkg):
    w = inputs.sweep_weight(0, device=DEV)
    rng = np.random.default_rng(9)
    sampled_block_case(pkg, w, [64, 512, 2048, 4096], _row_blocks(w.shape[0], 1, 6),
                       x_rows=lambda m: np.unique(np.concatenate([[0, m - 1], rng.integers(0, m, 14)])))


def test_prefill_large_weight_tile_order(pkg):
    """A weight whose codes exceed 64 MiB runs the prefill with the x tiles
    fastest on the grid (the smaller weights above run weight tiles
    fastest): block scales must still be read from the right tile row."""
    w = inputs.gaussian_bf16((16512, 4096), 0.02, 404, device=DEV)
    assert w.shape[0] * w.shape[1] > 64 << 20
    rng = np.random.default_rng(12)
    sampled_block_case(pkg, w, [64, 257, 600], _row_blocks(w.shape[0], 3, 12),
                       x_rows=lambda m: np.unique(np.concatenate([[0, m - 1], rng.integers(0, m, 14)])))


def test_mx_full_size(pkg):
    w = inputs.heavy_tail_weight(5, device=DEV)
    n, k = w.shape
    codes, e8m0 = pkg.mx_quantize(w)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 254)]))
    oc, oe = oracle.mx_quantize(bits(w[torch.from_numpy(rows).to(DEV)].cpu()))
    ridx = torch.from_numpy(rows).to(DEV)
    codes[ridx] = to_dev_bits(oc)
    e8m0[ridx] = to_dev_bits(oe)
    for m in (1, 8, 16, 24, 32):
        x = inputs.activations(m, k, 40 + m, device=DEV)
        y = pkg.mx_gemv(x, codes, e8m0)
        torch.cuda.synchronize()
        check_mx_gemv(y, bits(x.cpu()), rows, oc, oe)


@pytest.mark.parametrize("m", [1, 4, 8, 16])
@pytest.mark.parametrize("case", ["wide_range", "tiny", "huge", "single_spike"])
def test_x_dynamic_range(pkg, m, case):
    """Activations with extreme ranges inside one 32-column slice: the f16
    operand path rescales each slice by a power of two (exact for values
    within 2^-31 of the slice maximum), so results stay within tolerance."""
    w = inputs.gaussian_bf16((384, 1024), 0.02, 77)
    oc, os_ = oracle.block_quantize(bits(w))
    g = torch.Generator().manual_seed(5)
    base = torch.randn((m, 1024), generator=g)
    if case == "wide_range":
        expo = torch.randint(-30, 30, (m, 1024), generator=g).to(torch.float32)
        x = base * torch.pow(10.0, expo)
    elif case == "tiny":
        x = base * 1e-35
    elif case == "huge":
        x = base * 1e30
    else:
        x = base.clone()
        x[:, 37] = 3e20
    x = x.to(torch.bfloat16)
    for path in (0, PATH_GENERIC):
        y = pkg.gemv(x.to(DEV), to_dev_bits(oc), torch.from_numpy(os_).to(DEV), path=path)
        rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(3)}
        check_block_gemv(y, bits(x), rows_q)


# ----------------------------------- prepared x (fp8bs_gemv_ws, workspace)
def ws_for(pkg, m, k, fill=0xFF):
    """A workspace of the size gemv_ws needs, filled with NaN bytes: its
    contents on entry must not matter."""
    return torch.full((pkg.gemv_ws_bytes(m, k),), fill, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("m", [1, 2, 5, 8, 9, 13, 16, 17, 24, 31, 32])
def test_ws_tiny_ragged(pkg, m):
    w = inputs.tiny_ragged_weight(0)
    n, k = w.shape
    oc, os_ = oracle.block_quantize(bits(w))
    x = inputs.activations(m, k, 70 + m)
    y, raw = guarded_empty((m, n), torch.bfloat16, DEV)
    pkg.gemv_ws(x.to(DEV), to_dev_bits(oc), torch.from_numpy(os_).to(DEV), ws_for(pkg, m, k), y=y)
    torch.cuda.synchronize()
    assert guard_intact(raw, m * n * 2)
    rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(-(-n // 128))}
    check_block_gemv(y, bits(x), rows_q)


@pytest.mark.parametrize("n,k", [(37, 48), (129, 272), (513, 1024), (64, 4096), (300, 16)])
@pytest.mark.parametrize("m", [1, 8, 19, 32])
def test_ws_small_shapes(pkg, n, k, m):
    w = inputs.gaussian_bf16((n, k), 0.02, n * 31 + k)
    oc, os_ = oracle.block_quantize(bits(w))
    x = inputs.activations(m, k, 7)
    y = pkg.gemv_ws(x.to(DEV), to_dev_bits(oc), torch.from_numpy(os_).to(DEV), ws_for(pkg, m, k))
    rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(-(-n // 128))}
    check_block_gemv(y, bits(x), rows_q)


def test_ws_sweep_shape_all_m(pkg):
    w = inputs.sweep_weight(0, device=DEV)
    n, k = w.shape
    codes, scales = pkg.quantize(w)
    rows_q = {}
    for rb in _row_blocks(n, 2, 5):
        c, s = oracle.block_quantize(bits(w[rb * 128:rb * 128 + 128].cpu()))
        rows_q[int(rb)] = (c, s[0])
    install_block_rows(codes, scales, rows_q)
    ws = ws_for(pkg, 32, k)
    for m in range(1, 33):
        x = inputs.activations(m, k, 11 + m, device=DEV)
        y = pkg.gemv_ws(x, codes, scales, ws)   # one workspace reused by every call
        torch.cuda.synchronize()
        check_block_gemv(y, bits(x.cpu()), rows_q)


@pytest.mark.parametrize("m", [4, 16, 32])
@pytest.mark.parametrize("case", ["wide_range", "tiny", "huge", "single_spike"])
def test_ws_x_dynamic_range(pkg, m, case):
    """The prepared f16 copy of x takes one power of two per (row, K block):
    activations spanning 60 decades, all tiny, all huge, or one spike per
    row stay within tolerance."""
    w = inputs.gaussian_bf16((384, 1024), 0.02, 77)
    oc, os_ = oracle.block_quantize(bits(w))
    g = torch.Generator().manual_seed(5)
    base = torch.randn((m, 1024), generator=g)
    if case == "wide_range":
        x = base * torch.pow(10.0, torch.randint(-30, 30, (m, 1024), generator=g).to(torch.float32))
    elif case == "tiny":
        x = base * 1e-35
    elif case == "huge":
        x = base * 1e30
    else:
        x = base.clone()
        x[:, 37] = 3e20
    x = x.to(torch.bfloat16)
    y = pkg.gemv_ws(x.to(DEV), to_dev_bits(oc), torch.from_numpy(os_).to(DEV), ws_for(pkg, m, 1024))
    rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(3)}
    check_block_gemv(y, bits(x), rows_q)


def test_ws_every_code_exact_and_prefill_ignores_it(pkg):
    codes_list = [c for c in range(256) if c not in (0x7F, 0xFF)]
    n, k = len(codes_list), 32
    w = np.zeros((n, k), dtype=np.uint8)
    w[:, 3] = codes_list
    scales = np.ones((-(-n // 128), 1), dtype=np.float32)
    want = np.array([oracle.double_to_bf16(0.0 + v) for v in table()[codes_list]], dtype=np.uint16)
    for m in (1, 9, 32, 40):   # 40: the prefill path, which needs no workspace
        x = np.zeros((m, k), dtype=np.uint16)
        x[:, 3] = 0x3F80
        y = pkg.gemv_ws(bf16_dev(x), to_dev_bits(w), torch.from_numpy(scales).to(DEV), ws_for(pkg, m, k))
        got = bits(y.cpu())
        for i in range(m):
            assert np.array_equal(got[i], want)


def test_repeat_is_deterministic(pkg):
    w = inputs.rotation_weight(1, 1, device=DEV)
    codes, scales = pkg.quantize(w)
    x = inputs.activations(16, w.shape[1], 3, device=DEV)
    y1 = pkg.gemv(x, codes, scales)
    y2 = pkg.gemv(x, codes, scales)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_no_device_error(pkg):
    assert pkg.check_device_error() == 0
