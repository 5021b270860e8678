"""GPU parity for per-row and per-tensor FP8 (one fp32 scale per output row,
or one per weight; FreeToken PR #389): quantizers bit-exact against the
oracle, the GEMV on every path within the tolerance of oracle/tolerance.py,
with exact checks where the result is fixed exactly (every code through a
one-hot x, one-hot columns, x = 0).

Every GEMV input on a checked output comes from the seeded generators and
the oracle's own quantizer, never from the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import PATH_DECODE, PATH_GENERIC, PATH_PREFILL, inputs
from oracle import tolerance

from gpu_helpers import bits, guard_intact, guarded_empty, lib_or_skip, table

pytestmark = pytest.mark.gpu
DEV = "cuda"
PATHS = [PATH_DECODE, PATH_GENERIC, PATH_PREFILL]
MODES = ["row", "tensor"]


@pytest.fixture(scope="module")
def pkg():
    return lib_or_skip()


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def bf16_dev(a_bits):
    return torch.from_numpy(np.ascontiguousarray(a_bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def oracle_quant(mode, w_bits, rows=None):
    return (oracle.row_quantize if mode == "row" else oracle.tensor_quantize)(w_bits, rows=rows)


def gpu_quant(pkg, mode, w_dev, offset=0):
    n, k = w_dev.shape
    if offset:
        buf = torch.empty(n * k + offset, dtype=torch.bfloat16, device=DEV)
        src = buf[offset:].view(n, k)
        src.copy_(w_dev)
        w_dev = src
    codes, craw = guarded_empty((n, k), torch.uint8, DEV)
    ns = n if mode == "row" else 1
    scales, sraw = guarded_empty((ns,), torch.float32, DEV)
    if mode == "row":
        pkg.row_quantize(w_dev, codes=codes, scales=scales)
    else:
        pkg.tensor_quantize(w_dev, codes=codes, scale=scales)
    torch.cuda.synchronize()
    assert guard_intact(craw, n * k) and guard_intact(sraw, ns * 4)
    return codes, scales


def assert_quant_equal(pkg, mode, w_cpu, offset=0):
    c, s = gpu_quant(pkg, mode, w_cpu.to(DEV), offset)
    oc, os_ = oracle_quant(mode, bits(w_cpu))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    cg = c.cpu().numpy()
    bad = np.argwhere(cg != oc)
    assert bad.size == 0, (bad[:5], cg[tuple(bad[0])], oc[tuple(bad[0])])


def wmax_rows(codes, scales):
    s = np.broadcast_to(np.asarray(scales, dtype=np.float64).ravel(), (codes.shape[0],))
    return np.abs(table()[codes]).max(axis=1) * s


def check_gemv(y_dev, x_bits, codes, scales, rows=None):
    """y_dev[:, rows] against the oracle's fp64 GEMV over those rows; codes
    and scales are the full arrays the GEMV read."""
    y64 = oracle.row_gemv(x_bits, codes, scales, rows=rows)
    if rows is None:
        y = bits(y_dev.cpu())
        cr = codes
        sr = scales
    else:
        y = bits(y_dev[:, torch.as_tensor(rows, device=y_dev.device)].cpu())
        cr = codes[rows]
        sr = scales[rows] if scales.shape[0] > 1 else scales
    st = tolerance.gemv_errors(y, y64, x_bits, wmax_rows(cr, sr))
    assert tolerance.gemv_ok(st), st
    return st


# --------------------------------------------------------------- quantize
SHAPES = [(1, 1), (1, 8), (7, 5), (3, 40), (129, 257), (300, 33), (256, 1024), (64, 7168), (2, 20000)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n,k", SHAPES)
def test_quantize_shapes(pkg, mode, n, k):
    assert_quant_equal(pkg, mode, inputs.gaussian_bf16((n, k), 0.02, 200 + n + k))


@pytest.mark.parametrize("mode", MODES)
def test_quantize_heavy_tail_and_outliers(pkg, mode):
    assert_quant_equal(pkg, mode, inputs.tiny_ragged_weight(0))
    assert_quant_equal(pkg, mode, inputs.heavy_tail_weight(7, shape=(300, 704), frac=0.01))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("offset", [1, 4])
def test_unaligned_source_takes_scalar_kernel(pkg, mode, offset):
    assert_quant_equal(pkg, mode, inputs.gaussian_bf16((130, 264), 0.02, 56), offset=offset)


def special_weight():
    """Zero row (with -0), subnormal row, a 448 row, the largest bf16 value,
    values on rounding midpoints when divided."""
    w = bits(inputs.gaussian_bf16((64, 512), 0.02, 9)).copy()
    w[3] = 0
    w[3, 7] = 0x8000
    w[4] = 0x0001
    w[4, 9] = 0x8005
    w[5] = 0x3F80
    w[5, 100] = 0x43E0
    w[6] = 0x7F7F
    w[6, 1] = 0xFF7F
    w[7] = 0x4040
    return torch.from_numpy(w.view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("mode", MODES)
def test_quantize_special_values(pkg, mode):
    assert_quant_equal(pkg, mode, special_weight())


def test_zero_tensor(pkg):
    c, s = gpu_quant(pkg, "tensor", torch.zeros((33, 96), dtype=torch.bfloat16, device=DEV))
    assert s.item() == 1.0 and int(c.sum()) == 0


def test_quantize_full_size_sampled(pkg):
    """lm_head [152064, 4096] per row (sampled rows) and the [18432, 7168]
    heavy-tail weight per tensor (amax over all of it, sampled rows)."""
    w = inputs.lm_head_weight(2, device=DEV)
    codes, scales = pkg.row_quantize(w)
    torch.cuda.synchronize()
    n = w.shape[0]
    rng = np.random.default_rng(4)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 126)]))
    ridx = torch.from_numpy(rows).to(DEV)
    oc, os_ = oracle.row_quantize(bits(w[ridx].cpu()))
    assert np.array_equal(codes[ridx].cpu().numpy(), oc)
    assert np.array_equal(scales[ridx].cpu().numpy().view(np.uint32), os_.view(np.uint32))
    # every row's amax element encodes to +-448, no NaN code anywhere
    assert int(((codes & 0x7F).amax(dim=1) != 0x7E).sum()) == 0
    assert int(((codes & 0x7F) == 0x7F).sum()) == 0
    del codes, scales, w

    w = inputs.heavy_tail_weight(5, device=DEV)
    codes, scale = pkg.tensor_quantize(w)
    torch.cuda.synchronize()
    n = w.shape[0]
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 30)]))
    oc, os_ = oracle.tensor_quantize(bits(w.cpu()), rows=rows)
    assert scale.cpu().numpy().view(np.uint32)[0] == os_.view(np.uint32)[0]
    assert np.array_equal(codes[torch.from_numpy(rows).to(DEV)].cpu().numpy(), oc)


# ------------------------------------------------------------------- GEMV
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("m", [1, 8, 9, 32, 40, 130])
def test_every_code_decodes_exactly(pkg, mode, path, m):
    """Row i holds code i at column 3 and x = e_3; with scale 1 (per row or
    per tensor) y[:, i] = bf16(dec(i)) exactly."""
    codes_list = [c for c in range(256) if c not in (0x7F, 0xFF)]
    n, k = len(codes_list), 32
    w = np.zeros((n, k), dtype=np.uint8)
    w[:, 3] = codes_list
    scales = np.ones(n if mode == "row" else 1, dtype=np.float32)
    x = np.zeros((m, k), dtype=np.uint16)
    x[:, 3] = 0x3F80
    y = bits(pkg.row_gemv(bf16_dev(x), dev_u8(w), dev_f32(scales), path=path).cpu())
    want = np.array([oracle.double_to_bf16(0.0 + v) for v in table()[codes_list]], dtype=np.uint16)
    for i in range(m):
        assert np.array_equal(y[i], want), np.argwhere(y[i] != want)[:5]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("path", PATHS)
def test_one_hot_columns(pkg, mode, path):
    """x = e_c gives y[n] = bf16(fl32(dec(q[n, c]) * s_n)) exactly: the fp32
    sum is the decoded code, multiplied once by the row's scale."""
    w = inputs.tiny_ragged_weight(0)
    n, k = w.shape
    oc, os_ = oracle_quant(mode, bits(w))
    cols = [0, 1, 127, 128, 300, 640, 703]
    x = np.zeros((len(cols), k), dtype=np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = 0x3F80
    y = bits(pkg.row_gemv(bf16_dev(x), dev_u8(oc), dev_f32(os_), path=path).cpu())
    s = np.broadcast_to(os_, (n,)).astype(np.float32)
    for i, c in enumerate(cols):
        prod = (table()[oc[:, c]].astype(np.float32) * s).astype(np.float32)
        want = np.array([oracle.double_to_bf16(0.0 + float(v)) for v in prod], dtype=np.uint16)
        assert np.array_equal(y[i], want), (c, np.argwhere(y[i] != want)[:5])


@pytest.mark.parametrize("mode", MODES)
def test_zero_input_gives_zero(pkg, mode):
    oc, os_ = oracle_quant(mode, bits(inputs.gaussian_bf16((256, 512), 0.02, 3)))
    for path in PATHS:
        y = pkg.row_gemv(torch.zeros((4, 512), dtype=torch.bfloat16, device=DEV), dev_u8(oc), dev_f32(os_),
                         path=path)
        assert int((y.view(torch.int16) & 0x7FFF).abs().sum()) == 0


def small_case(pkg, mode, w, m, path, seed=7):
    n, k = w.shape
    oc, os_ = oracle_quant(mode, bits(w))
    x = inputs.activations(m, k, seed)
    y, raw = guarded_empty((m, n), torch.bfloat16, DEV)
    pkg.row_gemv(x.to(DEV), dev_u8(oc), dev_f32(os_), y=y, path=path)
    torch.cuda.synchronize()
    assert guard_intact(raw, m * n * 2)
    return check_gemv(y, bits(x), oc, os_)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("m", [1, 4, 8, 9, 16, 17, 32, 33, 64, 130])
def test_tiny_ragged_all_m(pkg, mode, path, m):
    small_case(pkg, mode, inputs.tiny_ragged_weight(0), m, path)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n,k", [(1, 16), (5, 300), (37, 48), (129, 272), (300, 7), (513, 1024), (64, 4096)])
@pytest.mark.parametrize("m", [1, 8, 19, 32, 100])
def test_small_shapes(pkg, mode, n, k, m):
    small_case(pkg, mode, inputs.gaussian_bf16((n, k), 0.02, n * 13 + k), m, 0)


# ------------------------------------------------------ full-size, sampled
def sampled_case(pkg, mode, w_dev, ms, nrows, seed, x_rows=None):
    n, k = w_dev.shape
    codes, scales = (pkg.row_quantize if mode == "row" else pkg.tensor_quantize)(w_dev)
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, nrows)]))
    ridx = torch.from_numpy(rows).to(DEV)
    if mode == "row":
        oc, os_ = oracle.row_quantize(bits(w_dev[ridx].cpu()))
        scales[ridx] = dev_f32(os_)
        full_s = None
    else:
        oc, os_ = oracle.tensor_quantize(bits(w_dev.cpu()), rows=rows)
        scales.copy_(dev_f32(os_))
        full_s = os_
    codes[ridx] = dev_u8(oc)
    for m in ms:
        x = inputs.activations(m, k, seed + m, device=DEV)
        y = pkg.row_gemv(x, codes, scales)
        torch.cuda.synchronize()
        xb = bits(x.cpu())
        mr = x_rows(m) if x_rows else np.arange(m)
        y64 = oracle.row_gemv(xb[mr], oc, os_ if full_s is None else full_s)
        yg = bits(y[torch.as_tensor(mr, device=DEV)][:, ridx].cpu())
        st = tolerance.gemv_errors(yg, y64, xb[mr], wmax_rows(oc, os_))
        assert tolerance.gemv_ok(st), (m, st)


@pytest.mark.parametrize("mode", MODES)
def test_lm_head_full_size(pkg, mode):
    sampled_case(pkg, mode, inputs.lm_head_weight(2, device=DEV), [1, 4, 8, 16], 200, 1)


@pytest.mark.parametrize("j", range(4))
def test_rotation_shapes_per_row(pkg, j):
    sampled_case(pkg, "row", inputs.rotation_weight(0, j, device=DEV), [1, 8, 16, 32], 100, j)


def test_prefill_shapes_sampled(pkg):
    rng = np.random.default_rng(9)
    sampled_case(pkg, "row", inputs.sweep_weight(0, device=DEV), [64, 512, 2048, 4096], 100, 6,
                 x_rows=lambda m: np.unique(np.concatenate([[0, m - 1], rng.integers(0, m, 14)])))


def test_repeat_is_deterministic(pkg):
    w = inputs.rotation_weight(1, 1, device=DEV)
    codes, scales = pkg.row_quantize(w)
    for m in (16, 200):
        x = inputs.activations(m, w.shape[1], 3, device=DEV)
        y1 = pkg.row_gemv(x, codes, scales)
        y2 = pkg.row_gemv(x, codes, scales)
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_no_device_error(pkg):
    assert pkg.check_device_error() == 0
