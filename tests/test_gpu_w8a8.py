"""GPU parity for the W8A8 route (FreeToken PR #389): dynamic per-tensor
activation quantization bit-exact against the oracle, and the e4m3 x e4m3
GEMM on every path within the tolerance of oracle/tolerance.py against the
oracle's fp64 W8A8 result, with exact checks where the result is fixed
exactly (every weight code through a one-hot x, power-of-two scales).

The GEMM's inputs (both code tensors and both scales) on every checked
output come from the seeded generators and the oracle's own quantizers.
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


@pytest.fixture(scope="module")
def pkg():
    return lib_or_skip()


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(DEV) if dtype is None else t.to(dtype).to(DEV)


def f32dev(v):
    return torch.tensor(np.asarray(v, dtype=np.float32).ravel()[:1], device=DEV)


def deq_bits(codes, scale):
    """bf16 bits of dec(codes) * scale (for the tolerance's ||x||)."""
    v = torch.from_numpy(table()[codes] * float(np.ravel(scale)[0])).to(torch.bfloat16)
    return bits(v)


def check(y_dev, xq, sx, wq, sw, rows=None, x_rows=None):
    xr = np.arange(xq.shape[0]) if x_rows is None else x_rows
    y64 = oracle.w8a8_gemv(xq[xr], sx, wq, sw, rows=rows)
    yg = y_dev[torch.as_tensor(xr, device=y_dev.device)]
    if rows is not None:
        yg = yg[:, torch.as_tensor(rows, device=y_dev.device)]
    wsel = wq if rows is None else wq[rows]
    wmax = np.abs(table()[wsel]).max(axis=1) * float(np.ravel(sw)[0])
    st = tolerance.gemv_errors(bits(yg.cpu()), y64, deq_bits(xq[xr], sx), wmax)
    assert tolerance.gemv_ok(st), st
    return st


# ----------------------------------------------------- activation quantize
@pytest.mark.parametrize("m,k", [(1, 1), (1, 8), (1, 4096), (8, 4096), (16, 7168), (64, 1024), (65, 1024),
                                 (300, 33), (512, 4096)])
def test_act_quantize_bit_exact(pkg, m, k):
    x = inputs.activations(m, k, 10 + m + k)
    codes, craw = guarded_empty((m, k), torch.uint8, DEV)
    scale, sraw = guarded_empty((1,), torch.float32, DEV)
    pkg.act_quantize(x.to(DEV), codes=codes, scale=scale)
    torch.cuda.synchronize()
    assert guard_intact(craw, m * k) and guard_intact(sraw, 4)
    oc, os_ = oracle.act_quantize(bits(x))
    assert scale.cpu().numpy().view(np.uint32)[0] == os_.view(np.uint32)[0]
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("offset", [1, 4])
def test_act_quantize_unaligned(pkg, offset):
    x = inputs.activations(8, 264, 3)
    buf = torch.empty(8 * 264 + offset, dtype=torch.bfloat16, device=DEV)
    xs = buf[offset:].view(8, 264)
    xs.copy_(x)
    codes, scale = pkg.act_quantize(xs)
    oc, os_ = oracle.act_quantize(bits(x))
    assert scale.item() == float(os_[0]) and np.array_equal(codes.cpu().numpy(), oc)


def test_act_quantize_zero_and_extremes(pkg):
    codes, scale = pkg.act_quantize(torch.zeros((4, 100), dtype=torch.bfloat16, device=DEV))
    assert scale.item() == 1.0 and int(codes.sum()) == 0
    x = inputs.activations(4, 100, 5)
    x[1, 7] = 3e30
    x[2, 9] = -1e-30
    codes, scale = pkg.act_quantize(x.to(DEV))
    oc, os_ = oracle.act_quantize(bits(x))
    assert scale.item() == float(os_[0]) and np.array_equal(codes.cpu().numpy(), oc)


# ------------------------------------------------------------- exact GEMM
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("m", [1, 8, 9, 32, 40, 300])
def test_every_code_exact(pkg, path, m):
    """Weight row i holds code i at column 3, x codes hold 1.0 (0x38) at
    column 3, sx = 2^-3, sw = 2^-5: y[:, i] = bf16(dec(i) / 256) exactly."""
    codes_list = [c for c in range(256) if c not in (0x7F, 0xFF)]
    n, k = len(codes_list), 32
    w = np.zeros((n, k), dtype=np.uint8)
    w[:, 3] = codes_list
    xq = np.zeros((m, k), dtype=np.uint8)
    xq[:, 3] = 0x38
    y = pkg.w8a8_gemm(dev(xq), f32dev(2.0 ** -3), dev(w), f32dev(2.0 ** -5), path=path)
    got = bits(y.cpu())
    want = np.array([oracle.double_to_bf16(0.0 + v / 256.0) for v in table()[codes_list]], dtype=np.uint16)
    for i in range(m):
        assert np.array_equal(got[i], want), np.argwhere(got[i] != want)[:5]


@pytest.mark.parametrize("path", PATHS)
def test_zero_x(pkg, path):
    wq, sw = oracle.tensor_quantize(bits(inputs.gaussian_bf16((256, 512), 0.02, 3)))
    y = pkg.w8a8_gemm(torch.zeros((40, 512), dtype=torch.uint8, device=DEV), f32dev(1.0), dev(wq), dev(sw), path=path)
    assert int((y.view(torch.int16) & 0x7FFF).abs().sum()) == 0


# ------------------------------------------------------------ tolerance
def small_case(pkg, w, m, path, seed=7):
    n, k = w.shape
    wq, sw = oracle.tensor_quantize(bits(w))
    xq, sx = oracle.act_quantize(bits(inputs.activations(m, k, seed)))
    y, raw = guarded_empty((m, n), torch.bfloat16, DEV)
    pkg.w8a8_gemm(dev(xq), dev(sx), dev(wq), dev(sw), y=y, path=path)
    torch.cuda.synchronize()
    assert guard_intact(raw, m * n * 2)
    return check(y, xq, sx, wq, sw)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("m", [1, 4, 8, 9, 16, 17, 32, 33, 64, 130, 257])
def test_tiny_ragged_all_m(pkg, path, m):
    small_case(pkg, inputs.tiny_ragged_weight(0), m, path)


@pytest.mark.parametrize("n,k", [(1, 16), (5, 300), (37, 48), (129, 272), (300, 7), (513, 1024), (64, 4096)])
@pytest.mark.parametrize("m", [1, 8, 19, 32, 100])
def test_small_shapes(pkg, n, k, m):
    small_case(pkg, inputs.gaussian_bf16((n, k), 0.02, n * 11 + k), m, 0)


def test_linear_matches_two_calls(pkg):
    w = inputs.gaussian_bf16((300, 512), 0.02, 12)
    wq, sw = pkg.tensor_quantize(w.to(DEV))
    x = inputs.activations(8, 512, 13, device=DEV)
    y1 = pkg.w8a8_linear(x, wq, sw)
    xq, sx = pkg.act_quantize(x)
    y2 = pkg.w8a8_gemm(xq, sx, wq, sw)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


# ------------------------------------------------------ full-size, sampled
def sampled_case(pkg, w_dev, ms, nrows, seed, x_rows=None):
    n, k = w_dev.shape
    wq, sw = pkg.tensor_quantize(w_dev)
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, nrows)]))
    owq, osw = oracle.tensor_quantize(bits(w_dev.cpu()), rows=rows)
    wq[torch.from_numpy(rows).to(DEV)] = dev(owq)
    sw.copy_(dev(osw))
    for m in ms:
        x = inputs.activations(m, k, seed + m)
        xq, sx = oracle.act_quantize(bits(x))
        y = pkg.w8a8_gemm(dev(xq), dev(sx), wq, sw)
        torch.cuda.synchronize()
        xr = x_rows(m) if x_rows else None
        y64 = oracle.w8a8_gemv(xq if xr is None else xq[xr], sx, owq, osw)
        yg = y if xr is None else y[torch.as_tensor(xr, device=DEV)]
        yg = bits(yg[:, torch.from_numpy(rows).to(DEV)].cpu())
        wmax = np.abs(table()[owq]).max(axis=1) * float(osw[0])
        st = tolerance.gemv_errors(yg, y64, deq_bits(xq if xr is None else xq[xr], sx), wmax)
        assert tolerance.gemv_ok(st), (m, st)


def test_lm_head_full_size(pkg):
    sampled_case(pkg, inputs.lm_head_weight(2, device=DEV), [1, 8, 16], 200, 1)


def test_prefill_shapes_sampled(pkg):
    rng = np.random.default_rng(9)
    sampled_case(pkg, inputs.sweep_weight(0, device=DEV), [64, 512, 2048, 4096], 100, 6,
                 x_rows=lambda m: np.unique(np.concatenate([[0, m - 1], rng.integers(0, m, 14)])))


def test_prefill_more_tiles_than_ctas(pkg):
    """180 output tiles of 128 weight rows x 256 x rows for at most 152
    persistent CTAs: CTAs take a second tile into the other accumulator;
    every output is checked."""
    n, k, m = 20 * 128, 256, 9 * 256
    w = inputs.gaussian_bf16((n, k), 0.02, 31)
    owq, osw = oracle.tensor_quantize(bits(w))
    x = inputs.activations(m, k, 32)
    xq, sx = oracle.act_quantize(bits(x))
    y = pkg.w8a8_gemm(dev(xq), dev(sx), dev(owq), dev(osw), path=PATH_PREFILL)
    torch.cuda.synchronize()
    check(y, xq, sx, owq, osw)


def test_repeat_is_deterministic(pkg):
    w = inputs.rotation_weight(1, 1, device=DEV)
    wq, sw = pkg.tensor_quantize(w)
    for m in (16, 300):
        x = inputs.activations(m, w.shape[1], 3, device=DEV)
        y1 = pkg.w8a8_linear(x, wq, sw)
        y2 = pkg.w8a8_linear(x, wq, sw)
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_no_device_error(pkg):
    assert pkg.check_device_error() == 0
