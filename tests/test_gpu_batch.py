"""GPU parity: the batched GEMV (fp8bs_gemv_batch / mxfp8_gemv_batch).

A batch must give, op by op, what fp8bs_gemv gives for that op in the
batch's order: every output is held to the oracle's fp64 result under the
GEMV tolerance, on inputs that come from the seeded generators and the
oracle's own quantizer.  The ordering cases build their intermediate values
from the oracle alone: a one-hot x makes the first GEMV's output exact
(bf16(fl32(dec(q) * s))), so the second GEMV's expected result is the
oracle's on those exact values, and a premature read of the first output
(pre-filled with NaN) cannot pass.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import PATH_DECODE, PATH_GENERIC, inputs

from gpu_helpers import (bits, check_block_gemv, check_mx_gemv, guard_intact, guarded_empty, install_block_rows,
                         lib_or_skip, table)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    return lib_or_skip()


def bf16_dev(a_bits: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a_bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def _row_blocks(n, count, seed):
    nb = -(-n // 128)
    rng = np.random.default_rng(seed)
    return sorted(set([0, nb - 1] + list(rng.integers(0, nb, count))))


@pytest.fixture(scope="module")
def rotation_layers(pkg):
    """Two layers of the decode rotation (8 projection weights, 312 row
    tiles): quantized on the GPU, with sampled 128-row blocks overwritten by
    the oracle's codes and scales (the checked rows)."""
    out = []
    for layer in range(2):
        for j in range(4):
            w = inputs.rotation_weight(layer, j, device=DEV)
            codes, scales = pkg.quantize(w)
            rows_q = {}
            for rb in _row_blocks(w.shape[0], 2, 10 * layer + j):
                c, s = oracle.block_quantize(bits(w[rb * 128:rb * 128 + 128].cpu()))
                rows_q[int(rb)] = (c, s[0])
            install_block_rows(codes, scales, rows_q)
            out.append((codes, scales, rows_q))
            del w
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("path", [0, PATH_DECODE])
@pytest.mark.parametrize("m", [1, 3, 8, 9, 16, 17, 24, 32])
def test_rotation_layers(pkg, rotation_layers, m, path):
    ops, xs = [], []
    for i, (codes, scales, _) in enumerate(rotation_layers):
        x = inputs.activations(m, codes.shape[1], 60 + 7 * i + m, device=DEV)
        xs.append(x)
        ops.append((x, codes, scales))
    ys = pkg.gemv_batch(ops, path=path)
    torch.cuda.synchronize()
    for x, y, (_, _, rows_q) in zip(xs, ys, rotation_layers):
        check_block_gemv(y, bits(x.cpu()), rows_q)


RAGGED = [(320, 704), (129, 272), (37, 48), (1, 16), (513, 1024), (300, 16), (128, 128), (255, 4096)]


@pytest.mark.parametrize("m", [1, 5, 8, 13, 24, 32])
def test_ragged_shapes_in_one_launch(pkg, m):
    """Ragged row and K tiles of several weights in one batched launch
    (forced), every output checked in full, y guarded against overruns."""
    ops, cases = [], []
    for i, (n, k) in enumerate(RAGGED):
        w = inputs.tiny_ragged_weight(0) if (n, k) == (320, 704) else inputs.gaussian_bf16((n, k), 0.02, 31 * n + k)
        oc, os_ = oracle.block_quantize(bits(w))
        x = inputs.activations(m, k, 90 + i)
        y, raw = guarded_empty((m, n), torch.bfloat16, DEV)
        ops.append((x.to(DEV), torch.from_numpy(oc).to(DEV), torch.from_numpy(os_).to(DEV), y))
        cases.append((x, y, raw, oc, os_))
    pkg.gemv_batch(ops, path=PATH_DECODE)
    torch.cuda.synchronize()
    for x, y, raw, oc, os_ in cases:
        n = oc.shape[0]
        assert guard_intact(raw, y.numel() * 2)
        rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(-(-n // 128))}
        check_block_gemv(y, bits(x), rows_q)


def test_more_ops_than_one_launch_holds(pkg):
    """230 small weights (more than the 96-op table of one launch): the
    batch is split over several launches and every op is still computed."""
    rng = np.random.default_rng(4)
    ops, cases = [], []
    for i in range(230):
        n = int(rng.integers(1, 300))
        k = 16 * int(rng.integers(1, 40))
        w = inputs.gaussian_bf16((n, k), 0.02, 1000 + i)
        oc, os_ = oracle.block_quantize(bits(w))
        x = inputs.activations(4, k, 2000 + i)
        ops.append((x.to(DEV), torch.from_numpy(oc).to(DEV), torch.from_numpy(os_).to(DEV)))
        cases.append((x, oc, os_))
    ys = pkg.gemv_batch(ops, path=PATH_DECODE)
    torch.cuda.synchronize()
    for (x, oc, os_), y in zip(cases, ys):
        n = oc.shape[0]
        rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(-(-n // 128))}
        check_block_gemv(y, bits(x), rows_q)


def one_hot_case(n, k, m, seed):
    """A weight quantized by the oracle and an x of m one-hot rows (distinct
    columns); returns the exact bf16 bits of x . dequant(W)^T."""
    w = inputs.gaussian_bf16((n, k), 0.02, seed)
    oc, os_ = oracle.block_quantize(bits(w))
    cols = np.random.default_rng(seed).choice(k, size=m, replace=False)
    x = np.zeros((m, k), dtype=np.uint16)
    y = np.zeros((m, n), dtype=np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = 0x3F80
        prod = (table()[oc[:, c]].astype(np.float32) * os_[np.arange(n) // 128, c // 128]).astype(np.float32)
        y[i] = [oracle.double_to_bf16(0.0 + float(v)) for v in prod]
    return x, oc, os_, y


@pytest.mark.parametrize("path", [0, PATH_DECODE])
@pytest.mark.parametrize("m", [1, 8, 16, 32])
def test_chained_output_feeds_next_input(pkg, m, path):
    """op 1 reads op 0's output as its x, op 2 overwrites op 0's x, op 3
    writes the same output as op 2 (read-after-write, write-after-read and
    write-after-write in one batch): each op sees the state the sequence of
    single calls would leave."""
    xa, qa, sa, ya = one_hot_case(384, 256, m, 5)            # exact y of op 0
    wb = inputs.gaussian_bf16((256, 384), 0.02, 6)
    qb, sb = oracle.block_quantize(bits(wb))
    xc_next, qc, sc, yc = one_hot_case(256, 512, m, 7)        # op 2 writes x of op 0 (m x 256)
    xd, qd, sd, yd = one_hot_case(256, 640, m, 8)             # op 3 writes the same buffer
    x0 = bf16_dev(xa)
    y0 = torch.full((m, 384), float("nan"), dtype=torch.bfloat16, device=DEV)  # read before written -> NaN
    y1 = torch.empty((m, 256), dtype=torch.bfloat16, device=DEV)
    dev = lambda a: torch.from_numpy(a).to(DEV)
    ops = [(x0, dev(qa), dev(sa), y0),
           (y0, dev(qb), dev(sb), y1),
           (bf16_dev(xc_next), dev(qc), dev(sc), x0),
           (bf16_dev(xd), dev(qd), dev(sd), x0)]
    pkg.gemv_batch(ops, path=path)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y0.cpu()), ya)
    rows_q = {rb: (qb[rb * 128:rb * 128 + 128], sb[rb]) for rb in range(2)}
    check_block_gemv(y1, ya, rows_q)
    # x0 was overwritten by op 2, then op 3 (the last writer wins)
    assert np.array_equal(bits(x0.cpu()), yd)


@pytest.mark.parametrize("m", [1, 8, 16, 32])
def test_mx_batch(pkg, m):
    shapes = [(300, 704), (1024, 2560), (129, 272), (2560, 3072)]
    ops, cases = [], []
    for i, (n, k) in enumerate(shapes):
        w = inputs.heavy_tail_weight(3 + i, shape=(n, k), frac=0.01)
        oc, oe = oracle.mx_quantize(bits(w))
        x = inputs.activations(m, k, 70 + i)
        ops.append((x.to(DEV), torch.from_numpy(oc).to(DEV), torch.from_numpy(oe).to(DEV)))
        cases.append((x, oc, oe))
    for path in (0, PATH_DECODE, PATH_GENERIC):
        ys = pkg.mx_gemv_batch(ops, path=path)
        torch.cuda.synchronize()
        for (x, oc, oe), y in zip(cases, ys):
            check_mx_gemv(y, bits(x), np.arange(oc.shape[0]), oc, oe)


def test_batch_in_cuda_graph(pkg, rotation_layers):
    """The batched call captures into a CUDA graph (its op table lives in the
    launch parameters); a replay gives the eager result bit for bit."""
    m = 8
    ops = [(inputs.activations(m, c.shape[1], 300 + i, device=DEV), c, s) for i, (c, s, _) in
           enumerate(rotation_layers)]
    want = [y.clone() for y in pkg.gemv_batch(ops)]
    ys = [torch.empty_like(y) for y in want]
    ops_y = [(x, c, s, y) for (x, c, s), y in zip(ops, ys)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkg.gemv_batch(ops_y)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for y in ys:
        y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkg.gemv_batch(ops_y)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(want, ys):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_no_device_error(pkg):
    assert pkg.check_device_error() == 0
