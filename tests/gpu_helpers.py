"""Helpers for the GPU parity tests (imported only by tests marked gpu)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import inputs
from oracle import tolerance

TABLE = None


def table():
    global TABLE
    if TABLE is None:
        TABLE = oracle.e4m3_decode_table()
    return TABLE


def lib_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_block_scaled_02_gb300 import build
    build.build()
    import fp8_block_scaled_02_gb300 as pkg
    pkg.lib()
    return pkg


def bits(t: torch.Tensor) -> np.ndarray:
    return inputs.bf16_bits(t)


def oracle_block_rows(w_cpu_bits: np.ndarray, row_blocks):
    """Oracle block quantization of whole 128-row blocks (a row's codes and
    scales depend only on its own 128-row block).  Returns
    {rb: (codes [rows, K], scales [K/128])}."""
    out = {}
    n = w_cpu_bits.shape[0]
    for rb in row_blocks:
        sub = np.ascontiguousarray(w_cpu_bits[rb * 128:min(n, rb * 128 + 128)])
        c, s = oracle.block_quantize(sub)
        out[int(rb)] = (c, s[0])
    return out


def install_block_rows(codes_gpu, scales_gpu, rows_q):
    """Overwrite the GPU weight buffers with the oracle's codes/scales for
    the sampled row blocks, so the GEMV's checked outputs depend on oracle
    inputs only."""
    for rb, (c, s) in rows_q.items():
        codes_gpu[rb * 128: rb * 128 + c.shape[0]].copy_(torch.from_numpy(c))
        scales_gpu[rb].copy_(torch.from_numpy(s))


def check_block_gemv(y_gpu, x_cpu_bits, rows_q, m_rows=None):
    """Compare the GEMV output on the sampled row blocks with the oracle."""
    rows = np.concatenate([np.arange(rb * 128, rb * 128 + c.shape[0]) for rb, (c, _) in rows_q.items()])
    codes = np.concatenate([c for c, _ in rows_q.values()])
    kb = next(iter(rows_q.values()))[1].shape[0]
    scales = np.zeros((rows.max() // 128 + 1, kb), dtype=np.float32)
    for rb, (_, s) in rows_q.items():
        scales[rb] = s
    # oracle over the gathered rows: build a compact weight whose row j is rows[j]
    xb = x_cpu_bits if m_rows is None else x_cpu_bits[m_rows]
    y64 = np.zeros((xb.shape[0], len(rows)))
    off = 0
    for rb, (c, s) in rows_q.items():
        y64[:, off:off + c.shape[0]] = oracle.block_gemv(xb, c, s[None, :])
        off += c.shape[0]
    y = bits(y_gpu[:, torch.from_numpy(rows).to(y_gpu.device)])
    if m_rows is not None:
        y = y[m_rows]
    wmax = np.abs(table()[codes] * np.repeat(scales[rows // 128].astype(np.float64), 128, axis=1)[:, :codes.shape[1]]).max(axis=1)
    st = tolerance.gemv_errors(y, y64, xb, wmax)
    assert tolerance.gemv_ok(st), st
    return st


def check_mx_gemv(y_gpu, x_cpu_bits, rows, codes_rows, e8m0_rows):
    y64 = oracle.mx_gemv(x_cpu_bits, codes_rows, e8m0_rows)
    y = bits(y_gpu[:, torch.as_tensor(rows, device=y_gpu.device)])
    st = tolerance.gemv_errors(y, y64, x_cpu_bits, tolerance.mx_wmax_rows(codes_rows, e8m0_rows, table()))
    assert tolerance.gemv_ok(st), st
    return st


def guarded_empty(shape, dtype, device, guard=4096, fill=0x5A):
    """A tensor view followed by a guard band filled with a sentinel."""
    numel = int(np.prod(shape))
    itemsize = torch.empty((), dtype=dtype).element_size()
    raw = torch.full((numel * itemsize + guard,), fill, dtype=torch.uint8, device=device)
    view = raw[: numel * itemsize].view(dtype).view(*shape)
    return view, raw


def guard_intact(raw, numel_bytes, fill=0x5A) -> bool:
    return bool((raw[numel_bytes:] == fill).all().item())
