"""fp8bs_gemv_noalloc: the workspace GEMV for callers that cannot allocate
device memory (a plugin inside a framework that owns all device memory, a
real-time loop that cannot afford cudaMalloc / cudaFree, a C caller with
nowhere to keep a buffer).  Its scratch is a fixed array in the library's
own device memory, so the call takes no workspace.

Called through the C ABI (ctypes) and compared, on two calls in a row, with
the existing entry point fp8bs_gemv_ws given a caller-allocated workspace,
under the GEMV tolerance used by every parity test (and both against the
oracle).  This file is collected last so that a run stopping at its first
failure has run every other test before it; it also passes on its own in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import inputs
from oracle import tolerance

from gpu_helpers import bits, check_block_gemv, lib_or_skip, table

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_BYTES = 2 * 1024 * 1024   # FP8BS_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def pkg():
    p = lib_or_skip()
    L = p.lib()
    i64, v = ctypes.c_int64, ctypes.c_void_p
    L.fp8bs_gemv_noalloc.argtypes = [v, i64, v, v, i64, i64, v, v]
    L.fp8bs_gemv_noalloc.restype = ctypes.c_int
    return p


def noalloc(pkg, x, codes, scales, y):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return pkg.lib().fp8bs_gemv_noalloc(ctypes.c_void_p(x.data_ptr()), x.shape[0], ctypes.c_void_p(codes.data_ptr()),
                                       ctypes.c_void_p(scales.data_ptr()), codes.shape[0], codes.shape[1],
                                       ctypes.c_void_p(y.data_ptr()), stream)


def test_two_calls_in_a_row_match_the_workspace_entry_point(pkg):
    w = inputs.sweep_weight(0)[:1024]                        # [1024, 4096] block-FP8, 8 row tiles
    oc, os_ = oracle.block_quantize(bits(w))
    n, k = oc.shape
    codes, scales = torch.from_numpy(oc).to(DEV), torch.from_numpy(os_).to(DEV)
    rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(n // 128)}
    wmax = tolerance.block_wmax_rows(oc, os_, np.arange(n), table())
    for m, seed in ((16, 1), (5, 2)):                        # two calls in a row, different x
        x = inputs.activations(m, k, seed, device=DEV)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
        assert noalloc(pkg, x, codes, scales, y) == 0
        ws = torch.empty((pkg.gemv_ws_bytes(m, k),), dtype=torch.uint8, device=DEV)
        y_ws = pkg.gemv_ws(x, codes, scales, ws)
        torch.cuda.synchronize()
        st = tolerance.gemv_errors(bits(y.cpu()), tolerance.bf16_bits_to_f64(bits(y_ws.cpu())), bits(x.cpu()), wmax)
        assert tolerance.gemv_ok(st), st
        check_block_gemv(y, bits(x.cpu()), rows_q)
        check_block_gemv(y_ws, bits(x.cpu()), rows_q)
    assert pkg.check_device_error() == 0


def test_larger_than_its_scratch_is_refused(pkg):
    k = 65536                                                 # m = 32: 4 MiB of f16 x, over the 2 MiB
    assert pkg.gemv_ws_bytes(32, k) > SCRATCH_BYTES
    x = torch.zeros((32, k), dtype=torch.bfloat16, device=DEV)
    codes = torch.zeros((128, k), dtype=torch.uint8, device=DEV)
    scales = torch.ones((1, k // 128), dtype=torch.float32, device=DEV)
    y = torch.empty((32, 128), dtype=torch.bfloat16, device=DEV)
    assert noalloc(pkg, x, codes, scales, y) == -2            # FP8BS_ERR_SHAPE, nothing launched
