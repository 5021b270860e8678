"""Failure detection on the GPU without a fault: a bounded wait that runs out
sets the device error word instead of hanging, the host reads (and clears)
it, and the context keeps computing correct results afterwards.

The wait that runs out is the library's own probe (fp8bs_debug_wait_expiry):
one thread waits on a barrier nothing completes, with the same bounded wait
every pipelined kernel uses, and gives up after about 2 s.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import inputs

from gpu_helpers import bits, check_block_gemv, lib_or_skip

pytestmark = pytest.mark.gpu
DEV = "cuda"
FULL_WAIT = 1  # bit of the error word set by a consumer-side wait that gave up


@pytest.fixture(scope="module")
def pkg():
    return lib_or_skip()


def small_gemv_matches_oracle(pkg):
    """One ragged block-FP8 GEMV, its codes and scales from the oracle."""
    w = inputs.tiny_ragged_weight(0)
    oc, os_ = oracle.block_quantize(bits(w))
    x = inputs.activations(3, w.shape[1], 9)
    y = pkg.gemv(x.to(DEV), torch.from_numpy(oc).to(DEV), torch.from_numpy(os_).to(DEV))
    torch.cuda.synchronize()
    rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(os_.shape[0])}
    check_block_gemv(y, bits(x), rows_q)


def test_wait_expiry_sets_the_error_word_and_the_context_survives(pkg):
    assert pkg.check_device_error() == 0
    t0 = time.monotonic()
    pkg.debug_wait_expiry()
    word = pkg.check_device_error()  # synchronises: includes the whole wait
    elapsed = time.monotonic() - t0
    assert word & FULL_WAIT
    assert 1.0 < elapsed < 60.0, elapsed  # the bound is about 2 s of device time
    assert pkg.check_device_error() == 0  # reading the word cleared it
    small_gemv_matches_oracle(pkg)
    assert pkg.check_device_error() == 0


def test_wait_expiry_on_a_side_stream(pkg):
    s = torch.cuda.Stream()
    pkg.debug_wait_expiry(stream=s)
    assert pkg.check_device_error(stream=s) & FULL_WAIT
    small_gemv_matches_oracle(pkg)
