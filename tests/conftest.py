import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def golden():
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        return json.load(f)


def e4m3_values_torch() -> np.ndarray:
    """Decode of all 256 codes by torch's float8_e4m3fn (an independent
    library, executed, not read)."""
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bitwise_e4m3_encode(v) -> np.ndarray:
    """An independent round-to-nearest-even, saturating e4m3 encoder written
    as arithmetic on each value's binade (numpy, vectorised); the oracle's
    encoder is a brute-force nearest search, so the two share no method."""
    v = np.asarray(v, dtype=np.float32)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v).astype(np.float64)
    out = np.zeros(a.shape, dtype=np.uint8)
    nz = a > 0
    f, ex = np.frexp(a[nz])             # a = f * 2^ex, f in [0.5, 1)
    e = ex - 1                          # a in [2^e, 2^(e+1))
    qexp = np.maximum(e, -6) - 3        # e4m3 quantum in this binade
    t = np.ldexp(a[nz], -qexp)
    r = np.rint(t)                      # numpy rint: half to even
    val = np.minimum(np.ldexp(r, qexp), 448.0)
    code = np.zeros(val.shape, dtype=np.int64)
    pos = val > 0
    f2, ex2 = np.frexp(val[pos])
    e2 = ex2 - 1
    sub = e2 < -6
    mant_norm = np.rint(np.ldexp(val[pos], -e2) * 8 - 8).astype(np.int64)
    mant_sub = np.rint(np.ldexp(val[pos], 9)).astype(np.int64)
    c = np.where(sub, mant_sub, ((e2 + 7) << 3) | mant_norm)
    code[pos] = c
    out[nz] = code.astype(np.uint8)
    return out | sign


def ulp_bf16(v) -> np.ndarray:
    """Spacing of bf16 values at |v| (2^-133 in the subnormal range)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    return np.ldexp(1.0, np.maximum(ex - 1, -126) - 7)
