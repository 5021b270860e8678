"""Every binary32 bit pattern, in fixed slices that host threads check in
parallel (the oracle and numpy release the GIL while they work)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

SLICE = 1 << 22
ALL = 1 << 32
FINITE = ALL - (1 << 24)  # exponent field 255 (Inf, NaN): 2 signs x 2^23 mantissas


def f32_slice(base: int):
    """The binary32 values with bit patterns base .. base + SLICE - 1 and a
    mask of the finite ones."""
    bits = np.arange(base, base + SLICE, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    return f, np.isfinite(f)


def workers() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1))


def sweep(check, bases=None):
    """check(base) -> (mismatches, values checked) for every slice; returns
    the totals."""
    bases = range(0, ALL, SLICE) if bases is None else bases
    with ThreadPoolExecutor(workers()) as ex:
        results = list(ex.map(check, bases))
    return sum(r[0] for r in results), sum(r[1] for r in results)
