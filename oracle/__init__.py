"""CPU oracle for block-scaled FP8 / MXFP8 quantization and the W8A16 GEMV.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain, slow, independent
statement of what the library computes (``fp8bs_oracle.c``, plain C11 in
binary32/binary64).  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it; the product path never does, and
the two share no code.

This module compiles ``fp8bs_oracle.c`` with gcc (``-O2 -ffp-contract=off``,
no fast-math) into ``oracle/_build/liboracle.so`` and wraps it with ctypes
over numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8bs_oracle.c")
_HDR = os.path.join(_HERE, "fp8bs_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

TILE = 128
MX_GROUP = 32


def build(force: bool = False) -> str:
    """Compile the oracle shared library (if stale) and return its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= newest_src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode_f32_array.argtypes = [p, i64, p]
        lib.oracle_e4m3_encode_f32_array.restype = None
        lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_block_quantize.argtypes = [p, i64, i64, p, p]
        lib.oracle_block_quantize_tile.argtypes = [p, i64, i64, i64, i64, p, p]
        lib.oracle_mx_quantize.argtypes = [p, i64, i64, p, p]
        lib.oracle_mx_quantize_rows.argtypes = [p, i64, i64, p, i64, p, p]
        lib.oracle_block_gemv.argtypes = [p, i64, p, p, i64, i64, p, i64, p]
        lib.oracle_mx_gemv.argtypes = [p, i64, p, p, i64, i64, p, i64, p]
        lib.oracle_row_quantize_rows.argtypes = [p, i64, i64, p, i64, p, p]
        lib.oracle_tensor_quantize_rows.argtypes = [p, i64, i64, p, i64, p, p]
        lib.oracle_row_gemv.argtypes = [p, i64, p, p, i64, i64, i64, p, i64, p]
        lib.oracle_w8a8_gemv.argtypes = [p, i64, ctypes.c_float, p, ctypes.c_float, i64, i64, p, i64, p]
        lib.oracle_moe_gemv.argtypes = [p, i64, p, i64, p, p, i64, i64, i64, p, i64, p]
        f32, f64 = ctypes.c_float, ctypes.c_double
        lib.oracle_kv_append.argtypes = [p, i64, i64, i64, p, f32, p]
        lib.oracle_kv_attention.argtypes = [p, i64, i64, i64, i64, p, p, f32, f32, p, i64, p, i64, f64, p]
        for f in ("oracle_block_quantize", "oracle_block_quantize_tile",
                  "oracle_mx_quantize", "oracle_mx_quantize_rows",
                  "oracle_block_gemv", "oracle_mx_gemv",
                  "oracle_row_quantize_rows", "oracle_tensor_quantize_rows",
                  "oracle_row_gemv", "oracle_w8a8_gemv", "oracle_moe_gemv", "oracle_kv_append",
                  "oracle_kv_attention"):
            getattr(lib, f).restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def _bits16(w) -> np.ndarray:
    """Accept a numpy uint16 array of bf16 bit patterns (or a torch bf16
    tensor on the CPU) and return a C-contiguous uint16 numpy array."""
    if not isinstance(w, np.ndarray):
        import torch
        assert w.dtype == torch.bfloat16 and w.device.type == "cpu", (w.dtype, w.device)
        w = w.contiguous().view(torch.int16).numpy().view(np.uint16)
    w = np.ascontiguousarray(w)
    assert w.dtype == np.uint16, w.dtype
    return w


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


# ---------------------------------------------------------------- scalars
def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def e4m3_encode_f32(v) -> np.ndarray:
    """Element-wise e4m3 encode of binary32 values (brute force)."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.zeros(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_f32_array(_ptr(v), v.size, _ptr(out))
    return out


def double_to_bf16(v: float) -> int:
    return int(_load().oracle_double_to_bf16(float(v)))


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits) & 0xFFFF)


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(i) for i in range(256)], dtype=np.float64)


# ---------------------------------------------------------------- arrays
def block_quantize(w) -> tuple[np.ndarray, np.ndarray]:
    """w: [N,K] bf16 bits -> (codes u8 [N,K], scales f32 [ceil(N/128), ceil(K/128)])."""
    w = _bits16(w)
    n, k = w.shape
    codes = np.zeros((n, k), dtype=np.uint8)
    scales = np.zeros((cdiv(n, TILE), cdiv(k, TILE)), dtype=np.float32)
    _load().oracle_block_quantize(_ptr(w), n, k, _ptr(codes), _ptr(scales))
    return codes, scales


def block_quantize_tiles(w, tiles) -> tuple[np.ndarray, np.ndarray]:
    """Quantize only the listed (bn, bk) tiles; other entries stay 0."""
    w = _bits16(w)
    n, k = w.shape
    codes = np.zeros((n, k), dtype=np.uint8)
    scales = np.zeros((cdiv(n, TILE), cdiv(k, TILE)), dtype=np.float32)
    lib = _load()
    for bn, bk in tiles:
        lib.oracle_block_quantize_tile(_ptr(w), n, k, int(bn), int(bk),
                                       _ptr(codes), _ptr(scales))
    return codes, scales


def mx_quantize(w) -> tuple[np.ndarray, np.ndarray]:
    """w: [N,K] bf16 bits -> (codes u8 [N,K], e8m0 u8 [N, ceil(K/32)])."""
    w = _bits16(w)
    n, k = w.shape
    codes = np.zeros((n, k), dtype=np.uint8)
    e8m0 = np.zeros((n, cdiv(k, MX_GROUP)), dtype=np.uint8)
    _load().oracle_mx_quantize(_ptr(w), n, k, _ptr(codes), _ptr(e8m0))
    return codes, e8m0


def mx_quantize_rows(w, rows) -> tuple[np.ndarray, np.ndarray]:
    """Quantize only the listed rows of w; returns arrays of the listed rows."""
    w = _bits16(w)
    n, k = w.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    codes = np.zeros((n, k), dtype=np.uint8)
    e8m0 = np.zeros((n, cdiv(k, MX_GROUP)), dtype=np.uint8)
    _load().oracle_mx_quantize_rows(_ptr(w), n, k, _ptr(rows), len(rows),
                                    _ptr(codes), _ptr(e8m0))
    return codes[rows], e8m0[rows]


def _rows_arg(rows, n):
    if rows is None:
        return None, n
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert rows.ndim == 1 and (len(rows) == 0 or (rows.min() >= 0 and rows.max() < n))
    return rows, len(rows)


def block_gemv(x, codes: np.ndarray, scales: np.ndarray, rows=None) -> np.ndarray:
    """fp64 y[M, len(rows)] = x . (dec(codes) * s)^T over the listed rows."""
    x = _bits16(x)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    m, k = x.shape
    n, k2 = codes.shape
    assert k == k2 and scales.shape == (cdiv(n, TILE), cdiv(k, TILE))
    rows, nrows = _rows_arg(rows, n)
    y = np.zeros((m, nrows), dtype=np.float64)
    _load().oracle_block_gemv(_ptr(x), m, _ptr(codes), _ptr(scales), n, k,
                              None if rows is None else _ptr(rows), nrows, _ptr(y))
    return y


def mx_gemv(x, codes: np.ndarray, e8m0: np.ndarray, rows=None) -> np.ndarray:
    """fp64 y[M, len(rows)] = x . (dec(codes) * 2^(E-127))^T over the listed rows."""
    x = _bits16(x)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    e8m0 = np.ascontiguousarray(e8m0, dtype=np.uint8)
    m, k = x.shape
    n, k2 = codes.shape
    assert k == k2 and e8m0.shape == (n, cdiv(k, MX_GROUP))
    rows, nrows = _rows_arg(rows, n)
    y = np.zeros((m, nrows), dtype=np.float64)
    _load().oracle_mx_gemv(_ptr(x), m, _ptr(codes), _ptr(e8m0), n, k,
                           None if rows is None else _ptr(rows), nrows, _ptr(y))
    return y


def row_quantize(w, rows=None) -> tuple[np.ndarray, np.ndarray]:
    """Per-row FP8: w [N,K] bf16 bits -> (codes u8 [N,K], scales f32 [N]).
    With ``rows``, only those rows are quantized and returned (in order)."""
    w = _bits16(w)
    n, k = w.shape
    rows, nrows = _rows_arg(rows, n)
    codes = np.zeros((n, k), dtype=np.uint8)
    scales = np.zeros((n,), dtype=np.float32)
    _load().oracle_row_quantize_rows(_ptr(w), n, k, None if rows is None else _ptr(rows),
                                     nrows, _ptr(codes), _ptr(scales))
    if rows is None:
        return codes, scales
    return codes[rows], scales[rows]


def tensor_quantize(w, rows=None) -> tuple[np.ndarray, np.ndarray]:
    """Per-tensor FP8: w [N,K] bf16 bits -> (codes u8 [N,K], scale f32 [1]).
    The amax is always taken over the whole tensor; with ``rows`` only
    those rows are encoded and returned (in order)."""
    w = _bits16(w)
    n, k = w.shape
    rows, nrows = _rows_arg(rows, n)
    codes = np.zeros((n, k), dtype=np.uint8)
    scale = np.zeros((1,), dtype=np.float32)
    _load().oracle_tensor_quantize_rows(_ptr(w), n, k, None if rows is None else _ptr(rows),
                                        nrows, _ptr(codes), _ptr(scale))
    if rows is None:
        return codes, scale
    return codes[rows], scale


def row_gemv(x, codes: np.ndarray, scales: np.ndarray, rows=None) -> np.ndarray:
    """fp64 y[M, len(rows)] = x . (dec(codes) * s_row)^T.  ``scales`` is the
    per-row vector [N] or the per-tensor scalar [1] (broadcast)."""
    x = _bits16(x)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(np.asarray(scales, dtype=np.float32).ravel())
    m, k = x.shape
    n, k2 = codes.shape
    assert k == k2 and scales.shape in ((n,), (1,))
    stride = 1 if scales.shape == (n,) and n > 1 else 0
    rows, nrows = _rows_arg(rows, n)
    y = np.zeros((m, nrows), dtype=np.float64)
    _load().oracle_row_gemv(_ptr(x), m, _ptr(codes), _ptr(scales), stride, n, k,
                            None if rows is None else _ptr(rows), nrows, _ptr(y))
    return y


def act_quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """Dynamic per-tensor activation quantization: x [M,K] bf16 bits ->
    (codes u8 [M,K], scale f32 [1]); the per-tensor rule applied to x."""
    return tensor_quantize(x)


def w8a8_gemv(xcodes: np.ndarray, sx, wcodes: np.ndarray, sw, rows=None) -> np.ndarray:
    """fp64 y[M, len(rows)] = sx * sw * dec(xcodes) . dec(wcodes)^T."""
    xcodes = np.ascontiguousarray(xcodes, dtype=np.uint8)
    wcodes = np.ascontiguousarray(wcodes, dtype=np.uint8)
    m, k = xcodes.shape
    n, k2 = wcodes.shape
    assert k == k2
    rows, nrows = _rows_arg(rows, n)
    y = np.zeros((m, nrows), dtype=np.float64)
    _load().oracle_w8a8_gemv(_ptr(xcodes), m, float(np.float32(np.ravel(sx)[0])), _ptr(wcodes),
                             float(np.float32(np.ravel(sw)[0])), n, k,
                             None if rows is None else _ptr(rows), nrows, _ptr(y))
    return y


def moe_gemv(x, ids, codes: np.ndarray, scales: np.ndarray, rows=None) -> np.ndarray:
    """fp64 y[M, topk, len(rows)]: (token t, slot j) = block GEMV of x[t] with
    expert ids[t, j]; codes [E, N, K], scales [E, ceil(N/128), ceil(K/128)]."""
    x = _bits16(x)
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    m, k = x.shape
    e, n, k2 = codes.shape
    assert k == k2 and ids.shape[0] == m and scales.shape == (e, cdiv(n, TILE), cdiv(k, TILE))
    topk = ids.shape[1]
    rows, nrows = _rows_arg(rows, n)
    y = np.zeros((m, topk, nrows), dtype=np.float64)
    _load().oracle_moe_gemv(_ptr(x), m, _ptr(ids), topk, _ptr(codes), _ptr(scales), e, n, k,
                            None if rows is None else _ptr(rows), nrows, _ptr(y))
    return y


def kv_append(x, slots, scale, cache: np.ndarray) -> np.ndarray:
    """Quantize x [T, Hkv, D] (bf16 bits) into a copy of cache
    [num_blocks, page_size, Hkv, D] at the flat token slots."""
    x = _bits16(x)
    t, hkv, d = x.shape
    slots = np.ascontiguousarray(np.asarray(slots, dtype=np.int32))
    out = np.ascontiguousarray(cache, dtype=np.uint8).copy()
    assert out.shape[2:] == (hkv, d) and slots.shape == (t,)
    assert t == 0 or (slots.min() >= 0 and slots.max() < out.shape[0] * out.shape[1])
    _load().oracle_kv_append(_ptr(x), t, hkv, d, _ptr(slots), float(np.float32(np.ravel(scale)[0])), _ptr(out))
    return out


def kv_attention(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, sm_scale) -> np.ndarray:
    """fp64 decode attention: q [B, Hq, D] bf16 bits, caches [num_blocks,
    page_size, Hkv, D] e4m3, block_table [B, max_blocks] int32, seq_lens [B]."""
    q = _bits16(q)
    b, hq, d = q.shape
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint8)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint8)
    nb, page, hkv, d2 = k_cache.shape
    assert d2 == d and v_cache.shape == k_cache.shape and hq % hkv == 0
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    assert bt.shape[0] == b and sl.shape == (b,)
    assert np.all(sl <= bt.shape[1] * page)
    o = np.zeros((b, hq, d), dtype=np.float64)
    _load().oracle_kv_attention(_ptr(q), b, hq, hkv, d, _ptr(k_cache), _ptr(v_cache),
                                float(np.float32(np.ravel(k_scale)[0])), float(np.float32(np.ravel(v_scale)[0])),
                                _ptr(bt), bt.shape[1], _ptr(sl), page, float(sm_scale), _ptr(o))
    return o


def to_bf16_bits(y64: np.ndarray) -> np.ndarray:
    """Round each fp64 value to bf16 (nearest, ties to even)."""
    lib = _load()
    flat = np.asarray(y64, dtype=np.float64).ravel()
    out = np.fromiter((lib.oracle_double_to_bf16(float(v)) for v in flat),
                      dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(y64))
