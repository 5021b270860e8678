"""fp8_block_scaled_02_gb300 -- block-scaled FP8 / MXFP8 / per-row FP8 W8A16 on GB300.

A thin Python binding over the C ABI in ``include/fp8bs.h`` (``libfp8bs.so``,
built from ``csrc/`` for sm_103a).  Every function here only marshals
arguments -- device pointers, sizes and the current CUDA stream -- and calls
the library; all computation runs in the library's kernels.  There is no CPU
fallback: if the shared library has not been built, or a tensor is not on a
CUDA device, the call raises.

Functions (names follow the C entry points):
    quantize(w)            -> (codes u8 [N,K], scales f32 [ceil(N/128), ceil(K/128)])
    gemv(x, codes, scales) -> y bf16 [M,N]
    mx_quantize(w)         -> (codes u8 [N,K], e8m0 u8 [N, ceil(K/32)])
    mx_gemv(x, codes, e8m0)-> y bf16 [M,N]
    row_quantize(w)        -> (codes u8 [N,K], scales f32 [N])       (fp8row_*)
    tensor_quantize(w)     -> (codes u8 [N,K], scale f32 [1])        (fp8tensor_*)
    row_gemv(x, codes, s)  -> y bf16 [M,N]; s is [N] (per row) or [1] (per tensor)
    act_quantize(x)        -> (x codes u8 [M,K], scale f32 [1])      (fp8act_quantize)
    w8a8_gemm(xq, sx, wq, sw) -> y bf16 [M,N]                        (w8a8_gemm)
    w8a8_linear(x, wq, sw) -> y bf16 [M,N]: act_quantize then w8a8_gemm
    moe_gemv(x, ids, codes, scales) -> y bf16 [M, topk, N]            (fp8bs_moe_gemv)
        codes [E,N,K], scales [E, ceil(N/128), ceil(K/128)], ids int32 [M, topk]
    kv_append(x, slots, scale, cache)    FP8 KV cache append (fp8kv_append), in place
    kv_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                        max_seq_len, sm_scale) -> o bf16 [B, Hq, 128]   (fp8kv_decode_attention)
    check_device_error()   -> the kernels' error word (synchronises; reading clears it)
    select_path(m, n, k)   -> the kernel path an AUTO call takes (host only)
    debug_wait_expiry(), debug_encode_f32(first_bits, count)   test hooks (fp8bs_debug_*)
"""
from __future__ import annotations

import ctypes
import os
import threading

PATH_AUTO, PATH_DECODE, PATH_PREFILL, PATH_GENERIC = 0, 1, 2, 3
PATH_NAMES = {PATH_AUTO: "auto", PATH_DECODE: "decode", PATH_PREFILL: "prefill", PATH_GENERIC: "generic"}

STATUS = {0: "FP8BS_OK", -1: "FP8BS_ERR_NULL", -2: "FP8BS_ERR_SHAPE", -3: "FP8BS_ERR_BLOCK",
          -4: "FP8BS_ERR_ALIGN", -5: "FP8BS_ERR_CUDA", -6: "FP8BS_ERR_DEVICE", -7: "FP8BS_ERR_PATH"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfp8bs.so")
_lock = threading.Lock()
_lib = None


class Fp8bsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({strerror(status)})")


def lib() -> ctypes.CDLL:
    """The loaded libfp8bs.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "or `python fp8_block_scaled_02_gb300/build.py`")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.fp8bs_quantize.argtypes = [p, i64, i64, i32, p, p, p]
        L.fp8bs_gemv.argtypes = [p, i64, p, p, i64, i64, p, p]
        L.fp8bs_gemv_ex.argtypes = [p, i64, p, p, i64, i64, p, i32, p]
        L.mxfp8_quantize.argtypes = [p, i64, i64, p, p, p]
        L.mxfp8_gemv.argtypes = [p, i64, p, p, i64, i64, p, p]
        L.mxfp8_gemv_ex.argtypes = [p, i64, p, p, i64, i64, p, i32, p]
        L.fp8row_quantize.argtypes = [p, i64, i64, p, p, p]
        L.fp8tensor_quantize.argtypes = [p, i64, i64, p, p, p]
        L.fp8row_gemv.argtypes = [p, i64, p, p, i64, i64, p, p]
        L.fp8row_gemv_ex.argtypes = [p, i64, p, p, i64, i64, p, i32, p]
        L.fp8tensor_gemv.argtypes = [p, i64, p, p, i64, i64, p, p]
        L.fp8tensor_gemv_ex.argtypes = [p, i64, p, p, i64, i64, p, i32, p]
        L.fp8act_quantize.argtypes = [p, i64, i64, p, p, p]
        L.fp8bs_moe_gemv.argtypes = [p, i64, p, i64, p, p, i64, i64, i64, p, p]
        L.fp8kv_append.argtypes = [p, i64, i64, i64, p, p, p, i64, p]
        L.fp8kv_decode_attention.argtypes = [p, p, p, p, p, p, i64, p, i64, i64, i64, i64, i64, i64, i64,
                                             ctypes.c_float, p, p]
        L.w8a8_gemm.argtypes = [p, i64, p, p, p, i64, i64, p, p]
        L.w8a8_gemm_ex.argtypes = [p, i64, p, p, p, i64, i64, p, i32, p]
        L.fp8bs_select_path.argtypes = [i64, i64, i64, p, p, i32]
        L.fp8bs_strerror.argtypes = [i32]
        L.fp8bs_strerror.restype = ctypes.c_char_p
        L.fp8bs_check_device_error.argtypes = [p, ctypes.POINTER(ctypes.c_uint32)]
        L.fp8bs_debug_wait_expiry.argtypes = [p]
        L.fp8bs_debug_encode_f32.argtypes = [ctypes.c_uint32, i64, p, p]
        L.fp8bs_version.argtypes = []
        for f in ("fp8bs_quantize", "fp8bs_gemv", "fp8bs_gemv_ex", "mxfp8_quantize", "mxfp8_gemv",
                  "mxfp8_gemv_ex", "fp8row_quantize", "fp8tensor_quantize", "fp8row_gemv", "fp8row_gemv_ex",
                  "fp8tensor_gemv", "fp8tensor_gemv_ex", "fp8act_quantize", "w8a8_gemm", "w8a8_gemm_ex",
                  "fp8bs_moe_gemv", "fp8kv_append", "fp8kv_decode_attention",
                  "fp8bs_select_path", "fp8bs_check_device_error", "fp8bs_debug_wait_expiry",
                  "fp8bs_debug_encode_f32", "fp8bs_version"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
        return L


def strerror(status: int) -> str:
    try:
        return lib().fp8bs_strerror(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(status: int, what: str):
    if status != 0:
        raise Fp8bsError(status, what)


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def quantize(w, block: int = 128, codes=None, scales=None, stream=None):
    """Block-FP8 load-time quantization of a bf16 [N, K] CUDA tensor."""
    import torch
    n, k = w.shape
    if codes is None:
        codes = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((cdiv(n, 128), cdiv(k, 128)), dtype=torch.float32, device=w.device)
    _check(lib().fp8bs_quantize(_dev(w, torch.bfloat16, "w"), n, k, int(block), _dev(codes, torch.uint8, "codes"),
                                _dev(scales, torch.float32, "scales"), _stream(stream)), "fp8bs_quantize")
    return codes, scales


def gemv(x, codes, scales, y=None, path: int = PATH_AUTO, stream=None):
    """y[M, N] = x[M, K] . dequant(codes, scales)^T (bf16 out, fp32 accumulate)."""
    import torch
    m, k = x.shape
    n = codes.shape[0]
    if codes.shape[1] != k:
        raise ValueError("codes and x disagree on K")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    _check(lib().fp8bs_gemv_ex(_dev(x, torch.bfloat16, "x"), m, _dev(codes, torch.uint8, "codes"),
                               _dev(scales, torch.float32, "scales"), n, k, _dev(y, torch.bfloat16, "y"),
                               int(path), _stream(stream)), "fp8bs_gemv")
    return y


def mx_quantize(w, codes=None, e8m0=None, stream=None):
    """MXFP8 load-time quantization of a bf16 [N, K] CUDA tensor."""
    import torch
    n, k = w.shape
    if codes is None:
        codes = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    if e8m0 is None:
        e8m0 = torch.empty((n, cdiv(k, 32)), dtype=torch.uint8, device=w.device)
    _check(lib().mxfp8_quantize(_dev(w, torch.bfloat16, "w"), n, k, _dev(codes, torch.uint8, "codes"),
                                _dev(e8m0, torch.uint8, "e8m0"), _stream(stream)), "mxfp8_quantize")
    return codes, e8m0


def mx_gemv(x, codes, e8m0, y=None, path: int = PATH_AUTO, stream=None):
    """y[M, N] = x[M, K] . dequant_mx(codes, e8m0)^T."""
    import torch
    m, k = x.shape
    n = codes.shape[0]
    if codes.shape[1] != k:
        raise ValueError("codes and x disagree on K")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    _check(lib().mxfp8_gemv_ex(_dev(x, torch.bfloat16, "x"), m, _dev(codes, torch.uint8, "codes"),
                               _dev(e8m0, torch.uint8, "e8m0"), n, k, _dev(y, torch.bfloat16, "y"),
                               int(path), _stream(stream)), "mxfp8_gemv")
    return y


def row_quantize(w, codes=None, scales=None, stream=None):
    """Per-row FP8 load-time quantization: one fp32 scale per row of w."""
    import torch
    n, k = w.shape
    if codes is None:
        codes = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((n,), dtype=torch.float32, device=w.device)
    _check(lib().fp8row_quantize(_dev(w, torch.bfloat16, "w"), n, k, _dev(codes, torch.uint8, "codes"),
                                 _dev(scales, torch.float32, "scales"), _stream(stream)), "fp8row_quantize")
    return codes, scales


def tensor_quantize(w, codes=None, scale=None, stream=None):
    """Per-tensor FP8 load-time quantization: one fp32 scale for all of w."""
    import torch
    n, k = w.shape
    if codes is None:
        codes = torch.empty((n, k), dtype=torch.uint8, device=w.device)
    if scale is None:
        scale = torch.empty((1,), dtype=torch.float32, device=w.device)
    _check(lib().fp8tensor_quantize(_dev(w, torch.bfloat16, "w"), n, k, _dev(codes, torch.uint8, "codes"),
                                    _dev(scale, torch.float32, "scale"), _stream(stream)), "fp8tensor_quantize")
    return codes, scale


def row_gemv(x, codes, scales, y=None, path: int = PATH_AUTO, stream=None):
    """y[M, N] = x[M, K] . (dec(codes) * s_row)^T.  ``scales`` of shape [N]
    calls fp8row_gemv, of shape [1] fp8tensor_gemv."""
    import torch
    m, k = x.shape
    n = codes.shape[0]
    if codes.shape[1] != k:
        raise ValueError("codes and x disagree on K")
    per_row = tuple(scales.shape) == (n,) and n > 1
    if not per_row and tuple(scales.shape) not in ((1,), ()):
        raise ValueError("scales must have shape [N] (per row) or [1] (per tensor)")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    fn = lib().fp8row_gemv_ex if per_row else lib().fp8tensor_gemv_ex
    _check(fn(_dev(x, torch.bfloat16, "x"), m, _dev(codes, torch.uint8, "codes"),
              _dev(scales, torch.float32, "scales"), n, k, _dev(y, torch.bfloat16, "y"), int(path),
              _stream(stream)), "fp8row_gemv" if per_row else "fp8tensor_gemv")
    return y


def moe_gemv(x, ids, codes, scales, y=None, stream=None):
    """Grouped block-FP8 GEMV over routed experts: y[t, j] = x[t] . dequant(W[ids[t, j]])^T."""
    import torch
    m, k = x.shape
    e, n, k2 = codes.shape
    topk = ids.shape[1]
    if k2 != k or ids.shape[0] != m:
        raise ValueError("x, ids and codes disagree on M or K")
    if y is None:
        y = torch.empty((m, topk, n), dtype=torch.bfloat16, device=x.device)
    _check(lib().fp8bs_moe_gemv(_dev(x, torch.bfloat16, "x"), m, _dev(ids, torch.int32, "ids"), topk,
                                _dev(codes, torch.uint8, "codes"), _dev(scales, torch.float32, "scales"), e, n, k,
                                _dev(y, torch.bfloat16, "y"), _stream(stream)), "fp8bs_moe_gemv")
    return y


def kv_append(x, slots, scale, cache, stream=None):
    """Quantize new keys or values x [T, Hkv, 128] bf16 into the e4m3 cache
    [num_blocks, page_size, Hkv, 128] at flat token slots (in place)."""
    import torch
    t, hkv, d = x.shape
    nb, page, hkv2, d2 = cache.shape
    if (hkv2, d2) != (hkv, d):
        raise ValueError("x and cache disagree on kv heads or head_dim")
    _check(lib().fp8kv_append(_dev(x, torch.bfloat16, "x"), t, hkv, d, _dev(slots, torch.int32, "slots"),
                              _dev(scale, torch.float32, "scale"), _dev(cache, torch.uint8, "cache"), nb * page,
                              _stream(stream)), "fp8kv_append")
    return cache


def kv_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, max_seq_len: int,
                        sm_scale: float, out=None, stream=None):
    """Paged decode attention over the FP8 KV cache: q [B, Hq, 128] bf16."""
    import torch
    b, hq, d = q.shape
    nb, page, hkv, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape) or block_table.shape[0] != b:
        raise ValueError("q, caches and block table disagree")
    if out is None:
        out = torch.empty((b, hq, d), dtype=torch.bfloat16, device=q.device)
    _check(lib().fp8kv_decode_attention(_dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.uint8, "k_cache"),
                                        _dev(v_cache, torch.uint8, "v_cache"), _dev(k_scale, torch.float32, "k_scale"),
                                        _dev(v_scale, torch.float32, "v_scale"),
                                        _dev(block_table, torch.int32, "block_table"), block_table.shape[1],
                                        _dev(seq_lens, torch.int32, "seq_lens"), b, hq, hkv, d, page, nb,
                                        int(max_seq_len), float(sm_scale), _dev(out, torch.bfloat16, "out"),
                                        _stream(stream)), "fp8kv_decode_attention")
    return out


def act_quantize(x, codes=None, scale=None, stream=None):
    """Dynamic per-tensor e4m3 quantization of bf16 activations [M, K]."""
    import torch
    m, k = x.shape
    if codes is None:
        codes = torch.empty((m, k), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((1,), dtype=torch.float32, device=x.device)
    _check(lib().fp8act_quantize(_dev(x, torch.bfloat16, "x"), m, k, _dev(codes, torch.uint8, "codes"),
                                 _dev(scale, torch.float32, "scale"), _stream(stream)), "fp8act_quantize")
    return codes, scale


def w8a8_gemm(xq, sx, wq, sw, y=None, path: int = PATH_AUTO, stream=None):
    """y[M, N] = sx * sw * dec(xq) . dec(wq)^T (e4m3 x e4m3, fp32 accumulate, bf16 out)."""
    import torch
    m, k = xq.shape
    n = wq.shape[0]
    if wq.shape[1] != k:
        raise ValueError("x codes and weight codes disagree on K")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=xq.device)
    _check(lib().w8a8_gemm_ex(_dev(xq, torch.uint8, "xq"), m, _dev(sx, torch.float32, "sx"),
                              _dev(wq, torch.uint8, "wq"), _dev(sw, torch.float32, "sw"), n, k,
                              _dev(y, torch.bfloat16, "y"), int(path), _stream(stream)), "w8a8_gemm")
    return y


def w8a8_linear(x, wq, sw, y=None, xq=None, sx=None, path: int = PATH_AUTO, stream=None):
    """The W8A8 route end to end: quantize x per tensor, then w8a8_gemm."""
    xq, sx = act_quantize(x, codes=xq, scale=sx, stream=stream)
    return w8a8_gemm(xq, sx, wq, sw, y=y, path=path, stream=stream)


def select_path(m: int, n: int, k: int, x_ptr: int = 0, codes_ptr: int = 0, mx: bool = False) -> int:
    """Path the AUTO dispatch would take (host-only; pointers only matter for alignment)."""
    return lib().fp8bs_select_path(m, n, k, ctypes.c_void_p(x_ptr), ctypes.c_void_p(codes_ptr), int(mx))


def debug_wait_expiry(stream=None) -> None:
    """Launch the library's wait-expiry probe (fp8bs_debug_wait_expiry): one
    thread gives up a bounded wait after about 2 s and sets the error word."""
    _check(lib().fp8bs_debug_wait_expiry(_stream(stream)), "fp8bs_debug_wait_expiry")


def debug_encode_f32(first_bits: int, count: int, out=None, stream=None):
    """The quantizers' e4m3 encode step on the binary32 bit patterns
    first_bits .. first_bits + count - 1 (fp8bs_debug_encode_f32); returns
    uint8 codes on the device."""
    import torch
    if out is None:
        out = torch.empty(count, dtype=torch.uint8, device="cuda")
    if out.numel() < count:
        raise ValueError("out holds fewer than count bytes")
    _check(lib().fp8bs_debug_encode_f32(first_bits, count, _dev(out, torch.uint8, "out"), _stream(stream)),
           "fp8bs_debug_encode_f32")
    return out


def check_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the kernels' error word."""
    word = ctypes.c_uint32(0)
    st = lib().fp8bs_check_device_error(_stream(stream), ctypes.byref(word))
    if st not in (0, -6):
        raise Fp8bsError(st, "fp8bs_check_device_error")
    return int(word.value)
