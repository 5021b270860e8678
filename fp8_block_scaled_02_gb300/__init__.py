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
    gemv_ws(x, codes, scales, workspace) -> y bf16 [M,N]        (fp8bs_gemv_ws)
    gemv_batch([(x, codes, scales[, y]), ...]) -> [y, ...]   (fp8bs_gemv_batch)
    GemvBatch(ops)() -> [y, ...]                  (fp8bs_gemv_batch, op table built once)
    mx_gemv_batch([(x, codes, e8m0[, y]), ...]) -> [y, ...]  (mxfp8_gemv_batch)
    row_quantize(w)        -> (codes u8 [N,K], scales f32 [N])       (fp8row_*)
    tensor_quantize(w)     -> (codes u8 [N,K], scale f32 [1])        (fp8tensor_*)
    row_gemv(x, codes, s)  -> y bf16 [M,N]; s is [N] (per row) or [1] (per tensor)
    act_quantize(x)        -> (x codes u8 [M,K], scale f32 [1])      (fp8act_quantize)
    w8a8_gemm(xq, sx, wq, sw) -> y bf16 [M,N]                        (w8a8_gemm)
    w8a8_linear(x, wq, sw) -> y bf16 [M,N]: act_quantize then w8a8_gemm
    moe_gemv(x, ids, codes, scales) -> y bf16 [M, topk, N]            (fp8bs_moe_gemv)
    moe_gemv_ws(x, ids, codes, scales, workspace) -> y                (fp8bs_moe_gemv_ws)
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


class GemvOp(ctypes.Structure):
    """fp8bs_gemv_op: one GEMV of a batch (device pointers, sizes)."""
    _fields_ = [("x_bf16", ctypes.c_void_p), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("y_bf16", ctypes.c_void_p), ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


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
        L.fp8bs_gemv_ws_bytes.argtypes = [i64, i64]
        L.fp8bs_gemv_ws_bytes.restype = i64
        L.fp8bs_gemv_ws.argtypes = [p, i64, p, p, i64, i64, p, p, i64, p]
        L.fp8bs_gemv_batch.argtypes = [p, i64, i64, p]
        L.fp8bs_gemv_batch_ex.argtypes = [p, i64, i64, i32, p]
        L.mxfp8_gemv_batch.argtypes = [p, i64, i64, p]
        L.mxfp8_gemv_batch_ex.argtypes = [p, i64, i64, i32, p]
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
        L.fp8bs_moe_gemv_ws.argtypes = [p, i64, p, i64, p, p, i64, i64, i64, p, p, i64, p]
        L.fp8bs_moe_gemv_ws_bytes.argtypes = [i64, i64, i64, i64]
        L.fp8bs_moe_gemv_ws_bytes.restype = i64
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
        for f in ("fp8bs_quantize", "fp8bs_gemv", "fp8bs_gemv_ex", "fp8bs_gemv_ws", "fp8bs_gemv_batch",
                  "fp8bs_gemv_batch_ex",
                  "mxfp8_gemv_batch", "mxfp8_gemv_batch_ex", "mxfp8_quantize", "mxfp8_gemv",
                  "mxfp8_gemv_ex", "fp8row_quantize", "fp8tensor_quantize", "fp8row_gemv", "fp8row_gemv_ex",
                  "fp8tensor_gemv", "fp8tensor_gemv_ex", "fp8act_quantize", "w8a8_gemm", "w8a8_gemm_ex",
                  "fp8bs_moe_gemv", "fp8bs_moe_gemv_ws", "fp8kv_append", "fp8kv_decode_attention",
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


def _stream(stream, device=None):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


class _Args:
    """Checks one call's tensors before anything is launched.

    ``need(name, t, dtype, numel=..., shape=...)`` records a tensor; sizes
    are checked first (ValueError, for any device), then that every tensor
    sits on the device of the first one (ValueError), then CUDA, dtype and
    contiguity (TypeError / ValueError).  ``ptr(name)`` gives the device
    address once ``check()`` has passed; ``device`` is where the call runs."""

    def __init__(self):
        self.items = []

    def need(self, name, t, dtype, numel=None, shape=None):
        import torch
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
        if numel is not None and t.numel() != numel:
            raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
        self.items.append((name, t, dtype))
        return self

    def check(self):
        first = self.items[0][1].device
        for name, t, _ in self.items:
            if t.device != first:
                raise ValueError(f"{name} is on {t.device}, the call's tensors on {first}")
        for name, t, dtype in self.items:
            if t.device.type != "cuda":
                raise TypeError(f"{name} must be a CUDA tensor")
            if t.dtype != dtype:
                raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        self.device = first
        self.ptrs = {name: ctypes.c_void_p(t.data_ptr()) for name, t, _ in self.items}
        return self

    def ptr(self, name):
        return self.ptrs[name]


def _run(args: _Args, what: str, fn, *call_args, stream=None):
    """Call the library on the device of the call's tensors, on that
    device's current stream unless one is given."""
    import torch
    with torch.cuda.device(args.device):
        _check(fn(*call_args, _stream(stream, args.device)), what)


def _shape2(t, name):
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got {t.dim()}-D")
    return t.shape


def _new(t, shape, dtype, like):
    import torch
    return torch.empty(shape, dtype=dtype, device=like.device) if t is None else t


def quantize(w, block: int = 128, codes=None, scales=None, stream=None):
    """Block-FP8 load-time quantization of a bf16 [N, K] CUDA tensor."""
    import torch
    n, k = _shape2(w, "w")
    codes = _new(codes, (n, k), torch.uint8, w)
    scales = _new(scales, (cdiv(n, 128), cdiv(k, 128)), torch.float32, w)
    a = _Args().need("w", w, torch.bfloat16).need("codes", codes, torch.uint8, numel=n * k) \
        .need("scales", scales, torch.float32, numel=cdiv(n, 128) * cdiv(k, 128)).check()
    _run(a, "fp8bs_quantize", lib().fp8bs_quantize, a.ptr("w"), n, k, int(block), a.ptr("codes"), a.ptr("scales"),
         stream=stream)
    return codes, scales


def _gemv_args(x, codes, y, scales, sdtype, snumel, check=True):
    import torch
    m, k = _shape2(x, "x")
    n, k2 = _shape2(codes, "codes")
    if k2 != k:
        raise ValueError("codes and x disagree on K")
    y = _new(y, (m, n), torch.bfloat16, x)
    a = _Args().need("x", x, torch.bfloat16).need("codes", codes, torch.uint8) \
        .need("scales", scales, sdtype, numel=snumel(n, k)).need("y", y, torch.bfloat16, numel=m * n)
    return (a.check() if check else a), m, n, k, y


def _block_numel(n, k):
    return cdiv(n, 128) * cdiv(k, 128)


def gemv(x, codes, scales, y=None, path: int = PATH_AUTO, stream=None):
    """y[M, N] = x[M, K] . dequant(codes, scales)^T (bf16 out, fp32 accumulate)."""
    import torch
    a, m, n, k, y = _gemv_args(x, codes, y, scales, torch.float32, _block_numel)
    _run(a, "fp8bs_gemv", lib().fp8bs_gemv_ex, a.ptr("x"), m, a.ptr("codes"), a.ptr("scales"), n, k, a.ptr("y"),
         int(path), stream=stream)
    return y


def gemv_ws_bytes(m: int, k: int) -> int:
    """Bytes of device workspace gemv_ws needs (fp8bs_gemv_ws_bytes)."""
    v = lib().fp8bs_gemv_ws_bytes(m, k)
    if v < 0:
        raise Fp8bsError(int(v), "fp8bs_gemv_ws_bytes")
    return int(v)


def gemv_ws(x, codes, scales, workspace, y=None, stream=None):
    """gemv with caller-provided device scratch (fp8bs_gemv_ws): x is
    converted once per call to f16 in `workspace` (a uint8 CUDA tensor of at
    least gemv_ws_bytes(M, K) bytes) and the decode kernel reads that copy."""
    import torch
    a, m, n, k, y = _gemv_args(x, codes, y, scales, torch.float32, _block_numel, check=False)
    a.need("workspace", workspace, torch.uint8).check()
    _run(a, "fp8bs_gemv_ws", lib().fp8bs_gemv_ws, a.ptr("x"), m, a.ptr("codes"), a.ptr("scales"), n, k, a.ptr("y"),
         a.ptr("workspace"), workspace.numel(), stream=stream)
    return y


def _batch_ops(ops, mx):
    import torch
    arr = (GemvOp * max(1, len(ops)))()
    if not ops:
        return arr, 0, [], None
    m = _shape2(ops[0][0], "x")[0]
    sdtype = torch.uint8 if mx else torch.float32
    snumel = (lambda n, k: n * cdiv(k, 32)) if mx else _block_numel
    # every op's sizes first (nothing about devices), then devices and dtypes
    for i, op in enumerate(ops):
        if _shape2(op[0], f"op {i} x")[0] != m:
            raise ValueError("every op of a batch has the same M")
        if len(op) > 3 and op[3] is not None:
            _gemv_args(op[0], op[1], op[3], op[2], sdtype, snumel, check=False)
        else:
            n = _shape2(op[1], f"op {i} codes")[0]
            _Args().need("scales", op[2], sdtype, numel=snumel(n, op[0].shape[1]))
    first = ops[0][0].device
    for i, op in enumerate(ops):
        for name, tt in zip(("x", "codes", "scales", "y"), op):
            if tt is not None and tt.device != first:
                raise ValueError(f"op {i} {name} is on {tt.device}, the batch on {first}")
    ys = []
    device = None
    for i, op in enumerate(ops):
        y = op[3] if len(op) > 3 else None
        a, _, n, k, y = _gemv_args(op[0], op[1], y, op[2], sdtype, snumel)
        if device is None:
            device = a.device
        elif a.device != device:
            raise ValueError(f"op {i} is on {a.device}, the batch on {device}")
        ys.append(y)
        arr[i] = GemvOp(a.ptr("x").value, a.ptr("codes").value, a.ptr("scales").value, a.ptr("y").value, n, k)
    return arr, m, ys, device


def _run_batch(fn, what, ops, mx, path, stream):
    import torch
    arr, m, ys, device = _batch_ops(ops, mx)
    if not ops:
        return ys
    with torch.cuda.device(device):
        _check(fn(ctypes.cast(arr, ctypes.c_void_p), len(ops), m, int(path), _stream(stream, device)), what)
    return ys


def gemv_batch(ops, path: int = PATH_AUTO, stream=None):
    """A sequence of block-FP8 GEMVs (fp8bs_gemv_batch): ops is a list of
    (x [M,K], codes, scales[, y]) with one M; returns the list of y.  Same
    results as calling gemv on each op in order."""
    return _run_batch(lib().fp8bs_gemv_batch_ex, "fp8bs_gemv_batch", ops, False, path, stream)


class GemvBatch:
    """A prepared sequence of block-FP8 GEMVs (fp8bs_gemv_batch): the op
    table is built once, so calling it only enqueues the launches.  ops as
    for gemv_batch."""

    def __init__(self, ops, path: int = PATH_AUTO):
        self.arr, self.m, self.ys, self.device = _batch_ops(ops, False)
        self.count = len(ops)
        self.path = path
        self.ops = ops  # keeps the tensors alive

    def __call__(self, stream=None):
        import torch
        if not self.count:
            return self.ys
        with torch.cuda.device(self.device):
            _check(lib().fp8bs_gemv_batch_ex(ctypes.cast(self.arr, ctypes.c_void_p), self.count, self.m,
                                             int(self.path), _stream(stream, self.device)), "fp8bs_gemv_batch")
        return self.ys


def mx_gemv_batch(ops, path: int = PATH_AUTO, stream=None):
    """A sequence of MXFP8 GEMVs (mxfp8_gemv_batch): ops is a list of
    (x [M,K], codes, e8m0[, y]) with one M; returns the list of y."""
    return _run_batch(lib().mxfp8_gemv_batch_ex, "mxfp8_gemv_batch", ops, True, path, stream)


def mx_quantize(w, codes=None, e8m0=None, stream=None):
    """MXFP8 load-time quantization of a bf16 [N, K] CUDA tensor."""
    import torch
    n, k = _shape2(w, "w")
    codes = _new(codes, (n, k), torch.uint8, w)
    e8m0 = _new(e8m0, (n, cdiv(k, 32)), torch.uint8, w)
    a = _Args().need("w", w, torch.bfloat16).need("codes", codes, torch.uint8, numel=n * k) \
        .need("e8m0", e8m0, torch.uint8, numel=n * cdiv(k, 32)).check()
    _run(a, "mxfp8_quantize", lib().mxfp8_quantize, a.ptr("w"), n, k, a.ptr("codes"), a.ptr("e8m0"), stream=stream)
    return codes, e8m0


def mx_gemv(x, codes, e8m0, y=None, path: int = PATH_AUTO, stream=None):
    """y[M, N] = x[M, K] . dequant_mx(codes, e8m0)^T."""
    import torch
    a, m, n, k, y = _gemv_args(x, codes, y, e8m0, torch.uint8, lambda n, k: n * cdiv(k, 32))
    _run(a, "mxfp8_gemv", lib().mxfp8_gemv_ex, a.ptr("x"), m, a.ptr("codes"), a.ptr("scales"), n, k, a.ptr("y"),
         int(path), stream=stream)
    return y


def _rowwise_quantize(fn, what, w, codes, scales, count, stream):
    import torch
    n, k = _shape2(w, "w")
    codes = _new(codes, (n, k), torch.uint8, w)
    scales = _new(scales, (count(n),), torch.float32, w)
    a = _Args().need("w", w, torch.bfloat16).need("codes", codes, torch.uint8, numel=n * k) \
        .need("scales", scales, torch.float32, numel=count(n)).check()
    _run(a, what, fn, a.ptr("w"), n, k, a.ptr("codes"), a.ptr("scales"), stream=stream)
    return codes, scales


def row_quantize(w, codes=None, scales=None, stream=None):
    """Per-row FP8 load-time quantization: one fp32 scale per row of w."""
    return _rowwise_quantize(lib().fp8row_quantize, "fp8row_quantize", w, codes, scales, lambda n: n, stream)


def tensor_quantize(w, codes=None, scale=None, stream=None):
    """Per-tensor FP8 load-time quantization: one fp32 scale for all of w."""
    return _rowwise_quantize(lib().fp8tensor_quantize, "fp8tensor_quantize", w, codes, scale, lambda n: 1, stream)


def row_gemv(x, codes, scales, y=None, path: int = PATH_AUTO, stream=None):
    """y[M, N] = x[M, K] . (dec(codes) * s_row)^T.  ``scales`` of shape [N]
    calls fp8row_gemv, of shape [1] fp8tensor_gemv."""
    import torch
    n = _shape2(codes, "codes")[0]
    per_row = tuple(scales.shape) == (n,) and n > 1
    if not per_row and tuple(scales.shape) not in ((1,), ()):
        raise ValueError("scales must have shape [N] (per row) or [1] (per tensor)")
    a, m, n, k, y = _gemv_args(x, codes, y, scales, torch.float32, lambda n, k: n if per_row else 1)
    fn = lib().fp8row_gemv_ex if per_row else lib().fp8tensor_gemv_ex
    _run(a, "fp8row_gemv" if per_row else "fp8tensor_gemv", fn, a.ptr("x"), m, a.ptr("codes"), a.ptr("scales"), n,
         k, a.ptr("y"), int(path), stream=stream)
    return y


def _moe_args(x, ids, codes, scales, y):
    import torch
    m, k = _shape2(x, "x")
    if codes.dim() != 3:
        raise ValueError("codes must be [E, N, K]")
    e, n, k2 = codes.shape
    topk = _shape2(ids, "ids")[1]
    if k2 != k or ids.shape[0] != m:
        raise ValueError("x, ids and codes disagree on M or K")
    y = _new(y, (m, topk, n), torch.bfloat16, x)
    a = _Args().need("x", x, torch.bfloat16).need("ids", ids, torch.int32) \
        .need("codes", codes, torch.uint8) \
        .need("scales", scales, torch.float32, numel=e * cdiv(n, 128) * cdiv(k, 128)) \
        .need("y", y, torch.bfloat16, numel=m * topk * n)
    return a, m, topk, e, n, k, y


def moe_gemv(x, ids, codes, scales, y=None, stream=None):
    """Grouped block-FP8 GEMV over routed experts: y[t, j] = x[t] . dequant(W[ids[t, j]])^T."""
    a, m, topk, e, n, k, y = _moe_args(x, ids, codes, scales, y)
    a.check()
    _run(a, "fp8bs_moe_gemv", lib().fp8bs_moe_gemv, a.ptr("x"), m, a.ptr("ids"), topk, a.ptr("codes"),
         a.ptr("scales"), e, n, k, a.ptr("y"), stream=stream)
    return y


def moe_gemv_ws_bytes(m: int, topk: int, num_experts: int, k: int) -> int:
    """Bytes of device workspace moe_gemv_ws needs (fp8bs_moe_gemv_ws_bytes)."""
    v = lib().fp8bs_moe_gemv_ws_bytes(m, topk, num_experts, k)
    if v < 0:
        raise Fp8bsError(int(v), "fp8bs_moe_gemv_ws_bytes")
    return int(v)


def moe_gemv_ws(x, ids, codes, scales, workspace, y=None, stream=None):
    """moe_gemv with caller-provided device scratch (fp8bs_moe_gemv_ws): more
    than 32 tokens run as one grouped tensor-core GEMM over the routed
    experts; `workspace` is a uint8 CUDA tensor of at least
    moe_gemv_ws_bytes(M, topk, E, K) bytes."""
    import torch
    a, m, topk, e, n, k, y = _moe_args(x, ids, codes, scales, y)
    a.need("workspace", workspace, torch.uint8).check()
    _run(a, "fp8bs_moe_gemv_ws", lib().fp8bs_moe_gemv_ws, a.ptr("x"), m, a.ptr("ids"), topk, a.ptr("codes"),
         a.ptr("scales"), e, n, k, a.ptr("y"), a.ptr("workspace"), workspace.numel(), stream=stream)
    return y


def kv_append(x, slots, scale, cache, stream=None):
    """Quantize new keys or values x [T, Hkv, 128] bf16 into the e4m3 cache
    [num_blocks, page_size, Hkv, 128] at flat token slots (in place)."""
    import torch
    if x.dim() != 3 or cache.dim() != 4:
        raise ValueError("x must be [T, Hkv, 128] and cache [num_blocks, page_size, Hkv, 128]")
    t, hkv, d = x.shape
    nb, page, hkv2, d2 = cache.shape
    if (hkv2, d2) != (hkv, d):
        raise ValueError("x and cache disagree on kv heads or head_dim")
    a = _Args().need("x", x, torch.bfloat16).need("slots", slots, torch.int32, numel=t) \
        .need("scale", scale, torch.float32, numel=1).need("cache", cache, torch.uint8).check()
    _run(a, "fp8kv_append", lib().fp8kv_append, a.ptr("x"), t, hkv, d, a.ptr("slots"), a.ptr("scale"),
         a.ptr("cache"), nb * page, stream=stream)
    return cache


def kv_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, max_seq_len: int,
                        sm_scale: float, out=None, stream=None):
    """Paged decode attention over the FP8 KV cache: q [B, Hq, 128] bf16."""
    import torch
    if q.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("q must be [B, Hq, 128] and the caches [num_blocks, page_size, Hkv, 128]")
    b, hq, d = q.shape
    nb, page, hkv, d2 = k_cache.shape
    bt_rows, max_blocks = _shape2(block_table, "block_table")
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape) or bt_rows != b:
        raise ValueError("q, caches and block table disagree")
    out = _new(out, (b, hq, d), torch.bfloat16, q)
    a = _Args().need("q", q, torch.bfloat16).need("k_cache", k_cache, torch.uint8) \
        .need("v_cache", v_cache, torch.uint8).need("k_scale", k_scale, torch.float32, numel=1) \
        .need("v_scale", v_scale, torch.float32, numel=1).need("block_table", block_table, torch.int32) \
        .need("seq_lens", seq_lens, torch.int32, numel=b).need("out", out, torch.bfloat16, numel=b * hq * d).check()
    _run(a, "fp8kv_decode_attention", lib().fp8kv_decode_attention, a.ptr("q"), a.ptr("k_cache"),
         a.ptr("v_cache"), a.ptr("k_scale"), a.ptr("v_scale"), a.ptr("block_table"), max_blocks,
         a.ptr("seq_lens"), b, hq, hkv, d, page, nb, int(max_seq_len), float(sm_scale), a.ptr("out"), stream=stream)
    return out


def act_quantize(x, codes=None, scale=None, stream=None):
    """Dynamic per-tensor e4m3 quantization of bf16 activations [M, K]."""
    import torch
    m, k = _shape2(x, "x")
    codes = _new(codes, (m, k), torch.uint8, x)
    scale = _new(scale, (1,), torch.float32, x)
    a = _Args().need("x", x, torch.bfloat16).need("codes", codes, torch.uint8, numel=m * k) \
        .need("scale", scale, torch.float32, numel=1).check()
    _run(a, "fp8act_quantize", lib().fp8act_quantize, a.ptr("x"), m, k, a.ptr("codes"), a.ptr("scale"),
         stream=stream)
    return codes, scale


def w8a8_gemm(xq, sx, wq, sw, y=None, path: int = PATH_AUTO, stream=None):
    """y[M, N] = sx * sw * dec(xq) . dec(wq)^T (e4m3 x e4m3, fp32 accumulate, bf16 out)."""
    import torch
    m, k = _shape2(xq, "xq")
    n, k2 = _shape2(wq, "wq")
    if k2 != k:
        raise ValueError("x codes and weight codes disagree on K")
    y = _new(y, (m, n), torch.bfloat16, xq)
    a = _Args().need("xq", xq, torch.uint8).need("sx", sx, torch.float32, numel=1).need("wq", wq, torch.uint8) \
        .need("sw", sw, torch.float32, numel=1).need("y", y, torch.bfloat16, numel=m * n).check()
    _run(a, "w8a8_gemm", lib().w8a8_gemm_ex, a.ptr("xq"), m, a.ptr("sx"), a.ptr("wq"), a.ptr("sw"), n, k,
         a.ptr("y"), int(path), stream=stream)
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
    a = _Args().need("out", out, torch.uint8).check()
    _run(a, "fp8bs_debug_encode_f32", lib().fp8bs_debug_encode_f32, first_bits, count, a.ptr("out"), stream=stream)
    return out


def check_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the kernels' error word."""
    word = ctypes.c_uint32(0)
    st = lib().fp8bs_check_device_error(_stream(stream), ctypes.byref(word))
    if st not in (0, -6):
        raise Fp8bsError(st, "fp8bs_check_device_error")
    return int(word.value)
