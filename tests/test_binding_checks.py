"""The Python binding refuses a call whose tensors do not fit each other
before anything is launched (CPU only).

Sizes are checked first, for tensors on any device, so a wrong-sized scale,
code, exponent or output buffer raises ValueError here without a GPU; with
every size right, a tensor on another device than the call's first tensor
raises ValueError, and CPU tensors raise TypeError ("must be a CUDA
tensor").  The library is never called with such arguments, so a short
buffer can never be read or written past its end by a kernel.
"""
import pytest
import torch

import fp8_block_scaled_02_gb300 as fp8bs

BF, U8, F32, I32 = torch.bfloat16, torch.uint8, torch.float32, torch.int32


def t(shape, dtype, device="cpu"):
    return torch.zeros(shape, dtype=dtype, device=device)


M, N, K = 3, 300, 256
NB, KB = 3, 2          # ceil(300/128), ceil(256/128)


@pytest.mark.parametrize("call", [
    lambda: fp8bs.gemv(t((M, K), BF), t((N, K), U8), t((NB, KB - 1), F32)),           # scales short
    lambda: fp8bs.gemv(t((M, K), BF), t((N, K), U8), t((NB, KB), F32), y=t((M, N - 1), BF)),  # y short
    lambda: fp8bs.gemv(t((M, K), BF), t((N, K + 16), U8), t((NB, KB), F32)),          # K disagrees
    lambda: fp8bs.gemv(t((M, K), BF), t((N * K,), U8), t((NB, KB), F32)),             # codes not 2-D
    lambda: fp8bs.mx_gemv(t((M, K), BF), t((N, K), U8), t((N, K // 32 - 1), U8)),     # e8m0 short
    lambda: fp8bs.quantize(t((N, K), BF), scales=t((NB - 1, KB), F32)),
    lambda: fp8bs.quantize(t((N, K), BF), codes=t((N - 1, K), U8)),
    lambda: fp8bs.mx_quantize(t((N, K), BF), e8m0=t((N, 7), U8)),
    lambda: fp8bs.row_quantize(t((N, K), BF), scales=t((N - 1,), F32)),
    lambda: fp8bs.tensor_quantize(t((N, K), BF), scale=t((2,), F32)),
    lambda: fp8bs.row_gemv(t((M, K), BF), t((N, K), U8), t((N - 1,), F32)),
    lambda: fp8bs.moe_gemv(t((M, K), BF), t((M, 2), I32), t((4, N, K), U8), t((4, NB, KB - 1), F32)),
    lambda: fp8bs.moe_gemv(t((M, K), BF), t((M, 2), I32), t((4, N, K), U8), t((4, NB, KB), F32),
                           y=t((M, 1, N), BF)),
    lambda: fp8bs.moe_gemv(t((M, K), BF), t((M + 1, 2), I32), t((4, N, K), U8), t((4, NB, KB), F32)),
    lambda: fp8bs.act_quantize(t((M, K), BF), scale=t((2,), F32)),
    lambda: fp8bs.w8a8_gemm(t((M, K), U8), t((1,), F32), t((N, K), U8), t((2,), F32)),
    lambda: fp8bs.kv_append(t((4, 8, 128), BF), t((5,), I32), t((1,), F32), t((16, 16, 8, 128), U8)),
    lambda: fp8bs.kv_decode_attention(t((2, 32, 128), BF), t((16, 16, 8, 128), U8), t((16, 16, 8, 128), U8),
                                      t((1,), F32), t((1,), F32), t((2, 4), I32), t((3,), I32), 64, 0.1),
    lambda: fp8bs.gemv_batch([(t((M, K), BF), t((N, K), U8), t((NB, KB), F32)),
                              (t((M + 1, K), BF), t((N, K), U8), t((NB, KB), F32))]),          # M differs
    lambda: fp8bs.gemv_batch([(t((M, K), BF), t((N, K), U8), t((NB, KB), F32)),
                              (t((M, K), BF), t((N, K), U8), t((NB, 1), F32))]),               # op 1 scales short
    lambda: fp8bs.mx_gemv_batch([(t((M, K), BF), t((N, K), U8), t((N, 2), U8))]),
])
def test_size_mismatch_raises_value_error(call):
    with pytest.raises(ValueError):
        call()


def test_tensors_on_different_devices_raise():
    # "meta" stands in for a second device; the sizes are right
    with pytest.raises(ValueError, match="is on"):
        fp8bs.gemv(t((M, K), BF, "meta"), t((N, K), U8), t((NB, KB), F32))
    with pytest.raises(ValueError, match="is on"):
        fp8bs.gemv_batch([(t((M, K), BF), t((N, K), U8), t((NB, KB), F32)),
                          (t((M, K), BF, "meta"), t((N, K), U8, "meta"), t((NB, KB), F32, "meta"))])


def test_right_sizes_on_the_cpu_are_refused_as_not_cuda():
    with pytest.raises(TypeError, match="CUDA"):
        fp8bs.gemv(t((M, K), BF), t((N, K), U8), t((NB, KB), F32))
    with pytest.raises(TypeError, match="CUDA"):
        fp8bs.mx_gemv_batch([(t((M, K), BF), t((N, K), U8), t((N, K // 32), U8))])


def test_wrong_dtype_is_refused():
    with pytest.raises(TypeError):
        fp8bs.gemv(t((M, K), F32, "meta"), t((N, K), U8, "meta"), t((NB, KB), F32, "meta"))
