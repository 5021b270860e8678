"""The C ABI's execution contract on the GPU: every call only enqueues work on
the given stream, allocates nothing and branches on shapes only, so a
sequence of calls captures into a CUDA graph and replays to the same bits;
calls on a side stream order with that stream; m = 0 is a no-op.
"""
import numpy as np
import pytest
import torch

from fp8_block_scaled_02_gb300 import PATH_DECODE, PATH_GENERIC, PATH_PREFILL, inputs

from gpu_helpers import lib_or_skip

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    return lib_or_skip()


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


def test_graph_capture_replays_bit_exact(pkg):
    w = inputs.gaussian_bf16((1000, 1536), 0.02, 1).to(DEV)
    codes, scales = pkg.quantize(w)
    mcodes, e8m0 = pkg.mx_quantize(w)
    rcodes, rscales = pkg.row_quantize(w)
    tcodes, tscale = pkg.tensor_quantize(w)
    E, n, k = 6, 256, 1536
    moe_c = torch.stack([pkg.quantize(inputs.gaussian_bf16((n, k), 0.02, 10 + e).to(DEV))[0] for e in range(E)])
    moe_s = torch.stack([pkg.quantize(inputs.gaussian_bf16((n, k), 0.02, 10 + e).to(DEV))[1] for e in range(E)])
    ids = torch.tensor([[0, 5], [3, 1], [2, 0], [4, 3]], dtype=torch.int32, device=DEV)
    q, kk, vv, tbl, sl = inputs.kv_layer(2, [300, 77], 30, 32, 8, 128, 16, 3, device=DEV)
    kc = torch.zeros((30, 16, 8, 128), dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    ks = torch.tensor([0.01], device=DEV)
    vs = torch.tensor([0.01], device=DEV)
    slots = torch.arange(30 * 16, dtype=torch.int32, device=DEV)
    pkg.kv_append(kk.view(-1, 8, 128), slots, ks, kc)
    pkg.kv_append(vv.view(-1, 8, 128), slots, vs, vc)

    xs = {m: inputs.activations(m, 1536, 20 + m, device=DEV) for m in (1, 4, 13, 40, 300)}
    outs = {}

    def work():
        r = []
        for m, x in xs.items():
            r.append(pkg.gemv(x, codes, scales))
            r.append(pkg.mx_gemv(x, mcodes, e8m0))
            r.append(pkg.row_gemv(x, rcodes, rscales))
            r.append(pkg.row_gemv(x, tcodes, tscale))
            r.append(pkg.w8a8_linear(x, tcodes, tscale))
        r.append(pkg.moe_gemv(xs[4], ids, moe_c, moe_s))
        r.append(pkg.kv_decode_attention(q, kc, vc, ks, vs, tbl, sl, 300, 0.088))
        return r

    eager = work()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        work()  # warm-up on the capture stream (per-device set-up happens here, outside capture)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        captured = work()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert len(eager) == len(captured)
    for i, (a, b) in enumerate(zip(eager, captured)):
        assert same_bits(a, b), i
    assert pkg.check_device_error() == 0


def test_side_stream_orders_with_its_stream(pkg):
    w = inputs.gaussian_bf16((2048, 2048), 0.02, 2).to(DEV)
    x = inputs.activations(8, 2048, 3, device=DEV)
    codes, scales = pkg.quantize(w)
    ref = pkg.gemv(x, codes, scales)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c2, s2 = pkg.quantize(w)
        y2 = pkg.gemv(x, c2, s2, stream=s)
    s.synchronize()
    assert same_bits(ref, y2)


@pytest.mark.parametrize("path", [0, PATH_DECODE, PATH_GENERIC, PATH_PREFILL])
def test_zero_rows_is_a_noop(pkg, path):
    w = inputs.gaussian_bf16((256, 256), 0.02, 4).to(DEV)
    codes, scales = pkg.quantize(w)
    y = torch.full((0, 256), 3.0, dtype=torch.bfloat16, device=DEV)
    pkg.gemv(torch.empty((0, 256), dtype=torch.bfloat16, device=DEV), codes, scales, y=y, path=path)
    rc, rs = pkg.row_quantize(w)
    pkg.row_gemv(torch.empty((0, 256), dtype=torch.bfloat16, device=DEV), rc, rs, y=y, path=path)
    torch.cuda.synchronize()
    assert pkg.check_device_error() == 0


def test_long_ragged_k_all_paths(pkg):
    """k = 7168 + 16: the last K block is 16 wide on every path."""
    import oracle
    from gpu_helpers import bits, check_block_gemv
    n, k = 300, 7184
    w = inputs.gaussian_bf16((n, k), 0.02, 5)
    oc, os_ = oracle.block_quantize(bits(w))
    rows_q = {rb: (oc[rb * 128:rb * 128 + 128], os_[rb]) for rb in range(3)}
    for m, path in ((1, PATH_DECODE), (20, PATH_DECODE), (70, PATH_PREFILL), (3, PATH_GENERIC)):
        x = inputs.activations(m, k, 6 + m)
        y = pkg.gemv(x.to(DEV), torch.from_numpy(oc).to(DEV), torch.from_numpy(os_).to(DEV), path=path)
        check_block_gemv(y, bits(x), rows_q)
