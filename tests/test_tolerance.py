"""The acceptance tests (oracle/tolerance.py) are tight enough to catch the
mistakes a block-FP8 / MXFP8 GEMV or an FP8 KV decode-attention kernel
plausibly makes (CPU only).

GEMV: a kernel-like result in numpy -- fp32 partial sums per K block (block
scales) or per 32-element group (MX), the scale applied to the fp32 partial,
one bf16 rounding at the end -- once correctly and once with one planted
mistake.  Attention: the oracle's own result rounded to bf16, and the oracle
run on inputs that carry one planted mistake.  The acceptance test must pass
the first and reject the second, against the oracle's fp64 result.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import inputs
from oracle import tolerance


def to_bf16_bits(y64: np.ndarray) -> np.ndarray:
    return inputs.bf16_bits(torch.from_numpy(np.ascontiguousarray(y64, dtype=np.float32)).to(torch.bfloat16))


def x_f32(xb):
    return (xb.astype(np.uint32) << 16).view(np.float32)


def kernel_like_block(xb, codes, scales, bug=None):
    """fp32 partial per (row, K block) x scale, fp32 sum, bf16 rounding; `bug`
    plants one mistake."""
    table = oracle.e4m3_decode_table().astype(np.float32)
    x = x_f32(xb)
    m, k = x.shape
    n = codes.shape[0]
    nb, kb_n = scales.shape
    deq = table[codes]                                     # unscaled weights, fp32
    y = np.zeros((m, n), dtype=np.float32)
    for kb in range(kb_n):
        if bug == "drop_last_block" and kb == kb_n - 1:
            continue
        c0, c1 = kb * 128, min(k, kb * 128 + 128)
        xs = x[:, c0:c1]
        if bug == "x_rows_shifted":
            xs = np.roll(xs, 1, axis=0)
        part = xs @ deq[:, c0:c1].T                        # fp32 partial [m, n]
        for rb in range(nb):
            r0, r1 = rb * 128, min(n, rb * 128 + 128)
            s = scales[rb, kb]
            if bug == "next_k_block_scale":
                s = scales[rb, (kb + 1) % kb_n]
            elif bug == "next_row_block_scale":
                s = scales[(rb + 1) % nb, kb]
            elif bug == "transposed_scale_grid":
                s = scales.T.reshape(nb, kb_n)[rb, kb]     # same buffer read with the other stride
            elif bug == "scale_applied_twice":
                s = s * s
            elif bug == "sign_of_one_block" and kb == 1:
                s = -s
            y[:, r0:r1] += np.float32(s) * part[:, r0:r1]
    return to_bf16_bits(y)


def kernel_like_mx(xb, codes, e8m0, bug=None):
    table = oracle.e4m3_decode_table().astype(np.float32)
    x = x_f32(xb)
    m, k = x.shape
    deq = table[codes]
    groups = e8m0.shape[1]
    y = np.zeros((m, codes.shape[0]), dtype=np.float32)
    for g in range(groups):
        c0, c1 = g * 32, min(k, g * 32 + 32)
        part = x[:, c0:c1] @ deq[:, c0:c1].T
        E = e8m0[:, g].astype(np.int64)
        if bug == "next_group_exponent":
            E = e8m0[:, (g + 1) % groups].astype(np.int64)
        elif bug == "bias_126":
            E = E + 1
        y += np.ldexp(np.float32(1.0), (E - 127))[None, :].astype(np.float32) * part
    return to_bf16_bits(y)


@pytest.fixture(scope="module")
def block_case():
    w = inputs.bf16_bits(inputs.gaussian_bf16((384, 704), 0.02, 5))   # 3 x 6 tiles, ragged K
    xb = inputs.bf16_bits(inputs.activations(4, 704, 6))
    codes, scales = oracle.block_quantize(w)
    y64 = oracle.block_gemv(xb, codes, scales)
    wmax = tolerance.block_wmax_rows(codes, scales, np.arange(codes.shape[0]), oracle.e4m3_decode_table())
    return xb, codes, scales, y64, wmax


@pytest.fixture(scope="module")
def mx_case():
    w = inputs.bf16_bits(inputs.gaussian_bf16((256, 704), 0.02, 7))
    xb = inputs.bf16_bits(inputs.activations(4, 704, 8))
    codes, e8m0 = oracle.mx_quantize(w)
    y64 = oracle.mx_gemv(xb, codes, e8m0)
    wmax = tolerance.mx_wmax_rows(codes, e8m0, oracle.e4m3_decode_table())
    return xb, codes, e8m0, y64, wmax


def test_correct_block_kernel_passes(block_case):
    xb, codes, scales, y64, wmax = block_case
    st = tolerance.gemv_errors(kernel_like_block(xb, codes, scales), y64, xb, wmax)
    assert tolerance.gemv_ok(st), st


@pytest.mark.parametrize("bug", ["drop_last_block", "x_rows_shifted", "next_k_block_scale",
                                 "next_row_block_scale", "transposed_scale_grid", "scale_applied_twice",
                                 "sign_of_one_block"])
def test_block_kernel_mistakes_fail(block_case, bug):
    xb, codes, scales, y64, wmax = block_case
    st = tolerance.gemv_errors(kernel_like_block(xb, codes, scales, bug), y64, xb, wmax)
    assert not tolerance.gemv_ok(st), (bug, st)


def test_correct_mx_kernel_passes(mx_case):
    xb, codes, e8m0, y64, wmax = mx_case
    st = tolerance.gemv_errors(kernel_like_mx(xb, codes, e8m0), y64, xb, wmax)
    assert tolerance.gemv_ok(st), st


@pytest.mark.parametrize("bug", ["next_group_exponent", "bias_126"])
def test_mx_kernel_mistakes_fail(mx_case, bug):
    xb, codes, e8m0, y64, wmax = mx_case
    st = tolerance.gemv_errors(kernel_like_mx(xb, codes, e8m0, bug), y64, xb, wmax)
    assert not tolerance.gemv_ok(st), (bug, st)


# ------------------------------------------------------ decode attention
@pytest.fixture(scope="module")
def kv_case():
    hq, hkv, page, blocks = 8, 2, 16, 16
    q, k, v, tbl, sl = inputs.kv_layer(2, [37, 70], blocks, hq, hkv, 128, page, seed=3)
    kb = inputs.bf16_bits(k).reshape(-1, hkv, 128)
    vb = inputs.bf16_bits(v).reshape(-1, hkv, 128)
    _, ks = oracle.tensor_quantize(kb.reshape(-1, 128))
    _, vs = oracle.tensor_quantize(vb.reshape(-1, 128))
    slots = np.arange(blocks * page, dtype=np.int32)
    empty = np.zeros((blocks, page, hkv, 128), dtype=np.uint8)
    kc = oracle.kv_append(kb, slots, ks, empty)
    vc = oracle.kv_append(vb, slots, vs, empty)
    qb = inputs.bf16_bits(q)
    sm = 128 ** -0.5
    o64 = oracle.kv_attention(qb, kc, vc, ks, vs, tbl.numpy(), sl.numpy(), sm)
    vmax = np.abs(oracle.e4m3_decode_table()[vc]).max() * float(vs[0])
    return dict(q=qb, kc=kc, vc=vc, ks=ks, vs=vs, tbl=tbl.numpy(), sl=sl.numpy(), sm=sm, o64=o64, vmax=vmax)


def kv_accepts(c, o):
    o_bf16 = tolerance.bf16_bits_to_f64(to_bf16_bits(o))
    return bool(np.all(np.abs(o_bf16 - c["o64"]) <= tolerance.kv_attention_bound(o_bf16, c["o64"], c["vmax"])))


def test_correct_attention_passes(kv_case):
    assert kv_accepts(kv_case, kv_case["o64"])


@pytest.mark.parametrize("bug", ["k_scale_twice", "v_scale_missing", "last_token_dropped", "gqa_head_shifted",
                                 "no_sm_scale", "block_table_shifted"])
def test_attention_mistakes_fail(kv_case, bug):
    c = dict(kv_case)
    q, ks, vs, tbl, sl, sm = c["q"], c["ks"], c["vs"], c["tbl"].copy(), c["sl"].copy(), c["sm"]
    if bug == "k_scale_twice":
        ks = ks * ks
    elif bug == "v_scale_missing":
        vs = np.ones_like(vs)
    elif bug == "last_token_dropped":
        sl = sl - 1
    elif bug == "gqa_head_shifted":
        q = np.roll(q, 4, axis=1)          # query head h read as the group of head h + 4
    elif bug == "no_sm_scale":
        sm = 1.0
    elif bug == "block_table_shifted":
        tbl = np.roll(tbl, 1, axis=1)
    o = oracle.kv_attention(q, c["kc"], c["vc"], ks, vs, tbl, sl, sm)
    assert not kv_accepts(kv_case, o), bug


# ------------------------------------------------- the rel-L2 count threshold
def test_one_correctly_rounded_output_can_exceed_the_rel_l2_bar():
    """The premise of REL_L2_MIN_COUNT: rounding ONE exact result to the
    nearest bf16 (the oracle's own rounding, ties to even) can leave a
    relative error of almost 2^-8 = 3.9e-3, above the 2e-3 bar.  So rel-L2
    is a statistic over many outputs: a one-output GEMV that rounds
    correctly must pass (element-wise bound only), and would fail if rel-L2
    applied to it."""
    y64 = np.array([[1.0 + 2.0 ** -8 - 2.0 ** -30]])          # just below the midpoint of 1 and 1 + 2^-7
    yb = np.array([[oracle.double_to_bf16(float(y64[0, 0]))]], dtype=np.uint16)
    assert yb[0, 0] == 0x3F80                                   # rounds to 1.0
    x = np.array([[0x3F80]], dtype=np.uint16)                   # x = 1, K = 1
    st = tolerance.gemv_errors(yb, y64, x, np.array([float(y64[0, 0])]))
    assert st["rel_l2"] > 3.8e-3 > 2e-3
    assert st["max_ratio"] <= 1.0
    assert tolerance.gemv_ok(st)
    assert st["count"] < tolerance.REL_L2_MIN_COUNT
    # the same single output counted as part of a large output would fail
    assert not tolerance.gemv_ok(dict(st, count=tolerance.REL_L2_MIN_COUNT))


def test_threshold_count_of_correctly_rounded_outputs_meets_the_bar():
    """At the threshold itself the statistic is reliable: 400 seeded draws
    of 256 N(0,1) results, each rounded correctly by the oracle, all stay
    below 2e-3 (the worst draw is reported), so REL_L2_MIN_COUNT does not
    exempt outputs large enough for rel-L2 to mean something."""
    rng = np.random.default_rng(11)
    n = tolerance.REL_L2_MIN_COUNT
    worst = 0.0
    for _ in range(400):
        y64 = rng.standard_normal((1, n))
        yb = oracle.to_bf16_bits(y64)
        y = tolerance.bf16_bits_to_f64(yb)
        worst = max(worst, float(np.linalg.norm(y - y64) / np.linalg.norm(y64)))
    assert worst < 2e-3, worst


def test_a_256_output_row_can_miss_the_bar_when_rounded_correctly():
    """The statistic is reliable over a call's outputs, not over every row of
    256: in the grouped-MoE case with activations near 1e-35 (8 experts of
    [256, 1024] from the seeded generators, top-2 routing of 64 tokens), the
    correctly rounded bf16 of the fp64 result of token 40, slot 0 alone has
    relative L2 error just above 2e-3 while every element meets its bound;
    over all 128 (token, slot) rows of the call the statistic is far below
    the bar.  This is why the MoE parity tests take relative L2 over the
    call."""
    e_count, n, k, m, topk = 8, 256, 1024, 64, 2
    codes, scales = [], []
    for i in range(e_count):
        c, s = oracle.block_quantize(inputs.bf16_bits(inputs.gaussian_bf16((n, k), 0.02, 61 + i)))
        codes.append(c)
        scales.append(s)
    codes, scales = np.stack(codes), np.stack(scales)
    rng = np.random.default_rng(17)
    ids = np.stack([rng.choice(e_count, size=topk, replace=False) for _ in range(m)]).astype(np.int32)
    g = torch.Generator().manual_seed(6)
    xb = inputs.bf16_bits((torch.randn((m, k), generator=g) * 1e-35).to(torch.bfloat16))
    y64 = oracle.moe_gemv(xb, ids, codes, scales)                 # [m, topk, n]
    yb = oracle.to_bf16_bits(y64.reshape(m * topk, n)).reshape(m, topk, n)
    table = oracle.e4m3_decode_table()
    e = ids[40, 0]
    wmax = tolerance.block_wmax_rows(codes[e], scales[e], np.arange(n), table)
    st = tolerance.gemv_errors(yb[40, 0][None, :], y64[40, 0][None, :], xb[40][None, :], wmax)
    assert st["count"] == tolerance.REL_L2_MIN_COUNT
    assert st["max_ratio"] <= 1.0 and st["rel_l2"] > 2e-3, st
    y = tolerance.bf16_bits_to_f64(yb)
    assert float(np.linalg.norm(y - y64) / np.linalg.norm(y64)) < 1.8e-3
