"""Pins for the oracle's FP8 KV-cache append and decode attention (CPU only).

InfiniLM PR #586 (Summary): an E4M3 KV cache with per-layer fp32 k_scale /
v_scale for paged attention.  The append is the per-tensor rule with the
given static scale; attention is softmax(q . K^T * sm_scale) . V over the
dequantized cache.  Pins: the per-tensor quantizer's codes, numpy float64
attention on an independently gathered, torch-decoded cache, closed forms
(one token; equal keys -> mean of V; sm_scale = 0 -> mean of V), invariance
under relocating pages, GQA grouping, and empty sequences.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import e4m3_values_torch
from fp8_block_scaled_02_gb300 import inputs


def bits_of(t):
    return inputs.bf16_bits(t)


def quantized_layer(batch, lens, blocks, hq=8, hkv=2, d=128, page=16, seed=0):
    q, k, v, table, sl = inputs.kv_layer(batch, lens, blocks, hq, hkv, d, page, seed)
    kb, vb = bits_of(k), bits_of(v)
    _, ks = oracle.tensor_quantize(kb.reshape(-1, d))
    _, vs = oracle.tensor_quantize(vb.reshape(-1, d))
    slots = np.arange(blocks * page, dtype=np.int32)
    empty = np.zeros((blocks, page, hkv, d), dtype=np.uint8)
    kc = oracle.kv_append(kb.reshape(-1, hkv, d), slots, ks, empty)
    vc = oracle.kv_append(vb.reshape(-1, hkv, d), slots, vs, empty)
    return bits_of(q), kc, vc, ks, vs, table.numpy(), sl.numpy()


def test_append_is_the_per_tensor_rule():
    x = bits_of(inputs.gaussian_bf16((6, 2 * 128), 1.0, 3)).reshape(6, 2, 128)
    codes, s = oracle.tensor_quantize(x.reshape(6, -1))
    cache = np.full((2, 4, 2, 128), 0x11, dtype=np.uint8)
    slots = np.array([7, 0, 3, 4, 1, 6], dtype=np.int32)
    out = oracle.kv_append(x, slots, s, cache)
    flat = out.reshape(8, 2, 128)
    for t, sl in enumerate(slots):
        assert np.array_equal(flat[sl].reshape(-1), codes[t])
    untouched = sorted(set(range(8)) - set(slots.tolist()))
    assert np.all(flat[untouched] == 0x11)


def numpy_attention(q, kc, vc, ks, vs, table, lens, sm):
    t = e4m3_values_torch()
    b, hq, d = q.shape
    _, page, hkv, _ = kc.shape
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = np.zeros((b, hq, d))
    for bi in range(b):
        idx = [table[bi, i // page] * page + i % page for i in range(lens[bi])]
        kk = t[kc.reshape(-1, hkv, d)[idx]] * float(ks[0])
        vv = t[vc.reshape(-1, hkv, d)[idx]] * float(vs[0])
        for h in range(hq):
            g = h // (hq // hkv)
            s = sm * (kk[:, g, :] @ qf[bi, h])
            p = np.exp(s - s.max())
            out[bi, h] = (p / p.sum()) @ vv[:, g, :]
    return out


@pytest.mark.parametrize("lens", [[1], [16], [17, 40], [100, 3, 64]])
def test_vs_numpy(lens):
    q, kc, vc, ks, vs, table, sl = quantized_layer(len(lens), lens, 16, seed=len(lens))
    o = oracle.kv_attention(q, kc, vc, ks, vs, table, sl, 1 / np.sqrt(128))
    ref = numpy_attention(q, kc, vc, ks, vs, table, sl, 1 / np.sqrt(128))
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_single_token_returns_its_value():
    q, kc, vc, ks, vs, table, sl = quantized_layer(1, [1], 4, seed=5)
    o = oracle.kv_attention(q, kc, vc, ks, vs, table, sl, 0.1)
    t = e4m3_values_torch()
    blk = table[0, 0]
    for h in range(8):
        assert np.array_equal(o[0, h], t[vc[blk, 0, h // 4]] * float(vs[0]))


def test_equal_keys_or_zero_scale_give_the_mean_of_v():
    q, kc, vc, ks, vs, table, sl = quantized_layer(1, [37], 4, seed=6)
    t = e4m3_values_torch()
    idx = [table[0, i // 16] * 16 + i % 16 for i in range(37)]
    mean = (t[vc.reshape(-1, 2, 128)[idx]] * float(vs[0])).mean(axis=0)
    o0 = oracle.kv_attention(q, kc, vc, ks, vs, table, sl, 0.0)
    for h in range(8):
        assert np.allclose(o0[0, h], mean[h // 4], rtol=1e-13, atol=1e-15)
    kc2 = kc.copy()
    kc2[:] = kc[table[0, 0], 0]        # every key equal to the first
    o1 = oracle.kv_attention(q, kc2, vc, ks, vs, table, sl, 0.3)
    assert np.allclose(o1, o0, rtol=1e-12, atol=1e-15)


def test_relocating_pages_is_invariant():
    q, kc, vc, ks, vs, table, sl = quantized_layer(2, [33, 20], 8, seed=7)
    o = oracle.kv_attention(q, kc, vc, ks, vs, table, sl, 0.09)
    perm = np.array([5, 2, 7, 0, 3, 6, 1, 4])   # block i moves to perm[i]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    o2 = oracle.kv_attention(q, kc2, vc2, ks, vs, perm[table].astype(np.int32), sl, 0.09)
    assert np.array_equal(o, o2)


def test_gqa_grouping_and_empty_sequence():
    q, kc, vc, ks, vs, table, sl = quantized_layer(2, [20, 0], 4, seed=8)
    q[0, 1] = q[0, 0]                   # heads 0 and 1 share kv head 0
    o = oracle.kv_attention(q, kc, vc, ks, vs, table, sl, 0.09)
    assert np.array_equal(o[0, 0], o[0, 1])
    assert np.all(o[1] == 0)
    kc2 = kc.copy()
    kc2[..., 1, :] ^= 0x08              # perturb kv head 1 only
    o2 = oracle.kv_attention(q, kc2, vc, ks, vs, table, sl, 0.09)
    assert np.array_equal(o2[0, :4], o[0, :4]) and not np.array_equal(o2[0, 4:], o[0, 4:])
