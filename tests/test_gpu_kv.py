"""GPU parity for the FP8 E4M3 paged KV cache (InfiniLM PR #586): the append
bit-exact against the oracle, and split-KV decode attention against the
oracle's fp64 attention on caches the oracle wrote.

Tolerance (a reading; the pages give none for attention): the output is a
convex combination of dequantized values, so every error term scales with
max|V|: fp32 scores and softmax (relative ~1e-6), the attention weights
entering the V sum as f16 (relative 2^-11 each, at most 2^-11 max|V| in
total), fp32 accumulation; then one bf16 rounding.  Checked:
|o - o64| <= 2^-10 max_l |V_l| + 1/2 ulp_bf16(max(|o|, |o64|)).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import inputs
from oracle import tolerance
from oracle.tolerance import bf16_bits_to_f64

from gpu_helpers import bits, lib_or_skip, table

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    return lib_or_skip()


def oracle_layer(batch, lens, blocks, hq, hkv, page, seed):
    """Inputs plus caches written by the oracle's append (all slots)."""
    q, k, v, tbl, sl = inputs.kv_layer(batch, lens, blocks, hq, hkv, 128, page, seed)
    kb, vb = bits(k).reshape(-1, hkv, 128), bits(v).reshape(-1, hkv, 128)
    _, ks = oracle.tensor_quantize(kb.reshape(-1, 128))
    _, vs = oracle.tensor_quantize(vb.reshape(-1, 128))
    slots = np.arange(blocks * page, dtype=np.int32)
    empty = np.zeros((blocks, page, hkv, 128), dtype=np.uint8)
    kc = oracle.kv_append(kb, slots, ks, empty)
    vc = oracle.kv_append(vb, slots, vs, empty)
    return q, kc, vc, ks, vs, tbl, sl


def run(pkg, q, kc, vc, ks, vs, tbl, sl, sm, max_len=None):
    max_len = int(sl.max()) if max_len is None else max_len
    return pkg.kv_decode_attention(q.to(DEV), torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV),
                                   torch.from_numpy(ks).to(DEV), torch.from_numpy(vs).to(DEV), tbl.to(DEV),
                                   sl.to(DEV), max_len, sm)


def check(o_dev, q, kc, vc, ks, vs, tbl, sl, sm):
    o64 = oracle.kv_attention(bits(q), kc, vc, ks, vs, tbl.numpy(), sl.numpy(), sm)
    o = bf16_bits_to_f64(bits(o_dev.cpu()))
    vmax = np.nanmax(np.abs(table()[vc])) * float(vs[0])  # NaN codes may sit in unused slots
    bound = tolerance.kv_attention_bound(o, o64, vmax)
    err = np.abs(o - o64)
    assert np.all(np.isfinite(o))
    assert np.all(err <= bound), (err.max(), (err / bound).max())
    return float((err / bound).max())


# ------------------------------------------------------------------ append
@pytest.mark.parametrize("t,hkv", [(1, 8), (5, 2), (33, 8), (7, 1)])
def test_append_bit_exact(pkg, t, hkv):
    blocks, page = 6, 16
    x = inputs.gaussian_bf16((t, hkv * 128), 1.0, 70 + t).view(t, hkv, 128)
    rng = np.random.default_rng(t)
    slots = rng.choice(blocks * page, size=t, replace=False).astype(np.int32)
    _, s = oracle.tensor_quantize(bits(x).reshape(t, -1))
    cache0 = rng.integers(0, 0x7F, (blocks, page, hkv, 128), dtype=np.uint8)
    want = oracle.kv_append(bits(x), slots, s, cache0)
    cache = torch.from_numpy(cache0).to(DEV)
    pkg.kv_append(x.to(DEV), torch.from_numpy(slots).to(DEV), torch.from_numpy(s).to(DEV), cache)
    assert np.array_equal(cache.cpu().numpy(), want)
    assert pkg.check_device_error() == 0


def test_append_bad_slot_is_skipped_and_reported(pkg):
    x = inputs.gaussian_bf16((2, 128), 1.0, 3).view(2, 1, 128)
    cache = torch.zeros((2, 16, 1, 128), dtype=torch.uint8, device=DEV)
    pkg.kv_append(x.to(DEV), torch.tensor([5, 99], dtype=torch.int32, device=DEV),
                  torch.tensor([0.01], device=DEV), cache)
    assert pkg.check_device_error() != 0
    c = cache.cpu().numpy().reshape(32, 128)
    assert np.any(c[5] != 0) and np.all(np.delete(c, 5, axis=0) == 0)


# --------------------------------------------------------------- attention
@pytest.mark.parametrize("lens", [[1], [15], [16], [17], [100], [1000], [3, 70, 0, 257]])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 2), (4, 1)])
def test_attention_small(pkg, lens, hq, hkv):
    blocks = sum((n + 15) // 16 for n in lens) + 3
    q, kc, vc, ks, vs, tbl, sl = oracle_layer(len(lens), lens, blocks, hq, hkv, 16, len(lens) + hq)
    sm = 1 / np.sqrt(128)
    o = run(pkg, q, kc, vc, ks, vs, tbl, sl, sm)
    check(o, q, kc, vc, ks, vs, tbl, sl, sm)
    assert pkg.check_device_error() == 0


@pytest.mark.parametrize("page", [32, 64, 256])
def test_attention_page_sizes(pkg, page):
    lens = [700, 65, 1]
    blocks = sum((n + page - 1) // page for n in lens) + 2
    q, kc, vc, ks, vs, tbl, sl = oracle_layer(3, lens, blocks, 32, 8, page, page)
    o = run(pkg, q, kc, vc, ks, vs, tbl, sl, 0.0883)
    check(o, q, kc, vc, ks, vs, tbl, sl, 0.0883)


def test_single_token_is_exact(pkg):
    """One token: p = 1, so o = bf16(fl32(dec(v) * v_scale)) exactly."""
    q, kc, vc, ks, vs, tbl, sl = oracle_layer(2, [1, 1], 4, 32, 8, 16, 9)
    o = bits(run(pkg, q, kc, vc, ks, vs, tbl, sl, 0.3).cpu())
    for b in range(2):
        blk = int(tbl[b, 0])
        for h in range(32):
            prod = (table()[vc[blk, 0, h // 4]].astype(np.float32) * vs[0]).astype(np.float32)
            want = np.array([oracle.double_to_bf16(float(v)) for v in prod], dtype=np.uint16)
            assert np.array_equal(o[b, h], want), (b, h)


def test_empty_sequences_give_zero(pkg):
    q, kc, vc, ks, vs, tbl, sl = oracle_layer(3, [0, 40, 0], 6, 32, 8, 16, 10)
    o = run(pkg, q, kc, vc, ks, vs, tbl, sl, 0.1)
    assert int((o[0].view(torch.int16) & 0x7FFF).abs().sum()) == 0
    assert int((o[2].view(torch.int16) & 0x7FFF).abs().sum()) == 0
    check(o, q, kc, vc, ks, vs, tbl, sl, 0.1)


def test_nan_codes_in_unused_slots_do_not_leak(pkg):
    """Slots past a sequence's end inside its last page hold NaN codes."""
    q, kc, vc, ks, vs, tbl, sl = oracle_layer(1, [21], 4, 32, 8, 16, 11)
    blk = int(tbl[0, 1])
    kc[blk, 5:] = 0x7F
    vc[blk, 5:] = 0xFF
    o = run(pkg, q, kc, vc, ks, vs, tbl, sl, 0.1)
    check(o, q, kc, vc, ks, vs, tbl, sl, 0.1)


def test_bad_block_id_is_reported(pkg):
    q, kc, vc, ks, vs, tbl, sl = oracle_layer(1, [40], 4, 32, 8, 16, 12)
    tbl = tbl.clone()
    tbl[0, 1] = 1000
    o = run(pkg, q, kc, vc, ks, vs, tbl, sl, 0.1)
    torch.cuda.synchronize()
    assert pkg.check_device_error() != 0
    assert bool(torch.isfinite(o.float()).all())


@pytest.mark.parametrize("batch,length", [(1, 16384), (8, 4096), (2, 1023)])
def test_attention_full_size(pkg, batch, length):
    """The pages' decode shapes: Qwen3-8B layer (32 q heads, 8 kv heads,
    head_dim 128), page 16, one sequence of 16k tokens or 8 of 4k."""
    lens = [length] * batch
    blocks = batch * ((length + 15) // 16) + 5
    q, kc, vc, ks, vs, tbl, sl = oracle_layer(batch, lens, blocks, 32, 8, 16, batch)
    sm = 1 / np.sqrt(128)
    o = run(pkg, q, kc, vc, ks, vs, tbl, sl, sm)
    check(o, q, kc, vc, ks, vs, tbl, sl, sm)
    assert pkg.check_device_error() == 0


def test_repeat_is_deterministic(pkg):
    q, kc, vc, ks, vs, tbl, sl = oracle_layer(2, [3000, 2000], 400, 32, 8, 16, 13)
    o1 = run(pkg, q, kc, vc, ks, vs, tbl, sl, 0.09)
    o2 = run(pkg, q, kc, vc, ks, vs, tbl, sl, 0.09)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_many_sequences(pkg):
    """More (sequence, kv head) pairs than SMs: no KV split at all."""
    rng = np.random.default_rng(14)
    lens = [int(v) for v in rng.integers(0, 700, 24)]
    blocks = sum((n + 15) // 16 for n in lens) + 4
    q, kc, vc, ks, vs, tbl, sl = oracle_layer(24, lens, blocks, 32, 8, 16, 14)
    o = run(pkg, q, kc, vc, ks, vs, tbl, sl, 0.0883)
    check(o, q, kc, vc, ks, vs, tbl, sl, 0.0883)
    assert pkg.check_device_error() == 0
