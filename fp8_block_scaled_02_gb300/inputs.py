"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds random-number generation only -- none of the method's
arithmetic -- so both the CUDA path and the CPU oracle can consume the very
same tensors.  Every generator takes an explicit seed and a device; on a
given device the output is a pure function of (shape, seed).

Workloads (the weight shapes the pages measure):
  * tiny ragged       W [320, 704] ~ N(0, 0.02^2), 4 outliers of +-1.5
  * lm_head           W [152064, 4096], rows N(0, 0.02^2) * r_n,
                      r_n log-uniform in [0.5, 2]          (FreeToken PR #636)
  * rotation          48 layers x {[8192,2560], [2560,3072], [6656,2560],
                      [2560,3072]} ~ N(0, 0.02^2)           (FreeToken PR #389)
  * sweep / prefill   W [12288, 4096] ~ N(0, 0.02^2)
  * MXFP8             W [18432, 7168] ~ N(0, 0.02^2) with 0.1% of entries
                      replaced by 0.02 * t_3 (Student t, 3 d.o.f.)
  * activations       x [M, K] ~ N(0, 1)
All tensors are produced in fp32 and rounded once to bf16 (nearest-even).
"""
from __future__ import annotations

import math

import torch

WEIGHT_STD = 0.02

TINY_SHAPE = (320, 704)
LM_HEAD_SHAPE = (152064, 4096)
ROTATION_SHAPES = ((8192, 2560), (2560, 3072), (6656, 2560), (2560, 3072))
ROTATION_LAYERS = 48
SWEEP_SHAPE = (12288, 4096)
MX_SHAPE = (18432, 7168)
MOE_EXPERTS = 256            # routed experts; top-12 of 256 per token (Atlas quantize_fp8_bs.rs notes)
MOE_TOPK = 12
MOE_SHAPE = (2048, 4096)     # [n, k] of one expert's projection


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def gaussian_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def activations(m: int, k: int, seed: int, device="cpu") -> torch.Tensor:
    """x [M, K] bf16 ~ N(0, 1)."""
    return gaussian_bf16((m, k), 1.0, seed, device)


def tiny_ragged_weight(seed: int = 0, device="cpu") -> torch.Tensor:
    """[320, 704] ~ N(0, 0.02^2) with 4 outliers (+1.5, -1.5, +1.5, -1.5)
    at seeded distinct positions."""
    n, k = TINY_SHAPE
    g = _gen(seed, device)
    t = torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * WEIGHT_STD
    pos = torch.randperm(n * k, generator=g, device=device)[:4]
    vals = torch.tensor([1.5, -1.5, 1.5, -1.5], device=device)
    t.view(-1)[pos] = vals
    return t.to(torch.bfloat16)


def tiny_ragged_outliers(seed: int = 0):
    """(row, col, value) of the 4 outliers of tiny_ragged_weight(seed) on CPU."""
    n, k = TINY_SHAPE
    g = _gen(seed, "cpu")
    torch.randn((n, k), generator=g, dtype=torch.float32)
    pos = torch.randperm(n * k, generator=g)[:4].tolist()
    return [(p // k, p % k, v) for p, v in zip(pos, (1.5, -1.5, 1.5, -1.5))]


def lm_head_weight(seed: int = 2, device="cpu", shape=LM_HEAD_SHAPE) -> torch.Tensor:
    """rows N(0, 0.02^2) scaled by r_n, r_n log-uniform in [0.5, 2]."""
    n, k = shape
    g = _gen(seed, device)
    t = torch.randn((n, k), generator=g, device=device, dtype=torch.float32)
    u = torch.rand((n, 1), generator=g, device=device, dtype=torch.float32)
    r = torch.exp(math.log(0.5) + u * (math.log(2.0) - math.log(0.5)))
    t.mul_(WEIGHT_STD * r)
    return t.to(torch.bfloat16)


def rotation_weight(layer: int, j: int, device="cpu") -> torch.Tensor:
    """Weight j (0..3) of rotation layer `layer`; each has its own seed."""
    shape = ROTATION_SHAPES[j]
    return gaussian_bf16(shape, WEIGHT_STD, 1000 + 4 * layer + j, device)


def sweep_weight(copy: int = 0, device="cpu") -> torch.Tensor:
    return gaussian_bf16(SWEEP_SHAPE, WEIGHT_STD, 4000 + copy, device)


def heavy_tail_weight(seed: int = 5, device="cpu", shape=MX_SHAPE,
                      frac: float = 0.001) -> torch.Tensor:
    """N(0, 0.02^2) with round(frac*N*K) seeded positions replaced by
    0.02 * t_3, where t_3 = z / sqrt(chi2_3 / 3)."""
    n, k = shape
    g = _gen(seed, device)
    t = torch.randn((n, k), generator=g, device=device, dtype=torch.float32)
    t.mul_(WEIGHT_STD)
    cnt = max(1, int(round(frac * n * k)))
    pos = torch.randint(0, n * k, (cnt,), generator=g, device=device)
    z = torch.randn((cnt,), generator=g, device=device, dtype=torch.float32)
    c = torch.randn((cnt, 3), generator=g, device=device, dtype=torch.float32)
    t3 = z / torch.sqrt((c * c).sum(dim=1) / 3.0)
    t.view(-1)[pos] = WEIGHT_STD * t3
    return t.to(torch.bfloat16)


def moe_expert_weight(e: int, device="cpu", shape=MOE_SHAPE) -> torch.Tensor:
    """Expert e's bf16 [n, k] weight ~ N(0, 0.02^2), seed 6000 + e."""
    return gaussian_bf16(shape, 0.02, 6000 + e, device)


def moe_routing(m: int, topk: int = MOE_TOPK, experts: int = MOE_EXPERTS, seed: int = 0) -> torch.Tensor:
    """int32 [m, topk] expert ids, distinct within each token (a top-k
    selection), uniformly random with the given seed."""
    g = _gen(7000 + seed, "cpu")
    return torch.stack([torch.randperm(experts, generator=g)[:topk] for _ in range(m)]).to(torch.int32)


# FP8 KV cache decode attention (InfiniLM PR #586's paged FP8 KV cache on a
# Qwen3-8B-shaped layer: 32 query heads, 8 KV heads, head_dim 128).
KV_Q_HEADS = 32
KV_HEADS = 8
KV_HEAD_DIM = 128
KV_PAGE = 16


def kv_layer(batch: int, seq_lens, num_blocks: int, q_heads: int = KV_Q_HEADS, kv_heads: int = KV_HEADS,
             head_dim: int = KV_HEAD_DIM, page_size: int = KV_PAGE, seed: int = 0, device="cpu"):
    """Seeded inputs of one decode-attention call: q [B, Hq, D] ~ N(0, 1),
    bf16 keys / values [num_blocks, page_size, Hkv, D] ~ N(0, 1), and a block
    table [B, max_blocks] int32 that gives every sequence its own randomly
    chosen, randomly ordered blocks (max_blocks = the longest sequence's
    block count; unused entries 0)."""
    lens = [int(v) for v in seq_lens]
    need = [(n + page_size - 1) // page_size for n in lens]
    max_blocks = max(1, max(need))
    assert sum(need) <= num_blocks
    g = _gen(9000 + seed, "cpu")
    q = torch.randn((batch, q_heads, head_dim), generator=g).to(torch.bfloat16)
    k = torch.randn((num_blocks, page_size, kv_heads, head_dim), generator=g).to(torch.bfloat16)
    v = torch.randn((num_blocks, page_size, kv_heads, head_dim), generator=g).to(torch.bfloat16)
    perm = torch.randperm(num_blocks, generator=g)
    table = torch.zeros((batch, max_blocks), dtype=torch.int32)
    off = 0
    for b in range(batch):
        table[b, :need[b]] = perm[off:off + need[b]].to(torch.int32)
        off += need[b]
    dev = torch.device(device)
    return (q.to(dev), k.to(dev), v.to(dev), table.to(dev),
            torch.tensor(lens, dtype=torch.int32).to(dev))


def bf16_bits(t: torch.Tensor):
    """CPU numpy uint16 view of a bf16 tensor (copying from the device if needed)."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
