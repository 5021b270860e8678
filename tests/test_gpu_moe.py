"""GPU parity for the grouped MoE block-FP8 GEMV (Atlas quantize_fp8_bs.rs:
routed experts as block-FP8 weights): every (token, slot) output within the
tolerance of oracle/tolerance.py against the oracle's per-expert fp64 GEMV,
one-hot columns exact, out-of-range ids reported and left unwritten, and
only the selected experts' outputs depend on their weights.

The experts' codes and scales come from the oracle's quantizer (small
cases) or are installed from it for the sampled experts (full size).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_scaled_02_gb300 import inputs
from oracle import tolerance

from gpu_helpers import bits, guard_intact, guarded_empty, lib_or_skip, table

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pkg():
    return lib_or_skip()


def experts(e, n, k, seed):
    codes, scales = [], []
    for i in range(e):
        c, s = oracle.block_quantize(bits(inputs.gaussian_bf16((n, k), 0.02, seed + i)))
        codes.append(c)
        scales.append(s)
    return np.stack(codes), np.stack(scales)


def route(m, topk, e, seed):
    """Distinct experts per token (top-k routing), seeded."""
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(e, size=topk, replace=False) for _ in range(m)]).astype(np.int32)


def check(y_dev, x_bits, ids, codes, scales):
    m, topk = ids.shape
    y64 = oracle.moe_gemv(x_bits, ids, codes, scales)
    yb = bits(y_dev.cpu())
    for t in range(m):
        for j in range(topk):
            e = ids[t, j]
            s = np.repeat(scales[e].astype(np.float64), 128, axis=0)[:codes.shape[1]]
            wmax = np.abs(table()[codes[e]] * np.repeat(s, 128, axis=1)[:, :codes.shape[2]]).max(axis=1)
            st = tolerance.gemv_errors(yb[t, j][None, :], y64[t, j][None, :], x_bits[t][None, :], wmax)
            assert tolerance.gemv_ok(st), (t, j, st)


@pytest.mark.parametrize("m", [1, 2, 5, 8, 9, 16, 17, 32, 33])
@pytest.mark.parametrize("E,n,k,topk", [(8, 256, 512, 2), (16, 320, 704, 4), (6, 130, 256, 6), (32, 128, 128, 12)])
def test_moe_small(pkg, m, E, n, k, topk):
    codes, scales = experts(E, n, k, 100 + E + n)
    ids = route(m, topk, E, m + E)
    x = inputs.activations(m, k, 3 + m)
    y, raw = guarded_empty((m, topk, n), torch.bfloat16, DEV)
    pkg.moe_gemv(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(codes).to(DEV),
                 torch.from_numpy(scales).to(DEV), y=y)
    torch.cuda.synchronize()
    assert guard_intact(raw, m * topk * n * 2)
    check(y, bits(x), ids, codes, scales)
    assert pkg.check_device_error() == 0


def test_one_hot_exact(pkg):
    """x = e_c: y[t, j, r] = bf16(fl32(dec(q_e[r, c]) * s_e[r/128, c/128]))."""
    E, n, k = 4, 200, 256
    codes, scales = experts(E, n, k, 7)
    ids = np.array([[3, 1], [0, 2], [2, 3]], dtype=np.int32)
    cols = [5, 130, 255]
    x = np.zeros((3, k), dtype=np.uint16)
    for t, c in enumerate(cols):
        x[t, c] = 0x3F80
    y = pkg.moe_gemv(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(DEV), torch.from_numpy(ids).to(DEV),
                     torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV))
    yb = bits(y.cpu())
    for t, c in enumerate(cols):
        for j in range(2):
            e = ids[t, j]
            prod = (table()[codes[e][:, c]].astype(np.float32) * scales[e][np.arange(n) // 128, c // 128]).astype(np.float32)
            want = np.array([oracle.double_to_bf16(0.0 + float(v)) for v in prod], dtype=np.uint16)
            assert np.array_equal(yb[t, j], want), (t, j)


def test_out_of_range_id_sets_error_and_skips(pkg):
    E, n, k = 4, 128, 128
    codes, scales = experts(E, n, k, 9)
    ids = np.array([[1, 9], [-3, 2]], dtype=np.int32)
    x = inputs.activations(2, k, 4)
    y = torch.full((2, 2, n), 7.0, dtype=torch.bfloat16, device=DEV)
    pkg.moe_gemv(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(codes).to(DEV),
                 torch.from_numpy(scales).to(DEV), y=y)
    assert pkg.check_device_error() != 0
    yc = y.cpu().float()
    assert torch.all(yc[0, 1] == 7.0) and torch.all(yc[1, 0] == 7.0)
    y64 = oracle.moe_gemv(bits(x), np.where((ids >= 0) & (ids < E), ids, 0).astype(np.int32), codes, scales)
    for t, j in ((0, 0), (1, 1)):
        st = tolerance.gemv_errors(bits(y[t, j][None, :].cpu()), y64[t, j][None, :], bits(x)[t][None, :],
                                   np.full(n, np.abs(table()[codes]).max() * scales.max()))
        assert tolerance.gemv_ok(st)


def test_duplicate_id_within_a_token_sets_error(pkg):
    """ids of one token must be distinct (a top-k selection); a token that
    lists an expert twice is flagged in the device error word (only its
    lowest slot is written), and the other tokens' outputs are unaffected."""
    E, n, k = 4, 128, 128
    codes, scales = experts(E, n, k, 10)
    ids = np.array([[2, 2], [0, 3]], dtype=np.int32)
    x = inputs.activations(2, k, 5)
    y = torch.full((2, 2, n), 7.0, dtype=torch.bfloat16, device=DEV)
    pkg.moe_gemv(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(codes).to(DEV),
                 torch.from_numpy(scales).to(DEV), y=y)
    assert pkg.check_device_error() & 16       # ERRBIT_INDEX
    y64 = oracle.moe_gemv(bits(x), ids, codes, scales)
    for t, j in ((0, 0), (1, 0), (1, 1)):
        st = tolerance.gemv_errors(bits(y[t, j][None, :].cpu()), y64[t, j][None, :], bits(x)[t][None, :],
                                   np.full(n, np.abs(table()[codes]).max() * scales.max()))
        assert tolerance.gemv_ok(st)
    assert torch.all(y[0, 1].cpu().float() == 7.0)
    assert pkg.check_device_error() == 0       # reading cleared it


def test_unselected_experts_are_not_read(pkg):
    """Poisoning the weights of experts no token selected changes nothing."""
    E, n, k = 8, 128, 256
    codes, scales = experts(E, n, k, 11)
    ids = np.array([[0, 5], [5, 2]], dtype=np.int32)
    x = inputs.activations(2, k, 6).to(DEV)
    c = torch.from_numpy(codes).to(DEV)
    s = torch.from_numpy(scales).to(DEV)
    i = torch.from_numpy(ids).to(DEV)
    y1 = pkg.moe_gemv(x, i, c, s)
    for e in (1, 3, 4, 6, 7):
        c[e] = 0x7E
        s[e] = 1e30
    y2 = pkg.moe_gemv(x, i, c, s)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_full_size_sampled(pkg):
    """256 experts of [2048, 4096] (2.1 GB of codes), top-12, M = 1, 8, 16:
    the oracle checks the slots of a few sampled experts, whose codes and
    scales are installed from the oracle's quantizer."""
    E, n, k, topk = 256, 2048, 4096, 12
    w_all = torch.empty((E, n, k), dtype=torch.uint8, device=DEV)
    s_all = torch.empty((E, n // 128, k // 128), dtype=torch.float32, device=DEV)
    for e in range(E):
        c, s = pkg.quantize(inputs.moe_expert_weight(e, device=DEV))
        w_all[e] = c
        s_all[e] = s
    sample = [0, 17, 255]
    oc, os_ = experts_from(sample)
    for i, e in enumerate(sample):
        w_all[e] = torch.from_numpy(oc[i]).to(DEV)
        s_all[e] = torch.from_numpy(os_[i]).to(DEV)
    for m in (1, 8, 16):
        ids = inputs.moe_routing(m, topk, E, seed=m).numpy()
        for i, e in enumerate(sample):  # make sure every sampled expert is selected
            t = i % m
            if e not in ids[t]:
                ids[t, i] = e
        x = inputs.activations(m, k, 60 + m)
        y = pkg.moe_gemv(x.to(DEV), torch.from_numpy(ids).to(DEV), w_all, s_all)
        torch.cuda.synchronize()
        yb = bits(y.cpu())
        xb = bits(x)
        for i, e in enumerate(sample):
            for t, j in zip(*np.nonzero(ids == e)):
                y64 = oracle.block_gemv(xb[t][None, :], oc[i], os_[i])
                wmax = tolerance.block_wmax_rows(oc[i], os_[i], np.arange(n), table())
                st = tolerance.gemv_errors(yb[t, j][None, :], y64, xb[t][None, :], wmax)
                assert tolerance.gemv_ok(st), (m, e, t, j, st)
    assert pkg.check_device_error() == 0


def experts_from(sample):
    codes, scales = [], []
    for e in sample:
        c, s = oracle.block_quantize(bits(inputs.moe_expert_weight(e)))
        codes.append(c)
        scales.append(s)
    return codes, scales


# ------------------------------------------- grouped tensor-core GEMM (m > 32)
def ws(pkg, m, topk, e, k):
    """A routing workspace, pre-filled with garbage: its contents on entry
    must not matter."""
    return torch.full((max(1, pkg.moe_gemv_ws_bytes(m, topk, e, k)),), 0xA5, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("m", [33, 64, 130, 300])
@pytest.mark.parametrize("E,n,k,topk", [(8, 256, 512, 2), (16, 320, 704, 4), (6, 130, 256, 6), (32, 128, 128, 12)])
def test_moe_grouped_small(pkg, m, E, n, k, topk):
    codes, scales = experts(E, n, k, 100 + E + n)
    ids = route(m, topk, E, m + E)
    x = inputs.activations(m, k, 3 + m)
    y, raw = guarded_empty((m, topk, n), torch.bfloat16, DEV)
    pkg.moe_gemv_ws(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(codes).to(DEV),
                    torch.from_numpy(scales).to(DEV), ws(pkg, m, topk, E, k), y=y)
    torch.cuda.synchronize()
    assert guard_intact(raw, m * topk * n * 2)
    check(y, bits(x), ids, codes, scales)
    assert pkg.check_device_error() == 0


def test_moe_grouped_many_tiles_per_expert(pkg):
    """Skewed routing: every token picks experts 0 and 1 (300 pairs each, two
    256-pair tiles per expert, the second partial), the other experts get
    none and their weights are NaN codes that must never be read."""
    E, n, k, m, topk = 4, 256, 512, 300, 2
    codes, scales = experts(E, n, k, 77)
    codes[2:] = 0x7F
    ids = np.tile(np.array([[0, 1]], dtype=np.int32), (m, 1))
    ids[::3] = ids[::3, ::-1]
    x = inputs.activations(m, k, 9)
    y = pkg.moe_gemv_ws(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(codes).to(DEV),
                        torch.from_numpy(scales).to(DEV), ws(pkg, m, topk, E, k))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y.float()).all())
    check(y, bits(x), ids, codes, scales)
    assert pkg.check_device_error() == 0


def test_moe_grouped_pair_counts_across_box_and_mma_edges(pkg):
    """One routing whose experts receive pair counts on both sides of every
    32-row x box, 16-wide MMA-N step, 64-column epilogue half and 128-pair
    expert tile edge (up to three tiles per expert; tokens shuffled): each
    expert tile loads only the x boxes holding its pairs and runs its MMAs
    at N = pairs rounded up to 16; every output is checked in full."""
    counts = [1, 15, 16, 17, 31, 32, 33, 0, 63, 64, 65, 127, 128, 129, 191, 192, 193, 255, 256, 257, 383, 384, 385, 5]
    E, n, k = len(counts), 256, 512
    codes, scales = experts(E, n, k, 41)
    ids = np.repeat(np.arange(E, dtype=np.int32), counts)
    np.random.default_rng(8).shuffle(ids)
    ids = ids[:, None]
    m = ids.shape[0]
    x = inputs.activations(m, k, 12)
    y, raw = guarded_empty((m, 1, n), torch.bfloat16, DEV)
    pkg.moe_gemv_ws(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(codes).to(DEV),
                    torch.from_numpy(scales).to(DEV), ws(pkg, m, 1, E, k), y=y)
    torch.cuda.synchronize()
    assert guard_intact(raw, m * n * 2)
    yb, xb = bits(y.cpu()), bits(x)
    for e in range(E):
        toks = np.nonzero(ids[:, 0] == e)[0]
        assert len(toks) == counts[e]
        if not len(toks):
            continue
        y64 = oracle.block_gemv(xb[toks], codes[e], scales[e])
        wmax = tolerance.block_wmax_rows(codes[e], scales[e], np.arange(n), table())
        st = tolerance.gemv_errors(yb[toks, 0], y64, xb[toks], wmax)
        assert tolerance.gemv_ok(st), (e, counts[e], st)
    assert pkg.check_device_error() == 0


def test_moe_grouped_decode_tile_edges(pkg):
    """Few pairs per expert on average (pairs <= 32 * E): the call streams each
    selected expert once per tile of up to 32 of its pairs through the decode
    kernel.  Counts on both sides of the 32- and 64-pair tile edges, plus
    experts nobody picked; every output checked in full."""
    counts = [1, 31, 32, 33, 63, 64, 65, 0, 5, 96, 97] + [0] * 29
    E, n, k = len(counts), 256, 512
    assert sum(counts) <= 32 * E
    codes, scales = experts(E, n, k, 43)
    ids = np.repeat(np.arange(E, dtype=np.int32), counts)
    np.random.default_rng(9).shuffle(ids)
    ids = ids[:, None]
    m = ids.shape[0]
    x = inputs.activations(m, k, 14)
    y, raw = guarded_empty((m, 1, n), torch.bfloat16, DEV)
    pkg.moe_gemv_ws(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(codes).to(DEV),
                    torch.from_numpy(scales).to(DEV), ws(pkg, m, 1, E, k), y=y)
    torch.cuda.synchronize()
    assert guard_intact(raw, m * n * 2)
    yb, xb = bits(y.cpu()), bits(x)
    for e in range(E):
        toks = np.nonzero(ids[:, 0] == e)[0]
        if not len(toks):
            continue
        y64 = oracle.block_gemv(xb[toks], codes[e], scales[e])
        wmax = tolerance.block_wmax_rows(codes[e], scales[e], np.arange(n), table())
        st = tolerance.gemv_errors(yb[toks, 0], y64, xb[toks], wmax)
        assert tolerance.gemv_ok(st), (e, counts[e], st)
    assert pkg.check_device_error() == 0


@pytest.mark.parametrize("case", ["wide_range", "blockwise", "tiny", "huge", "single_spike"])
def test_moe_grouped_decode_tiles_x_dynamic_range(pkg, case):
    """The decode tiles read an f16 copy of the routed x rows with one power
    of two per (row, 128-column K block) and tile-local factors: activations
    spanning 60 decades, magnitudes that jump by up to 2^80 from one K block
    to the next, all tiny, all huge, or one spike per row stay within
    tolerance for every (token, slot)."""
    E, n, k, m, topk = 8, 256, 1024, 64, 2
    assert m * topk <= 32 * E
    codes, scales = experts(E, n, k, 61)
    ids = route(m, topk, E, 17)
    g = torch.Generator().manual_seed(6)
    base = torch.randn((m, k), generator=g)
    if case == "wide_range":
        x = base * torch.pow(10.0, torch.randint(-30, 30, (m, k), generator=g).to(torch.float32))
    elif case == "blockwise":
        expo = torch.randint(-40, 40, (m, k // 128), generator=g).to(torch.float32)
        x = base * torch.pow(2.0, expo).repeat_interleave(128, dim=1)
    elif case == "tiny":
        x = base * 1e-35
    elif case == "huge":
        x = base * 1e30
    else:
        x = base.clone()
        x[:, 37] = 3e20
    x = x.to(torch.bfloat16)
    y = pkg.moe_gemv_ws(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(codes).to(DEV),
                        torch.from_numpy(scales).to(DEV), ws(pkg, m, topk, E, k))
    torch.cuda.synchronize()
    check_call(y, bits(x), ids, codes, scales)
    assert pkg.check_device_error() == 0


def check_call(y_dev, x_bits, ids, codes, scales):
    """The GEMV tolerance with its relative-L2 statistic taken over all the
    call's outputs (as the dense tests take it) and the element bound per
    (token, slot): in the "tiny" case above, the correctly rounded bf16 of
    the fp64 result of output row (40, 0) alone has relative L2 error
    2.0035e-3, so a per-row statistic of 256 outputs would reject the exact
    answer."""
    m, topk = ids.shape
    y64 = oracle.moe_gemv(x_bits, ids, codes, scales)
    yb = bits(y_dev.cpu())
    yf = tolerance.bf16_bits_to_f64(yb)
    for t in range(m):
        for j in range(topk):
            e = ids[t, j]
            s = np.repeat(scales[e].astype(np.float64), 128, axis=0)[:codes.shape[1]]
            wmax = np.abs(table()[codes[e]] * np.repeat(s, 128, axis=1)[:, :codes.shape[2]]).max(axis=1)
            st = tolerance.gemv_errors(yb[t, j][None, :], y64[t, j][None, :], x_bits[t][None, :], wmax)
            assert st["finite"] and st["max_ratio"] <= 1.0, (t, j, st)
    rel_l2 = float(np.linalg.norm(yf - y64) / np.linalg.norm(y64))
    assert tolerance.gemv_ok({"finite": True, "max_ratio": 0.0, "rel_l2": rel_l2, "count": yf.size}), rel_l2


def test_moe_grouped_out_of_range_id(pkg):
    E, n, k, m, topk = 8, 256, 256, 40, 2
    codes, scales = experts(E, n, k, 5)
    ids = route(m, topk, E, 3)
    ids[7, 1] = 99
    ids[20, 0] = -1
    x = inputs.activations(m, k, 4)
    y = torch.full((m, topk, n), 7.0, dtype=torch.bfloat16, device=DEV)
    pkg.moe_gemv_ws(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(codes).to(DEV),
                    torch.from_numpy(scales).to(DEV), ws(pkg, m, topk, E, k), y=y)
    assert pkg.check_device_error() & 16
    yc = y.cpu().float()
    assert torch.all(yc[7, 1] == 7.0) and torch.all(yc[20, 0] == 7.0)
    good = np.ones((m, topk), dtype=bool)
    good[7, 1] = good[20, 0] = False
    safe = np.where(good, ids, 0).astype(np.int32)
    y64 = oracle.moe_gemv(bits(x), safe, codes, scales)
    yb = bits(y.cpu())
    for t, j in zip(*np.nonzero(good)):
        e = ids[t, j]
        wmax = np.abs(table()[codes[e]] * np.repeat(np.repeat(scales[e].astype(np.float64), 128, axis=0)[:n],
                                                      128, axis=1)[:, :k]).max(axis=1)
        st = tolerance.gemv_errors(yb[t, j][None, :], y64[t, j][None, :], bits(x)[t][None, :], wmax)
        assert tolerance.gemv_ok(st), (t, j, st)


@pytest.mark.parametrize("m", [64, 512, 2048])
def test_moe_grouped_full_size_sampled(pkg, m):
    """256 experts of [2048, 4096], top-12: the sampled experts' codes and
    scales come from the oracle; every (token, slot) routed to one of them is
    checked on 128 sampled weight rows."""
    E, (n, k), topk = inputs.MOE_EXPERTS, inputs.MOE_SHAPE, inputs.MOE_TOPK
    codes = torch.empty((E, n, k), dtype=torch.uint8, device=DEV)
    scales = torch.empty((E, n // 128, k // 128), dtype=torch.float32, device=DEV)
    for e in range(E):
        c, s_ = pkg.quantize(inputs.moe_expert_weight(e, device=DEV))
        codes[e] = c
        scales[e] = s_
    ids = inputs.moe_routing(m, topk, E, seed=m).numpy().astype(np.int32)
    sample = sorted(set(int(v) for v in ids[:4].ravel()))[:6]
    rows = np.arange(640, 768)
    oc, os_ = {}, {}
    for e in sample:
        w = inputs.moe_expert_weight(e)
        c, s = oracle.block_quantize(bits(w))
        codes[e] = torch.from_numpy(c).to(DEV)
        scales[e] = torch.from_numpy(s).to(DEV)
        oc[e], os_[e] = c, s
    x = inputs.activations(m, k, 800 + m)
    y = pkg.moe_gemv_ws(x.to(DEV), torch.from_numpy(ids).to(DEV), codes, scales, ws(pkg, m, topk, E, k))
    torch.cuda.synchronize()
    yb, xb = bits(y.cpu()), bits(x)
    for e in sample:
        pairs = np.argwhere(ids == e)
        y64 = oracle.block_gemv(xb[pairs[:, 0]], oc[e], os_[e], rows=rows)
        wmax = tolerance.block_wmax_rows(oc[e][rows], os_[e], rows, table())
        got = np.stack([yb[t, j][rows] for t, j in pairs])
        st = tolerance.gemv_errors(got, y64, xb[pairs[:, 0]], wmax)
        assert tolerance.gemv_ok(st), (e, st)
    assert pkg.check_device_error() == 0
