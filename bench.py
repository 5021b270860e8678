"""Benchmark of the block-FP8 W8A16 decode GEMV on GB300.

Default workload (one "step"): the lm_head weight [152064, 4096] quantized to
128x128 block FP8 at load time, then one GEMV call at each of M = 1, 4, 8, 16
(bf16 x, bf16 logits out).  The weight (623 MB of codes) is larger than L2,
so every call streams it from HBM.  Metric: algorithmic HBM bytes
(codes + scales + x + y) per second over the step, in GB/s; per-M us/call,
GB/s and fraction of HBM bandwidth are reported alongside.

Other workloads (--workload): rotation (48 layers x 4 projection weights,
192 GEMVs per step, CUDA-graph captured), sweep ([12288, 4096], M = 1..32
over 8 rotated copies), mx ([18432, 7168] MXFP8 GEMV, M = 1, 8, 16 over 4
copies), quantize ([18432, 7168] block, MXFP8, per-row and per-tensor
load-time quantization), prefill ([12288, 4096] at M = 512, 2048, 4096 on the
tensor cores), rowwise (the lm_head weight with one scale per row and with
one per tensor, M = 1, 8, 16).  --scales row|tensor runs the rotation and
prefill workloads on per-row / per-tensor FP8 instead of 128x128 blocks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload lm_head|rotation|sweep|mx|quantize|prefill|rowwise]
                  [--m M] [--scales block|row|tensor]

N > 1 runs one independent replica per GPU (the path needs no collective);
the reported value is the aggregate over ranks of bytes moved divided by the
slowest rank's time.  --impl reference times the CPU oracle (plain C, one
host core) on a bounded sample of the same workload and metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HBM_NOMINAL_GBS = 8000.0


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


KERNEL_SOURCES = {
    "decode_kernel": ["decode.cu", "common.cuh"],
    "gemv_batch_kernel": ["decode.cu", "common.cuh"],
    "prefill_kernel": ["prefill.cu", "common.cuh"],
    "block_quantize_kernel": ["quantize.cu", "common.cuh"],
}


def kernel_source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    base = kernel.split("<")[0]
    for f in KERNEL_SOURCES.get(base, []):
        with open(os.path.join(ROOT, "fp8_block_scaled_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
    the committed ncu capture in profiles/traffic.json, or None if the kernel's
    source has changed since those counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d[f"{kernel} {workload}"]
        if e["source_sha256"] != kernel_source_hash(kernel):
            return None
        return int(e["dram_bytes_per_launch"])
    except Exception:
        return None


def tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured, burst"
    except Exception:
        return 1900.0, "fallback"


def gemv_bytes(m, n, k, mx=False, scales="block"):
    if mx:
        sb = n * ((k + 31) // 32)
    elif scales == "row":
        sb = 4 * n
    elif scales == "tensor":
        sb = 4
    else:
        sb = 4 * ((n + 127) // 128) * ((k + 127) // 128)
    return n * k + sb + 2 * m * k + 2 * m * n


def quantizer(fp8bs, scales):
    """(quantize, gemv) pair of the binding for a scale layout."""
    if scales == "row":
        return fp8bs.row_quantize, fp8bs.row_gemv
    if scales == "tensor":
        return fp8bs.tensor_quantize, fp8bs.row_gemv
    return fp8bs.quantize, fp8bs.gemv


# ----------------------------------------------------------- clocks sampler
class Clocks:
    def __init__(self, path):
        self.path = path
        self.proc = None

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0],
                 "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 9:
                try:
                    rows.append((float(p[1]), float(p[2]), p[5:9]))
                except ValueError:
                    pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ ranks
def dist_setup(n_gpus):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return rank, world, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, v):
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, v):
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------- workloads
LM_HEAD_METRIC = "block-FP8 W8A16 GEMV HBM GB/s (lm_head, M=1,4,8,16)"


def lm_head_config(n, k, ms):
    return {"workload": "lm_head [152064,4096] block-FP8 (128x128 fp32 scales) W8A16 GEMV, one call at each "
                        "of M=1,4,8,16 per step (M > 8 through fp8bs_gemv_ws: x prepared once per call in a "
                        "workspace allocated before the timed region)", "n": n, "k": k, "ms": ms,
            "l2": "inputs larger than L2 (623 MB of codes per call)"}


def lm_head_call(fp8bs, m, x, codes, scales, y, ws):
    """The library's fastest call for this M: above M = 8 the workspace GEMV
    (f16 operands at every M) beats the bf16 decode on this weight."""
    if m > 8:
        fp8bs.gemv_ws(x, codes, scales, ws, y=y)
    else:
        fp8bs.gemv(x, codes, scales, y=y)


def lm_head_workload(torch, fp8bs, inputs, dev):
    ms = [1, 4, 8, 16]
    w = inputs.lm_head_weight(2, device=dev)
    n, k = w.shape
    codes, scales = fp8bs.quantize(w)
    del w
    xs = {m: inputs.activations(m, k, 100 + m, device=dev) for m in ms}
    ys = {m: torch.empty((m, n), dtype=torch.bfloat16, device=dev) for m in ms}
    ws = torch.empty((fp8bs.gemv_ws_bytes(max(ms), k),), dtype=torch.uint8, device=dev)
    calls = [(f"M={m}", m, gemv_bytes(m, n, k),
              (lambda m=m: lm_head_call(fp8bs, m, xs[m], codes, scales, ys[m], ws))) for m in ms]
    cfg = lm_head_config(n, k, ms)
    return dict(calls=calls, xs=xs, ys=ys, cfg=cfg, dominant=("decode_kernel<1,0,true>", [0, 1, 2]),
                codes=codes, scales=scales, ws=ws, n=n, k=k, mx=False,
                call_launches=[2 if m > 8 else 1 for m in ms])


def rotation_weights(fp8bs, inputs, dev, scales="block", layers=None):
    quant, _ = quantizer(fp8bs, scales)
    weights = []
    for l in range(inputs.ROTATION_LAYERS if layers is None else layers):
        for j in range(4):
            w = inputs.rotation_weight(l, j, device=dev)
            weights.append(quant(w))
            del w
    return weights


def rotation_workload(torch, fp8bs, inputs, dev, m, scales="block", batched=True, weights=None, layers=None):
    """48 layers x 4 projection weights, one GEMV each per step.  batched:
    the step is one fp8bs_gemv_batch call (the 192 GEMVs stream as two
    persistent launches); otherwise one fp8bs_gemv call per weight.
    `layers` < 48 gives a smaller case of the same kernels (profiling)."""
    layers = inputs.ROTATION_LAYERS if layers is None else layers
    quant, gemv = quantizer(fp8bs, scales)
    if weights is None:
        weights = rotation_weights(fp8bs, inputs, dev, scales, layers)
    shapes = [inputs.ROTATION_SHAPES[j] for _ in range(layers) for j in range(4)]
    xs = [inputs.activations(m, k, 7 + i, device=dev) for i, (n, k) in enumerate(shapes)]
    ys = [torch.empty((m, n), dtype=torch.bfloat16, device=dev) for (n, k) in shapes]
    batched = batched and scales == "block"
    ops = [(xs[i], c, s, ys[i]) for i, (c, s) in enumerate(weights)]

    def step():
        if batched:
            fp8bs.gemv_batch(ops)
        else:
            for i, (c, s) in enumerate(weights):
                gemv(xs[i], c, s, y=ys[i])
    total = sum(gemv_bytes(m, n, k, scales=scales) for (n, k) in shapes)
    kind = {"block": "block-FP8", "row": "per-row FP8", "tensor": "per-tensor FP8"}[scales]
    how = "one batched call (fp8bs_gemv_batch)" if batched else "one call per weight"
    cfg = {"workload": f"decode dense-projection rotation: {layers} layers x 4 {kind} weights "
                       f"([8192,2560],[2560,3072],[6656,2560],[2560,3072]), M={m}, {4 * layers} GEMVs per step, "
                       f"{how}, CUDA graph", "ms": [m],
           "l2": f"inputs larger than L2 ({total / 1e9:.2f} GB of codes per step)"}
    launches = -(-4 * layers // 96) if batched else 4 * layers
    mt = (m + 7) // 8
    dom = f"gemv_batch_kernel<{mt},0,{'true' if mt == 1 else 'false'}>" if batched else "decode_kernel"
    return dict(calls=[(f"rotation M={m}", m, total, step)], cfg=cfg, graph=True, launches_per_step=launches,
                dominant=(dom, [0]), xs=xs, ys=ys, weights=weights, ops=ops)


def sweep_workload(torch, fp8bs, inputs, dev, ms, ws=False):
    """ws: every call goes through fp8bs_gemv_ws (x prepared once per call
    in a caller-provided workspace, f16 operands at every M)."""
    copies = [fp8bs.quantize(inputs.sweep_weight(c, device=dev)) for c in range(8)]
    n, k = inputs.SWEEP_SHAPE
    work = torch.empty((fp8bs.gemv_ws_bytes(32, k),), dtype=torch.uint8, device=dev) if ws else None
    calls = []
    for m in ms:
        x = inputs.activations(m, k, 300 + m, device=dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)

        def fn(x=x, y=y):
            for c, s in copies:
                if ws:
                    fp8bs.gemv_ws(x, c, s, work, y=y)
                else:
                    fp8bs.gemv(x, c, s, y=y)
        calls.append((f"M={m}", m, 8 * gemv_bytes(m, n, k), fn))
    how = " (fp8bs_gemv_ws: x prepared once per call)" if ws else ""
    cfg = {"workload": f"M sweep: block-FP8 [12288,4096], one GEMV per M over 8 rotated weight copies (403 MB){how}",
           "n": n, "k": k, "ms": ms, "l2": "inputs larger than L2 (8 rotated copies)"}
    return dict(calls=calls, cfg=cfg, dominant=("decode_kernel", list(range(len(ms)))), gemvs_per_call=8,
                launches_per_call=16 if ws else 8)


def mx_workload(torch, fp8bs, inputs, dev):
    ms = [1, 8, 16]
    copies = []
    for c in range(4):
        w = inputs.heavy_tail_weight(5 + c, device=dev)
        copies.append(fp8bs.mx_quantize(w))
        del w
    n, k = inputs.MX_SHAPE
    calls = []
    for m in ms:
        x = inputs.activations(m, k, 500 + m, device=dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)

        def fn(x=x, y=y):
            for c, e in copies:
                fp8bs.mx_gemv(x, c, e, y=y)
        calls.append((f"M={m}", m, 4 * gemv_bytes(m, n, k, mx=True), fn))
    cfg = {"workload": "MXFP8 [18432,7168] (e8m0 per 32 K) W8A16 GEMV, M=1,8,16, 4 rotated copies",
           "n": n, "k": k, "ms": ms, "l2": "inputs larger than L2 (4 rotated copies, 528 MB)"}
    return dict(calls=calls, cfg=cfg, dominant=("decode_kernel<1,1,true>", [0, 1]), launches_per_call=4)


def prefill_launches(torch, m, n, k):
    """Kernel launches of one tcgen05 W8A16 prefill call (prefill.cu's split
    of the last wave): one launch of the full waves, plus one of the last
    wave's tiles split over K when that wave fills at most half the SMs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = -(-n // 128) * -(-m // 256)
    rem = tiles % sms
    return 2 if rem > 0 and 2 * rem <= sms and -(-k // 128) >= 2 else 1


def prefill_workload(torch, fp8bs, inputs, dev, scales="block"):
    ms = [512, 2048, 4096]
    quant, gemv = quantizer(fp8bs, scales)
    codes, sc = quant(inputs.sweep_weight(0, device=dev))
    n, k = inputs.SWEEP_SHAPE
    calls = []
    for m in ms:
        x = inputs.activations(m, k, 700 + m, device=dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        calls.append((f"M={m}", m, 2 * m * n * k, (lambda x=x, y=y: gemv(x, codes, sc, y=y))))
    kind = {"block": "block-FP8", "row": "per-row FP8", "tensor": "per-tensor FP8"}[scales]
    cfg = {"workload": f"prefill: {kind} [12288,4096] W8A16 GEMM on tcgen05, M=512,2048,4096", "n": n, "k": k,
           "ms": ms, "l2": "weight (50 MB) and x fit in L2; compute-bound"}
    dom = "prefill_kernel<0>" if scales == "block" else "prefill_kernel<2>"
    return dict(calls=calls, cfg=cfg, dominant=(dom, [0, 1, 2]), flops=True,
                call_launches=[prefill_launches(torch, m, n, k) for m in ms])


def mx_prefill_workload(torch, fp8bs, inputs, dev):
    """MXFP8 [18432, 7168] (0.1% Student-t entries) at prefill sizes on the
    tensor cores, the e8m0 group scales folded into the decoded weights."""
    ms = [512, 2048, 4096]
    w = inputs.heavy_tail_weight(5, device=dev)
    codes, e8m0 = fp8bs.mx_quantize(w)
    del w
    n, k = inputs.MX_SHAPE
    calls = []
    for m in ms:
        x = inputs.activations(m, k, 750 + m, device=dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        calls.append((f"M={m}", m, 2 * m * n * k, (lambda x=x, y=y: fp8bs.mx_gemv(x, codes, e8m0, y=y))))
    cfg = {"workload": "prefill: MXFP8 [18432,7168] W8A16 GEMM on tcgen05, M=512,2048,4096", "n": n, "k": k,
           "ms": ms, "l2": "weight (132 MB) about the size of L2; compute-bound"}
    return dict(calls=calls, cfg=cfg, dominant=("prefill_kernel<1>", [0, 1, 2]), flops=True,
                call_launches=[prefill_launches(torch, m, n, k) for m in ms])


def rowwise_workload(torch, fp8bs, inputs, dev):
    """lm_head [152064, 4096] with one fp32 scale per row and with one per
    tensor (FreeToken PR #389's per-row W8A16 route), M = 1, 8, 16."""
    ms = [1, 8, 16]
    w = inputs.lm_head_weight(2, device=dev)
    n, k = w.shape
    rq = fp8bs.row_quantize(w)
    tq = fp8bs.tensor_quantize(w)
    del w
    xs = {m: inputs.activations(m, k, 100 + m, device=dev) for m in ms}
    ys = {m: torch.empty((m, n), dtype=torch.bfloat16, device=dev) for m in ms}
    calls = [(f"row M={m}", m, gemv_bytes(m, n, k, scales="row"),
              (lambda m=m: fp8bs.row_gemv(xs[m], rq[0], rq[1], y=ys[m]))) for m in ms]
    calls += [(f"tensor M={m}", m, gemv_bytes(m, n, k, scales="tensor"),
               (lambda m=m: fp8bs.row_gemv(xs[m], tq[0], tq[1], y=ys[m]))) for m in ms]
    cfg = {"workload": "lm_head [152064,4096] per-row and per-tensor FP8 W8A16 GEMV, one call at each of "
                       "M=1,8,16 per layout per step", "n": n, "k": k, "ms": ms,
           "l2": "inputs larger than L2 (623 MB of codes per call)"}
    return dict(calls=calls, cfg=cfg, dominant=("decode_kernel<1,2,true>", [0, 1, 3, 4]))


def w8a8_workload(torch, fp8bs, inputs, dev):
    """lm_head [152064, 4096] per-tensor e4m3 weight x dynamically quantized
    e4m3 activations (FreeToken PR #389's W8A8 route), M = 1, 8, 16: the GEMM
    alone on pre-quantized x, and the whole linear (activation quantize +
    GEMM) per call."""
    ms = [1, 8, 16]
    w = inputs.lm_head_weight(2, device=dev)
    n, k = w.shape
    wq, sw = fp8bs.tensor_quantize(w)
    del w
    xs = {m: inputs.activations(m, k, 100 + m, device=dev) for m in ms}
    xq = {m: fp8bs.act_quantize(xs[m]) for m in ms}
    ys = {m: torch.empty((m, n), dtype=torch.bfloat16, device=dev) for m in ms}
    gb = lambda m: n * k + 4 + m * k + 4 + 2 * m * n
    calls = [(f"gemm M={m}", m, gb(m), (lambda m=m: fp8bs.w8a8_gemm(xq[m][0], xq[m][1], wq, sw, y=ys[m])))
             for m in ms]
    calls += [(f"linear M={m}", m, gb(m) + 2 * m * k,
               (lambda m=m: fp8bs.w8a8_linear(xs[m], wq, sw, y=ys[m], xq=xq[m][0], sx=xq[m][1]))) for m in ms]
    cfg = {"workload": "lm_head [152064,4096] W8A8 (per-tensor e4m3 weight, dynamic per-tensor e4m3 "
                       "activations): GEMM alone and activation-quantize + GEMM, M=1,8,16", "n": n, "k": k,
           "ms": ms, "l2": "inputs larger than L2 (623 MB of codes per call)"}
    return dict(calls=calls, cfg=cfg, dominant=("w8a8_decode_kernel<1>", [0, 1]),
                call_launches=[1, 1, 1, 2, 2, 2])


def w8a8_prefill_workload(torch, fp8bs, inputs, dev):
    ms = [512, 2048, 4096]
    wq, sw = fp8bs.tensor_quantize(inputs.sweep_weight(0, device=dev))
    n, k = inputs.SWEEP_SHAPE
    calls = []
    for m in ms:
        xq, sx = fp8bs.act_quantize(inputs.activations(m, k, 700 + m, device=dev))
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        calls.append((f"M={m}", m, 2 * m * n * k, (lambda xq=xq, sx=sx, y=y: fp8bs.w8a8_gemm(xq, sx, wq, sw, y=y))))
    cfg = {"workload": "prefill: W8A8 [12288,4096] e4m3 x e4m3 GEMM on tcgen05 (kind::f8f6f4), M=512,2048,4096",
           "n": n, "k": k, "ms": ms, "l2": "weight (50 MB) and x fit in L2; compute-bound"}
    return dict(calls=calls, cfg=cfg, dominant=("w8a8_prefill_kernel", [0, 1, 2]), flops=True, fp8=True)


def moe_workload(torch, fp8bs, inputs, dev):
    """Grouped MoE decode: 256 block-FP8 experts of [2048, 4096] (2.1 GB of
    codes), top-12 routing per token, M = 1, 8, 16 tokens.  Bytes per call
    count the experts the call's routing selects (each streamed once)."""
    E, (n, k), topk = inputs.MOE_EXPERTS, inputs.MOE_SHAPE, inputs.MOE_TOPK
    codes = torch.empty((E, n, k), dtype=torch.uint8, device=dev)
    scales = torch.empty((E, n // 128, k // 128), dtype=torch.float32, device=dev)
    for e in range(E):
        c, s_ = fp8bs.quantize(inputs.moe_expert_weight(e, device=dev))
        codes[e] = c
        scales[e] = s_
    ms = [1, 8, 16]
    calls = []
    for m in ms:
        ids_cpu = inputs.moe_routing(m, topk, E, seed=m)
        distinct = int(torch.unique(ids_cpu).numel())
        ids = ids_cpu.to(dev)
        x = inputs.activations(m, k, 800 + m, device=dev)
        y = torch.empty((m, topk, n), dtype=torch.bfloat16, device=dev)
        b = distinct * (n * k + 4 * (n // 128) * (k // 128)) + 2 * m * k + 4 * m * topk + 2 * m * topk * n
        calls.append((f"M={m} ({distinct} experts)", m, b,
                      (lambda x=x, ids=ids, y=y: fp8bs.moe_gemv(x, ids, codes, scales, y=y))))
    cfg = {"workload": "grouped MoE decode: 256 block-FP8 experts [2048,4096], top-12 routing, M=1,8,16",
           "experts": E, "n": n, "k": k, "topk": topk, "ms": ms,
           "l2": "inputs larger than L2 (12-144 experts x 8.4 MB selected per call)"}
    return dict(calls=calls, cfg=cfg, dominant=("decode_kernel<1,0,true,true>", [0, 1]))


def moe_prefill_workload(torch, fp8bs, inputs, dev, experts=None):
    """Grouped MoE at prefill sizes: 256 block-FP8 experts of [2048, 4096],
    top-12 routing, M = 512 and 2048 tokens through fp8bs_moe_gemv_ws (the
    routing grouped on the device, one grouped tcgen05 GEMM).  Work per call:
    2 * M * topk * N * K flops.  `experts`: fewer experts (a smaller case
    with more pairs per expert, for profiling)."""
    E, (n, k), topk = experts or inputs.MOE_EXPERTS, inputs.MOE_SHAPE, inputs.MOE_TOPK
    codes = torch.empty((E, n, k), dtype=torch.uint8, device=dev)
    scales = torch.empty((E, n // 128, k // 128), dtype=torch.float32, device=dev)
    for e in range(E):
        c, s_ = fp8bs.quantize(inputs.moe_expert_weight(e, device=dev))
        codes[e] = c
        scales[e] = s_
    ms = [512, 2048]
    calls, hbm = [], []
    for m in ms:
        ids = inputs.moe_routing(m, topk, E, seed=m).to(dev)
        # algorithmic bytes: every selected expert's codes and scales once,
        # x, the routing ids and y
        sel = int(torch.unique(ids).numel())
        hbm.append(sel * (n * k + 4 * (n // 128) * (k // 128)) + 2 * m * k + 4 * m * topk + 2 * m * topk * n)
        x = inputs.activations(m, k, 850 + m, device=dev)
        y = torch.empty((m, topk, n), dtype=torch.bfloat16, device=dev)
        work = torch.empty((fp8bs.moe_gemv_ws_bytes(m, topk, E, k),), dtype=torch.uint8, device=dev)
        calls.append((f"M={m}", m, 2 * m * topk * n * k,
                      (lambda x=x, ids=ids, y=y, work=work: fp8bs.moe_gemv_ws(x, ids, codes, scales, work, y=y))))
    path = lambda m: ("the decode kernel per 32-pair expert tile" if m * topk <= 32 * E
                      else "one grouped tcgen05 GEMM")
    cfg = {"workload": f"grouped MoE prefill: {E} block-FP8 experts [{n},{k}], top-{topk} routing, M=512,2048 "
                       f"(fp8bs_moe_gemv_ws: routing grouped on the device, then {path(512)} at M=512, "
                       f"{path(2048)} at M=2048)",
           "experts": E, "n": n, "k": k, "topk": topk, "ms": ms,
           "l2": f"inputs larger than L2 ({E * n * k / 1e9:.1f} GB of expert codes, nearly all selected)"}
    # M=512 (24 pairs per expert on average) takes the grouped decode path,
    # M=2048 (96) the tensor-core grouped GEMM
    return dict(calls=calls, cfg=cfg, dominant=("decode_kernel<4,0,true,true,true> + prefill_kernel<0,true,TX>", [0, 1]),
                flops=True, hbm_bytes=hbm,
                call_launches=[5, 5])


def kv_workload(torch, fp8bs, inputs, dev):
    """FP8 KV-cache split-KV decode attention on a Qwen3-8B-shaped layer (32 q
    heads, 8 kv heads, head_dim 128, page 16) at InfiniLM PR #586's decode
    shapes: batch 1 x 1k / 4k / 16k tokens and batch 8 x 1k / 4k.  Each call
    reads its sequences' K and V pages from a 2 GB cache pool through its own
    block table (8 rotations per shape, so nothing is L2-resident)."""
    hq, hkv, d, page = inputs.KV_Q_HEADS, inputs.KV_HEADS, inputs.KV_HEAD_DIM, inputs.KV_PAGE
    blocks = (1 << 30) // (page * hkv * d)         # 1 GB for K, 1 GB for V
    g = torch.Generator(device="cpu").manual_seed(11)
    k_cache = torch.randint(0, 0x7F, (blocks, page, hkv, d), dtype=torch.uint8, generator=g).to(dev)
    v_cache = torch.randint(0, 0x7F, (blocks, page, hkv, d), dtype=torch.uint8, generator=g).to(dev)
    ks = torch.tensor([0.01], device=dev)
    vs = torch.tensor([0.01], device=dev)
    shapes = [(1, 1024), (1, 4096), (1, 16384), (8, 1024), (8, 4096)]
    calls = []
    for bsz, length in shapes:
        nblk = (length + page - 1) // page
        perm = torch.randperm(blocks, generator=g)
        tables = [perm[r * bsz * nblk:(r + 1) * bsz * nblk].view(bsz, nblk).to(torch.int32).to(dev) for r in range(8)]
        lens = torch.full((bsz,), length, dtype=torch.int32, device=dev)
        q = inputs.activations(bsz * hq, d, 900 + length, device=dev).view(bsz, hq, d)
        out = torch.empty((bsz, hq, d), dtype=torch.bfloat16, device=dev)
        b = 8 * (2 * bsz * length * hkv * d + 4 * bsz * nblk + 4 * bsz * hq * d)

        def fn(tables=tables, lens=lens, q=q, out=out, length=length):
            for tb in tables:
                fp8bs.kv_decode_attention(q, k_cache, v_cache, ks, vs, tb, lens, length, d ** -0.5, out=out)
        calls.append((f"B={bsz} L={length}", bsz, b, fn))
    cfg = {"workload": "FP8 E4M3 paged KV cache decode attention (split-KV), 32 q / 8 kv heads, head_dim 128, "
                       "page 16; batch x context 1x1k, 1x4k, 1x16k, 8x1k, 8x4k", "q_heads": hq, "kv_heads": hkv,
           "head_dim": d, "page": page, "l2": "8 rotated block tables per shape over a 2 GB cache pool"}
    return dict(calls=calls, cfg=cfg, dominant=("kv_attn_kernel", [2, 4]), launches_per_call=8)


def quantize_workload(torch, fp8bs, inputs, dev):
    w = inputs.heavy_tail_weight(5, device=dev)
    n, k = w.shape
    codes = torch.empty((n, k), dtype=torch.uint8, device=dev)
    scales = torch.empty(((n + 127) // 128, (k + 127) // 128), dtype=torch.float32, device=dev)
    e8m0 = torch.empty((n, (k + 31) // 32), dtype=torch.uint8, device=dev)
    rs = torch.empty((n,), dtype=torch.float32, device=dev)
    ts = torch.empty((1,), dtype=torch.float32, device=dev)
    bq = 3 * n * k + 4 * scales.numel()
    mq = 3 * n * k + e8m0.numel()
    calls = [("block quantize", 0, bq, lambda: fp8bs.quantize(w, codes=codes, scales=scales)),
             ("mx quantize", 0, mq, lambda: fp8bs.mx_quantize(w, codes=codes, e8m0=e8m0)),
             ("row quantize", 0, 3 * n * k + 4 * n, lambda: fp8bs.row_quantize(w, codes=codes, scales=rs)),
             # per tensor: the weight is read twice (amax pass, then encode), 5 bytes per element moved
             ("tensor quantize", 0, 3 * n * k + 4, lambda: fp8bs.tensor_quantize(w, codes=codes, scale=ts))]
    cfg = {"workload": "load-time quantize of bf16 [18432,7168] (0.1% Student-t entries) to block FP8, "
                       "MXFP8, per-row and per-tensor FP8", "n": n, "k": k,
           "l2": "inputs larger than L2 (264 MB bf16 read per call)"}
    # per tensor: amax, encode and finalize kernels (plus a 4-byte memset)
    return dict(calls=calls, cfg=cfg, dominant=("block_quantize_kernel", [0]), call_launches=[1, 1, 1, 3])


# ------------------------------------------------------------------ timing
def time_calls(torch, calls, steps, warmup, pg, graph=False):
    """Run `warmup` untimed steps, then `steps` timed ones bracketed by one
    pair of CUDA events on the current stream (the whole timed region, ms),
    then `steps` more with events around each call (per-call mean ms)."""
    stream = torch.cuda.current_stream()
    run = [fn for _, _, _, fn in calls]
    if graph:
        g = []
        s = torch.cuda.Stream()
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            for fn in run:
                fn()
        stream.wait_stream(s)
        torch.cuda.synchronize()
        for fn in run:
            cg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(cg):
                fn()
            g.append(cg)
        run = [cg.replay for cg in g]
    for _ in range(warmup):
        for fn in run:
            fn()
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    # whole-job time: one event pair around all steps (an event between two
    # calls would separate them and stop the next launch from overlapping the
    # previous one's tail, which is not how the calls run in an application)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        for fn in run:
            fn()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    total = t0.elapsed_time(t1)
    # per-call breakdown: a second pass with events around every call
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in run]
          for _ in range(steps)]
    for s in range(steps):
        for i, fn in enumerate(run):
            ev[s][i][0].record(stream)
            fn()
            ev[s][i][1].record(stream)
    torch.cuda.synchronize()
    per = [statistics.fmean(ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(steps)) for i in range(len(run))]
    return per, total


def e2e_lm_head(torch, fp8bs, wl, steps, warmup, pg):
    """Same step through the public API with host buffers: every step copies
    each x from pinned host memory and reads each y back into pinned host
    memory, inside the timed region.  The copies run on their own streams
    (one per direction), ordered against the GEMVs by events, with x and y
    double-buffered across steps, so a call's read-back overlaps the next
    call's GEMV; the region ends after the last read-back has landed."""
    stream = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ms = wl["cfg"]["ms"]
    hx = {m: wl["xs"][m].cpu().pin_memory() for m in ms}
    hy = {m: [torch.empty(tuple(wl["ys"][m].shape), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
          for m in ms}
    dx = {m: [torch.empty_like(wl["xs"][m]) for _ in range(2)] for m in ms}
    dy = {m: [wl["ys"][m], torch.empty_like(wl["ys"][m])] for m in ms}
    ev = {(m, b, kind): torch.cuda.Event() for m in ms for b in range(2) for kind in ("x", "gemv", "y")}
    used = set()

    def step(i):
        b = i & 1
        for m in ms:
            if (m, b) in used:  # the GEMV that last read dx[m][b] has finished
                h2d_s.wait_event(ev[(m, b, "gemv")])
            with torch.cuda.stream(h2d_s):
                dx[m][b].copy_(hx[m], non_blocking=True)
                ev[(m, b, "x")].record(h2d_s)
            stream.wait_event(ev[(m, b, "x")])
            if (m, b) in used:  # dy[m][b]'s previous read-back has landed
                stream.wait_event(ev[(m, b, "y")])
            lm_head_call(fp8bs, m, dx[m][b], wl["codes"], wl["scales"], dy[m][b], wl["ws"])
            ev[(m, b, "gemv")].record(stream)
            d2h_s.wait_event(ev[(m, b, "gemv")])
            with torch.cuda.stream(d2h_s):
                hy[m][b].copy_(dy[m][b], non_blocking=True)
                ev[(m, b, "y")].record(d2h_s)
            used.add((m, b))
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(pg)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    h2d_s.wait_stream(stream)
    for i in range(steps):
        step(warmup + i)
    stream.wait_stream(h2d_s)
    stream.wait_stream(d2h_s)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    h2d = sum(hx[m].numel() * 2 for m in ms)
    d2h = sum(hy[m][0].numel() * 2 for m in ms)
    return t0.elapsed_time(t1), h2d, d2h


# ------------------------------------------------------------ CPU oracle
_ORACLE_CACHE = {}
ORACLE_GEMV_ROWS = 4096      # lm_head rows in the GEMV sample (M = 1, 4, 8, 16)
ORACLE_QUANT_ROWS = 1024     # lm_head rows in the quantize sample
ORACLE_ROT_ROWS = 1024       # rows of each rotation weight shape in the rotation GEMV sample


def _oracle_samples():
    """Seeded, bounded samples of the workloads (generated once, untimed):
    the first rows of the lm_head weight (bf16 bits), x for M = 1, 4, 8, 16,
    and for the rotation GEMV random finite e4m3 codes with positive scales
    for the first rows of each of the four projection shapes (a GEMV's time
    does not depend on its values)."""
    if "s" in _ORACLE_CACHE:
        return _ORACLE_CACHE["s"]
    import numpy as np
    import oracle
    from fp8_block_scaled_02_gb300 import inputs
    wq = inputs.bf16_bits(inputs.lm_head_weight(2, shape=(ORACLE_QUANT_ROWS, 4096)))
    wg = inputs.bf16_bits(inputs.lm_head_weight(2, shape=(ORACLE_GEMV_ROWS, 4096)))
    codes, scales = oracle.block_quantize(wg)
    xs = {m: inputs.bf16_bits(inputs.activations(m, 4096, 100 + m)) for m in (1, 4, 8, 16)}
    rng = np.random.default_rng(17)
    rot = []
    for j, (n, k) in enumerate(inputs.ROTATION_SHAPES):
        r = min(n, ORACLE_ROT_ROWS)
        c = rng.integers(0, 0x7F, size=(r, k), dtype=np.uint8) | (rng.integers(0, 2, size=(r, k), dtype=np.uint8) << 7)
        s = rng.uniform(1e-5, 1e-3, size=(-(-r // 128), -(-k // 128))).astype(np.float32)
        rot.append((c, s, inputs.bf16_bits(inputs.activations(1, k, 7 + j))))
    _ORACLE_CACHE["s"] = dict(wq=wq, codes=codes, scales=scales, xs=xs, rot=rot)
    return _ORACLE_CACHE["s"]


def _row_chunks(rows, threads, align=128):
    """Split [0, rows) into `threads` contiguous ranges on `align` boundaries."""
    blocks = -(-rows // align)
    per = -(-blocks // threads)
    out = []
    for t in range(threads):
        r0, r1 = t * per * align, min(rows, (t + 1) * per * align)
        if r0 < r1:
            out.append((r0, r1))
    return out


def _parallel(fn, chunks, threads):
    """Run fn(r0, r1) over the chunks on `threads` host threads (the oracle's
    C calls release the GIL); returns the wall time in seconds."""
    import concurrent.futures as cf
    t = time.perf_counter()
    if threads == 1:
        for c in chunks:
            fn(*c)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda c: fn(*c), chunks))
    return time.perf_counter() - t


ORACLE_MIN_SECONDS = 1.5     # each cpu_baseline measurement repeats its sample for at least this long


def _repeat(once, min_seconds):
    """Run once() (which returns its seconds) until min_seconds have passed;
    returns (total seconds, repetitions)."""
    total, reps = 0.0, 0
    while reps == 0 or total < min_seconds:
        total += once()
        reps += 1
    return total, reps


def oracle_gemv_step(threads, ms=(1, 4, 8, 16), min_seconds=0.0):
    """The oracle's fp64 block GEMV on the lm_head sample, one call at each M
    (the bench step's M sweep) with its rows split over `threads` host
    threads, repeated for at least min_seconds.  Returns (GB/s in the
    metric's units, seconds)."""
    import oracle
    s = _oracle_samples()
    rows = s["codes"].shape[0]
    chunks = _row_chunks(rows, threads)

    def once():
        secs = 0.0
        for m in ms:
            x = s["xs"][m]
            secs += _parallel(lambda r0, r1: oracle.block_gemv(x, s["codes"][r0:r1],
                                                               s["scales"][r0 // 128:-(-r1 // 128)]), chunks, threads)
        return secs
    secs, reps = _repeat(once, min_seconds)
    nbytes = reps * sum(gemv_bytes(m, rows, 4096) for m in ms)
    return nbytes / secs / 1e9, secs


def oracle_runs(threads_list):
    """The CPU oracle as it stands, timed on the host cores: block quantize
    and MXFP8 quantize of the lm_head sample, the fp64 GEMV of the lm_head
    sample at M = 1 and of the rotation sample at M = 1, each with 1 and with
    all host threads (rows split into contiguous 128-row ranges).  Each
    measurement repeats its sample for at least ORACLE_MIN_SECONDS."""
    import oracle
    s = _oracle_samples()
    out = []
    rq = s["wq"].shape[0]
    qbytes = 3 * rq * 4096
    for t in threads_list:
        chunks = _row_chunks(rq, t)
        for op, fn in (("block_quantize", oracle.block_quantize), ("mx_quantize", oracle.mx_quantize)):
            sec, reps = _repeat(lambda: _parallel(lambda r0, r1: fn(s["wq"][r0:r1]), chunks, t), ORACLE_MIN_SECONDS)
            out.append({"op": op, "workload": f"lm_head [{rq} of 152064 rows, 4096]", "cores": t,
                        "gb_s": round(reps * qbytes / sec / 1e9, 5), "seconds": round(sec, 3), "repetitions": reps})
        v, sec = oracle_gemv_step(t, ms=(1,), min_seconds=ORACLE_MIN_SECONDS)
        out.append({"op": "block_gemv", "workload": f"lm_head M=1 [{s['codes'].shape[0]} of 152064 rows, 4096]",
                    "cores": t, "gb_s": round(v, 5), "seconds": round(sec, 3)})

        def rotation_once():
            sec = 0.0
            for c, sc, x in s["rot"]:
                sec += _parallel(lambda r0, r1: oracle.block_gemv(x, c[r0:r1], sc[r0 // 128:-(-r1 // 128)]),
                                 _row_chunks(c.shape[0], t), t)
            return sec
        sec, reps = _repeat(rotation_once, ORACLE_MIN_SECONDS)
        rate = reps * sum(gemv_bytes(1, c.shape[0], c.shape[1]) for c, _, _ in s["rot"]) / sec
        out.append({"op": "block_gemv", "workload": "rotation M=1 (first 1024 rows of each projection shape)",
                    "cores": t, "gb_s": round(rate / 1e9, 5), "seconds": round(sec, 3), "repetitions": reps,
                    "ms_per_rotation_step": round(1e3 * 2.5829e9 / rate, 1)})
    return out


def oracle_sample_desc(threads):
    return (f"oracle block_gemv (plain C, fp64, as it stands) on {threads} host thread(s), rows split in 128-row "
            f"ranges: the first {ORACLE_GEMV_ROWS} of the 152064 lm_head rows, K=4096, one call at each of "
            f"M=1,4,8,16, the sample repeated for at least {ORACLE_MIN_SECONDS} s")


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# --------------------------------------------------------------- summaries
def summarize(wl, per, total_ms, steps, workload):
    """(value, unit, per_call, roofline) of one timed workload: per-call
    rates from the per-call events; the roofline of the workload's dominant
    kernel = its algorithmic bytes (flops) over its event time, against the
    measured peak."""
    peak, peak_kind = measured_peaks()
    calls = wl["calls"]
    flops = wl.get("flops", False)
    scale_unit = 1e12 if flops else 1e9
    unit = "TFLOP/s" if flops else "GB/s"
    tpeak, tpeak_kind = tensor_peak()
    if wl.get("fp8"):
        # e4m3 tensor-core peak: the measured bf16 peak times the nominal
        # fp8 : bf16 ratio (4.5 : 2.25 PFLOP/s dense)
        tpeak, tpeak_kind = 2.0 * tpeak, tpeak_kind + " x 2 (fp8 : bf16 nominal)"
    step_bytes = sum(b for _, _, b, _ in calls)
    value = step_bytes * steps / (total_ms * 1e-3) / scale_unit
    per_call = {}
    hbm_bytes = wl.get("hbm_bytes")   # a contraction's algorithmic HBM bytes per call, where it has them
    for i, ((name, m, b, _), t) in enumerate(zip(calls, per)):
        lp = wl.get("gemvs_per_call", wl.get("launches_per_call", 1))   # us per GEMV / kernel call
        rate = b / (t * 1e-3) / scale_unit
        if flops:
            per_call[name] = {"us_per_call": round(1e3 * t / lp, 3), "tflop_s": round(rate, 1),
                              "frac_of_peak": round(rate / tpeak, 4)}
            if hbm_bytes:
                gbs = hbm_bytes[i] / (t * 1e-3) / 1e9
                per_call[name].update(gb_s=round(gbs, 1), frac_of_measured_hbm=round(gbs / peak, 4),
                                      bound="hbm" if hbm_bytes[i] / peak > b / 1e3 / tpeak else "tensor")
        else:
            per_call[name] = {"us_per_call": round(1e3 * t / lp, 3), "gb_s": round(rate, 1),
                              "frac_of_8TBps": round(rate / HBM_NOMINAL_GBS, 4),
                              "frac_of_measured": round(rate / peak, 4)}
    dom_name, dom_idx = wl["dominant"]
    dom_bytes = sum(calls[i][2] for i in dom_idx)
    dom_ms = sum(per[i] for i in dom_idx)
    achieved = dom_bytes / (dom_ms * 1e-3) / scale_unit
    if flops and hbm_bytes and sum(hbm_bytes[i] for i in dom_idx) / peak > dom_bytes / 1e3 / tpeak:
        # more time in the bytes than in the flops at the peaks: bound by HBM
        hb = sum(hbm_bytes[i] for i in dom_idx)
        gbs = hb / (dom_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": dom_name, "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                    "frac": round(gbs / peak, 4), "peak_kind": f"hbm_gbs ({peak_kind})",
                    "traffic": measured_traffic(dom_name, workload),
                    "tensor": {"achieved": round(achieved, 1), "peak": tpeak, "unit": "TFLOP/s",
                               "frac": round(achieved / tpeak, 4)}}
    elif flops:
        roofline = {"bound": "tensor", "kernel": dom_name, "achieved": round(achieved, 1), "peak": tpeak,
                    "unit": "TFLOP/s", "frac": round(achieved / tpeak, 4),
                    "peak_kind": f"bf16_tflops ({tpeak_kind})", "traffic": None,
                    "dtype": "e4m3" if wl.get("fp8") else "bf16"}
    else:
        roofline = {"bound": "hbm", "kernel": dom_name, "achieved": round(achieved, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": f"hbm_gbs ({peak_kind})",
                    "traffic": measured_traffic(dom_name, workload)}
    return value, unit, per_call, roofline


def extra_configs(torch, fp8bs, inputs, dev, steps, warmup):
    """The other measured configurations, each timed like the main workload
    (warm-up, one event pair over the timed steps, then events around every
    call) with its own roofline record: the 48-layer rotation at M = 1, 8,
    16, 32 (one batched call per step), the [12288, 4096] M sweep at M = 1,
    9, 17, 25, 32, the tcgen05 prefill at M = 512, 2048, 4096, the MXFP8
    GEMV at M = 1, 8, 16 and its tcgen05 prefill at M = 512, 2048, 4096,
    and the block / MXFP8 / per-row / per-tensor
    load-time quantizers.  Returns ({name: record}, kernel launches)."""
    out, launches = {}, 0

    def run(name, wl, workload):
        nonlocal launches
        per, total = time_calls(torch, wl["calls"], steps, warmup, None, graph=wl.get("graph", False))
        value, unit, per_call, roofline = summarize(wl, per, total, steps, workload)
        out[name] = {"workload": wl["cfg"]["workload"], "value": round(value, 2), "unit": unit,
                     "ms_per_step": round(total / steps, 4), "per_call": per_call, "roofline": roofline}
        lpc = wl.get("call_launches", [wl.get("launches_per_call", 1)] * len(wl["calls"]))
        launches += 2 * steps * sum(lpc) * wl.get("launches_per_step", 1)   # timed pass + per-call pass
        torch.cuda.synchronize()
        if fp8bs.check_device_error() != 0:
            raise RuntimeError(f"device error word set while timing {name}")

    weights = rotation_weights(fp8bs, inputs, dev)
    for m in (1, 8, 16, 32):
        run(f"rotation M={m}", rotation_workload(torch, fp8bs, inputs, dev, m, weights=weights), "rotation")
    del weights
    run("sweep", sweep_workload(torch, fp8bs, inputs, dev, [1, 9, 17, 25, 32]), "sweep")
    run("prefill", prefill_workload(torch, fp8bs, inputs, dev), "prefill")
    run("mx", mx_workload(torch, fp8bs, inputs, dev), "mx")
    run("mx_prefill", mx_prefill_workload(torch, fp8bs, inputs, dev), "mx_prefill")
    run("quantize", quantize_workload(torch, fp8bs, inputs, dev), "quantize")
    torch.cuda.empty_cache()
    return out, launches


# -------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="lm_head",
                    choices=["lm_head", "rotation", "sweep", "mx", "mx_prefill", "quantize", "prefill", "rowwise", "w8a8",
                             "moe_prefill",
                             "w8a8_prefill", "moe", "kv"])
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--layers", type=int, default=None, help="rotation: fewer layers than 48 (a smaller case)")
    ap.add_argument("--experts", type=int, default=None,
                    help="moe_prefill: fewer experts than 256 (a smaller case)")
    ap.add_argument("--single", action="store_true", help="rotation: one GEMV call per weight, not one batch")
    ap.add_argument("--ws", action="store_true", help="sweep: call fp8bs_gemv_ws (x prepared in a workspace)")
    ap.add_argument("--scales", default="block", choices=["block", "row", "tensor"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="lm_head: skip the other configurations (rotation, sweep, prefill, MXFP8, quantize)")
    ap.add_argument("--clocks-file", default=os.path.join(tempfile.gettempdir(), "fp8bs_bench_clocks.csv"),
                    help="raw nvidia-smi samples taken during the timed region (summarised in the JSON line)")
    args = ap.parse_args()
    warmup = max(3, args.warmup)
    peak, peak_kind = measured_peaks()

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        # the oracle as it stands on all host cores; each step is the bounded
        # lm_head sample of oracle_gemv_step (the cpu_baseline leg's sample)
        threads = host_cores()
        for _ in range(warmup):
            oracle_gemv_step(threads)
        per_step = [oracle_gemv_step(threads) for _ in range(args.steps)]
        value = statistics.fmean(v for v, _ in per_step)
        ms_step = 1e3 * statistics.fmean(s for _, s in per_step)
        # the same metric, unit and config as this file's own lm_head line;
        # the oracle processes a sample of the rows (cpu_baseline.sample)
        line = {"impl": "reference", "metric": LM_HEAD_METRIC,
                "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": len(per_step),
                "warmup": warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": dict(lm_head_config(152064, 4096, [1, 4, 8, 16]), parallelism=f"replicas x{args.gpus}"),
                "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                 "sample": oracle_sample_desc(threads)},
                "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    rank, world, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import fp8_block_scaled_02_gb300 as fp8bs
    from fp8_block_scaled_02_gb300 import inputs
    fp8bs.lib()

    if args.workload == "lm_head":
        wl = lm_head_workload(torch, fp8bs, inputs, dev)
    elif args.workload == "rotation":
        wl = rotation_workload(torch, fp8bs, inputs, dev, args.m, args.scales, batched=not args.single,
                               layers=args.layers)
    elif args.workload == "sweep":
        wl = sweep_workload(torch, fp8bs, inputs, dev, list(range(1, 33)), ws=args.ws)
    elif args.workload == "mx":
        wl = mx_workload(torch, fp8bs, inputs, dev)
    elif args.workload == "prefill":
        wl = prefill_workload(torch, fp8bs, inputs, dev, args.scales)
    elif args.workload == "mx_prefill":
        wl = mx_prefill_workload(torch, fp8bs, inputs, dev)
    elif args.workload == "rowwise":
        wl = rowwise_workload(torch, fp8bs, inputs, dev)
    elif args.workload == "w8a8":
        wl = w8a8_workload(torch, fp8bs, inputs, dev)
    elif args.workload == "w8a8_prefill":
        wl = w8a8_prefill_workload(torch, fp8bs, inputs, dev)
    elif args.workload == "moe":
        wl = moe_workload(torch, fp8bs, inputs, dev)
    elif args.workload == "moe_prefill":
        wl = moe_prefill_workload(torch, fp8bs, inputs, dev, experts=args.experts)
    elif args.workload == "kv":
        wl = kv_workload(torch, fp8bs, inputs, dev)
    else:
        wl = quantize_workload(torch, fp8bs, inputs, dev)
    torch.cuda.synchronize()
    if fp8bs.check_device_error() != 0:
        raise RuntimeError("device error word set during set-up")

    calls = wl["calls"]
    os.makedirs(os.path.dirname(args.clocks_file), exist_ok=True)
    with Clocks(args.clocks_file) as clk:
        per, total_ms = time_calls(torch, calls, args.steps, warmup, pg, graph=wl.get("graph", False))
    clocks = clk.summary() if rank == 0 else None
    if fp8bs.check_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    step_bytes = sum(b for _, _, b, _ in calls)
    total_ms = max_over_ranks(pg, total_ms)
    all_bytes = sum_over_ranks(pg, step_bytes * args.steps)
    _, unit, per_call, roofline = summarize(wl, per, total_ms, args.steps, args.workload)
    value = all_bytes / (total_ms * 1e-3) / (1e12 if wl.get("flops", False) else 1e9)

    e2e = None
    if args.workload == "lm_head":
        e2e_ms, h2d, d2h = e2e_lm_head(torch, fp8bs, wl, max(1, args.steps // 4), warmup, pg)
        e2e_ms = max_over_ranks(pg, e2e_ms)
        e_bytes = sum_over_ranks(pg, step_bytes * max(1, args.steps // 4))
        e2e = {"value": round(e_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == "lm_head":
        threads = host_cores()
        v, _ = oracle_gemv_step(threads, min_seconds=ORACLE_MIN_SECONDS)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": oracle_sample_desc(threads), "runs": oracle_runs(sorted({1, threads}))}

    per_call_launches = wl.get("call_launches", [wl.get("launches_per_call", 1)] * len(calls))
    launches = args.steps * sum(per_call_launches) * wl.get("launches_per_step", 1)
    cfg = dict(wl["cfg"], parallelism=f"replicas x{world}")

    extras = None
    if args.workload == "lm_head" and world == 1 and not args.no_extras:
        del wl, calls
        torch.cuda.empty_cache()
        with Clocks(args.clocks_file + ".extras") as clk2:
            recs, extra_launches = extra_configs(torch, fp8bs, inputs, dev, min(args.steps, 20), warmup)
        extras = {"clocks": clk2.summary(), "gpu_launches": extra_launches, **recs}

    if rank == 0:
        line = {"metric": LM_HEAD_METRIC if args.workload == "lm_head"
                else f"{args.workload} {unit}",
                "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
                "warmup": warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x bf16 -> fp32", "data": "synthetic",
                "config": cfg,
                "per_call": per_call, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "clocks": clocks, "gpu_launches": launches}
        if extras is not None:
            line["configs"] = extras
        print(json.dumps(line))
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
