#!/usr/bin/env python
"""Benchmark: block-sparse attention throughput on one GB300 (per rank).

One step = one block-sparse attention forward, O = softmax(scale Q K^T on the
layout) V, over one batch of the workload (default: the banded workload,
Z=4 H=16 S=8192 D=128 B=128 bf16, block band |i-j| <= 4).  The fused kernel
does SDD -> softmax -> DSD in one pass.  Throughput counts nonzero-block FLOPs
only: 4 * B^2 * D per present block per batch entry.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-sparse attention TFLOP/s (nonzero-block FLOPs) and % of GB300 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
W_ATTENTION = ("band", "strided", "bigbird", "tiny")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="band", choices=["band", "strided", "bigbird", "tiny"])
    p.add_argument("--no-ops", action="store_true", help="skip the per-op section")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other workloads' attention / softmax / spMM section")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="target oracle CPU time")
    p.add_argument("--skip-cpu", action="store_true", help="no CPU-baseline leg (profiling runs)")
    p.add_argument("--skip-e2e", action="store_true", help="no end-to-end leg (profiling runs)")
    p.add_argument("--split", action="store_true",
                   help="under torchrun: split ONE batch of the workload across the ranks by nnz-balanced "
                        "(batch, head) ranges (strong scaling) instead of one batch per rank (weak scaling)")
    p.add_argument("--graph", action="store_true",
                   help="replay each step from a captured CUDA graph (launch-bound workloads)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if self.proc is None or not self.lines:
            return None
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ helpers --

def workload(name):
    from sparse_attention_layout_gb300 import workloads as W
    return W.ATTENTION_WORKLOADS[name]


def nonzero_flops(lay, B, D, Z):
    return 4.0 * B * B * D * int(lay.sum()) * Z


def input_bytes(w):
    return 4 * w.Z * w.H * w.S * w.D * (2 if w.dtype != "f32" else 4)


def config_of(w, lay, path_name, flush):
    nnz = int(lay.sum())
    if flush is None:
        l2 = "host run (no GPU caches involved)"
    elif flush:
        l2 = (f"L2 flushed before every timed step (Q, K, V, O total {input_bytes(w) / 1e6:.1f} MB fit in L2): "
              "a buffer of twice the L2 size is written outside the timed spans, each step timed by its own events")
    else:
        l2 = f"inputs larger than L2: Q, K, V, O total {input_bytes(w) / 1e6:.0f} MB, no flush"
    return {
        "workload": f"{w.name}: Z{w.Z} H{w.H} S{w.S} D{w.D} B{w.B} {w.dtype}, "
                    f"{nnz} of {w.H * w.nb * w.nb} blocks present ({100.0 * nnz / (w.H * w.nb * w.nb):.1f}%)",
        "Z": w.Z, "H": w.H, "S": w.S, "D": w.D, "block": w.B, "nnz_blocks": nnz,
        "mask": ["none", "dense", "diag_causal"][w.mask_kind], "scale": w.scale,
        "path": path_name,
        "l2": l2,
    }


def kernel_source_sha():
    """Hash of the fused attention kernel's own sources (the kernel whose DRAM
    traffic profiles/traffic.json records)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "sparse_attention_layout_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if not f.startswith("tc_attention"):
            continue
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def launches_per_call(bsp, L, Z, dtype, device):
    """Kernels one bsp_attention call launches: the fused kernel, plus the
    combine pass when its schedule cuts tiles."""
    import torch
    from sparse_attention_layout_gb300 import workloads as W
    n_sm = torch.cuda.get_device_properties(device).multi_processor_count
    sc = bsp.bsp_diag_attention_schedule(L, Z, n_sm, W.torch_dtype(dtype))
    return 1 + (len(sc["combine"]) > 0)


def traffic_for(kernel, wname):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(f"{kernel}:{wname}")
    if not e or e.get("source_sha") != kernel_source_sha():
        return None
    return e.get("bytes_per_launch")


def cpu_oracle_sample(w, lay, Q, K, V, target_s, seed=0):
    """Time the oracle on a seeded sample of rows; returns (TFLOP/s, rows, seconds)."""
    import oracle
    orc = oracle.Oracle()
    rng = np.random.default_rng(seed)
    total_rows = w.Z * w.H * w.S
    rows_blocks = lay.sum(axis=2)  # [H, nb]

    def flops_of(sel):
        zh, r = sel // w.S, sel % w.S
        h = zh % w.H
        return float(np.sum(4.0 * w.B * w.D * rows_blocks[h, r // w.B]))

    n = 64
    while True:
        sel = np.sort(rng.choice(total_rows, size=min(n, total_rows), replace=False))
        t0 = time.perf_counter()
        orc.attention(lay, w.B, Q, K, V, w.scale, w.mask_kind, None, sel=sel)
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= total_rows:
            return flops_of(sel) / dt / 1e12, int(sel.size), dt, orc.num_threads()
        n = min(total_rows, int(n * max(2.0, min(16.0, 1.2 * target_s / max(dt, 1e-3)))))


# --------------------------------------------------------------- reference --

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload(args.workload)
    lay = w.layout()
    Q, K, V = w.qkv()
    import oracle
    orc = oracle.Oracle()
    rng = np.random.default_rng(123)
    total_rows = w.Z * w.H * w.S
    rows_blocks = lay.sum(axis=2)
    per_step = max(16, min(total_rows, 256))
    # calibrate the sample so one step is about 0.5 s of CPU work
    sel = np.sort(rng.choice(total_rows, size=per_step, replace=False))
    t0 = time.perf_counter()
    orc.attention(lay, w.B, Q, K, V, w.scale, w.mask_kind, None, sel=sel)
    dt = time.perf_counter() - t0
    per_step = int(max(16, min(total_rows, per_step * 0.5 / max(dt, 1e-4))))
    flops = 0.0
    for _ in range(args.warmup):
        sel = np.sort(rng.choice(total_rows, size=per_step, replace=False))
        orc.attention(lay, w.B, Q, K, V, w.scale, w.mask_kind, None, sel=sel)
    t_total = 0.0
    for _ in range(args.steps):
        sel = np.sort(rng.choice(total_rows, size=per_step, replace=False))
        zh, r = sel // w.S, sel % w.S
        flops += float(np.sum(4.0 * w.B * w.D * rows_blocks[zh % w.H, r // w.B]))
        t0 = time.perf_counter()
        orc.attention(lay, w.B, Q, K, V, w.scale, w.mask_kind, None, sel=sel)
        t_total += time.perf_counter() - t0
    value = flops / t_total / 1e12
    sample = f"{per_step} random rows of {total_rows} per step (all heads and batch entries)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, lay, "fp64 CPU oracle (dense-mask definition)", None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours --

def max_over_ranks(ms: float, world: int, device: str) -> float:
    """Slowest rank's time: the job finishes when the last rank does.  The
    only collective of the multi-GPU path (no data-path exchange)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_value(flops_per_rank: float, world: int, ms_step: float) -> float:
    """Whole-job TFLOP/s: every rank processes its own batch of the workload."""
    return flops_per_rank * world / (ms_step * 1e-3) / 1e12


_FLUSH = None


def time_launches(fn, n, stream, warmup=3):
    """Average device time of fn over n calls, each timed by its own events
    after a write of twice the L2 size (outside the timed span), so that no
    call finds its inputs in L2 left there by the previous one."""
    import torch
    global _FLUSH
    if _FLUSH is None:
        _FLUSH = torch.empty(2 * torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size,
                             dtype=torch.uint8, device="cuda")
    for _ in range(warmup):  # first launches load the module and build tensor maps
        fn()
    torch.cuda.synchronize()
    spans = []
    for _ in range(n):
        _FLUSH.fill_(1)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b_.record(stream)
        spans.append((a, b_))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b_) for a, b_ in spans) / n  # ms per call


def per_op_section(w, lay, L, q, k, v, pk, bsp, stream):
    """Times each step of the unfused chain and the general spMM modes (every
    call cold in L2)."""
    import torch
    from sparse_attention_layout_gb300 import workloads as W
    out = {}
    elt = 2 if w.dtype != "f32" else 4
    Z, B, D, nnz = w.Z, w.B, w.D, int(lay.sum())
    P = bsp.bsp_sdd(L, q, k)
    ms = time_launches(lambda: bsp.bsp_sdd(L, q, k, P), 10, stream)
    out["sdd"] = {"ms": ms, "TFLOP/s": 2.0 * B * B * D * nnz * Z / ms / 1e9,
                  "GB/s": (Z * nnz * B * B * elt) / ms / 1e6}
    # the other operand orientations: an operand stored [K][S] is read MN-major
    if w.dtype != "f32":
        qt, kt = q.transpose(-1, -2).contiguous(), k.transpose(-1, -2).contiguous()
        out["sdd_trans"] = {}
        for ta, tb in ((0, 0), (1, 0), (1, 1)):
            a_op, b_op = (qt if ta else q), (k if tb else kt)
            ms = time_launches(lambda: bsp.bsp_sdd(L, a_op, b_op, P, trans_a=ta, trans_b=tb), 10, stream)
            out["sdd_trans"][f"ta{ta}_tb{tb}"] = {"ms": ms, "GB/s": (Z * nnz * B * B * elt) / ms / 1e6}
        del qt, kt
    X = P.clone()
    ms = time_launches(lambda: bsp.bsp_softmax(L, X, P, w.scale, w.mask_kind), 10, stream)
    sbytes = 2.0 * Z * nnz * B * B * elt
    out["softmax"] = {"ms": ms, "GB/s": sbytes / ms / 1e6,
                      "frac_of_hbm": sbytes / ms / 1e6 / pk["hbm_gbs"],
                      "algorithmic_bytes": sbytes}
    O = torch.empty_like(q)
    ms = time_launches(lambda: bsp.bsp_dsd(L, P, v, O), 10, stream)
    out["dsd"] = {"ms": ms, "TFLOP/s": 2.0 * B * B * D * nnz * Z / ms / 1e9}
    ms = time_launches(lambda: bsp.attention_unfused(L, q, k, v, w.scale, w.mask_kind), 5, stream)
    out["attention_unfused_chain"] = {"ms": ms, "TFLOP/s": nonzero_flops(lay, B, D, Z) / ms / 1e9}
    # SDD and softmax fused (scores never in HBM), then DSD
    ms = time_launches(lambda: bsp.bsp_sdd_softmax(L, q, k, P, w.scale, w.mask_kind), 10, stream)
    out["sdd_softmax"] = {"ms": ms, "GB/s_of_P": (Z * nnz * B * B * elt) / ms / 1e6}
    ms = time_launches(lambda: bsp.bsp_dsd(L, bsp.bsp_sdd_softmax(L, q, k, P, w.scale, w.mask_kind), v, O), 5,
                       stream)
    out["attention_sdd_softmax_dsd"] = {"ms": ms, "TFLOP/s": nonzero_flops(lay, B, D, Z) / ms / 1e9}
    # backward: softmax backward on the chain's P, and the whole attention
    # backward (recomputes P; 5 block matmuls of 2 B^2 D each per block)
    dY = torch.randn_like(P)
    dX = torch.empty_like(P)
    ms = time_launches(lambda: bsp.bsp_softmax_backward(L, P, dY, dX, w.scale), 10, stream)
    byt = 3.0 * P.numel() * P.element_size()
    out["softmax_backward"] = {"ms": ms, "GB/s": byt / ms / 1e6, "frac_of_hbm": byt / ms / 1e6 / pk["hbm_gbs"],
                               "algorithmic_bytes": byt}
    del dY, dX
    gO = torch.randn_like(q)
    ms = time_launches(lambda: bsp.attention_backward(L, q, k, v, gO, w.scale, w.mask_kind), 5, stream)
    fl = 10.0 * B * B * D * nnz * Z
    out["attention_backward"] = {"ms": ms, "TFLOP/s": fl / ms / 1e9, "flops_counted": "10 B^2 D per block",
                                 "api": "bsp_attention_backward (recomputes the softmax statistics)"}
    # the autograd path: the forward keeps O and the rows' log-sum-exp
    Of, lse = bsp.bsp_attention_lse(L, q, k, v, None, None, w.scale, w.mask_kind)
    ms = time_launches(lambda: bsp.attention_backward_lse(L, q, k, v, Of, gO, lse, w.scale, w.mask_kind), 5,
                       stream)
    out["attention_backward_lse"] = {"ms": ms, "TFLOP/s": fl / ms / 1e9, "flops_counted": "10 B^2 D per block",
                                     "api": "bsp_attention_backward_lse (O and lse of bsp_attention_lse)"}
    del P, X, O, gO, Of, lse
    # general spMM at 10 % density (8192^2 sparse, 8192x4096 dense, block 32)
    sp = W.SPMM
    lay4 = sp.layout(0.10)
    L4 = bsp.bsp_layout_compile(lay4, sp.B)
    A = sp.sparse_values(L4.nnz, 0.10).cuda()
    Bd = sp.dense_dsd(0.10).cuda()
    Ad = sp.dense_dds(0.10).cuda()
    C1 = bsp.bsp_dsd(L4, A, Bd)
    ms = time_launches(lambda: bsp.bsp_dsd(L4, A, Bd, C1), 10, stream)
    fl = 2.0 * sp.B * sp.B * sp.N * L4.nnz
    out["dsd_spmm_10pct"] = {"ms": ms, "TFLOP/s": fl / ms / 1e9, "frac_of_bf16_peak": fl / ms / 1e9 / pk["bf16_tflops"]}
    C2 = bsp.bsp_dds(L4, Ad, A)
    ms = time_launches(lambda: bsp.bsp_dds(L4, Ad, A, C2), 10, stream)
    out["dds_spmm_10pct"] = {"ms": ms, "TFLOP/s": fl / ms / 1e9, "frac_of_bf16_peak": fl / ms / 1e9 / pk["bf16_tflops"]}
    del A, Bd, Ad, C1, C2
    # the same shapes at the other block sizes, 10 % and 50 % density
    out["spmm_blocks"] = {}
    for bs, spb in W.SPMM_BLOCKS.items():
        for dens in W.SPMM_BLOCK_DENSITIES:
            layb = spb.layout(dens)
            Lb = bsp.bsp_layout_compile(layb, bs)
            A = spb.sparse_values(Lb.nnz, dens).cuda()
            Bd, Ad = spb.dense_dsd(dens).cuda(), spb.dense_dds(dens).cuda()
            C1, C2 = bsp.bsp_dsd(Lb, A, Bd), bsp.bsp_dds(Lb, Ad, A)
            fl = 2.0 * bs * bs * spb.N * Lb.nnz
            ms1 = time_launches(lambda: bsp.bsp_dsd(Lb, A, Bd, C1), 10, stream)
            ms2 = time_launches(lambda: bsp.bsp_dds(Lb, Ad, A, C2), 10, stream)
            out["spmm_blocks"][f"B{bs}_{int(round(dens * 100))}pct"] = {
                "dsd_ms": ms1, "dsd_TFLOP/s": fl / ms1 / 1e9, "dds_ms": ms2, "dds_TFLOP/s": fl / ms2 / 1e9,
                "frac_of_bf16_peak": [fl / ms1 / 1e9 / pk["bf16_tflops"], fl / ms2 / 1e9 / pk["bf16_tflops"]]}
            del A, Bd, Ad, C1, C2, Lb
    return out


# nominal dense tensor-core rates per GPU (PFLOP/s): bf16 2.25, tf32 1.1
TF32_PER_BF16 = 1.1 / 2.25
# the fp32 attention kernel takes each fp32 product as three TF32 products
TF32_PRODUCTS = 3


def attention_roofline(w, achieved, pk, pk_kind):
    if w.dtype != "f32":
        peak, src = pk["bf16_tflops"], f"bf16_tflops (burst) of {pk_kind}"
        extra = {}
    else:
        # fp32 runs on the tensor cores as three TF32 products (hi*hi + hi*lo
        # + lo*hi); its peak is the TF32 rate: the measured bf16 peak times the
        # nominal tf32 / bf16 ratio.  `frac` counts the algorithmic FLOPs,
        # `issued_frac` the tensor-core FLOPs issued for them.
        peak = pk["bf16_tflops"] * TF32_PER_BF16 if pk.get("bf16_tflops") else None
        src = f"tf32 = bf16_tflops (burst) of {pk_kind} x 1.1 / 2.25 (nominal ratio)"
        extra = {"tf32_products_per_fp32_product": TF32_PRODUCTS,
                 "issued_frac": TF32_PRODUCTS * achieved / peak if peak else None}
    return {"bound": "tensor", "kernel": "attention", "achieved": achieved, "peak": peak, "peak_source": src,
            "unit": "TFLOP/s", "frac": achieved / peak if peak else None, **extra}


def workload_section(w, bsp, stream, steps, warmup, pk, pk_kind, local):
    """One attention workload timed the way the headline is (W warm-ups, K
    timed launches, L2 flushed before each step when the inputs fit in L2,
    clocks sampled during the timed steps), plus its softmax on SDD-shaped
    input (every call cold in L2), each against its own roofline."""
    import torch
    lay = w.layout()
    L = bsp.bsp_layout_compile(lay, w.B)
    Qc, Kc, Vc = w.qkv()
    q, k, v = (t.cuda() for t in (Qc, Kc, Vc))
    o = torch.empty_like(q)
    flops = nonzero_flops(lay, w.B, w.D, w.Z)
    l2_bytes = torch.cuda.get_device_properties(local).L2_cache_size
    flush = input_bytes(w) < 2 * l2_bytes
    scratch = torch.empty(2 * l2_bytes if flush else 0, dtype=torch.uint8, device="cuda")
    for _ in range(max(3, warmup)):
        bsp.bsp_attention(L, q, k, v, o, w.scale, w.mask_kind)
    torch.cuda.synchronize()
    if bsp.bsp_status_check(L) != 0:
        raise RuntimeError(f"device status after warm-up of {w.name}")
    with ClockSampler(local) as clk:
        spans = []
        if flush:
            for _ in range(steps):
                scratch.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                bsp.bsp_attention(L, q, k, v, o, w.scale, w.mask_kind)
                e1.record(stream)
                spans.append((e0, e1))
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                bsp.bsp_attention(L, q, k, v, o, w.scale, w.mask_kind)
            e1.record(stream)
            spans.append((e0, e1))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b_) for a, b_ in spans) / steps
        # softmax of SDD-shaped input in the workload's dtype
        X = W_randn((w.Z, L.nnz, w.B, w.B), w.dtype, 77).cuda()
        Y = torch.empty_like(X)
        sms = time_launches(lambda: bsp.bsp_softmax(L, X, Y, w.scale, w.mask_kind), steps, stream)
        # its backward: Y that softmax's output, dY random of the same shape
        G = W_randn((w.Z, L.nnz, w.B, w.B), w.dtype, 79).cuda()
        dX = torch.empty_like(X)
        sbms = time_launches(lambda: bsp.bsp_softmax_backward(L, Y, G, dX, w.scale), steps, stream)
        del Y, G, dX
        # 16-bit workloads: the backward from the forward's O and log-sum-exp
        # (the autograd path), every call cold in L2
        bwd = None
        if w.dtype != "f32":
            gO = W_randn(tuple(q.shape), w.dtype, 78).cuda()
            Of, lse = bsp.bsp_attention_lse(L, q, k, v, None, None, w.scale, w.mask_kind)
            bms = time_launches(lambda: bsp.attention_backward_lse(L, q, k, v, Of, gO, lse, w.scale, w.mask_kind),
                                5, stream)
            bfl = 2.5 * flops  # 10 B^2 D per block against the forward's 4 B^2 D
            bwd = {"ms": bms, "TFLOP/s": bfl / bms / 1e9, "flops_counted": "10 B^2 D per block",
                   "api": "bsp_attention_backward_lse (O and lse of bsp_attention_lse)"}
            del gO, Of, lse
    clocks = clk.summary()
    achieved = flops / (ms * 1e-3) / 1e12
    sbytes = 2.0 * X.numel() * X.element_size()
    gbs = sbytes / sms / 1e6
    sbbytes = 1.5 * sbytes  # Y and dY read, dX written
    sbgbs = sbbytes / sbms / 1e6
    out = {
        "config": config_of(w, lay, "fused attention kernel", flush),
        "attention": {"ms": ms, "TFLOP/s": achieved, "gpu_launches": steps * launches_per_call(bsp, L, w.Z, w.dtype, local),
                      "roofline": dict(attention_roofline(w, achieved, pk, pk_kind),
                                       traffic=traffic_for("attention", w.name), algorithmic_flops_per_launch=flops)},
        "softmax": {"ms": sms, "GB/s": gbs,
                    "roofline": {"bound": "hbm", "kernel": "softmax", "achieved": gbs, "peak": pk["hbm_gbs"],
                                 "peak_source": f"hbm_gbs of {pk_kind}", "unit": "GB/s",
                                 "frac": gbs / pk["hbm_gbs"], "algorithmic_bytes_per_launch": sbytes}},
        "softmax_backward": {"ms": sbms, "GB/s": sbgbs,
                             "roofline": {"bound": "hbm", "kernel": "softmax backward", "achieved": sbgbs,
                                          "peak": pk["hbm_gbs"], "peak_source": f"hbm_gbs of {pk_kind}",
                                          "unit": "GB/s", "frac": sbgbs / pk["hbm_gbs"],
                                          "algorithmic_bytes_per_launch": sbbytes}},
        "clocks": clocks,
    }
    if bwd is not None:
        out["attention_backward_lse"] = bwd
    del X, q, k, v, o, scratch
    return out


def spmm_section(bsp, stream, steps, pk, pk_kind, local, B=32, density=0.25):
    """DSD and DDS on the general spMM workload (8192^2 sparse, 8192 x 4096
    dense, bf16) at one block size and density, every call cold in L2."""
    import torch
    from sparse_attention_layout_gb300 import workloads as W
    sp = W.SPMM_BLOCKS[B]
    lay = sp.layout(density)
    L = bsp.bsp_layout_compile(lay, B)
    A = sp.sparse_values(L.nnz, density).cuda()
    Bd, Ad = sp.dense_dsd(density).cuda(), sp.dense_dds(density).cuda()
    C1, C2 = bsp.bsp_dsd(L, A, Bd), bsp.bsp_dds(L, Ad, A)
    fl = 2.0 * B * B * sp.N * L.nnz
    with ClockSampler(local) as clk:
        ms1 = time_launches(lambda: bsp.bsp_dsd(L, A, Bd, C1), steps, stream)
        ms2 = time_launches(lambda: bsp.bsp_dds(L, Ad, A, C2), steps, stream)
    out = {"workload": f"spmm: sparse {sp.S}x{sp.S} (block {B}, {L.nnz} of {(sp.S // B) ** 2} blocks, "
                       f"{100 * density:.0f}%) x dense {sp.S}x{sp.N}, bf16",
           "clocks": clk.summary()}
    for name, ms in (("dsd", ms1), ("dds", ms2)):
        t = fl / ms / 1e9
        out[name] = {"ms": ms, "TFLOP/s": t,
                     "roofline": {"bound": "tensor", "kernel": "spmm_group", "achieved": t,
                                  "peak": pk["bf16_tflops"], "peak_source": f"bf16_tflops (burst) of {pk_kind}",
                                  "unit": "TFLOP/s", "frac": t / pk["bf16_tflops"]}}
    del A, Bd, Ad, C1, C2
    return out


def W_randn(shape, dtype, seed):
    from sparse_attention_layout_gb300 import workloads as W
    return W.randn(shape, dtype, seed)


def run_ours(args):
    import torch
    import torch.distributed as dist
    from sparse_attention_layout_gb300 import build as b
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        b.build()
    if world > 1:
        dist.barrier()
    from sparse_attention_layout_gb300 import bsp

    w = workload(args.workload)
    lay_full = lay = w.layout()
    split = args.split and world > 1
    if split:
        # this rank's share of ONE batch: a contiguous range of (batch, head)
        # pairs balanced by present blocks, run as batch 1 with those heads
        from sparse_attention_layout_gb300 import partition
        u0, u1, lay = partition.shard_layout(lay_full, w.Z, rank, world)
        Qc, Kc, Vc = (t.reshape(1, w.Z * w.H, w.S, w.D)[:, u0:u1].contiguous() for t in w.qkv())
        args.no_ops = args.no_workloads = args.skip_e2e = True
    else:
        Qc, Kc, Vc = w.qkv(shard=rank)  # each rank: its own batch (weak scaling)
    Zr = 1 if split else w.Z
    stream = torch.cuda.current_stream()
    L = bsp.bsp_layout_compile(lay, w.B) if lay.shape[0] else None
    q, k, v = (t.cuda() for t in (Qc, Kc, Vc))
    o = torch.empty_like(q)
    pk, pk_kind = peaks()

    def step():
        if L is not None:
            bsp.bsp_attention(L, q, k, v, o, w.scale, w.mask_kind)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    status = bsp.bsp_status_check(L) if L is not None else 0
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")
    if args.graph:
        # one step captured once and replayed: the kernel launch without the
        # per-call host work (argument checks, tensor-map encoding)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        with torch.cuda.graph(graph):
            step()
        step = graph.replay
        for _ in range(3):
            step()
        torch.cuda.synchronize()

    # inputs that fit in L2 are timed cold: flush before every step, outside
    # the timed spans
    l2_bytes = torch.cuda.get_device_properties(local).L2_cache_size
    flush = input_bytes(w) < 2 * l2_bytes
    scratch = torch.empty(2 * l2_bytes if flush else 0, dtype=torch.uint8, device="cuda")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        if flush:
            spans = []
            for _ in range(args.steps):
                scratch.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                step()
                e1.record(stream)
                spans.append((e0, e1))
            torch.cuda.synchronize()
            total_ms = sum(a.elapsed_time(b_) for a, b_ in spans)
        else:
            start.record(stream)
            for _ in range(args.steps):
                step()
            end.record(stream)
            torch.cuda.synchronize()
            total_ms = start.elapsed_time(end)
        if world > 1:
            dist.barrier()
    ms = max_over_ranks(total_ms, world, "cuda")
    ms_step = ms / args.steps
    flops = nonzero_flops(lay, w.B, w.D, Zr)  # this rank's launch
    if split:
        value = nonzero_flops(lay_full, w.B, w.D, w.Z) / (ms_step * 1e-3) / 1e12  # one batch / slowest rank
    else:
        value = weak_value(flops, world, ms_step)
    achieved = flops / (ms_step * 1e-3) / 1e12  # one attention launch per step

    # end to end through the C ABI with host buffers: bsp_attention_host takes
    # the pinned host inputs and output; every step copies Q, K, V in and O
    # out (slices of half the batch, copies overlapped with the kernels; slices
    # of one batch entry measured 0.6 % slower: twice the copies)
    Qh, Kh, Vh = (t.pin_memory() for t in (Qc, Kc, Vc))
    Oh = torch.empty_like(Qc).pin_memory()
    ws = None if split else torch.empty(bsp.bsp_attention_host_workspace(L, Qc.dtype, w.D, max(1, w.Z // 2)),
                                        dtype=torch.uint8, device="cuda")

    def e2e_step():
        bsp.bsp_attention_host(L, Qh, Kh, Vh, Oh, w.scale, w.mask_kind, workspace=ws, reserved_workspace=True)

    e2e_ms = None
    if not args.skip_e2e:
        # one pair of events around all the steps: a step's input copies may
        # start during the previous step's tail, so only the whole run's span
        # counts every copy
        e2e_steps = max(3, min(args.steps, 20))
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_start.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e_end.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e_start.elapsed_time(e_end) / e2e_steps
    h2d = 3 * Qc.numel() * Qc.element_size()
    d2h = Oh.numel() * Oh.element_size()

    ops = None
    if not args.no_ops and rank == 0:
        ops = per_op_section(w, lay, L, q, k, v, pk, bsp, stream)
    torch.cuda.synchronize()
    # the other attention workloads and the spMM workload at 25 %, each with
    # its own clocks and rooflines (rank 0; the headline above is the job's)
    workloads = None
    if not args.no_workloads and rank == 0:
        del q, k, v, o
        torch.cuda.empty_cache()
        workloads = {}
        for name in W_ATTENTION:
            if name != w.name:
                workloads[name] = workload_section(workload(name), bsp, stream, args.steps, args.warmup, pk,
                                                   pk_kind, local)
        workloads["spmm_B32_25pct"] = spmm_section(bsp, stream, min(args.steps, 10), pk, pk_kind, local)
        torch.cuda.synchronize()

    if rank != 0:
        if world > 1:
            dist.barrier()
        return
    cpu = None
    if not args.skip_cpu:
        cpu_val, cpu_rows, cpu_s, cores = cpu_oracle_sample(w, lay_full, *((w.qkv() if split else (Qc, Kc, Vc))),
                                                            args.cpu_seconds)
        cpu = {"value": cpu_val, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{cpu_rows} random rows of {w.Z * w.H * w.S} ({cpu_s:.1f} s, fp64, OpenMP)"}
    if world > 1:
        dist.barrier()
    clocks = clk.summary()
    roof = attention_roofline(w, achieved, pk, pk_kind)
    roof["traffic"] = traffic_for("attention", w.name)
    roof["algorithmic_flops_per_launch"] = flops
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "strong" if split else "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config_of(w, lay_full, "fused attention kernel" + (", replayed from a CUDA graph" if args.graph else "")
                            + (f", one batch split over {world} ranks by nnz-balanced (batch, head) ranges"
                               if split else ""), flush),
        "gpu_launches": args.steps * launches_per_call(bsp, L, Zr, w.dtype, local) if L is not None else 0,
        "roofline": roof,
        "e2e": None if e2e_ms is None else {
            "value": flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "api": "bsp_attention_host (C ABI, pinned host buffers, workspace reserved to the handle)"},
        "cpu_baseline": cpu,
        "clocks": clocks,
        "lib": bsp.lib_path(),
    }
    if ops is not None:
        line["ops"] = ops
    if workloads is not None:
        line["workloads"] = workloads
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
