"""Benchmark of the block-sparse attention hot path on GB300.

One step = forward + backward (rowsum, dK/dV launch, dQ launch) of
block-sparse attention over one batch of synthetic input, with the
compiled MaskInfo (forward and dK/dV orientations) resident on the device.
The default workload is GQA 32/8 causal attention at 8192 tokens, D = 128
(2016 of 4096 blocks skipped per head).

Metric: TFLOP/s over executed blocks.  Forward counts 4*128*128*D FLOP per
executed (label 1 or 2) block and query head; backward counts 2.5x the
forward (five GEMMs: one score recompute, dP, dV, dK, dQ); label-0 blocks
count nothing.  The JSON line also carries the roofline of the dominant
kernel, the oracle timed on the host cores, an end-to-end number through
the public API with host buffers, and clocks sampled during the timed
region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import WORKLOADS, bernoulli_mask, qkvdo  # noqa: E402

METRIC = "splash fwd/bwd TFLOP/s over executed blocks; % of GB300 bf16 tensor peak"
DEFAULT_WORKLOAD = "gqa_causal_s8192"
L2_FLUSH_BYTES = 512 << 20


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": d["bf16_tflops"], "bf16_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


KERNEL_NAMES = {"fwd": "fwd_kernel", "dkv": "dkv_kernel", "dq": "dq_kernel"}


def traffic_per_launch(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu capture, or None when there
    is no capture for this workload or the kernel source changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        ent = json.load(f).get(workload, {}).get(KERNEL_NAMES[kernel])
    if not ent or not ent.get("valid"):
        return None
    src = os.path.join(ROOT, "block_sparse_attention_process_gb300", "csrc", ent["source"])
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != ent["source_sha"]:
            return None
    return ent["bytes_per_launch"]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device=None) -> float:
    """The largest x over the ranks of the default process group (x itself
    when there is none or it has one rank)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_rank: float, seconds: float, world: int) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's time."""
    return world * flop_per_rank / seconds / 1e12


def mask_kwargs(w):
    if w.mask.kind == "local":
        return {"local_left": w.mask.left, "local_right": w.mask.right}
    if w.mask.kind == "chunked":
        return {"chunk": w.mask.chunk}
    return {}


def flops(w, n_exec_per_head):
    fwd = n_exec_per_head * w.B * w.Hq * 4 * 128 * 128 * w.D
    return fwd, 2.5 * fwd


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            self.proc.wait(timeout=5)
        self.file.flush()

    def summary(self):
        self.file.seek(0)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class Prepared:
    """One workload's inputs, compiled MaskInfo (both orientations) and output
    buffers, resident on the device."""

    def __init__(self, bsa, w, dev, seed_offset=0):
        self.bsa, self.w, self.dev = bsa, w, dev
        self.q, self.k, self.v, self.do = qkvdo(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed + seed_offset)
        self.dense_h = bernoulli_mask(w.S, w.mask.p, w.mask.seed) if w.mask.kind == "dense" else None
        self.qd, self.kd, self.vd, self.dod = (t.to(dev) for t in (self.q, self.k, self.v, self.do))
        self.dense_d = None if self.dense_h is None else torch.from_numpy(self.dense_h).to(dev)
        t0 = time.perf_counter()
        self.info, self.dkv = self.compile()
        torch.cuda.synchronize()
        self.compile_cold_ms = (time.perf_counter() - t0) * 1e3
        warm = []
        for _ in range(3):
            t0 = time.perf_counter()
            i2, d2 = self.compile()
            torch.cuda.synchronize()
            warm.append((time.perf_counter() - t0) * 1e3)
            i2.destroy()
            d2.destroy()
        self.compile_ms = sorted(warm)[1]
        d = self.info.desc()
        self.n_exec = (d.n_partial + d.n_full) // d.heads
        self.o = torch.empty_like(self.qd)
        self.lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(self.qd)
        self.dk = torch.empty_like(self.kd)
        self.dv = torch.empty_like(self.vd)
        self.dsum = torch.empty_like(self.lse)

    def compile(self):
        w, bsa = self.w, self.bsa
        info = bsa.mask_compile(w.mask.kind, w.S, w.S, dense=self.dense_d, **mask_kwargs(w))
        dkv = bsa.mask_compile(w.mask.kind, w.S, w.S, dense=self.dense_d, orientation="dkv", **mask_kwargs(w))
        return info, dkv

    def step(self, stream, evs=None, phases=False):
        """forward, rowsum, dK/dV, dQ; with `evs` (5 events) one between
        launches, or with `phases` (3 events) one before the forward, one
        between the forward and the backward and one after the backward (the
        backward's three launches follow each other as in a training step)."""
        bsa = self.bsa
        between = evs is not None and not phases
        if evs is not None:
            evs[0].record(stream)
        bsa.fwd(self.qd, self.kd, self.vd, self.info, o=self.o, lse=self.lse)
        if evs is not None:
            evs[1].record(stream)
        bsa.bwd_rowsum(self.o, self.dod, dsum=self.dsum)
        if between:
            evs[2].record(stream)
        bsa.bwd_dkv(self.qd, self.kd, self.vd, self.o, self.lse, self.dod, self.dsum, self.dkv, dk=self.dk,
                    dv=self.dv)
        if between:
            evs[3].record(stream)
        bsa.bwd_dq(self.qd, self.kd, self.vd, self.o, self.lse, self.dod, self.dsum, self.info, dq=self.dq)
        if between:
            evs[4].record(stream)
        elif evs is not None:
            evs[2].record(stream)

    def time_steps(self, stream, flush, n):
        """Whole steps, events only at step boundaries; L2 flushed between
        steps outside the events.  Returns the per-step times in ms."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            flush.zero_()
            evs[i][0].record(stream)
            self.step(stream)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) for e in evs]

    def time_kernels(self, stream, flush, n):
        """The same steps with an event between launches: mean ms per kernel."""
        kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
        for i in range(n):
            flush.zero_()
            self.step(stream, kevs[i])
        torch.cuda.synchronize()
        per = {"fwd": [], "rowsum": [], "dkv": [], "dq": [], "step": []}
        for e in kevs:
            per["fwd"].append(e[0].elapsed_time(e[1]))
            per["rowsum"].append(e[1].elapsed_time(e[2]))
            per["dkv"].append(e[2].elapsed_time(e[3]))
            per["dq"].append(e[3].elapsed_time(e[4]))
            per["step"].append(e[0].elapsed_time(e[4]))
        # the backward as one phase: its launches back to back, no event between them
        pevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        for i in range(n):
            flush.zero_()
            self.step(stream, pevs[i], phases=True)
        torch.cuda.synchronize()
        per["bwd_phase"] = [e[1].elapsed_time(e[2]) for e in pevs]
        return {k: sum(v) / len(v) for k, v in per.items()}


# Backward work split between the two launches in proportion to the GEMMs each
# executes (dK/dV: S^T, dP^T, dV, dK; dQ: S, dP, dQ): the algorithmic
# backward is 5 GEMMs of the 7 executed, so each launch is credited 5/7 of
# its executed FLOP.
ALG_BWD = 5.0 / 7.0


def kernel_table(w, n_exec, ms, pk, mhz, n_sms):
    """Per-kernel throughput for one workload: algorithmic TFLOP/s and its
    fraction of the measured bf16 peak, executed ("hardware") TFLOP/s, and SM
    cycles per executed block and q head at the sampled SM clock."""
    gemm = n_exec * w.B * w.Hq * 2 * 128 * 128 * w.D
    executed = {"fwd": 2 * gemm, "dkv": 4 * gemm, "dq": 3 * gemm}
    alg = {"fwd": 2 * gemm, "dkv": 4 * gemm * ALG_BWD, "dq": 3 * gemm * ALG_BWD}
    blocks = n_exec * w.B * w.Hq
    out = {}
    for k in executed:
        t = ms[k] * 1e-3
        out[k] = {"ms": round(ms[k], 4),
                  "tflops_alg": round(alg[k] / t / 1e12, 1),
                  "frac_alg": round(alg[k] / t / 1e12 / pk["bf16_tflops"], 4),
                  "tflops_executed": round(executed[k] / t / 1e12, 1),
                  "frac_executed": round(executed[k] / t / 1e12 / pk["bf16_tflops"], 4)}
        if mhz:
            out[k]["sm_cycles_per_block"] = round(t * mhz * 1e6 * n_sms / blocks, 1)
            out[k]["tensor_cycles_per_block"] = {"fwd": 2, "dkv": 4, "dq": 3}[k] * 2 * 128 * 128 * w.D // 8192
    # the backward: its three launches timed as one phase (as they run in a
    # step); the sum of the kernels timed one by one beside it
    sum_ms = ms["rowsum"] + ms["dkv"] + ms["dq"]
    bwd_ms = ms.get("bwd_phase", sum_ms)
    out["bwd"] = {"ms": round(bwd_ms, 4), "tflops_alg": round(5 * gemm / (bwd_ms * 1e-3) / 1e12, 1),
                  "frac_alg": round(5 * gemm / (bwd_ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                  "timed": "rowsum, dK/dV and dQ launched back to back, events around the three",
                  "sum_of_kernels_ms": round(sum_ms, 4),
                  "frac_alg_sum_of_kernels": round(5 * gemm / (sum_ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4)}
    out["rowsum"] = {"ms": round(ms["rowsum"], 4),
                     "gbs": round((4 * w.B * w.Hq * w.S * w.D + 4 * w.B * w.Hq * w.S) / (ms["rowsum"] * 1e-3) / 1e9,
                                  1)}
    return out


def run_gpu(args):
    import block_sparse_attention_process_gb300 as bsa
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    pk = peaks()
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count

    # ---------------------------------------------------------------- inputs (resident in HBM)
    P = Prepared(bsa, w, dev, seed_offset=rank)
    dense_compile = None if args.no_mask_bench else big_dense_compile(bsa, dev)
    perhead_compile = None if args.no_mask_bench else perhead_dense_compile(bsa, dev)
    n_exec = P.n_exec
    f_fwd, f_bwd = flops(w, n_exec)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        flush.zero_()
        P.step(stream)
    assert bsa.get_device_error() == 0

    # ---------------------------------------------------------------- timed region
    # Whole steps, events only at the step boundaries (the four launches of
    # a step follow each other as they would in training).
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        step_times = P.time_steps(stream, flush, args.steps)
    if ws > 1:
        torch.distributed.barrier()
    assert bsa.get_device_error() == 0
    step_ms = sum(step_times) / len(step_times)
    clocks = clk.summary()

    # Per-kernel breakdown (roofline of the dominant kernel): the same steps
    # again with an event between launches.
    with Clocks(local) as kclk:
        ms = P.time_kernels(stream, flush, args.steps)
    assert bsa.get_device_error() == 0
    kclocks = kclk.summary()
    step_ms = max_over_ranks(step_ms, dev)
    value = job_tflops(f_fwd + f_bwd, step_ms * 1e-3, ws)
    mhz = kclocks["sm_mhz"] or clocks["sm_mhz"]
    table = kernel_table(w, n_exec, ms, pk, mhz, n_sms)

    dom = max(("fwd", "dkv", "dq"), key=lambda k: ms[k])
    traffic = traffic_per_launch(args.workload, dom)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": table[dom]["tflops_alg"], "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": table[dom]["frac_alg"], "traffic": traffic,
                "frac_algorithmic": table[dom]["frac_alg"],
                "achieved_executed": table[dom]["tflops_executed"], "frac_executed": table[dom]["frac_executed"],
                "count": "algorithmic: forward 2 GEMMs per executed block and q head; backward 5 GEMMs, each "
                         "launch credited 5/7 of the GEMMs it executes (dK/dV 4, dQ 3); executed = every GEMM run",
                "sm_cycles_per_block": table[dom].get("sm_cycles_per_block"),
                "peak_source": f"{pk['source']} bf16 burst (of measured)" if pk["source"] == "measured"
                else "fallback bf16 burst"}

    # ---------------------------------------------------------------- sustained: seconds of steps
    sustained = None
    if args.sustained_s > 0:
        n = max(args.steps, int(math.ceil(args.sustained_s * 1e3 / max(step_ms, 1e-3))))
        torch.cuda.synchronize()
        with Clocks(local) as sclk:
            st = P.time_steps(stream, flush, n)
        assert bsa.get_device_error() == 0
        s_ms = sum(st) / len(st)
        s_val = (f_fwd + f_bwd) / (s_ms * 1e-3) / 1e12
        peak_s = pk["bf16_sustained"] or pk["bf16_tflops"]
        sustained = {"steps": n, "seconds": round(sum(st) * 1e-3, 2), "ms_per_step": round(s_ms, 4),
                     "value": round(s_val, 2), "unit": "TFLOP/s", "peak": peak_s,
                     "frac": round(s_val / peak_s, 4), "peak_source": "measured bf16 sustained",
                     "clocks": sclk.summary()}

    # ---------------------------------------------------------------- the other workloads
    others = {}
    if not args.no_workloads and ws == 1:
        others = other_workloads(bsa, args, dev, pk, n_sms, flush, stream)

    # ---------------------------------------------------------------- end to end through the public API
    e2e = run_e2e(bsa, w, P.q, P.k, P.v, P.do, P.dense_h, dev, args, f_fwd + f_bwd, ws)

    out = None
    if rank == 0:
        cpu = None if args.no_cpu_baseline or ws > 1 else cpu_baseline(w, P.dense_h, n_exec,
                                                                       seconds=args.cpu_seconds)
        out = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(step_ms, 4),
            "step_ms_spread": {"min": round(min(step_times), 4), "median": round(statistics.median(step_times), 4),
                               "max": round(max(step_times), 4)},
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 Q/K/V/dO; no dataset)",
            "config": {"workload": args.workload, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D,
                       "mask": w.mask.kind, "block": 128, "executed_blocks_per_head": n_exec,
                       "l2": "flushed between steps (512 MiB write, outside the timed events)",
                       "parallelism": f"replicas x{ws} (independent batches, no collective)"},
            "frac_of_peak": round(value / pk["bf16_tflops"], 4),
            "kernels_ms": {k: round(v, 4) for k, v in ms.items()},
            "kernels_note": ("kernels_ms from a second pass with an event between launches (bwd_phase: a third "
                             "pass with events only around the backward's three launches); value from whole steps"),
            "kernels": table,
            "fwd_tflops": table["fwd"]["tflops_alg"],
            "bwd_tflops": table["bwd"]["tflops_alg"],
            "rowsum_gbs": table["rowsum"]["gbs"],
            "mask_compile_ms": round(P.compile_ms, 3),
            "mask_compile_note": "both orientations, warm median of 3 (first, cold: %.3f ms)" % P.compile_cold_ms,
            "mask_dense_compile": dense_compile,
            "mask_dense_perhead_compile": perhead_compile,
            "roofline": roofline,
            "sustained": sustained,
            "workloads": others,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 4 * args.steps,
            "clocks": clocks,
            "clocks_kernel_pass": kclocks,
        }
        print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return out


def big_dense_compile(bsa, dev):
    """The dense-mask compiler on a large mask, where reading it dominates:
    16384 x 16384 bytes (256 MiB) of a causal pattern (all 128 diagonal
    blocks partial and equal), forward orientation, warm median of 3."""
    big_s = 16384
    idx = torch.arange(big_s, device=dev)
    big = (idx[:, None] >= idx[None, :]).to(torch.uint8)
    del idx
    bsa.mask_compile("dense", big_s, big_s, dense=big).destroy()
    dense_ms = []
    for _ in range(3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        bsa.mask_compile("dense", big_s, big_s, dense=big).destroy()
        dense_ms.append((time.perf_counter() - t0) * 1e3)
    del big
    ms = sorted(dense_ms)[1]
    return {"S": big_s, "mask_bytes": big_s * big_s, "ms": round(ms, 3),
            "gbs": round(big_s * big_s / (ms * 1e-3) / 1e9, 1),
            "note": "whole compile (classify, dedup, next-block and shrink passes, host syncs) of a "
                    "causal-pattern byte mask; GB/s = mask bytes / compile time"}


def perhead_dense_compile(bsa, dev, H=16, S=8192):
    """The dense-mask compiler on per-head masks: H heads of S x S bytes
    (1 GiB at 16 x 8192), a quarter each of scattered Bernoulli(0.1) heads
    (every block partial and distinct), causal-pattern heads, band heads
    |q - k| <= 700 and all-ones heads; forward orientation, warm median of
    3.  GB/s = mask bytes / compile time."""
    g = torch.Generator(device=dev).manual_seed(1)
    idx = torch.arange(S, device=dev)
    m = torch.empty((H, S, S), dtype=torch.uint8, device=dev)
    for h in range(H):
        k = h % 4
        if k == 0:
            m[h] = (torch.rand((S, S), generator=g, device=dev) < 0.1).to(torch.uint8)
        elif k == 1:
            m[h] = (idx[:, None] >= idx[None, :]).to(torch.uint8)
        elif k == 2:
            m[h] = ((idx[:, None] - idx[None, :]).abs() <= 700).to(torch.uint8)
        else:
            m[h] = 1
    info = bsa.mask_compile("dense", S, S, dense=m)
    d = info.desc()
    info.destroy()
    times = []
    for _ in range(3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        bsa.mask_compile("dense", S, S, dense=m).destroy()
        times.append((time.perf_counter() - t0) * 1e3)
    del m
    ms = sorted(times)[1]
    return {"heads": H, "S": S, "mask_bytes": H * S * S, "partial_blocks": int(d.n_partial),
            "stack_depth": int(d.num_partial), "ms": round(ms, 3), "gbs": round(H * S * S / (ms * 1e-3) / 1e9, 1),
            "note": "whole compile of a per-head dense mask (classify, dedup, next-block and shrink passes, "
                    "host syncs); GB/s = mask bytes / compile time"}


def run_mask_only(args):
    """--mask-only: the two dense-mask compile measurements alone (also the
    command the mask-compiler ncu captures run)."""
    import block_sparse_attention_process_gb300 as bsa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    out = {"mask_dense_compile": big_dense_compile(bsa, dev),
           "mask_dense_perhead_compile": perhead_dense_compile(bsa, dev)}
    print(json.dumps(out), flush=True)


def other_workloads(bsa, args, dev, pk, n_sms, flush, stream):
    """Every workload but the headline one, measured in the same run: forward,
    dK/dV, dQ and backward throughput at the algorithmic count, per-kernel
    times, SM cycles per block, mask compile time and the oracle timed on
    the host cores on a bounded sample of that workload."""
    out = {}
    for name in sorted(WORKLOADS):
        if name == args.workload:
            continue
        w = WORKLOADS[name]
        P = Prepared(bsa, w, dev)
        for _ in range(args.warmup):
            flush.zero_()
            P.step(stream)
        with Clocks(dev.index) as clk:
            ms = P.time_kernels(stream, flush, max(args.steps, 10))
            st = P.time_steps(stream, flush, max(args.steps, 10))
        assert bsa.get_device_error() == 0
        c = clk.summary()
        f_fwd, f_bwd = flops(w, P.n_exec)
        step_ms = sum(st) / len(st)
        ent = {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D, "mask": w.mask.kind,
               "executed_blocks_per_head": P.n_exec,
               "step_ms": round(step_ms, 4), "step_tflops": round((f_fwd + f_bwd) / (step_ms * 1e-3) / 1e12, 1),
               "kernels": kernel_table(w, P.n_exec, ms, pk, c["sm_mhz"], n_sms),
               "mask_compile_ms": round(P.compile_ms, 3), "clocks": c}
        if w.mask.kind == "dense":
            ent["mask_compile_gbs"] = round(2 * w.S * w.S / (P.compile_ms * 1e-3) / 1e9, 1)
        if not args.no_cpu_baseline:
            ent["cpu_baseline"] = cpu_baseline(w, P.dense_h, P.n_exec, seconds=args.cpu_seconds_other)
        out[name] = ent
        del P
        torch.cuda.empty_cache()
    return out


def run_e2e(bsa, w, q, k, v, do, dense_h, dev, args, total_flop, ws):
    """Same metric through the public API from pinned host buffers: H2D of the
    step's inputs, mask compile, forward, backward, D2H of the gradients."""
    qh, kh, vh, doh = (t.pin_memory() for t in (q, k, v, do))
    dense_hp = None if dense_h is None else torch.from_numpy(dense_h).pin_memory()
    outs_h = [torch.empty(q.shape, dtype=torch.bfloat16).pin_memory(),
              torch.empty(k.shape, dtype=torch.bfloat16).pin_memory(),
              torch.empty(v.shape, dtype=torch.bfloat16).pin_memory()]
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh, doh))
    if dense_hp is not None:
        h2d += dense_hp.numel()
    d2h = sum(t.numel() * t.element_size() for t in outs_h)

    side = torch.cuda.Stream(device=dev)  # copies that overlap the kernels
    cstream = torch.cuda.Stream(device=dev)  # the second mask compile
    # The forward runs in two KV-head-aligned halves, so that the first
    # half starts once its Q/K/V are in while the second half's are copied;
    # dQ runs in four parts, each going back to the host while the next is
    # computed.  The rowsum and dK/dV run once over all heads.  Heads are
    # independent, so the results are those of single calls over all heads.
    # (One part each when B > 1, where a head slice is not contiguous.)
    G = w.Hq // w.Hkv

    def parts(n):
        n = n if (w.B == 1 and w.Hkv % n == 0) else 1
        kv = w.Hkv // n
        return [(slice(c * kv * G, (c + 1) * kv * G), slice(c * kv, (c + 1) * kv)) for c in range(n)]
    fwd_parts, dq_parts = parts(2), parts(4)

    def one():
        main = torch.cuda.current_stream(dev)
        # Q, K, V (half by half) and then dO come in on the side stream while
        # MaskInfo is compiled on the main one (a computable mask does not
        # depend on the step's data; a dense one is copied in first, on the
        # main stream)
        qd, kd, vd, dod = (torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (qh, kh, vh, doh))
        side.wait_stream(main)
        qkv_in = []
        with torch.cuda.stream(side):
            for hs, gs in fwd_parts:
                qd[:, hs].copy_(qh[:, hs], non_blocking=True)
                kd[:, gs].copy_(kh[:, gs], non_blocking=True)
                vd[:, gs].copy_(vh[:, gs], non_blocking=True)
                qkv_in.append(torch.cuda.Event())
                qkv_in[-1].record(side)
            dod.copy_(doh, non_blocking=True)
            do_in = torch.cuda.Event()
            do_in.record(side)
        dd = None if dense_hp is None else dense_hp.to(dev, non_blocking=True)
        info = bsa.mask_compile(w.mask.kind, w.S, w.S, dense=dd, **mask_kwargs(w))
        # the dK/dV orientation right after, while the SMs are free (the
        # forward waits for its inputs anyway); on its own stream, each
        # compile returning once its MaskInfo is complete
        cstream.wait_stream(main)
        dkv = bsa.mask_compile(w.mask.kind, w.S, w.S, dense=dd, orientation="dkv", stream=cstream,
                               **mask_kwargs(w))
        o = torch.empty_like(qd)
        lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
        dsum = torch.empty_like(lse)
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        for ev, (hs, gs) in zip(qkv_in, fwd_parts):
            main.wait_event(ev)
            bsa.fwd(qd[:, hs], kd[:, gs], vd[:, gs], info, o=o[:, hs], lse=lse[:, hs])
        main.wait_event(do_in)
        bsa.bwd_rowsum(o, dod, dsum=dsum)
        main.wait_stream(cstream)
        bsa.bwd_dkv(qd, kd, vd, o, lse, dod, dsum, dkv, dk=dk, dv=dv)
        side.wait_stream(main)
        with torch.cuda.stream(side):  # dK and dV go back while dQ is computed
            outs_h[1].copy_(dk, non_blocking=True)
            outs_h[2].copy_(dv, non_blocking=True)
        for hs, gs in dq_parts:
            bsa.bwd_dq(qd[:, hs], kd[:, gs], vd[:, gs], o[:, hs], lse[:, hs], dod[:, hs], dsum[:, hs], info,
                       dq=dq[:, hs])
            side.wait_stream(main)
            with torch.cuda.stream(side):
                outs_h[0][:, hs].copy_(dq[:, hs], non_blocking=True)
        main.wait_stream(side)
        torch.cuda.synchronize()
        info.destroy()
        dkv.destroy()
        return outs_h

    for _ in range(max(1, args.warmup)):
        one()
    n = max(1, min(args.steps, 5))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        one()
    dt = max_over_ranks((time.perf_counter() - t0) / n, dev)
    return {"value": round(job_tflops(total_flop, dt, ws), 2), "unit": "TFLOP/s", "ms_per_step": round(dt * 1e3, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "includes": "H2D Q/K/V (two KV-head halves) and dO (side stream, during the mask compile and the "
                        "forward), mask compile (both orientations before the forward, the dkv one on a third "
                        "stream), fwd (per half), rowsum, dK/dV, dQ (four "
                        "parts), D2H dK/dV and each dQ part (side stream, behind its launch)",
            "parts": {"fwd": len(fwd_parts), "dq": len(dq_parts)}}


ORACLE_ROWS = 1024   # query rows per oracle sample (one row chunk of one head)


def oracle_setup(w, dense_h):
    """The oracle's mask (for its attention) and non-empty blocks per block row."""
    from oracle import mask_info as omi
    mask = {"kind": w.mask.kind, "kv_len": w.S}
    kw = {}
    if w.mask.kind == "local":
        kw = dict(left=w.mask.left, right=w.mask.right)
    elif w.mask.kind == "chunked":
        kw = dict(chunk=w.mask.chunk)
    elif w.mask.kind == "dense":
        mask.update(dense=dense_h)
    mask.update(kw)
    info = omi.compile_mask_info(w.mask.kind, w.S, w.S, dense=dense_h, **kw)
    per_row = (info.labels_unshrunk[0] != 0).sum(axis=1)
    return mask, per_row


def oracle_sample_step(w, inputs, mask, per_row, b, h, chunk):
    """The oracle's forward + backward for query rows [chunk*1024, +1024) of one
    (batch, q head): scores against every key, P, O, Dsum, dP, dS, dQ and that
    chunk's contributions to dK/dV.  Returns (seconds, executed-block FLOP)."""
    from oracle import attention as oatt
    q, k, v, do = inputs
    g = h // (w.Hq // w.Hkv)
    r0 = chunk * ORACLE_ROWS
    r1 = min(w.S, r0 + ORACLE_ROWS)
    f = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    base = oatt.mask_rows_for(mask, 0)
    rows_fn = lambda r: base(np.asarray(r) + r0)  # noqa: E731
    args = (f(q[b, h, r0:r1]), f(k[b, g]), f(v[b, g]), f(do[b, h, r0:r1]))
    t0 = time.perf_counter()
    oatt.head_backward(*args, rows_fn, 1 / math.sqrt(w.D))
    dt = time.perf_counter() - t0
    blocks = int(per_row[r0 // 128:r1 // 128].sum())
    return dt, 3.5 * blocks * 4 * 128 * 128 * w.D


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count()


def cpu_baseline(w, dense_h, n_exec, seconds=20.0):
    """The oracle (as it stands) on the host cores, on a bounded sample: 1024-row
    chunks of (batch, q head) slices of the workload, forward + backward, for
    about `seconds` of CPU work; reported in the same unit (TFLOP/s counted
    over the executed blocks of the rows processed)."""
    inputs = qkvdo(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed)
    mask, per_row = oracle_setup(w, dense_h)
    n_chunks = max(1, w.S // ORACLE_ROWS)
    spent, fl, n = 0.0, 0.0, 0
    while spent < seconds and n < w.B * w.Hq * n_chunks:
        dt, f = oracle_sample_step(w, inputs, mask, per_row, (n // n_chunks) % w.B, (n // n_chunks) % w.Hq,
                                   n % n_chunks)
        spent += dt
        fl += f
        n += 1
    return {"value": round(fl / spent / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} chunks of 1024 query rows (of {w.B * w.Hq * n_chunks}), fp64 fwd+bwd, {spent:.1f} s"}


def run_reference(args):
    """--impl reference: the oracle timed on the host cores, same metric/config.
    Each step is a bounded sample of the workload: one 1024-row chunk of one
    (batch, q head), forward + backward."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    dense_h = bernoulli_mask(w.S, w.mask.p, w.mask.seed) if w.mask.kind == "dense" else None
    inputs = qkvdo(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed)
    mask, per_row = oracle_setup(w, dense_h)
    n_chunks = max(1, w.S // ORACLE_ROWS)
    for i in range(args.warmup):
        oracle_sample_step(w, inputs, mask, per_row, 0, i % w.Hq, i % n_chunks)
    spent, fl = 0.0, 0.0
    for i in range(args.steps):
        dt, f = oracle_sample_step(w, inputs, mask, per_row, i % w.B, i % w.Hq, i % n_chunks)
        spent += dt
        fl += f
    value = fl / spent / 1e12
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(spent / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16-rounded inputs)",
        "config": {"workload": args.workload, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D,
                   "mask": w.mask.kind},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": "each step: one 1024-row chunk of one (batch, q-head) slice, fp64 fwd+bwd"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return out


KERNEL_SOURCES = {"fwd_kernel": "attn_fwd.cu", "rowsum_kernel": "attn_bwd_rowsum.cu", "dkv_kernel": "attn_bwd.cu",
                  "dq_kernel": "attn_bwd.cu"}


def ingest_ncu(report: str, workload: str):
    """Writes profiles/traffic.json's entry for `workload` from an ncu report
    of the bench (first launch of each attention kernel): DRAM bytes per
    launch, tied to the sha of the kernel's source file."""
    import csv
    import hashlib
    import io
    import re
    import subprocess
    raw = subprocess.run(["ncu", "-i", report, "--page", "raw", "--csv"], capture_output=True, text=True,
                         check=True).stdout
    rows = list(csv.reader(io.StringIO(raw)))
    hdr, units = rows[0], rows[1]
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}

    def val(r, name):
        i = hdr.index(name)
        return float(r[i].replace(",", "")) * scale[units[i]]

    path = os.path.join(ROOT, "profiles", "traffic.json")
    table = json.load(open(path)) if os.path.exists(path) else {}
    ent = {}
    for r in rows[2:]:
        names = re.findall(r"::(\w+)(?:<[^()]*>)?\(", r[hdr.index("Kernel Name")])
        k = names[-1] if names else ""
        if k not in KERNEL_SOURCES or k in ent:
            continue
        src = KERNEL_SOURCES[k]
        with open(os.path.join(ROOT, "block_sparse_attention_process_gb300", "csrc", src), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        rd, wr = val(r, "dram__bytes_read.sum"), val(r, "dram__bytes_write.sum")
        ent[k] = {"bytes_per_launch": int(rd + wr), "dram_read_mb": round(rd / 1e6, 6), "dram_write_mb": round(wr / 1e6, 6),
                  "source": src, "source_sha": sha, "valid": True}
    table[workload] = ent
    with open(path, "w") as f:
        json.dump(table, f, indent=1)
    print(json.dumps(ent))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--cpu-seconds-other", type=float, default=5.0,
                    help="oracle seconds per workload in the 'workloads' table")
    ap.add_argument("--sustained-s", type=float, default=3.0,
                    help="seconds of back-to-back steps timed against the sustained bf16 peak (0: off)")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mask-only", action="store_true", help="only the dense-mask compile measurements")
    ap.add_argument("--no-mask-bench", action="store_true",
                    help="skip the large dense-mask compile measurements (shorter runs for profiling)")
    ap.add_argument("--ingest-ncu", metavar="REPORT",
                    help="write profiles/traffic.json for --workload from an ncu report of this bench, then exit")
    args = ap.parse_args()
    if args.ingest_ncu:
        ingest_ncu(args.ingest_ncu, args.workload)
        return
    if args.warmup < 3 and args.impl == "gb300":
        ap.error("--warmup must be >= 3")
    if args.mask_only:
        run_mask_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
